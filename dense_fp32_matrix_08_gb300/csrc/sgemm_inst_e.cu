// Kernel instantiations of tile configurations 14 15 16 17 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
template <> VariantKernels variant_kernels<14>() { return make_kernels<VariantCfg<14>::type>(); }
template <> VariantKernels variant_kernels<15>() { return make_kernels<VariantCfg<15>::type>(); }
template <> VariantKernels variant_kernels<16>() { return make_kernels<VariantCfg<16>::type>(); }
template <> VariantKernels variant_kernels<17>() { return make_kernels<VariantCfg<17>::type>(); }
}  // namespace sgemm
