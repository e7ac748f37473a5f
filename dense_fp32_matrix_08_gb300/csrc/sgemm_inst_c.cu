// Kernel instantiations of tile configurations 8 9 10 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
template <> VariantKernels variant_kernels<8>() { return make_kernels<VariantCfg<8>::type>(); }
template <> VariantKernels variant_kernels<9>() { return make_kernels<VariantCfg<9>::type>(); }
template <> VariantKernels variant_kernels<10>() { return make_kernels<VariantCfg<10>::type>(); }
}  // namespace sgemm
