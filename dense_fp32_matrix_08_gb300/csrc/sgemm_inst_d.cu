// Kernel instantiations of tile configurations 11 12 13 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
template <> VariantKernels variant_kernels<11>() { return make_kernels<VariantCfg<11>::type>(); }
template <> VariantKernels variant_kernels<12>() { return make_kernels<VariantCfg<12>::type>(); }
template <> VariantKernels variant_kernels<13>() { return make_kernels<VariantCfg<13>::type>(); }
}  // namespace sgemm
