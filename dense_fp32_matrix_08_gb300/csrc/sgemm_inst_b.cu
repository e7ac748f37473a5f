// Kernel instantiations of tile configurations 5 6 7 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
template <> VariantKernels variant_kernels<5>() { return make_kernels<VariantCfg<5>::type>(); }
template <> VariantKernels variant_kernels<6>() { return make_kernels<VariantCfg<6>::type>(); }
template <> VariantKernels variant_kernels<7>() { return make_kernels<VariantCfg<7>::type>(); }
}  // namespace sgemm
