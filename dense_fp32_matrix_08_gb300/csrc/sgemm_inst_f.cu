// Kernel instantiations of tile configurations 18 19 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
template <> VariantKernels variant_kernels<18>() { return make_kernels<VariantCfg<18>::type>(); }
template <> VariantKernels variant_kernels<19>() { return make_kernels<VariantCfg<19>::type>(); }
}  // namespace sgemm
