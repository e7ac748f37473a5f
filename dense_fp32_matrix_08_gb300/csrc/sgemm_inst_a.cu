// Kernel instantiations of tile configurations 0 1 2 3 4 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
template <> VariantKernels variant_kernels<0>() { return make_kernels<VariantCfg<0>::type>(); }
template <> VariantKernels variant_kernels<1>() { return make_kernels<VariantCfg<1>::type>(); }
template <> VariantKernels variant_kernels<2>() { return make_kernels<VariantCfg<2>::type>(); }
template <> VariantKernels variant_kernels<3>() { return make_kernels<VariantCfg<3>::type>(); }
template <> VariantKernels variant_kernels<4>() { return make_kernels<VariantCfg<4>::type>(); }
}  // namespace sgemm
