// Kernel instantiations of tile configurations 8 9 10 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(8)
SGEMM_DEFINE_VARIANT(9)
SGEMM_DEFINE_VARIANT(10)
}  // namespace sgemm
