// Kernel instantiations of tile configurations 22 23 24 25 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(22)
SGEMM_DEFINE_VARIANT(23)
SGEMM_DEFINE_VARIANT(24)
SGEMM_DEFINE_VARIANT(25)
}  // namespace sgemm
