// Kernel instantiations of tile configurations 11 12 13 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(11)
SGEMM_DEFINE_VARIANT(12)
SGEMM_DEFINE_VARIANT(13)
}  // namespace sgemm
