// Kernel instantiations of tile configurations 14 15 16 17 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(14)
SGEMM_DEFINE_VARIANT(15)
SGEMM_DEFINE_VARIANT(16)
SGEMM_DEFINE_VARIANT(17)
}  // namespace sgemm
