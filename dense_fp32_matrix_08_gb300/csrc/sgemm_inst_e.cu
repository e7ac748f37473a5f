// Kernel instantiations of tile configurations 13 21 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(13)
SGEMM_DEFINE_VARIANT(21)
}  // namespace sgemm
