// Kernel instantiations of tile configurations 5 6 7 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(5)
SGEMM_DEFINE_VARIANT(6)
SGEMM_DEFINE_VARIANT(7)
}  // namespace sgemm
