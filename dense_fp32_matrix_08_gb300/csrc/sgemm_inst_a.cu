// Kernel instantiations of tile configurations 0 1 2 3 4 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(0)
SGEMM_DEFINE_VARIANT(1)
SGEMM_DEFINE_VARIANT(2)
SGEMM_DEFINE_VARIANT(3)
SGEMM_DEFINE_VARIANT(4)
}  // namespace sgemm
