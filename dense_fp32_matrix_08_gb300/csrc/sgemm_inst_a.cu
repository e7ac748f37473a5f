// Kernel instantiations of tile configurations 0 1 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(0)
SGEMM_DEFINE_VARIANT(1)
}  // namespace sgemm
