// Kernel instantiations of tile configurations 3 4 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(3)
SGEMM_DEFINE_VARIANT(4)
}  // namespace sgemm
