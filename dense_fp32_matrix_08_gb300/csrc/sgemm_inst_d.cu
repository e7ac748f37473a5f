// Kernel instantiations of tile configurations 5 8 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(5)
SGEMM_DEFINE_VARIANT(8)
}  // namespace sgemm
