// Kernel instantiations of tile configurations 2 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(2)
}  // namespace sgemm
