// Kernel instantiations of tile configurations 16 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(16)
}  // namespace sgemm
