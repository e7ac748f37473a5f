// Kernel instantiations of tile configurations 18 19 20 21 (see sgemm_variants.cuh).
#include "sgemm_variants.cuh"

namespace sgemm {
SGEMM_DEFINE_VARIANT(18)
SGEMM_DEFINE_VARIANT(19)
SGEMM_DEFINE_VARIANT(20)
SGEMM_DEFINE_VARIANT(21)
}  // namespace sgemm
