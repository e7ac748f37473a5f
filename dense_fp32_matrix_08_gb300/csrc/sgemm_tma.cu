// Instantiations and launcher of the TMA-fed FFMA2 GEMM (sgemm_ffma_tma.cuh).
#include <cuda_runtime.h>

#include <mutex>

#include "sgemm_ffma_tma.cuh"
#include "sgemm_internal.h"

namespace sgemm {
namespace {

// Instance table: index = VariantShape::inst of the TMA-fed variants in sgemm_plan.h.
using Tma0 = tma::TmaCfg<128, 16, 3, 2, true>;   // 128 x 128, 8 x 16 threads, 2 CTAs/SM
using Tma1 = tma::TmaCfg<96, 12, 2, 3, false>;   // 128 x 96, 8 x 12 threads, 3 CTAs/SM
using Tma2 = tma::TmaCfg<128, 16, 3, 2, false>;  // Tma0 without A double-buffering
using Tma3 = tma::TmaCfg<64, 8, 2, 4, false>;    // 128 x 64, 8 x 8 threads, 4 CTAs/SM
using Tma4 = tma::TmaCfg<96, 12, 2, 3, false, 1>;   // Tma1 on k-major A (A^T)
using Tma5 = tma::TmaCfg<128, 16, 3, 2, false, 1>;  // Tma2 on k-major A (A^T)
using Tma6 = tma::TmaCfg<96, 12, 2, 3, false, 2>;   // Tma1, A transposed in the CTA
using Tma7 = tma::TmaCfg<128, 16, 2, 2, false, 2>;  // 128 x 128, 2 stages, A transposed
using Tma8 = tma::TmaCfg<64, 8, 2, 4, false, 1>;    // 128 x 64 on k-major A, 4 CTAs/SM
using Tma9 = tma::TmaCfg<128, 16, 2, 2, false, 1>;  // 128 x 128 on k-major A, 2 stages
using Tma10 = tma::TmaCfg<64, 8, 2, 3, false, 2>;   // Tma8, A transposed in the CTA
constexpr int kInstances = 11;

std::once_flag g_once[64];
cudaError_t g_err[64];

template <class Cfg>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(tma::sgemm_tma_kernel<Cfg>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
}

template <class Cfg>
cudaError_t launch(const float *A, long long lda, const float *B, long long ldb,
                   const GemmParams &p, int ctas, int *status, cudaStream_t stream) {
  CUtensorMap map_a, map_b;
  // k-major A (AT): A points at A^T, K x M with row stride lda; [32 k][128 m] boxes
  const bool ok_a = Cfg::AMODE == 1
                        ? encode_map_2d(&map_a, A, p.K, p.M, lda, Cfg::BM, Cfg::BK, false)
                        : encode_map_2d(&map_a, A, p.M, p.K, lda, Cfg::BK, Cfg::BM, true);
  if (!ok_a ||
      !encode_map_2d(&map_b, B, p.K, p.N, ldb, Cfg::BN, Cfg::BK, false))
    return cudaErrorInvalidValue;
  return launch_1d(tma::sgemm_tma_kernel<Cfg>, ctas, Cfg::THREADS, Cfg::SMEM_BYTES,
                   p.cluster ? p.split : 1, stream, map_a, map_b, p, status);
}

}  // namespace

cudaError_t tma_setup() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(g_once[dev], [dev]() {
    cudaError_t err = set_smem<Tma0>();
    if (err == cudaSuccess) err = set_smem<Tma1>();
    if (err == cudaSuccess) err = set_smem<Tma2>();
    if (err == cudaSuccess) err = set_smem<Tma3>();
    if (err == cudaSuccess) err = set_smem<Tma4>();
    if (err == cudaSuccess) err = set_smem<Tma5>();
    if (err == cudaSuccess) err = set_smem<Tma6>();
    if (err == cudaSuccess) err = set_smem<Tma7>();
    if (err == cudaSuccess) err = set_smem<Tma8>();
    if (err == cudaSuccess) err = set_smem<Tma9>();
    if (err == cudaSuccess) err = set_smem<Tma10>();
    g_err[dev] = err;
  });
  return g_err[dev];
}

int tma_cluster_ctas(int inst, int cluster) {
  switch (inst) {
#define SGEMM_TMA_CLUSTER_CASE(i)                                                          \
  case i:                                                                                  \
    return cluster_ctas_of(tma::sgemm_tma_kernel<Tma##i>, Tma##i::THREADS, Tma##i::SMEM_BYTES, \
                           cluster);
    SGEMM_TMA_CLUSTER_CASE(0)
    SGEMM_TMA_CLUSTER_CASE(1)
    SGEMM_TMA_CLUSTER_CASE(2)
    SGEMM_TMA_CLUSTER_CASE(3)
    SGEMM_TMA_CLUSTER_CASE(4)
    SGEMM_TMA_CLUSTER_CASE(5)
    SGEMM_TMA_CLUSTER_CASE(6)
    SGEMM_TMA_CLUSTER_CASE(7)
    SGEMM_TMA_CLUSTER_CASE(8)
    SGEMM_TMA_CLUSTER_CASE(9)
    SGEMM_TMA_CLUSTER_CASE(10)
#undef SGEMM_TMA_CLUSTER_CASE
    default:
      return 0;
  }
}

cudaError_t launch_tma(int inst, const float *A, long long lda, const float *B, long long ldb,
                       const GemmParams &p, int ctas, int *status, cudaStream_t stream) {
  static_assert(kInstances == 11, "instance table");
  switch (inst) {
    case 0: return launch<Tma0>(A, lda, B, ldb, p, ctas, status, stream);
    case 1: return launch<Tma1>(A, lda, B, ldb, p, ctas, status, stream);
    case 2: return launch<Tma2>(A, lda, B, ldb, p, ctas, status, stream);
    case 3: return launch<Tma3>(A, lda, B, ldb, p, ctas, status, stream);
    case 4: return launch<Tma4>(A, lda, B, ldb, p, ctas, status, stream);
    case 5: return launch<Tma5>(A, lda, B, ldb, p, ctas, status, stream);
    case 6: return launch<Tma6>(A, lda, B, ldb, p, ctas, status, stream);
    case 7: return launch<Tma7>(A, lda, B, ldb, p, ctas, status, stream);
    case 8: return launch<Tma8>(A, lda, B, ldb, p, ctas, status, stream);
    case 9: return launch<Tma9>(A, lda, B, ldb, p, ctas, status, stream);
    case 10: return launch<Tma10>(A, lda, B, ldb, p, ctas, status, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sgemm
