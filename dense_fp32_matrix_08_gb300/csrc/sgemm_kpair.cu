// Instantiations and launchers of the K-paired TMA-fed GEMM (sgemm_ffma_kpair.cuh) and of
// the B -> B^T copy that gives it a K-major B when the caller's B is row-major.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sgemm_ffma_kpair.cuh"
#include "sgemm_internal.h"

namespace sgemm {

// Bt[n][k] = B[k][n]: B is K x N row-major (row stride ldb), Bt is N x K row-major (row
// stride ldbt). 64 x 64 tiles through shared memory (one padding column: the column-wise
// reads of the transpose cost at most two wavefronts). Each of the 256 threads has its 16
// loads of a tile in flight at once, 128-bit along B's rows when VEC (ldb % 4 == 0 and a
// 16-byte aligned B), and writes 128-bit groups of Bt's rows when vec_out (ldbt % 4 == 0,
// 16-byte aligned Bt); ragged edges fall back to masked 4-byte accesses. A warp reads and
// writes 256 contiguous bytes of two rows. Grid-stride over tiles.
template <bool VEC>
__global__ void __launch_bounds__(256) transpose_b_kernel(const float *__restrict__ B,
                                                          long long ldb, int K, int N,
                                                          float *__restrict__ Bt,
                                                          long long ldbt, int vec_out) {
  __shared__ float t[64][65];
  const long long tiles_n = (N + 63) / 64;
  const long long tiles = tiles_n * ((K + 63) / 64);
  const int tid = threadIdx.x;
  const int cg = tid & 15;  // 4-float column group
  const int ro = tid >> 4;  // row offset, + 16 i
  for (long long tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int k0 = (int)(tile / tiles_n) * 64;
    const int n0 = (int)(tile % tiles_n) * 64;
    float v[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = k0 + ro + 16 * i, n = n0 + 4 * cg;
      const float *src = B + (long long)k * ldb + n;
      if (VEC && k < K && n + 3 < N) {
        const float4 f = __ldcs(reinterpret_cast<const float4 *>(src));
        v[i][0] = f.x;
        v[i][1] = f.y;
        v[i][2] = f.z;
        v[i][3] = f.w;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[i][j] = (k < K && n + j < N) ? src[j] : 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) t[ro + 16 * i][4 * cg + j] = v[i][j];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int nl = ro + 16 * i, kl = 4 * cg;  // Bt row n0 + nl, columns k0 + kl .. + 3
      const int n = n0 + nl, k = k0 + kl;
      if (n >= N) continue;
      float *dst = Bt + (long long)n * ldbt + k;
      if (vec_out && k + 3 < K) {
        *reinterpret_cast<float4 *>(dst) =
            make_float4(t[kl][nl], t[kl + 1][nl], t[kl + 2][nl], t[kl + 3][nl]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (k + j < K) dst[j] = t[kl + j][nl];
      }
    }
    __syncthreads();
  }
}

namespace {
std::once_flag g_once[64];
cudaError_t g_err[64];

template <int S>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(kpair::sgemm_kpair_kernel<S>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kpair::smem_bytes<S>());
}
}  // namespace

cudaError_t kpair_setup() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(g_once[dev], [dev]() {
    cudaError_t err = set_smem<4>();
    if (err == cudaSuccess) err = set_smem<5>();
    if (err == cudaSuccess) err = set_smem<6>();
    g_err[dev] = err;
  });
  return g_err[dev];
}

cudaError_t launch_kpair(int stages, const CUtensorMap &map_a, const CUtensorMap &map_bt,
                         const GemmParams &p, int ctas, int *status, cudaStream_t stream) {
  switch (stages) {
    case 4:
      kpair::sgemm_kpair_kernel<4><<<ctas, kpair::THREADS, kpair::smem_bytes<4>(), stream>>>(
          map_a, map_bt, p, status);
      break;
    case 5:
      kpair::sgemm_kpair_kernel<5><<<ctas, kpair::THREADS, kpair::smem_bytes<5>(), stream>>>(
          map_a, map_bt, p, status);
      break;
    case 6:
      kpair::sgemm_kpair_kernel<6><<<ctas, kpair::THREADS, kpair::smem_bytes<6>(), stream>>>(
          map_a, map_bt, p, status);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_transpose_b(const float *B, long long ldb, int K, int N, float *Bt,
                               long long ldbt, int num_sms, cudaStream_t stream) {
  const long long tiles = ((long long)(N + 63) / 64) * ((K + 63) / 64);
  const long long cap = (long long)num_sms * 8;
  const int grid = (int)(tiles < cap ? (tiles > 0 ? tiles : 1) : cap);
  const bool vec = ldb % 4 == 0 && (reinterpret_cast<uintptr_t>(B) & 15u) == 0;
  const int vec_out = (ldbt % 4 == 0 && (reinterpret_cast<uintptr_t>(Bt) & 15u) == 0) ? 1 : 0;
  if (vec)
    transpose_b_kernel<true><<<grid, 256, 0, stream>>>(B, ldb, K, N, Bt, ldbt, vec_out);
  else
    transpose_b_kernel<false><<<grid, 256, 0, stream>>>(B, ldb, K, N, Bt, ldbt, vec_out);
  return cudaGetLastError();
}

}  // namespace sgemm
