// Instantiations and launchers of the K-paired TMA-fed GEMM (sgemm_ffma_kpair.cuh) and of
// the B -> B^T copy that gives it a K-major B when the caller's B is row-major.
#include <cuda_runtime.h>

#include <mutex>

#include "sgemm_ffma_kpair.cuh"
#include "sgemm_internal.h"

namespace sgemm {

// Bt[n][k] = B[k][n]: B is K x N row-major (row stride ldb), Bt is N x K row-major (row
// stride ldbt). 32 x 32 tiles through shared memory (one padding column, so the transposed
// reads hit 32 banks); 32 x 8 threads, 4 elements each; reads and writes are 128-byte rows.
// Grid-stride over tiles, the grid is a multiple of the SM count.
__global__ void __launch_bounds__(256) transpose_b_kernel(const float *__restrict__ B,
                                                          long long ldb, int K, int N,
                                                          float *__restrict__ Bt,
                                                          long long ldbt) {
  __shared__ float t[32][33];
  const long long tiles_n = (N + 31) / 32;
  const long long tiles = tiles_n * ((K + 31) / 32);
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (long long tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int k0 = (int)(tile / tiles_n) * 32;
    const int n0 = (int)(tile % tiles_n) * 32;
#pragma unroll
    for (int r = ty; r < 32; r += 8) {
      const int k = k0 + r, n = n0 + tx;
      if (k < K && n < N) t[r][tx] = B[(long long)k * ldb + n];
    }
    __syncthreads();
#pragma unroll
    for (int r = ty; r < 32; r += 8) {
      const int n = n0 + r, k = k0 + tx;
      if (n < N && k < K) Bt[(long long)n * ldbt + k] = t[tx][r];
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
  const long long tiles = ((long long)(N + 31) / 32) * ((K + 31) / 32);
  const long long cap = (long long)num_sms * 8;
  const int grid = (int)(tiles < cap ? (tiles > 0 ? tiles : 1) : cap);
  transpose_b_kernel<<<grid, dim3(32, 8), 0, stream>>>(B, ldb, K, N, Bt, ldbt);
  return cudaGetLastError();
}

}  // namespace sgemm
