// Instantiations and launchers of the thin-product streaming kernels (sgemm_thin.cuh).
#include <cuda_runtime.h>

#include <mutex>

#include "sgemm_internal.h"
#include "sgemm_thin.cuh"
#include "sgemm_thin_tma.cuh"

namespace sgemm {
namespace {

std::once_flag g_once[64];
cudaError_t g_err[64];

template <class F>
cudaError_t set_smem(F kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t thin_setup() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(g_once[dev], [dev]() {
    const size_t sm_m = thin::m::smem_bytes(thin::m::KMAX);
    const size_t sm_n = thin::n::smem_bytes(thin::n::KMAX);
    cudaError_t err = set_smem(thin::thin_m_kernel<true>, sm_m);
    if (err == cudaSuccess) err = set_smem(thin::thin_m_kernel<false>, sm_m);
    if (err == cudaSuccess) err = set_smem(thin::thin_n_kernel<true>, sm_n);
    if (err == cudaSuccess) err = set_smem(thin::thin_n_kernel<false>, sm_n);
    if (err == cudaSuccess)
      err = set_smem(thin::thin_tma_kernel<false>, thin::mt::smem_bytes(thin::mt::KMAX));
    if (err == cudaSuccess)
      err = set_smem(thin::thin_tma_kernel<true>, thin::mt::smem_bytes(thin::mt::KMAX));
    g_err[dev] = err;
  });
  return g_err[dev];
}

cudaError_t launch_thin_tma(bool thin_n, const thin::ThinParams &p, int *status,
                            cudaStream_t stream) {
  using namespace thin::mt;
  if (p.k_per_split <= 0 || p.k_per_split > KMAX || p.k_per_split % KB != 0)
    return cudaErrorInvalidValue;
  CUtensorMap map_s;
  const size_t smem = smem_bytes(p.k_per_split);
  if (thin_n) {  // A streams as [256 m][8 k] tiles, 32-byte swizzle
    if (!encode_map_2d_swizzle(&map_s, p.A, p.M, p.K, p.lda, KC, BNC, 32))
      return cudaErrorInvalidValue;
    const dim3 grid(p.tiles_m, p.split, p.tiles_n);
    thin::thin_tma_kernel<true><<<grid, THREADS, smem, stream>>>(map_s, p, status);
  } else {  // B streams as [8 k][256 n] tiles
    if (!encode_map_2d(&map_s, p.B, p.K, p.N, p.ldb, BNC, KC, false))
      return cudaErrorInvalidValue;
    const dim3 grid(p.tiles_n, p.split, p.tiles_m);
    thin::thin_tma_kernel<false><<<grid, THREADS, smem, stream>>>(map_s, p, status);
  }
  return cudaGetLastError();
}

cudaError_t launch_thin(bool thin_m, const thin::ThinParams &p, bool vec, cudaStream_t stream) {
  if (thin_m) {
    if (p.k_per_split <= 0 || p.k_per_split > thin::m::KMAX) return cudaErrorInvalidValue;
    const dim3 grid(p.tiles_n, p.split, p.tiles_m);
    const size_t smem = thin::m::smem_bytes(p.k_per_split);
    if (vec)
      thin::thin_m_kernel<true><<<grid, thin::m::THREADS, smem, stream>>>(p);
    else
      thin::thin_m_kernel<false><<<grid, thin::m::THREADS, smem, stream>>>(p);
  } else {
    if (p.k_per_split <= 0 || p.k_per_split > thin::n::KMAX) return cudaErrorInvalidValue;
    const dim3 grid(p.tiles_m, p.split, p.tiles_n);
    const size_t smem = thin::n::smem_bytes(p.k_per_split);
    if (vec)
      thin::thin_n_kernel<true><<<grid, thin::n::THREADS, smem, stream>>>(p);
    else
      thin::thin_n_kernel<false><<<grid, thin::n::THREADS, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace sgemm
