// Instantiations and launchers of the thin-product streaming kernels (sgemm_thin.cuh).
#include <cuda_runtime.h>

#include <mutex>

#include "sgemm_internal.h"
#include "sgemm_thin.cuh"
#include "sgemm_thin_cluster.cuh"
#include "sgemm_thin_tma.cuh"

namespace sgemm {
namespace {

std::once_flag g_once[64];
cudaError_t g_err[64];
int g_cluster_ctas[64][4];  // resident CTAs of the cluster kernel in clusters of 1, 2, 4, 8

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
    if (err == cudaSuccess) err = set_smem(thin::thin_cluster_kernel<false>, thin::cl::SMEM_BYTES);
    if (err == cudaSuccess) err = set_smem(thin::thin_cluster_kernel<true>, thin::cl::SMEM_BYTES);
    // How many CTAs of the cluster kernel can be resident at once, per cluster size: the
    // planner sizes grids against it (clusters are placed within one GPC each).
    for (int l = 0; l < 4 && err == cudaSuccess; ++l) {
      const int S = 1 << l;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1, S, 1);
      cfg.blockDim = dim3(thin::cl::THREADS, 1, 1);
      cfg.dynamicSmemBytes = thin::cl::SMEM_BYTES;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = 1;
      attr.val.clusterDim.y = S;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int n = 0;
      // a failed query leaves the capacity unknown (modelled) rather than failing the setup
      if (cudaOccupancyMaxActiveClusters(&n, thin::thin_cluster_kernel<false>, &cfg) !=
          cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
      g_cluster_ctas[dev][l] = n * S;
    }
    g_err[dev] = err;
  });
  return g_err[dev];
}

void thin_cluster_capacity(int ctas[4]) {
  int dev = 0;
  for (int l = 0; l < 4; ++l) ctas[l] = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return;
  if (thin_setup() != cudaSuccess) return;
  for (int l = 0; l < 4; ++l) ctas[l] = g_cluster_ctas[dev][l];
}

cudaError_t launch_thin_cluster(bool thin_n, const thin::ThinParams &p, int *status,
                                cudaStream_t stream) {
  using namespace thin::cl;
  const int S = p.split;
  if ((S != 1 && S != 2 && S != 4 && S != 8) || p.k_per_split <= 0 || p.k_per_split % KC != 0)
    return cudaErrorInvalidValue;
  CUtensorMap map_big, map_small;
  if (thin_n) {  // A streams as [128 m][8 k] boxes (32-byte swizzle), B as [8 k][16 n]
    if (!encode_map_2d_swizzle(&map_big, p.A, p.M, p.K, p.lda, KC, BW, 32) ||
        !encode_map_2d(&map_small, p.B, p.K, p.N, p.ldb, MT, KC, false))
      return cudaErrorInvalidValue;
  } else {  // B streams as [8 k][128 n] boxes, A as [16 m][8 k]
    if (!encode_map_2d(&map_big, p.B, p.K, p.N, p.ldb, BW, KC, false) ||
        !encode_map_2d(&map_small, p.A, p.M, p.K, p.lda, KC, MT, false))
      return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = thin_n ? dim3(p.tiles_m, S, p.tiles_n) : dim3(p.tiles_n, S, p.tiles_m);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  // programmatic dependent launch (the kernel waits for the previous grid before any
  // global access), and the cluster of the K slices
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = S;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = S > 1 ? 2 : 1;
  if (thin_n)
    return cudaLaunchKernelEx(&cfg, thin::thin_cluster_kernel<true>, map_big, map_small, p,
                              status);
  return cudaLaunchKernelEx(&cfg, thin::thin_cluster_kernel<false>, map_big, map_small, p,
                            status);
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
