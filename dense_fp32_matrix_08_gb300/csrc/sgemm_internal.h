// Library-internal helpers shared by the translation units of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace sgemm {

// One-time per-device setup (kernel attributes, SM count, workspace pool) for the current
// device; returns its status and the SM count.
cudaError_t device_setup(int *num_sms);

// The stream-ordered workspace pool of the current device (created by device_setup).
cudaMemPool_t workspace_pool();

// Tensor map (TMA descriptor) of a rows x cols row-major FP32 matrix with row stride ld
// elements (ld * 4 must be a multiple of 16 and ptr 16-byte aligned), box_cols x box_rows
// boxes, optional 128-byte swizzle (box_cols * 4 <= 128 then). Out-of-range elements of a
// box read as zero. Returns false if the driver rejects the description.
bool encode_map_2d(CUtensorMap *map, const float *ptr, long long rows, long long cols,
                   long long ld, int box_cols, int box_rows, bool swizzle128);
// The same with a chosen swizzle span: 0 (none), 32, 64 or 128 bytes (box_cols * 4 must
// equal the span when it is not 0).
bool encode_map_2d_swizzle(CUtensorMap *map, const float *ptr, long long rows, long long cols,
                           long long ld, int box_cols, int box_rows, int swizzle_bytes);

struct GemmParams;
struct Problem;

// Launch `kernel` on a 1-D grid, in thread-block clusters of `cluster` CTAs along x when
// cluster > 1 (grid a multiple of it), else as a plain launch. The launch allows
// programmatic dependent launch: its CTAs may be scheduled while the previous kernel in
// the stream finishes, so `kernel` must call griddep_wait() before touching global memory.
template <class... KArgs, class... Args>
cudaError_t launch_1d(void (*kernel)(KArgs...), int grid, int threads, size_t smem,
                      int cluster, cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)(cluster > 1 ? cluster : 1);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  if (cluster > 1 && grid % cluster != 0) return cudaErrorInvalidConfiguration;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Plan recorded by sgemm_f32_autotune for this problem (shape, flags, beta != 0) on a GPU
// with num_sms SMs: the forced variant and split to use. False when none is recorded.
bool tuned_lookup(const Problem &pr, bool beta_nz, int num_sms, int *variant, int *split);
namespace thin {
struct ThinParams;
}

// Thin-product streaming kernels (sgemm_thin.cuh): one-time kernel attributes for the
// current device, and a launch (thin_m: the thin-M kernel, else thin-N; vec: 128-bit loads
// of the streamed operand allowed).
cudaError_t thin_setup();
cudaError_t launch_thin(bool thin_m, const thin::ThinParams &p, bool vec, cudaStream_t stream);
// TMA-fed thin kernel (sgemm_thin_tma.cuh): thin-M (B TMA-addressable) or thin-N (A
// TMA-addressable); p.split CTAs along K, p.k_per_split a multiple of 8, at most 1024.
cudaError_t launch_thin_tma(bool thin_n, const thin::ThinParams &p, int *status,
                            cudaStream_t stream);
// Cluster thin kernel (sgemm_thin_cluster.cuh): thin-M (A and B TMA-addressable) or thin-N;
// p.split = the cluster size (1, 2, 4 or 8), p.k_per_split a multiple of 8. No workspace.
cudaError_t launch_thin_cluster(bool thin_n, const thin::ThinParams &p, int *status,
                                cudaStream_t stream);
// CTAs of the cluster thin kernel resident at once on the current device in clusters of
// 1, 2, 4 and 8 (zeros if unknown).
void thin_cluster_capacity(int ctas[4]);

// TMA-fed GEMM (sgemm_ffma_tma.cuh): one-time kernel attributes for the current device, and
// a launch of instance `inst` (VariantShape::inst) on row-major A (lda) and B (ldb); for
// the k-major instances A is A^T (K x M, row stride lda).
cudaError_t tma_setup();
cudaError_t launch_tma(int inst, const float *A, long long lda, const float *B, long long ldb,
                       const GemmParams &p, int ctas, int *status, cudaStream_t stream);
// CTAs of TMA-fed instance `inst` resident at once in clusters of `cluster` CTAs on the
// current device (cudaOccupancyMaxActiveClusters; 0 if the query fails).
int tma_cluster_ctas(int inst, int cluster);

// CTAs resident at once in clusters of S (index v * (kMaxClusterSplit + 1) + S) for every
// configuration that can finish split tiles in a cluster, on the current device; filled
// by device_setup. Null before setup.
const int *cluster_capacity_table();

// Occupancy query for a kernel launched in 1-D clusters of `cluster` CTAs.
template <class F>
int cluster_ctas_of(F kernel, int threads, size_t smem, int cluster) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)cluster;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n * cluster;
}

// K-paired TMA-fed GEMM (sgemm_ffma_kpair.cuh): one-time kernel attributes for the current
// device, and a launch with the given ring depth (4, 5 or 6 stages).
cudaError_t kpair_setup();
cudaError_t launch_kpair(int stages, const CUtensorMap &map_a, const CUtensorMap &map_bt,
                         const GemmParams &p, int ctas, int *status, cudaStream_t stream);

// Bt = B^T for a K x N row-major B (row stride ldb) into an N x K row-major Bt (row
// stride ldbt >= K).
cudaError_t launch_transpose_b(const float *B, long long ldb, int K, int N, float *Bt,
                               long long ldbt, int num_sms, cudaStream_t stream);

}  // namespace sgemm
