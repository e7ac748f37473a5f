// C ABI of the FP32 SGEMM library: argument checks, launch planning and dispatch.
// The operation and its contract are documented in include/sgemm_f32.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <limits>
#include <mutex>

#include "../../include/sgemm_f32.h"
#include "sgemm_aux.cuh"
#include "sgemm_ffma_kpair.cuh"
#include "sgemm_thin.cuh"
#include "sgemm_internal.h"
#include "sgemm_plan.h"
#include "sgemm_ptx.cuh"
#include "sgemm_variants.cuh"

namespace sgemm {

// The copy-fed kernels of configuration V, or none for a retired configuration.
template <int V>
VariantKernels kernels_if_built() {
  if constexpr (variant_built(V)) {
    return variant_kernels<V>();
  } else {
    return VariantKernels{};
  }
}

static const VariantKernels kKernels[kNumVariants] = {
#define SGEMM_KERNELS_ENTRY(v) kernels_if_built<v>(),
    SGEMM_FOR_EACH_VARIANT(SGEMM_KERNELS_ENTRY)
#undef SGEMM_KERNELS_ENTRY
    VariantKernels{},  // kTmaVariant: its own kernel (sgemm_tma.cu)
    VariantKernels{},  // K-paired variants: their own kernel (sgemm_kpair.cu)
    VariantKernels{},
    VariantKernels{},
    VariantKernels{},  // more TMA-fed instances (sgemm_tma.cu)
    VariantKernels{},
    VariantKernels{},
    VariantKernels{},  // thin-M and thin-N streaming kernels (sgemm_thin.cu)
    VariantKernels{},
    VariantKernels{},  // k-major TMA-fed instances (sgemm_tma.cu)
    VariantKernels{},
    VariantKernels{},  // TMA-fed instances transposing A in the CTA (sgemm_tma.cu)
    VariantKernels{},
    VariantKernels{},  // more k-major TMA-fed instances (sgemm_tma.cu)
    VariantKernels{},
    VariantKernels{},  // TMA-fed thin-M and thin-N kernels (sgemm_thin.cu)
    VariantKernels{},
    VariantKernels{},  // cluster thin-M and thin-N kernels (sgemm_thin.cu)
    VariantKernels{},
    VariantKernels{},  // TMA-fed 128 x 64 transposing A in the CTA (sgemm_tma.cu)
};
static_assert(kTmaVariant == 26 && kFirstKpairVariant == 27 && kThinMVariant == 33 &&
                  kThinNVariant == 34 && kThinTmaVariant == 41 &&
                  kThinClusterVariant == 43 && kNumVariants == 46,
              "the generic variants come first, then the TMA-fed and streaming ones");

// Device status word of the TMA-fed kernel (0 = fine; nonzero = a bounded wait gave up).
__device__ int g_ffma_status;

// ------------------------------------------------------------------------------------
// Per-device one-time setup: opt every kernel into its dynamic shared memory, cache the SM
// count, and ask the driver how many CTAs each cluster-capable configuration keeps
// resident in clusters of 2 .. 8 (the planner's cluster capacity).
constexpr int kMaxDevices = 64;
struct DeviceState {
  std::once_flag once;
  int num_sms = 0;
  int *status = nullptr;  // device address of g_ffma_status
  cudaMemPool_t pool = nullptr;  // split-K workspace pool of this device
  cudaError_t err = cudaSuccess;
  // CTAs resident at once in clusters of S, per configuration (cluster_capacity_table)
  int cluster_cap[kNumVariants * (kMaxClusterSplit + 1)] = {};
};
static DeviceState g_dev[kMaxDevices];

cudaError_t device_setup(int *num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceState &st = g_dev[dev];
  std::call_once(st.once, [&st, dev]() {
    int sms = 0;
    cudaError_t err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    for (int v = 0; v < kNumVariants && err == cudaSuccess; ++v)
      for (int a = 0; a < 3 && err == cudaSuccess; ++a)
        for (int b = 0; b < 3 && err == cudaSuccess; ++b)
          if (kKernels[v].k[a][b])
            err = cudaFuncSetAttribute(kKernels[v].k[a][b],
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kKernels[v].smem);
    if (err == cudaSuccess) err = tma_setup();
    if (err == cudaSuccess) err = thin_setup();
    if (err == cudaSuccess) err = kpair_setup();
    if (err == cudaSuccess)
      err = cudaGetSymbolAddress(reinterpret_cast<void **>(&st.status), g_ffma_status);
    // cluster capacities of the configurations that can finish split tiles in a cluster
    for (int v = 0; v < kNumVariants && err == cudaSuccess; ++v) {
      if (!cluster_split_ok(v, 2)) continue;
      KernelFn fn = nullptr;
      for (int a = 0; a < 3 && !fn; ++a)
        for (int b = 0; b < 3 && !fn; ++b) fn = kKernels[v].k[a][b];
      for (int S = 2; S <= kMaxClusterSplit; ++S)
        st.cluster_cap[v * (kMaxClusterSplit + 1) + S] =
            kVariants[v].tma ? tma_cluster_ctas(kVariants[v].inst, S)
            : fn != nullptr  ? cluster_ctas_of(fn, kVariants[v].threads,
                                               (size_t)kVariants[v].smem_bytes, S)
                             : 0;
    }
    // A pool of the library's own for split-K workspaces. It keeps freed memory (release
    // threshold: never), so a stream-ordered allocation of a recently freed size is a
    // cheap reuse instead of a fresh mapping; the default pool returns its memory at every
    // synchronisation. The pool holds at most the largest workspace the planner chooses
    // (64 MiB) plus whatever concurrent calls on several streams need at once.
    if (err == cudaSuccess) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      err = cudaMemPoolCreate(&st.pool, &props);
      if (err == cudaSuccess) {
        uint64_t keep = ~0ull;
        err = cudaMemPoolSetAttribute(st.pool, cudaMemPoolAttrReleaseThreshold, &keep);
      }
    }
    st.num_sms = sms;
    st.err = err;
  });
  *num_sms = st.num_sms;
  return st.err;
}

// make_plan evaluates a few hundred candidate layouts; a small per-thread cache keeps
// repeated calls on the same shape at a table lookup. The plan depends only on the shape,
// the special values of alpha and beta, the operand flags, the SM count (and, when known,
// the device's cluster capacity) and the forcing arguments.
static Plan cached_plan(const Problem &pr, float alpha, float beta, int num_sms, int force_v,
                        int force_split) {
  struct Entry {
    int M, N, K, num_sms, force_v, force_split;
    unsigned flags;  // alpha == 0, beta != 0, beta == 1, op(A) / op(B) transposed, TMA-able,
                     // planned with the device's measured cluster capacity
    bool valid;
    Plan plan;
  };
  constexpr int kEntries = 16;
  thread_local Entry cache[kEntries] = {};
  thread_local int next = 0;
  const unsigned flags = (alpha == 0.0f ? 1u : 0u) | (beta != 0.0f ? 2u : 0u) |
                         (beta == 1.0f ? 4u : 0u) | (pr.transa ? 8u : 0u) |
                         (pr.transb ? 16u : 0u) | (pr.tma_ok ? 32u : 0u) |
                         (pr.kpair_ok ? 64u : 0u) | (pr.b_kmajor ? 128u : 0u) |
                         (pr.a_tma ? 256u : 0u) | (pr.b_tma ? 512u : 0u) |
                         (pr.at_direct ? 1024u : 0u) |
                         (pr.cluster_cap != nullptr ? 2048u : 0u);  // measured capacity
  for (int i = 0; i < kEntries; ++i) {
    const Entry &e = cache[i];
    if (e.valid && e.M == pr.M && e.N == pr.N && e.K == pr.K && e.num_sms == num_sms &&
        e.force_v == force_v && e.force_split == force_split && e.flags == flags)
      return e.plan;
  }
  Entry &e = cache[next];
  next = (next + 1) % kEntries;
  e = Entry{pr.M, pr.N, pr.K, num_sms, force_v, force_split, flags, true,
            make_plan(pr, alpha, beta, num_sms, force_v, force_split)};
  return e.plan;
}

// SGEMM_F32_FORCE="v" or "v:s" (environment, read once per process) pins the automatic
// plan to configuration v with split argument s, as sgemm_f32_forced would: a benchmarking
// switch. Problems the configuration cannot run keep their automatic plan.
static bool env_force(int *v, int *s) {
  static int ev = -1, es = 0;
  static std::once_flag once;
  std::call_once(once, []() {
    const char *t = std::getenv("SGEMM_F32_FORCE");
    int a = -1, b = 0;
    if (t != nullptr && std::sscanf(t, "%d:%d", &a, &b) >= 1 && a >= 0 && a < kNumVariants &&
        b >= -64 && b <= 64) {
      ev = a;
      es = b;
    }
  });
  if (ev < 0) return false;
  *v = ev;
  *s = es;
  return true;
}

// The automatic plan: SGEMM_F32_FORCE if set and applicable, else a plan recorded by
// sgemm_f32_autotune, else the cost model.
static Plan automatic_plan(const Problem &pr, float alpha, float beta, int num_sms) {
  int v = -1, sp = 0;
  if (env_force(&v, &sp)) {
    const Plan pl = cached_plan(pr, alpha, beta, num_sms, v, sp);
    if (pl.variant >= 0 || alpha == 0.0f || pr.K == 0) return pl;
  }
  if (tuned_lookup(pr, beta != 0.0f, num_sms, &v, &sp))
    return cached_plan(pr, alpha, beta, num_sms, v, sp);
  return cached_plan(pr, alpha, beta, num_sms, -1, 0);
}

const int *cluster_capacity_table() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return g_dev[dev].err == cudaSuccess && g_dev[dev].num_sms > 0 ? g_dev[dev].cluster_cap
                                                                 : nullptr;
}

// One warp waits, with the kernels' own bounded wait, for a phase of an mbarrier that
// nothing ever completes; *out = 1 when the wait gave up, as it must (sgemm_f32_wait_selftest).
__global__ void wait_selftest_kernel(int *out) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = saddr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    mbar_init_fence();
  }
  __syncwarp();
  const bool done = mbar_wait(b, 0);  // no arrival is ever made
  if (threadIdx.x == 0) *out = done ? 0 : 1;
}

static int *status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return g_dev[dev].status;
}

cudaMemPool_t workspace_pool() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return g_dev[dev].pool;
}

static inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

static int grid_for_stream_kernel(long long work_items, int num_sms) {
  const long long blocks = (work_items + 255) / 256;
  const long long cap = (long long)num_sms * 8;
  return (int)std::max<long long>(1, std::min(blocks, cap));
}

// Launch shape of the split-K finish: small jobs (a few thousand float4 outputs, as for
// thin problems) in 64-thread blocks so that they spread over every SM instead of a few
// large blocks; large jobs in 256-thread blocks, at most 8 per SM, grid-stride.
static void reduce_shape(long long work_items, int num_sms, int *grid, int *block) {
  *block = work_items >= (long long)num_sms * 512 ? 256 : 64;
  const long long blocks = (work_items + *block - 1) / *block;
  const long long cap = (long long)num_sms * (2048 / *block);
  *grid = (int)std::max<long long>(1, std::min(blocks, cap));
}

// Enqueue the whole computation for a validated, non-empty problem.
static int run(const Problem &pr, const Plan &pl, float alpha, const float *A,
               const float *B, float beta, float *C, float *ws, int num_sms,
               cudaStream_t stream) {
  const bool vec_c = (pr.ldc % 4 == 0) && aligned16(C);
  if (pl.variant < 0) {  // alpha == 0 or K == 0: C = beta * C
    if (beta == 1.0f) return 0;
    const long long work = (long long)pr.M * ((pr.N + 3) / 4);
    scale_c_kernel<<<grid_for_stream_kernel(work, num_sms), 256, 0, stream>>>(
        C, pr.ldc, pr.M, pr.N, beta, vec_c ? 1 : 0);
    return (int)cudaGetLastError();
  }
  const VariantShape &vs = kVariants[pl.variant];
  if (vs.thin) {
    thin::ThinParams tp;
    tp.M = pr.M;
    tp.N = pr.N;
    tp.K = pr.K;
    tp.alpha = alpha;
    tp.beta = beta;
    tp.A = A;
    tp.lda = pr.lda;
    tp.B = B;
    tp.ldb = pr.ldb;
    tp.C = C;
    tp.ldc = pr.ldc;
    tp.ws = ws;
    tp.split = pl.split;
    tp.k_per_split = pl.k_per_split;
    tp.tiles_m = pl.tiles_m;
    tp.tiles_n = pl.tiles_n;
    tp.vec_c = vec_c ? 1 : 0;
    cudaError_t te;
    int parts = pl.split;  // partial tiles per C tile for the reduce kernel
    if (pl.pack_a || pl.pack_b) {  // the small operand, copied to aligned rows for TMA
      if (vs.thin < 5) return kErrBadVariant;  // (the planner makes no such plan)
      if (pl.pack_a) {
        pack_rows_kernel<<<grid_for_stream_kernel((long long)pr.M * ((pr.K + 3) / 4), num_sms),
                           256, 0, stream>>>(A, pr.lda, pr.M, pr.K, ws, pl.lda_p);
        tp.A = ws;
        tp.lda = pl.lda_p;
      } else {
        pack_rows_kernel<<<grid_for_stream_kernel((long long)pr.K * ((pr.N + 3) / 4), num_sms),
                           256, 0, stream>>>(B, pr.ldb, pr.K, pr.N, ws, pl.ldb_p);
        tp.B = ws;
        tp.ldb = pl.ldb_p;
      }
      tp.ws = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + pl.pre_bytes);
      te = cudaGetLastError();
      if (te != cudaSuccess) return (int)te;
    }
    if (vs.thin >= 5) {
      te = launch_thin_cluster(vs.thin == 6, tp, status_word(), stream);
      parts = 1;  // the cluster adds its slices itself
    } else if (vs.thin >= 3) {
      te = launch_thin_tma(vs.thin == 4, tp, status_word(), stream);
    } else {
      // 128-bit loads of the streamed operand: B rows (thin-M) or A rows (thin-N)
      const bool vec = vs.thin == 1 ? (pr.ldb % 4 == 0 && aligned16(B))
                                    : (pr.lda % 4 == 0 && aligned16(A));
      te = launch_thin(vs.thin == 1, tp, vec, stream);
    }
    if (te != cudaSuccess) return (int)te;
    if (parts > 1) {
      const long long tiles = (long long)pl.tiles_m * pl.tiles_n;
      const long long work = tiles * vs.BM * (vs.BN / 4);
      int rgrid = 1, rblock = 256;
      reduce_shape(work, num_sms, &rgrid, &rblock);
      tail_reduce_kernel<<<rgrid, rblock, 0, stream>>>(
          ws, 0, (int)tiles, parts, vs.BM, vs.BN, pl.tiles_m, pl.tiles_n, 1, pr.M, pr.N,
          alpha, beta, C, pr.ldc, vec_c ? 1 : 0);
      te = cudaGetLastError();
    }
    return (int)te;
  }
  GemmParams p;
  p.M = pr.M;
  p.N = pr.N;
  p.K = pr.K;
  p.alpha = alpha;
  p.beta = beta;
  p.A = A;
  p.lda = pr.lda;
  p.B = B;
  p.ldb = pr.ldb;
  p.C = C;
  p.ldc = pr.ldc;
  p.ws = ws;
  p.main_tiles = pl.main_tiles;
  p.split = pl.split;
  p.k_per_split = pl.k_per_split;
  p.tiles_m = pl.tiles_m;
  p.tiles_n = pl.tiles_n;
  p.group_m = pl.group_m;
  p.vec_c = vec_c ? 1 : 0;
  p.cluster = pl.cluster ? 1 : 0;
  if (pl.cluster && (!cluster_split_ok(pl.variant, pl.split) || pl.main_tiles != 0))
    return kErrBadVariant;  // (the planner makes no such plan)
  if (vs.kpair) {
    const float *Bt = B;
    long long ldbt = pr.ldb;
    if (pl.bt_bytes > 0) {  // row-major B: copy it to B^T (N x K) at the front of ws
      float *bt = ws;
      p.ws = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + pl.bt_bytes);
      cudaError_t te = launch_transpose_b(B, pr.ldb, pr.K, pr.N, bt, pl.ldbt, num_sms, stream);
      if (te != cudaSuccess) return (int)te;
      Bt = bt;
      ldbt = pl.ldbt;
    }
    ws = p.ws;
    CUtensorMap map_a, map_bt;
    if (!encode_map_2d(&map_a, A, pr.M, pr.K, pr.lda, kpair::BK, kpair::BM, true) ||
        !encode_map_2d(&map_bt, Bt, pr.N, pr.K, ldbt, kpair::BK, kpair::BN, true))
      return (int)cudaErrorInvalidValue;
    if (pl.ctas <= 0) return (int)cudaErrorInvalidConfiguration;
    cudaError_t ke = launch_kpair(vs.stages, map_a, map_bt, p, pl.ctas, status_word(), stream);
    if (ke != cudaSuccess) return (int)ke;
  } else if (vs.tma) {
    if (pl.ctas <= 0) return (int)cudaErrorInvalidConfiguration;
    // operands TMA cannot address are copied to aligned rows in the workspace first
    char *wsb = reinterpret_cast<char *>(ws);
    const float *Ap = A, *Bp = B;
    long long ldap = pr.lda, ldbp = pr.ldb;
    if (pl.at_a) {  // k-major instances read A^T
      float *dst = reinterpret_cast<float *>(wsb + pl.bt_bytes);
      cudaError_t te = launch_transpose_b(A, pr.lda, pr.M, pr.K, dst, pl.lda_p, num_sms, stream);
      if (te != cudaSuccess) return (int)te;
      Ap = dst;
      ldap = pl.lda_p;
    } else if (pl.pack_a) {
      float *dst = reinterpret_cast<float *>(wsb + pl.bt_bytes);
      const long long work = (long long)pr.M * ((pr.K + 3) / 4);
      pack_rows_kernel<<<grid_for_stream_kernel(work, num_sms), 256, 0, stream>>>(
          A, pr.lda, pr.M, pr.K, dst, pl.lda_p);
      Ap = dst;
      ldap = pl.lda_p;
    }
    if (pl.pack_b) {
      float *dst = reinterpret_cast<float *>(wsb + pl.bt_bytes + pl.pack_a_bytes);
      const long long work = (long long)pr.K * ((pr.N + 3) / 4);
      pack_rows_kernel<<<grid_for_stream_kernel(work, num_sms), 256, 0, stream>>>(
          B, pr.ldb, pr.K, pr.N, dst, pl.ldb_p);
      Bp = dst;
      ldbp = pl.ldb_p;
    }
    if (pl.pre_bytes > 0) {
      p.ws = reinterpret_cast<float *>(wsb + pl.pre_bytes);
      ws = p.ws;
    }
    cudaError_t ke = cudaGetLastError();
    if (ke == cudaSuccess)
      ke = launch_tma(vs.inst, Ap, ldap, Bp, ldbp, p, pl.ctas, status_word(), stream);
    if (ke != cudaSuccess) return (int)ke;
  } else {
  const int apath = !pr.transa ? APATH_N
                    : ((pr.lda % 4 == 0) && aligned16(A)) ? APATH_T16 : APATH_T4;
  const int bpath = pr.transb ? BPATH_T
                    : ((pr.ldb % 4 == 0) && aligned16(B)) ? BPATH_N16 : BPATH_N4;
  const KernelFn fn = kKernels[pl.variant].k[apath][bpath];
  if (fn == nullptr) return kErrBadVariant;  // forced variant without transposed paths
  if (pl.ctas <= 0) return (int)cudaErrorInvalidConfiguration;
  cudaError_t le = launch_1d(fn, pl.ctas, vs.threads, (size_t)vs.smem_bytes,
                             pl.cluster ? pl.split : 1, stream, p);
  if (le != cudaSuccess) return (int)le;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  const long long tail_tiles = (long long)pl.tiles_m * pl.tiles_n - pl.main_tiles;
  if (tail_tiles > 0 && !pl.cluster) {
    const long long work = (long long)tail_tiles * vs.BM * (vs.BN / 4);
    int rgrid = 1, rblock = 256;
    reduce_shape(work, num_sms, &rgrid, &rblock);
    tail_reduce_kernel<<<rgrid, rblock, 0, stream>>>(
        ws, pl.main_tiles, (int)tail_tiles, pl.split, vs.BM, vs.BN, pl.tiles_m, pl.tiles_n,
        pl.group_m, pr.M, pr.N, alpha, beta, C, pr.ldc, vec_c ? 1 : 0);
    e = cudaGetLastError();
  }
  return (int)e;
}

// Shared body of the computing entry points. ws_mode: 0 = allocate on the stream,
// 1 = caller workspace (ws, ws_bytes).
static int sgemm_entry(int M, int N, int K, float alpha, const float *A, int lda,
                       const float *B, int ldb, float beta, float *C, int ldc, int force_v,
                       int force_split, int ws_mode, void *ws, size_t ws_bytes,
                       cudaStream_t stream, int transa = 0, int transb = 0) {
  Problem pr{M, N, K, lda, ldb, ldc, transa, transb};
  pr.tma_ok = !transa && !transb && lda % 4 == 0 && ldb % 4 == 0 && aligned16(A) &&
              aligned16(B) && A != nullptr && B != nullptr;
  pr.kpair_ok = !transa && lda % 4 == 0 && aligned16(A) && A != nullptr && B != nullptr;
  pr.b_kmajor = transb && ldb % 4 == 0 && aligned16(B);
  pr.a_tma = !transa && lda % 4 == 0 && aligned16(A) && A != nullptr;
  pr.b_tma = !transb && ldb % 4 == 0 && aligned16(B) && B != nullptr;
  pr.at_direct = transa && lda % 4 == 0 && aligned16(A) && A != nullptr;
  int rc = (transa || transb) ? validate_ex(pr, alpha, A != nullptr, B != nullptr, C != nullptr)
                              : validate(pr, alpha, A != nullptr, B != nullptr, C != nullptr);
  if (rc != 0) return rc;
  if (M == 0 || N == 0) return 0;
  if (force_v >= kNumVariants || force_v < -1) return kErrBadVariant;
  if (force_v >= 0 && kVariants[force_v].tma && (transa || transb) &&
      !(kVariants[force_v].at && pr.at_direct && !transb))
    return kErrBadVariant;
  if (force_v >= 0 && kVariants[force_v].kpair && !pr.kpair_ok) return kErrBadVariant;
  int num_sms = 0;
  cudaError_t e = device_setup(&num_sms);
  if (e != cudaSuccess) return (int)e;
  thin_cluster_capacity(pr.cluster_ctas);
  pr.cluster_cap = cluster_capacity_table();
  Plan pl = (force_v < 0 && force_split == 0)
                ? automatic_plan(pr, alpha, beta, num_sms)
                : cached_plan(pr, alpha, beta, num_sms, force_v, force_split);
  // No candidate fitted (a forced configuration whose workspace exceeds the limits).
  if (pl.variant < 0 && alpha != 0.0f && K > 0) return force_v >= 0 ? kErrBadVariant
                                                                    : kErrWorkspace;
  // A caller workspace that cannot hold the plan's A^T copy gets the twin configuration
  // that transposes A in shared memory: the same tiles and k order, no copy.
  if (ws_mode == 1 && pl.ws_bytes > ws_bytes) pl = without_at_copy(pr, pl);
  float *wsp = nullptr;
  if (pl.ws_bytes > 0) {
    if (ws_mode == 1) {
      if (ws == nullptr || ws_bytes < pl.ws_bytes || !aligned16(ws)) return kErrWorkspace;
      wsp = static_cast<float *>(ws);
    } else {
      e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&wsp), pl.ws_bytes,
                                  workspace_pool(), stream);
      if (e != cudaSuccess) return (int)e;
    }
  }
  rc = run(pr, pl, alpha, A, B, beta, C, wsp, num_sms, stream);
  if (ws_mode == 0 && wsp != nullptr) {
    e = cudaFreeAsync(wsp, stream);
    if (rc == 0 && e != cudaSuccess) rc = (int)e;
  }
  return rc;
}

}  // namespace sgemm

using namespace sgemm;

extern "C" {

int sgemm_f32(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
              int ldb, float beta, float *C, int ldc, cudaStream_t stream) {
  return sgemm_entry(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, -1, 0, 0, nullptr, 0,
                     stream);
}

int sgemm_f32_ex(int transa, int transb, int M, int N, int K, float alpha, const float *A,
                 int lda, const float *B, int ldb, float beta, float *C, int ldc,
                 cudaStream_t stream) {
  Problem pr{M, N, K, lda, ldb, ldc, transa, transb};
  const int rc = validate_ex(pr, alpha, A != nullptr, B != nullptr, C != nullptr);
  if (rc != 0) return rc;
  return sgemm_entry(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, -1, 0, 0, nullptr, 0,
                     stream, transa, transb);
}

// Column-major C (m x n) = alpha op(A) op(B) + beta C is, read row-major, the n x m matrix
// C^T = alpha op(B)^T op(A)^T + beta C^T: the same call with the operands swapped and
// each operand's transpose flag applied to its row-major view ("Lecture 4 - GPU
// Acceleration", section 5.4, the swap trick for calling a column-major library on
// row-major tensors, used here the other way round).
int sgemm_f32_colmajor(int transa, int transb, int m, int n, int k, float alpha,
                       const float *A, int lda, const float *B, int ldb, float beta, float *C,
                       int ldc, cudaStream_t stream) {
  const int rc = validate_colmajor(transa, transb, m, n, k, lda, ldb, ldc, alpha,
                                   A != nullptr, B != nullptr, C != nullptr);
  if (rc != 0) return rc;
  return sgemm_entry(n, m, k, alpha, B, ldb, A, lda, beta, C, ldc, -1, 0, 0, nullptr, 0, stream,
                     transb, transa);
}

int sgemm_f32_ws(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                 int ldb, float beta, float *C, int ldc, void *workspace,
                 size_t workspace_bytes, cudaStream_t stream) {
  return sgemm_entry(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, -1, 0, 1, workspace,
                     workspace_bytes, stream);
}

int sgemm_f32_forced(int M, int N, int K, float alpha, const float *A, int lda,
                     const float *B, int ldb, float beta, float *C, int ldc, int variant,
                     int split, cudaStream_t stream) {
  return sgemm_entry(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, variant, split, 0,
                     nullptr, 0, stream);
}

int sgemm_f32_ex_forced(int transa, int transb, int M, int N, int K, float alpha,
                        const float *A, int lda, const float *B, int ldb, float beta, float *C,
                        int ldc, int variant, int split, cudaStream_t stream) {
  Problem pr{M, N, K, lda, ldb, ldc, transa, transb};
  const int rc = validate_ex(pr, alpha, A != nullptr, B != nullptr, C != nullptr);
  if (rc != 0) return rc;
  return sgemm_entry(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, variant, split, 0, nullptr,
                     0, stream, transa, transb);
}

int sgemm_f32_workspace_size(int M, int N, int K, int lda, int ldb, int ldc,
                             size_t *bytes) {
  return sgemm_f32_plan(M, N, K, lda, ldb, ldc, 1.0f, 1.0f, 0, nullptr, nullptr, nullptr,
                        nullptr, bytes);
}

int sgemm_f32_workspace_size_min(int M, int N, int K, int lda, int ldb, int ldc,
                                 size_t *bytes) {
  if (bytes) *bytes = 0;
  Problem pr{M, N, K, lda, ldb, ldc};
  pr.tma_ok = lda % 4 == 0 && ldb % 4 == 0;  // pointers assumed 16-byte aligned
  pr.kpair_ok = lda % 4 == 0;
  pr.a_tma = lda % 4 == 0;
  pr.b_tma = ldb % 4 == 0;
  int rc = validate(pr, 1.0f, true, true, true);
  if (rc != 0) return rc;
  if (M == 0 || N == 0) return 0;
  int num_sms = 0;
  cudaError_t e = device_setup(&num_sms);
  if (e != cudaSuccess) return (int)e;
  thin_cluster_capacity(pr.cluster_ctas);
  pr.cluster_cap = cluster_capacity_table();
  // the plan sgemm_f32_ws makes when the workspace cannot hold the A^T copy
  const Plan pl = without_at_copy(pr, automatic_plan(pr, 1.0f, 1.0f, num_sms));
  if (bytes) *bytes = pl.ws_bytes;
  return 0;
}

int sgemm_f32_plan(int M, int N, int K, int lda, int ldb, int ldc, float alpha, float beta,
                   int num_sms, int *variant, int *split, int *main_tiles, int *launches,
                   size_t *ws_bytes) {
  Problem pr{M, N, K, lda, ldb, ldc};
  pr.tma_ok = lda % 4 == 0 && ldb % 4 == 0;  // pointers assumed 16-byte aligned
  pr.kpair_ok = lda % 4 == 0;
  pr.a_tma = lda % 4 == 0;
  pr.b_tma = ldb % 4 == 0;
  int rc = validate(pr, alpha, true, true, true);
  if (rc != 0) return rc;
  if (num_sms <= 0) {  // the current device, with its own cluster capacity
    cudaError_t e = device_setup(&num_sms);
    if (e != cudaSuccess) return (int)e;
    thin_cluster_capacity(pr.cluster_ctas);
    pr.cluster_cap = cluster_capacity_table();
  }
  Plan pl;
  if (M == 0 || N == 0) {
    pl.variant = -1;
  } else {
    pl = automatic_plan(pr, alpha, beta, num_sms);
  }
  if (variant) *variant = pl.variant;
  if (split) *split = pl.split;
  if (main_tiles) *main_tiles = pl.main_tiles;
  if (launches) *launches = pl.launches;
  if (ws_bytes) *ws_bytes = pl.ws_bytes;
  return 0;
}

int sgemm_f32_num_variants(void) { return kNumVariants; }

int sgemm_f32_variant_info(int v, int *BM, int *BN, int *BK, int *threads, int *TM, int *TN,
                           int *stages) {
  if (v < 0 || v >= kNumVariants) return -1;
  const int built = variant_built(v) ? 0 : 1;
  const VariantShape &s = kVariants[v];
  if (BM) *BM = s.BM;
  if (BN) *BN = s.BN;
  if (BK) *BK = s.BK;
  if (threads) *threads = s.threads;
  if (TM) *TM = s.TM;
  if (TN) *TN = s.TN;
  if (stages) *stages = s.stages;
  return built;
}

int sgemm_f32_cluster_capacity(int variant, int cluster, int *ctas) {
  if (ctas) *ctas = 0;
  if (variant < 0 || variant >= kNumVariants) return -1;
  if (cluster < 1 || cluster > kMaxClusterSplit) return -2;
  if (ctas == nullptr) return -3;
  int num_sms = 0;
  cudaError_t e = device_setup(&num_sms);
  if (e != cudaSuccess) return (int)e;
  const VariantShape &s = kVariants[variant];
  if (s.thin >= 5) {  // cluster thin kernels: clusters of 1, 2, 4 or 8
    if ((cluster & (cluster - 1)) != 0) return 0;
    int t[4];
    thin_cluster_capacity(t);
    int l2 = 0;
    while ((1 << l2) < cluster) ++l2;
    *ctas = t[l2];
    return 0;
  }
  const int *cap = cluster_capacity_table();
  if (cap != nullptr && cluster >= 2 && variant_built(variant))
    *ctas = cap[variant * (kMaxClusterSplit + 1) + cluster];
  return 0;
}

const char *sgemm_f32_version(void) { return "sgemm_f32 0.1.0 sm_103a"; }

int sgemm_f32_wait_selftest(int *timed_out, float *seconds) {
  if (timed_out) *timed_out = 0;
  if (seconds) *seconds = 0.0f;
  int num_sms = 0;
  cudaError_t e = device_setup(&num_sms);
  if (e != cudaSuccess) return (int)e;
  int *d = nullptr;
  e = cudaMalloc(reinterpret_cast<void **>(&d), sizeof(int));
  if (e != cudaSuccess) return (int)e;
  cudaStream_t s = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  if (e == cudaSuccess) e = cudaMemsetAsync(d, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaEventRecord(e0, s);
  if (e == cudaSuccess) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(d);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaEventRecord(e1, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  int v = 0;
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaMemcpy(&v, d, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (s) cudaStreamDestroy(s);
  cudaFree(d);
  if (e != cudaSuccess) return (int)e;
  if (timed_out) *timed_out = v;
  if (seconds) *seconds = ms / 1000.0f;
  return 0;
}

int sgemm_f32_release_workspace(size_t *released_bytes) {
  if (released_bytes) *released_bytes = 0;
  int num_sms = 0;
  cudaError_t e = device_setup(&num_sms);  // (creates the empty pool on a first call)
  if (e != cudaSuccess) return (int)e;
  cudaMemPool_t pool = workspace_pool();
  if (pool == nullptr) return (int)cudaErrorInvalidDevice;
  uint64_t before = 0, after = 0;
  e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &before);
  if (e == cudaSuccess) e = cudaMemPoolTrimTo(pool, 0);
  if (e == cudaSuccess) e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &after);
  if (e != cudaSuccess) return (int)e;
  if (released_bytes) *released_bytes = (size_t)(before > after ? before - after : 0);
  return 0;
}

int sgemm_f32_status(int *status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_ffma_status, sizeof(int));
  if (e != cudaSuccess) return (int)e;
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_ffma_status, &zero, sizeof(int));
  if (status) *status = v;
  return (int)e;
}

}  // extern "C"
