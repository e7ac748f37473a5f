// Host-side argument checks and launch planning for the SGEMM library. Plain C++ (no CUDA
// types), so the same logic is exercised by CPU-only tests through sgemm_f32_plan().
#pragma once

#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <limits>

namespace sgemm {

constexpr int kErrWorkspace = -13;
constexpr int kErrBadVariant = -14;

struct Problem {
  int M, N, K, lda, ldb, ldc;
  int transa = 0, transb = 0;  // 1: op(X) = X_st^T (see sgemm_f32_ex)
  bool tma_ok = false;         // A, B 16-byte aligned with lda, ldb % 4 == 0 (TMA-fed kernel)
  bool a_tma = false;          // op(A) = A row-major, 16-byte aligned, lda % 4 == 0
  bool b_tma = false;          // op(B) = B row-major, 16-byte aligned, ldb % 4 == 0
  bool at_direct = false;      // op(A) = A_st^T with A_st (K x M) 16-byte aligned, lda % 4 == 0:
                               // A_st is the k-major A the at variants read, no copy needed
  bool kpair_ok = false;       // op(A) = A row-major, 16-byte aligned, lda % 4 == 0
  bool b_kmajor = false;       // op(B) = B_st^T with B_st 16-byte aligned, ldb % 4 == 0
  // CTAs of the cluster thin kernel that the device holds at once in clusters of 1, 2, 4
  // and 8 (queried from the driver; 0 = unknown, modelled by cluster_ctas)
  int cluster_ctas[4] = {0, 0, 0, 0};
  // CTAs of configuration v resident at once in clusters of S, at v * 9 + S (queried from
  // the driver; null = unknown)
  const int *cluster_cap = nullptr;
};

// Shape of one compiled tile configuration (mirrors TileConfig in sgemm_ffma.cuh).
struct VariantShape {
  int BM, BN, BK, threads, TM, TN, stages, min_blocks, mode, smem_bytes;
  double eff;  // modelled fraction of the FP32 pipe this configuration sustains
  bool automatic;  // considered by the automatic plan (others only when forced)
  bool trans_ok;   // compiled with the transposed-operand copy paths
  bool tma = false;  // the TMA-fed kernel (sgemm_ffma_tma.cuh), aligned row-major operands only
  bool kpair = false;  // the K-paired TMA-fed kernel (sgemm_ffma_kpair.cuh): K-major B
  int inst = 0;        // TMA-fed kernels: instance index of the launcher (sgemm_tma.cu)
  int thin = 0;        // streaming kernels: 1 thin-M, 2 thin-N (sgemm_thin.cuh), 3 TMA-fed
                       // thin-M, 4 TMA-fed thin-N (sgemm_thin_tma.cuh), 5 cluster thin-M,
                       // 6 cluster thin-N (sgemm_thin_cluster.cuh)
  bool at = false;     // TMA-fed kernel reading A k-major (A^T; copied first if row-major)
  int twin = -1;       // at variants: the variant with the same tiles and arithmetic that
                       // transposes A in shared memory instead (bitwise the same result)
};

// mode: 0 scalar FFMA, 1 FFMA2 with register broadcast, 2 FFMA2 with duplicated A in smem
constexpr int smem_of(int BM, int BN, int BK, int stages, int mode) {
  return stages * BK * (BM * (mode == 2 ? 2 : 1) + BN) * 4;
}

constexpr VariantShape kVariants[] = {
    {128, 256, 16, 256, 16, 8, 3, 1, 0, smem_of(128, 256, 16, 3, 0), 0.78, true, false},
    {128, 128, 16, 256, 8, 8, 4, 2, 0, smem_of(128, 128, 16, 4, 0), 0.72, true, false},
    {64, 64, 16, 128, 8, 4, 4, 4, 0, smem_of(64, 64, 16, 4, 0), 0.60, true, true},
    {16, 256, 32, 128, 8, 4, 3, 2, 0, smem_of(16, 256, 32, 3, 0), 0.50, true, true},
    {256, 16, 32, 128, 8, 4, 3, 2, 0, smem_of(256, 16, 32, 3, 0), 0.50, true, true},
    {128, 256, 16, 256, 8, 16, 3, 1, 1, smem_of(128, 256, 16, 3, 1), 0.86, true, false},
    {128, 256, 16, 256, 8, 16, 3, 1, 2, smem_of(128, 256, 16, 3, 2), 0.80, false, false},
    {128, 256, 32, 256, 8, 16, 3, 1, 2, smem_of(128, 256, 32, 3, 2), 0.80, false, false},
    {128, 128, 16, 256, 8, 8, 4, 2, 1, smem_of(128, 128, 16, 4, 1), 0.83, true, false},
    {128, 256, 16, 512, 8, 8, 3, 1, 1, smem_of(128, 256, 16, 3, 1), 0.80, false, false},
    {256, 128, 16, 512, 8, 8, 3, 1, 1, smem_of(256, 128, 16, 3, 1), 0.80, false, false},
    {128, 256, 32, 256, 8, 16, 3, 1, 1, smem_of(128, 256, 32, 3, 1), 0.80, false, false},
    {128, 256, 16, 256, 8, 16, 3, 1, 1, smem_of(128, 256, 16, 3, 1), 0.80, false, false},
    {128, 256, 16, 256, 8, 16, 4, 1, 1, smem_of(128, 256, 16, 4, 1), 0.88, true, false},
    {128, 64, 16, 128, 8, 8, 3, 2, 1, smem_of(128, 64, 16, 3, 1), 0.80, false, false},
    {128, 64, 16, 128, 8, 8, 4, 2, 1, smem_of(128, 64, 16, 4, 1), 0.80, false, false},
    {128, 128, 16, 128, 8, 16, 3, 2, 1, smem_of(128, 128, 16, 3, 1), 0.90, true, true},
    {128, 64, 16, 128, 8, 8, 3, 3, 1, smem_of(128, 64, 16, 3, 1), 0.80, false, false},
    {128, 256, 16, 256, 4, 32, 4, 1, 1, smem_of(128, 256, 16, 4, 1), 0.80, false, false},
    {128, 128, 16, 128, 4, 32, 3, 2, 1, smem_of(128, 128, 16, 3, 1), 0.80, false, false},
    {16, 512, 16, 128, 8, 8, 3, 2, 1, smem_of(16, 512, 16, 3, 1), 0.60, false, false},
    {128, 16, 32, 128, 4, 4, 4, 3, 0, smem_of(128, 16, 32, 4, 0), 0.55, true, false},
    {128, 128, 16, 128, 8, 16, 4, 2, 1, smem_of(128, 128, 16, 4, 1), 0.80, false, false},
    {128, 128, 32, 128, 8, 16, 3, 2, 1, smem_of(128, 128, 32, 3, 1), 0.80, false, false},
    {128, 128, 8, 128, 8, 16, 6, 2, 1, smem_of(128, 128, 8, 6, 1), 0.80, false, false},
    {128, 128, 16, 128, 8, 16, 3, 2, 2, smem_of(128, 128, 16, 3, 2), 0.80, false, false},
    // 26: TMA-fed 128 x 128 x 32, 3 stages, 2 CTAs/SM (its own kernel, see kTmaVariant)
    {128, 128, 32, 128, 8, 16, 3, 2, 1, smem_of(128, 128, 32, 3, 1), 0.96, true, false, true},
    // 27..29: K-paired TMA-fed 128 x 128 x 32, 8 warps, 1 CTA/SM, 4 / 5 / 6 stages; B is
    // read K-major (B^T), copied to a workspace first when the caller's B is row-major
    {128, 128, 32, 256, 8, 8, 4, 1, 3, smem_of(128, 128, 32, 4, 1), 0.88, true, true, false, true},
    {128, 128, 32, 256, 8, 8, 5, 1, 3, smem_of(128, 128, 32, 5, 1), 0.88, false, true, false, true},
    {128, 128, 32, 256, 8, 8, 6, 1, 3, smem_of(128, 128, 32, 6, 1), 0.88, false, true, false, true},
    // 30..32: more TMA-fed shapes: 128 x 96 (8 x 12 threads, 3 CTAs/SM, 2 stages); the 26
    // shape without A double-buffering; 128 x 64 (8 x 8 threads, 4 CTAs/SM, 2 stages)
    {128, 96, 32, 128, 8, 12, 2, 3, 1, smem_of(128, 96, 32, 2, 1), 0.97, true, false, true, false, 1},
    {128, 128, 32, 128, 8, 16, 3, 2, 1, smem_of(128, 128, 32, 3, 1), 0.90, false, false, true, false, 2},
    {128, 64, 32, 128, 8, 8, 2, 4, 1, smem_of(128, 64, 32, 2, 1), 0.955, true, false, true, false, 3},
    // 33, 34: streaming kernels for thin products (sgemm_thin.cuh): thin-M, 16 x 256 C tiles
    // (4 columns x 16 rows per thread, 4 k-groups, 2 CTAs/SM); thin-N, 1024 x 16 C tiles
    // (4 rows x 16 columns per thread, 1 CTA/SM). BK is the k batch of the streamed loads.
    {16, 256, 8, 256, 16, 4, 1, 2, 1, 0, 0.65, false, false, false, false, 0, 1},
    {1024, 16, 8, 256, 4, 16, 1, 1, 1, 0, 0.65, false, false, false, false, 0, 2},
    // 35, 36: the TMA-fed 128 x 96 and 128 x 128 shapes reading A k-major: A is copied to
    // A^T first, and the A tile arrives as [32 k][128 m] like the B tile. Their math loop
    // sustains ~9% more than 30 / 31 (measured 69.6 against 63.7 TFLOP/s at 8192^3).
    {128, 96, 32, 128, 8, 12, 2, 3, 1, smem_of(128, 96, 32, 2, 1), 1.06, true, false, true, false, 4, 0, true, 37},
    // 36 is forced-only: over 24 shapes from 200^3 to 3072^3 (every configuration and split
    // measured per call on GB300) it was 2-40% slower than the better of 35 and 39 on each.
    {128, 128, 32, 128, 8, 16, 3, 2, 1, smem_of(128, 128, 32, 3, 1), 1.04, false, false, true, false, 5, 0, true, 38},
    // 37, 38: the same two shapes reading A as stored and transposing each A tile in shared
    // memory (no workspace, no pre-pass; 128 x 128 with 2 stages to fit 2 CTAs/SM). They
    // are 3-5% slower than 35 / 36 at 8192^3 and 14-34% slower than the automatic choice
    // without them at 768^3 and 1536^3 (measured per call), so they are not automatic: they
    // are the twins that sgemm_f32_ws and sgemm_f32_noalloc take when their workspace cannot
    // hold the A^T copy
    {128, 96, 32, 128, 8, 12, 2, 3, 1, smem_of(128, 96, 32, 2, 1) + 16384, 1.028, false, false, true, false, 6},
    {128, 128, 32, 128, 8, 16, 2, 2, 1, smem_of(128, 128, 32, 2, 1) + 16384, 1.03, false, false, true, false, 7},
    // 39, 40: k-major A, 128 x 64 at 4 CTAs/SM and 128 x 128 with 2 stages. 39 is automatic
    // with its efficiency calibrated against 35 (1.8% slower at 8192^3, 13% faster at 3000^3,
    // 6% at 2048^3, where its 608 slots round the waves better)
    {128, 64, 32, 128, 8, 8, 2, 4, 1, smem_of(128, 64, 32, 2, 1), 1.04, true, false, true, false, 8, 0, true, 45},
    {128, 128, 32, 128, 8, 16, 2, 2, 1, smem_of(128, 128, 32, 2, 1), 1.0, false, false, true, false, 9, 0, true, 38},
    // 41: TMA-fed thin-M, 16 x 256 C tiles, 8 warps each streaming its own 8-k chunks of B
    // through 2 private stages, K slices reduced by the split-K finish (1 CTA/SM)
    {16, 256, 8, 256, 16, 8, 2, 1, 1, 0, 0.7, true, false, false, false, 0, 3},
    // 42: TMA-fed thin-N (C^T = B^T A^T on the same kernel): 256 x 16 C tiles, A streamed
    // as [256 m][8 k] chunks
    {256, 16, 8, 256, 8, 16, 2, 1, 1, 0, 0.7, true, false, false, false, 0, 4},
    // 43, 44: cluster thin-M / thin-N: 16 x 128 (128 x 16) C tiles, 16 warps streaming both
    // operands by TMA in 8-k chunks (16 x 4 outputs per lane, every warp over the whole
    // tile), the K slices of a tile one cluster of 1, 2, 4 or 8 CTAs reduced through
    // distributed shared memory (no workspace, one launch)
    {16, 128, 8, 512, 16, 4, 2, 1, 1, 0, 0.8, true, false, false, false, 0, 5},
    {128, 16, 8, 512, 4, 16, 2, 1, 1, 0, 0.8, true, false, false, false, 0, 6},
    // 45: 39's twin, transposing each A tile in shared memory (3 CTAs/SM; forced-only, and
    // the substitute for 39 when a caller workspace cannot hold the A^T copy)
    {128, 64, 32, 128, 8, 8, 2, 3, 1, smem_of(128, 64, 32, 2, 1) + 16384, 0.98, true, false, true, false, 10},
};
constexpr int kNumVariants = sizeof(kVariants) / sizeof(kVariants[0]);

// Copy-fed configurations that stay in the table, so that every index keeps its meaning, but
// are not compiled: neither the automatic plan nor sgemm_f32_autotune chose any of them on
// the shapes measured (the copy-fed configurations the plan can choose are 0-5, 8, 13, 16
// and 21). Forcing one returns -14.
constexpr int kRetiredVariants[] = {6, 7, 9, 10, 11, 12, 14, 15, 17, 18, 19, 20, 22, 23, 24, 25};
constexpr bool variant_built(int v) {
  for (int r : kRetiredVariants)
    if (r == v) return false;
  return v >= 0 && v < kNumVariants;
}
constexpr bool retired_are_forced_only() {
  for (int r : kRetiredVariants)
    if (kVariants[r].automatic || kVariants[r].trans_ok || kVariants[r].tma || kVariants[r].thin)
      return false;
  return true;
}
static_assert(retired_are_forced_only(), "only forced-only copy-fed configurations retire");
// Whether configuration v is the shared-memory-transpose twin of a k-major one.
constexpr bool is_transpose_twin(int v) {
  for (int u = 0; u < kNumVariants; ++u)
    if (kVariants[u].twin == v) return true;
  return false;
}
// The automatic plan takes a transpose twin only for K loops of at least this many K
// blocks: its per-block transpose and its fewer CTAs per SM do not pay on shorter ones
// (measured 9-10% behind configurations 32 / 39 at 2 and 4 K blocks, ahead at 8 and more).
constexpr int kTwinMinKBlocks = 8;

constexpr int kTmaVariant = 26;
constexpr int kFirstKpairVariant = 27;
constexpr int kThinMVariant = 33, kThinNVariant = 34;
constexpr int kThinMaxDim = 64;  // thin kernels considered for M (thin-M) or N (thin-N) <= this
// The cluster thin kernels (43, 44) are considered up to this M (thin-M) or N (thin-N):
// where the streamed operand stays in L2 they beat the tiled kernels well past 64, e.g.
// 5.1 against 6.0 us at 256^3, 6.5 against 10.1 at 384^3, 10.1 against 13.4 at
// 1024 x 128 x 1024 (per call, measured on GB300); the model decides.
constexpr int kThinClusterMaxDim = 1024;
constexpr int kThinMKmax = 512, kThinNKmax = 2048;  // K slice bounds (shared memory)
constexpr int kThinTmaVariant = 41, kThinTmaKmax = 1024;
constexpr int kThinClusterVariant = 43;  // 43 thin-M, 44 thin-N
constexpr int kMaxThinCluster = 8;
static_assert(kVariants[kTmaVariant].tma, "TMA variant index");
static_assert(kVariants[kFirstKpairVariant].kpair, "K-paired variant index");

struct Plan {
  int variant = -1;     // -1: no GEMM kernel (beta-scale only, or nothing)
  int main_tiles = 0;   // tiles computed whole by CTAs 0 .. main_tiles-1
  int split = 1;        // K slices of each remaining tile (1: no split-K)
  int k_per_split = 0;  // K elements per slice (multiple of BK)
  int tiles_m = 0, tiles_n = 0;
  int group_m = 1;
  int ctas = 0;         // GEMM grid size
  int launches = 0;
  // Workspace layout: [B^T copy | packed A | packed B | split-K partial tiles]; the first
  // three (pre_bytes in all) are written by pre-passes before the GEMM kernel.
  size_t ws_bytes = 0;
  size_t bt_bytes = 0;  // K-paired variants on a row-major B: its N x ldbt transpose
  long long ldbt = 0;
  // TMA-fed variants on row-major operands that TMA cannot address (ld % 4 != 0 or a
  // misaligned pointer): the operand is first copied to rows of ld_p = ceil4(cols) floats.
  bool pack_a = false, pack_b = false;
  long long lda_p = 0, ldb_p = 0;
  size_t pack_a_bytes = 0, pack_b_bytes = 0;
  // k-major TMA-fed variants: A^T (K x ldat) made by a transpose pre-pass (in pack_a_bytes)
  bool at_a = false;
  // every tile split (main_tiles == 0) into split <= 8 slices that run as one thread-block
  // cluster and add their partial tiles through distributed shared memory: no partial-tile
  // workspace, no reduce launch
  bool cluster = false;
  size_t pre_bytes = 0;
  double cycles = 0;    // modelled cost
};

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

constexpr int kMaxClusterSplit = 8;  // portable cluster size

// Whether a split of every tile of variant v into `split` slices can be finished inside a
// cluster: the GEMM kernels (not the thin or K-paired ones) whose shared memory holds a
// BM x BN FP32 tile, and 2 .. 8 slices.
inline bool cluster_split_ok(int v, int split) {
  const VariantShape &s = kVariants[v];
  return !s.thin && !s.kpair && split >= 2 && split <= kMaxClusterSplit &&
         (long long)s.BM * s.BN * 4 <= (long long)smem_of(s.BM, s.BN, s.BK, s.stages, s.mode);
}

// CTAs of the cluster thin kernel resident at once in clusters of S = 1 << l2 CTAs: the
// driver's figure when known, else a model of a GPU whose SMs sit in GPCs of about 19 SMs
// (a cluster never spans two): GB300 holds 144 CTAs in clusters of 4 and 120 in clusters of 8.
inline long long cluster_ctas(const Problem &p, int num_sms, int l2) {
  if (p.cluster_ctas[l2] > 0) return p.cluster_ctas[l2];
  static const double kFill[4] = {1.0, 1.0, 18.0 / 19.0, 15.0 / 19.0};
  const int S = 1 << l2;
  return std::max<long long>(S, (long long)(num_sms * kFill[l2]) / S * S);
}

// Modelled cost of a thin-product streaming kernel (variant v with s.thin != 0) with `split`
// K slices. The kernels stream one operand once and are bound by HBM at their shapes:
// the cost is the larger of the streamed bytes at ~2800 bytes/cycle for the chip (about
// 80% of the measured copy bandwidth) and the FMA work at the variant's efficiency, plus
// ~2000 cycles per launch. Partial tiles add their write and the reduce's read. The cluster
// kernels (thin 5, 6) take split = the cluster size (1, 2, 4 or 8), have no K bound and no
// partial tiles, and fill HBM once about 85% of the SMs stream (a TMA streaming probe
// reached the full copy bandwidth from 128 of 152 SMs).
// A cluster thin kernel's K slices add their partial tiles through distributed shared
// memory: two cluster barriers per wave (fitted with the GEMM kernels' fixed costs below).
constexpr double kThinClusterSplitCycles = 1500.0;

inline Plan model_thin(const Problem &p, int v, int split, int num_sms, bool beta_nz) {
  const VariantShape &s = kVariants[v];
  Plan pl;
  pl.variant = v;
  pl.tiles_m = (int)ceil_div(p.M, s.BM);
  pl.tiles_n = (int)ceil_div(p.N, s.BN);
  const bool cluster = s.thin >= 5;
  const bool streams_b = s.thin == 1 || s.thin == 3 || s.thin == 5;  // thin-M kinds stream B
  const int kq = 8;  // K slice granule (the load batch / TMA chunk of the thin kernels)
  long long kps = ceil_div(ceil_div(p.K, std::max(1, split)), kq) * kq;
  if (cluster) {
    int l2 = 0;
    while ((1 << l2) < split && l2 < 3) ++l2;
    split = 1 << l2;
    kps = std::max<long long>(kps, kq);
  } else {
    const int kmax = s.thin == 1 ? kThinMKmax : s.thin == 2 ? kThinNKmax : kThinTmaKmax;
    kps = std::min<long long>(std::max<long long>(kps, kq), kmax);
    split = (int)ceil_div(p.K, kps);
  }
  const long long tiles = (long long)pl.tiles_m * pl.tiles_n;
  const long long ctas = tiles * split;
  const double per_cta_fma = (double)s.BM * s.BN * (double)kps;
  const double rate = 128.0 * s.eff / s.min_blocks;  // FMA per cycle per resident CTA
  int l2 = 0;
  while ((1 << l2) < split) ++l2;
  const long long slots = cluster ? std::min<long long>(num_sms, cluster_ctas(p, num_sms, l2))
                                  : (long long)num_sms * s.min_blocks;
  const long long waves = ceil_div(ctas, slots);
  const double compute = (double)waves * per_cta_fma / rate;
  // streamed operand once per tile row (thin-M: B per row block) or column (thin-N: A)
  const double streamed = streams_b ? 4.0 * pl.tiles_m * (double)p.K * p.N
                                    : 4.0 * pl.tiles_n * (double)p.M * p.K;
  const double small = streams_b ? 4.0 * (double)p.M * p.K : 4.0 * (double)p.K * p.N;
  const int groups = cluster ? 1 : split;  // partial tiles per C tile in the workspace
  const double part = groups > 1 ? (double)tiles * groups * s.BM * s.BN * 4.0 : 0.0;
  const double mn_c = (double)p.M * p.N * 4.0 * (beta_nz ? 2.0 : 1.0);
  const double bytes = streamed + small + mn_c + 2.0 * part;
  pl.main_tiles = 0;
  pl.split = split;
  pl.k_per_split = (int)std::min<long long>(kps, 0x7ffffff8LL);
  pl.group_m = 1;
  pl.ctas = (int)std::min<long long>(ctas, 0x7fffffffLL);
  pl.launches = groups > 1 ? 2 : 1;
  pl.ws_bytes = groups > 1 ? (size_t)part : 0;
  // HBM is streamed at full speed only while enough SMs have work: scale the bandwidth by
  // the average fraction of CTA slots the grid fills over its waves (cluster kernels: of
  // 85% of the SMs). Each wave also pays ~3000 cycles of start-up (first copies in flight,
  // staging) and reduction that nothing hides.
  const double fill = cluster ? std::min(1.0, (double)ctas / (double)waves / (0.85 * num_sms))
                              : (double)ctas / (double)(waves * slots);
  pl.cycles = std::max(compute, bytes / (2800.0 * fill)) + 3000.0 * (double)waves +
              (cluster && split > 1 ? kThinClusterSplitCycles * (double)waves : 0.0) +
              2000.0 * pl.launches;
  // The cluster kernels read both operands by TMA. A small operand whose rows TMA cannot
  // address (row stride not a multiple of 16 bytes, or a misaligned base) is first copied
  // to aligned rows in the workspace: at most 64 rows (thin-M: A) or columns (thin-N: B).
  if (cluster && !(streams_b ? p.a_tma : p.b_tma)) {
    if (streams_b) {
      pl.pack_a = true;
      pl.lda_p = ceil_div(p.K, 4) * 4;
      pl.pack_a_bytes = (size_t)ceil_div((long long)p.M * pl.lda_p * 4, 256) * 256;
    } else {
      pl.pack_b = true;
      pl.ldb_p = ceil_div(p.N, 4) * 4;
      pl.pack_b_bytes = (size_t)ceil_div((long long)p.K * pl.ldb_p * 4, 256) * 256;
    }
    pl.pre_bytes = pl.pack_a_bytes + pl.pack_b_bytes;
    pl.ws_bytes += pl.pre_bytes;
    pl.launches += 1;
    pl.cycles += 2.0 * small / 3400.0 + 2000.0;  // read and written once, one launch
  }
  if (ctas > 0x7fffffffLL || pl.tiles_m > 65535 || pl.tiles_n > 65535 || split > 65535)
    pl.cycles = std::numeric_limits<double>::infinity();
  return pl;
}

// BLAS-style check: the first illegal argument, numbered from 1 in the sgemm_f32 order
// (M, N, K, alpha, A, lda, B, ldb, beta, C, ldc). A and B only have to be present when
// they are read (alpha != 0, K > 0, non-empty C); C whenever the view is non-empty.
// With transposed operands the stored A is K x M (lda >= M) and the stored B is N x K
// (ldb >= K), row-major.
inline int validate(const Problem &p, float alpha, bool hasA, bool hasB, bool hasC) {
  if (p.M < 0) return -1;
  if (p.N < 0) return -2;
  if (p.K < 0) return -3;
  const bool nonempty = p.M > 0 && p.N > 0;
  const bool reads_ab = nonempty && p.K > 0 && alpha != 0.0f;
  if (reads_ab && !hasA) return -5;
  if (p.lda < std::max(1, p.transa ? p.M : p.K)) return -6;
  if (reads_ab && !hasB) return -7;
  if (p.ldb < std::max(1, p.transb ? p.K : p.N)) return -8;
  if (nonempty && !hasC) return -10;
  if (p.ldc < std::max(1, p.N)) return -11;
  return 0;
}

// sgemm_f32_ex order: (transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc).
inline int validate_ex(const Problem &p, float alpha, bool hasA, bool hasB, bool hasC) {
  if (p.transa != 0 && p.transa != 1) return -1;
  if (p.transb != 0 && p.transb != 1) return -2;
  const int rc = validate(p, alpha, hasA, hasB, hasC);
  return rc < 0 ? rc - 2 : rc;
}

// Column-major (BLAS / cuBLAS) order and rules: (transa, transb, m, n, k, alpha, A, lda,
// B, ldb, beta, C, ldc); A is m x k (k x m when transposed), B is k x n (n x k), C m x n,
// each with ld >= its row count.
inline int validate_colmajor(int transa, int transb, int m, int n, int k, int lda, int ldb,
                             int ldc, float alpha, bool hasA, bool hasB, bool hasC) {
  if (transa != 0 && transa != 1) return -1;
  if (transb != 0 && transb != 1) return -2;
  if (m < 0) return -3;
  if (n < 0) return -4;
  if (k < 0) return -5;
  const bool nonempty = m > 0 && n > 0;
  const bool reads_ab = nonempty && k > 0 && alpha != 0.0f;
  if (reads_ab && !hasA) return -7;
  if (lda < std::max(1, transa ? k : m)) return -8;
  if (reads_ab && !hasB) return -9;
  if (ldb < std::max(1, transb ? n : k)) return -10;
  if (nonempty && !hasC) return -12;
  if (ldc < std::max(1, m)) return -13;
  return 0;
}

// Modelled cost, in SM cycles, of variant v with `main` whole tiles and the rest split
// into `split` K slices. `slots` CTAs run at once (SMs x CTAs per SM), each at 1/min_blocks
// of its SM's 128 FMA/cycle scaled by the variant's efficiency, plus ~2500 cycles of
// pipeline fill and epilogue per CTA; a slice also stores its BM x BN partial tile at the
// SM's share of the chip's bandwidth. Whole tiles run first (CTA order), then the slices.
// The GEMM overlaps with streaming its algorithmic bytes at ~3400 bytes/cycle for the
// chip. Split tiles add a reduction kernel afterwards: partials read, C read (beta != 0)
// and written, plus ~2000 cycles of launch.
// Fixed costs of the GEMM kernels' model, in SM cycles, fitted to per-call times measured
// on GB300 (CUDA graphs of back-to-back calls, inputs from HBM) over 30 shapes from 200^3 to
// 4096^3, thin and flat ones included, and every configuration and split of each: the
// model's choice among the measured plans came within 0.7% of the fastest on 24 of them.
// - kCtaFixedCycles: per CTA (whole tile or K slice): its start, first copies in flight
//   and epilogue, which a short K loop does not amortise;
// - kClusterFinishCycles: a split finished inside a cluster: its two cluster barriers,
//   the distributed-shared-memory reads and the sparser placement of clusters (at 1024^3
//   an 8-way cluster split and a 12-way split with the reduce kernel both take 50 us);
// - kGemmLaunchCycles: the GEMM launch itself (the thin kernels' model charges the same
//   kind of cost per launch).
constexpr double kCtaFixedCycles = 9000.0;
constexpr double kClusterFinishCycles = 12000.0;
constexpr double kGemmLaunchCycles = 2000.0;

inline Plan model_plan(const Problem &p, int v, long long main, int split, int num_sms,
                       bool beta_nz) {
  const VariantShape &s = kVariants[v];
  Plan pl;
  pl.variant = v;
  pl.tiles_m = (int)ceil_div(p.M, s.BM);
  pl.tiles_n = (int)ceil_div(p.N, s.BN);
  const long long tiles = (long long)pl.tiles_m * pl.tiles_n;
  const long long kt = ceil_div(p.K, s.BK);
  if (split <= 1 || main >= tiles) {
    split = 1;
    main = tiles;
  }
  const long long kt_per = ceil_div(kt, split);
  split = (int)ceil_div(kt, kt_per);  // no empty slices
  if (split == 1) main = tiles;
  const long long tail = tiles - main;
  const long long slots = (long long)num_sms * s.min_blocks;
  const double rate = 128.0 * s.eff / s.min_blocks;  // FMA per cycle per resident CTA
  const double t_full = (double)s.BM * s.BN * (double)(kt * s.BK) / rate + kCtaFixedCycles;
  const double t_slice = (double)s.BM * s.BN * (double)(kt_per * s.BK) / rate +
                         kCtaFixedCycles + (double)s.BM * s.BN * 4.0 / (3400.0 / num_sms);
  // CTAs start in index order, `slots` at a time: whole tiles first, then slices. A round
  // with fewer CTAs than slots leaves some SMs with fewer resident CTAs, which then run
  // faster, though less than in proportion: n of min_blocks CTAs on an SM take about
  // (n / min_blocks)^0.85 of their shared-SM time, and a CTA alone on its SM (4 warps,
  // one per scheduler, too few to keep the FP32 pipe busy) (1 / min_blocks)^0.6
  // (calibrated on 4096^3 and 8192^3, and on the last wave of 4099 x 3001 x 777).
  // Closed form (no loop over rounds): full rounds of whole tiles; one round mixing the
  // remaining whole tiles with the first slices; full rounds of slices; a last partial
  // round of slices.
  const long long slices = tail * split;
  auto partial = [&](long long n, double t) {
    if (n <= 0) return 0.0;
    const long long per_sm = ceil_div(n, num_sms);
    return t * std::pow((double)per_sm / s.min_blocks, per_sm == 1 ? 0.6 : 0.85);
  };
  double compute = (double)(main / slots) * t_full;
  const long long rem_full = main % slots;
  long long rem_slices = slices;
  if (rem_full > 0) {
    const long long mixed = std::min(slots - rem_full, rem_slices);
    rem_slices -= mixed;
    compute += partial(rem_full + mixed, t_full);
  }
  compute += (double)(rem_slices / slots) * t_slice;
  compute += partial(rem_slices % slots, t_slice);
  const double mn_c = (double)p.M * p.N * 4.0 * (beta_nz ? 2.0 : 1.0);
  double gemm_bytes = 4.0 * ((double)p.M * p.K + (double)p.K * p.N);
  double reduce = 0.0;
  const double part_bytes = (double)slices * s.BM * s.BN * 4.0;
  if (slices > 0) {
    const double tail_frac = (double)tail / (double)tiles;
    gemm_bytes += part_bytes + mn_c * (1.0 - tail_frac);
    reduce = (part_bytes + mn_c * tail_frac) / 3400.0 + 2000.0;
  } else {
    gemm_bytes += mn_c;
  }
  double bt_cycles = 0.0;
  if (s.kpair && !p.b_kmajor) {  // B -> B^T copy: K N floats read and written, one launch
    pl.ldbt = ceil_div(p.K, 4) * 4;
    pl.bt_bytes = (size_t)ceil_div((long long)p.N * pl.ldbt * 4, 256) * 256;
    bt_cycles = 8.0 * (double)p.K * p.N / 3400.0 + 2000.0;
  }
  if (s.at && !p.at_direct) {  // A^T first: M K floats read and written, one launch
    pl.at_a = true;
    pl.lda_p = ceil_div(p.M, 4) * 4;
    pl.pack_a_bytes = (size_t)ceil_div((long long)p.K * pl.lda_p * 4, 256) * 256;
    bt_cycles += 8.0 * (double)p.M * p.K / 3400.0 + 2000.0;
  }
  if (s.tma && !p.tma_ok) {  // aligned copies of the operands TMA cannot address
    if (!p.a_tma && !s.at) {
      pl.pack_a = true;
      pl.lda_p = ceil_div(p.K, 4) * 4;
      pl.pack_a_bytes = (size_t)ceil_div((long long)p.M * pl.lda_p * 4, 256) * 256;
      bt_cycles += 8.0 * (double)p.M * p.K / 3400.0 + 2000.0;
    }
    if (!p.b_tma) {
      pl.pack_b = true;
      pl.ldb_p = ceil_div(p.N, 4) * 4;
      pl.pack_b_bytes = (size_t)ceil_div((long long)p.K * pl.ldb_p * 4, 256) * 256;
      bt_cycles += 8.0 * (double)p.K * p.N / 3400.0 + 2000.0;
    }
  }
  pl.pre_bytes = pl.bt_bytes + pl.pack_a_bytes + pl.pack_b_bytes;
  // Clusters are placed within one GPC each, so fewer CTAs may be resident at once than
  // `slots`: take them only when that costs no extra wave (with the driver's figure; else
  // when a sixth of the slots to spare covers the loss).
  long long cap = (long long)(0.85 * (double)slots);
  if (p.cluster_cap != nullptr && split >= 2 && split <= kMaxClusterSplit)
    cap = p.cluster_cap[v * (kMaxClusterSplit + 1) + split];
  const bool cluster_fits = cap > 0 && ceil_div(slices, cap) <= ceil_div(slices, slots);
  if (main == 0 && cluster_split_ok(v, split) && cluster_fits) {
    // the cluster adds the slices in shared memory: no partial tiles in HBM and no reduce
    // launch; two cluster barriers and each CTA reading one tile's worth over DSMEM
    pl.cluster = true;
    gemm_bytes -= part_bytes;
    reduce = kClusterFinishCycles + (double)s.BM * s.BN * 4.0 / 64.0;
  }
  pl.main_tiles = (int)main;
  pl.split = split;
  pl.k_per_split = (int)(kt_per * s.BK);
  pl.group_m = std::min(16, pl.tiles_m);
  pl.ctas = (int)(main + slices);
  pl.launches = (slices > 0 && !pl.cluster ? 2 : 1) + (pl.bt_bytes > 0 ? 1 : 0) +
                (pl.pack_a || pl.at_a ? 1 : 0) + (pl.pack_b ? 1 : 0);
  pl.ws_bytes = pl.pre_bytes + (slices > 0 && !pl.cluster ? (size_t)part_bytes : 0);
  pl.cycles = std::max(compute, gemm_bytes / 3400.0) + reduce + bt_cycles + kGemmLaunchCycles;
  if (main + slices > 0x7fffffffLL) {  // grid too large for one launch
    pl.ctas = 0;
    pl.cycles = std::numeric_limits<double>::infinity();
  }
  return pl;
}

// The same plan with an at variant replaced by its twin, which transposes A in shared
// memory instead of reading a transposed copy: identical tiles, slices and k order (so
// bitwise the same result), without the A^T workspace or its launch. Only for an A that
// TMA can read as stored; otherwise the plan is returned unchanged.
inline Plan without_at_copy(const Problem &p, const Plan &pl) {
  if (pl.variant < 0 || !pl.at_a || !p.a_tma) return pl;
  const VariantShape &s = kVariants[pl.variant];
  if (s.twin < 0) return pl;
  Plan t = pl;
  t.variant = s.twin;
  t.at_a = false;
  t.pre_bytes -= pl.pack_a_bytes;
  t.ws_bytes -= pl.pack_a_bytes;
  t.pack_a_bytes = 0;
  t.lda_p = 0;
  t.launches -= 1;
  return t;
}

// Choose the tile configuration and the split-K layout. Candidates per variant: no split;
// every tile split in s slices; and, when the tiles do not fill the last wave, the full
// waves whole with only the last wave's tiles split (s chosen to fill that wave).
// force_v >= 0 pins the variant. force_split >= 1 splits every tile into that many slices
// (1: none); force_split == -1 takes the whole-waves-plus-split-tail layout with the
// automatic slice count, force_split <= -2 the same layout with -force_split slices;
// 0 leaves the choice to the model. The automatic choice takes the K-paired configurations
// only for a B that is already K-major (transposed and aligned): copying a row-major B to
// B^T first is never faster than the TMA-fed configuration on the same operands, so that
// copy happens only when such a configuration is forced.
inline Plan make_plan(const Problem &p, float alpha, float beta, int num_sms, int force_v,
                      int force_split) {
  Plan best;
  if (p.M == 0 || p.N == 0) return best;  // nothing to launch
  if (alpha == 0.0f || p.K == 0) {
    best.launches = (beta == 1.0f) ? 0 : 1;
    return best;
  }
  num_sms = std::max(1, num_sms);
  const bool beta_nz = beta != 0.0f;
  best.cycles = std::numeric_limits<double>::infinity();
  const double ws_cap = 64.0 * 1024 * 1024;  // largest split-K workspace the plan may use
  const size_t bt_cap = (size_t)2 << 30;  // largest pre-pass copies (B^T, packs) a plan makes
  auto consider = [&](const Plan &c) {
    if ((double)(c.ws_bytes - c.pre_bytes) > ws_cap && force_split < 1) return;
    if (c.pre_bytes > bt_cap) return;
    if (c.cycles < best.cycles * 0.999) best = c;  // prefer earlier (simpler) on ties
  };
  const int v_lo = force_v >= 0 ? force_v : 0;
  const int v_hi = force_v >= 0 ? force_v : kNumVariants - 1;
  const bool trans = p.transa || p.transb;
  for (int v = v_lo; v <= v_hi; ++v) {
    if (!variant_built(v)) continue;
    if (force_v < 0 && !kVariants[v].automatic) continue;
    const bool at_path = kVariants[v].at && p.at_direct && !p.transb;  // A_st is A^T
    if (trans && !kVariants[v].trans_ok && !at_path) continue;
    if (kVariants[v].tma && !p.tma_ok && (p.transa || p.transb) &&
        !(kVariants[v].at && p.at_direct && !p.transb))
      continue;
    if (kVariants[v].kpair && (!p.kpair_ok || (force_v < 0 && !p.b_kmajor))) continue;
    const VariantShape &s = kVariants[v];
    if (force_v < 0 && is_transpose_twin(v) && ceil_div(p.K, s.BK) < kTwinMinKBlocks) continue;
    // 16-wide tiles exist for thin problems: the automatic plan keeps them for those, and
    // there prefers the TMA-fed thin kernels where they apply (measured 10-25% faster than
    // the copy-fed 16-wide tiles on 16 x 4096 x 4096 and 4096 x 16 x 8192)
    if (force_v < 0 && s.thin < 5 &&
        ((s.BM <= 16 && p.M > kThinMaxDim) || (s.BN <= 16 && p.N > kThinMaxDim)))
      continue;
    if (force_v < 0 && !s.thin && !s.tma && !s.kpair &&
        ((s.BM <= 16 && p.b_tma && !p.transa) || (s.BN <= 16 && p.a_tma && !p.transb)))
      continue;
    if (s.thin) {
      const bool thin_n_kind = s.thin == 2 || s.thin == 4 || s.thin == 6;
      const int max_dim = s.thin >= 5 ? kThinClusterMaxDim : kThinMaxDim;
      if (force_v < 0 && (thin_n_kind ? p.N : p.M) > max_dim) continue;
      if (s.thin == 3 && (!p.b_tma || p.transa)) continue;  // B read by TMA as stored
      if (s.thin == 4 && (!p.a_tma || p.transb)) continue;  // A read by TMA as stored
      if (s.thin >= 5) {  // cluster kernels: both operands read by TMA, the streamed one as
                          // stored, the small one as stored or from an aligned copy
        if (!(s.thin == 5 ? p.b_tma : p.a_tma) || p.transa || p.transb) continue;
        if (force_split >= 1) {
          consider(model_thin(p, v, std::min(force_split, kMaxThinCluster), num_sms, beta_nz));
          continue;
        }
        for (int sp = 1; sp <= kMaxThinCluster; sp *= 2) {
          const long long kps = ceil_div(ceil_div(p.K, sp), 8) * 8;
          if (sp > 1 && (long long)(sp - 1) * kps >= p.K) break;  // no empty K slices
          consider(model_thin(p, v, sp, num_sms, beta_nz));
        }
        continue;
      }
      const int kmax = s.thin == 1 ? kThinMKmax : s.thin == 2 ? kThinNKmax : kThinTmaKmax;
      const int min_split = (int)ceil_div(p.K, kmax);
      if (force_split >= 1) {
        consider(model_thin(p, v, std::max(force_split, min_split), num_sms, beta_nz));
        continue;
      }
      for (int sp = min_split; sp <= std::max(min_split, 96); ++sp)
        consider(model_thin(p, v, sp, num_sms, beta_nz));
      continue;
    }
    const long long tiles = ceil_div(p.M, s.BM) * ceil_div(p.N, s.BN);
    const long long kt = ceil_div(p.K, s.BK);
    const int max_split = (int)std::min<long long>(64, kt);
    if (force_split >= 1) {
      consider(model_plan(p, v, 0, std::min(force_split, max_split), num_sms, beta_nz));
      continue;
    }
    const long long slots = (long long)num_sms * s.min_blocks;
    const long long main = (tiles / slots) * slots;
    const long long tail = tiles - main;
    if (force_split <= -1) {
      int sp = force_split == -1 ? (int)std::max<long long>(2, tail ? slots / tail : 2)
                                 : -force_split;
      sp = std::min(sp, max_split);
      consider(model_plan(p, v, tail > 0 ? main : tiles, sp, num_sms, beta_nz));
      continue;
    }
    consider(model_plan(p, v, tiles, 1, num_sms, beta_nz));
    for (int sp = 2; sp <= max_split; ++sp) consider(model_plan(p, v, 0, sp, num_sms, beta_nz));
    if (main > 0 && tail > 0) {
      const int sp = (int)std::min<long long>(max_split, std::max<long long>(2, slots / tail));
      consider(model_plan(p, v, main, sp, num_sms, beta_nz));
    }
  }
  return best;
}

}  // namespace sgemm
