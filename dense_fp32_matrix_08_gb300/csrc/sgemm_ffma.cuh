// FP32 FFMA GEMM main loop for sm_103a: C = alpha * A * B + beta * C, row-major.
//
// Design (one CTA computes a BM x BN tile of C, or one K slice of it under split-K):
//  * Staging: an S-stage ring of shared-memory tiles filled with cp.async, S-1 tiles in
//    flight while one is consumed (the double-buffered pipeline of "CUDA-Practice 04: from
//    shared-memory tiling to register outer products", double-buffering section,
//    generalised to S stages). Out-of-range elements are zero-filled by the copy itself
//    (src-size 0), so ragged M, N and K need no special tiles ("Lecture 4 - GPU
//    Acceleration", section 2.5: round the phase count up and load zeros past the edge).
//  * A is stored transposed in shared memory, As[k][m], so a thread's TM row values at one
//    k are contiguous and load with 128-bit LDS ("SGEMM six-level optimisation", section 8,
//    kernel K6: A transposed in smem so both operands are read as float4). The transpose
//    happens in the copy: each 4-byte cp.async reads A[m][k] and writes As[k][m].
//  * The naive transposed store is bank-conflicted (same page, section 8 part 5 lists
//    padding fallbacks that still leave ~4-way conflicts). Here the 16-byte chunk index of
//    each As row is XOR-swizzled with k: chunk' = chunk ^ (k & 7). A warp writes an 8 (k) x
//    4 (m) block per copy instruction and reads 16-byte chunks of one k row, both of which
//    then hit 32 distinct banks.
//  * Register tiling: each thread owns a TM x TN accumulator tile, made of (TM/4) x (TN/4)
//    4x4 sub-blocks spread over a warp tile WM x WN ("GPU GEMM optimisation, part 2",
//    kernel 10 warptiling: block -> warp -> thread). Per k step a thread loads TM/4 + TN/4
//    float4 fragments and issues TM * TN FFMA (the register outer product of "CUDA-Practice
//    04", register-tiling section). Fragments for step k+1 load while step k computes.
//  * Epilogue: alpha/beta applied in registers; float4 loads / stores of C when aligned and
//    in range, masked scalar accesses at the ragged edge. beta == 0 never reads C.
//  * Block order: tiles are visited in groups of GROUP_M tile-rows so that CTAs resident at
//    the same time share A row-panels and B column-panels in L2 ("GPU GEMM optimisation,
//    part 2", grid-orientation and block-swizzling remarks).
#pragma once

#include <cstdint>
#include <type_traits>

#include <cuda_runtime.h>

namespace sgemm {

struct GemmParams {
  int M, N, K;
  float alpha, beta;
  const float *A;
  long long lda;
  const float *B;
  long long ldb;
  float *C;
  long long ldc;
  // Work decomposition. CTAs 0 .. main_tiles-1 compute whole tiles (tile = CTA index, all
  // of K) and write C. The remaining tiles are split along K into `split` slices of
  // k_per_split elements; CTA main_tiles + u handles slice u % split of tile
  // main_tiles + u / split and writes its BM x BN partial tile to ws[u] (BM * BN floats,
  // row-major). A reduction kernel then finishes those tiles in slice order.
  float *ws;
  int main_tiles;
  int split;
  int k_per_split;    // multiple of BK
  int tiles_m, tiles_n;
  int group_m;        // tile-rows per L2 group
  int vec_c;          // 1: C is 16-byte aligned with ldc % 4 == 0 (128-bit epilogue)
  // 1: every tile is split (main_tiles == 0, split <= 8) and the grid is launched in
  // clusters of `split` CTAs, one per slice of a tile: the slices are added through
  // distributed shared memory (cluster_split_finish) instead of the workspace
  int cluster;
};

// ------------------------------------------------------------------------------------
// PTX wrappers (cp.async family, available sm_80+; compiled here for sm_103a).

// Programmatic dependent launch: wait until the grids this one depends on (the previous
// kernel in the stream, when this kernel was launched with programmatic stream
// serialization) have completed and their memory is visible. A no-op otherwise. Called
// before the kernel's first global-memory access, so that a launch may start while the
// previous kernel is finishing without reading anything it has not yet written.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// Programmatic dependent launch: this CTA no longer needs its SM for the main loop, so the
// next kernel in the stream (if launched with programmatic stream serialization) may be
// scheduled once every CTA of this grid has called this or exited. Only a scheduling hint:
// the next kernel's griddep_wait() still waits for this grid to complete, epilogue stores
// included. Called after the main loop, so the next kernel's prologue overlaps the epilogue.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 4-byte async copy; src_bytes == 0 writes zero to shared memory and reads nothing.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// 16-byte async copy bypassing L1; bytes past src_bytes (0..16) are zero-filled.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------------------------
// Tile configuration. All sizes are compile-time; static_asserts spell out which
// combinations are legal (the template-parameter legality idea of "GPU GEMM optimisation,
// part 2", autotuning section).
//
// MODE selects how the register outer product is issued:
//   0  scalar FFMA, one accumulator per instruction;
//   1  packed FFMA2 (fma.rn.f32x2) on accumulator pairs along N, the A value broadcast
//      into both halves of a register pair in registers;
//   2  packed FFMA2 with the broadcast done by the copy: every A element is stored twice in
//      shared memory, so 128-bit fragment loads return ready-made {a_i, a_i, a_i+1, a_i+1}.
// FFMA2 does the same FP32 work per pipe cycle as FFMA but needs half the issue slots,
// which leaves room for the fragment loads, copies and address arithmetic to overlap.
template <int BM_, int BN_, int BK_, int WM_, int WN_, int TM_, int TN_, int STAGES_,
          int MIN_BLOCKS_, int MODE_ = 0>
struct TileConfig {
  static constexpr int BM = BM_, BN = BN_, BK = BK_;
  static constexpr int WM = WM_, WN = WN_, TM = TM_, TN = TN_;
  static constexpr int STAGES = STAGES_, MIN_BLOCKS = MIN_BLOCKS_, MODE = MODE_;
  static constexpr int AW = (MODE == 2) ? 2 : 1;  // floats stored per A element
  static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
  static constexpr int NWARPS = WARPS_M * WARPS_N;
  static constexpr int NT = NWARPS * 32;
  static constexpr int LM = WM / TM, LN = WN / TN;  // lanes along M and N in a warp
  static constexpr int FM = TM / 4, FN = TN / 4;    // float4 fragments per k step
  static constexpr int A_STAGE = BK * BM * AW, B_STAGE = BK * BN;  // floats per stage
  static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
  // A copy: one warp instruction moves an 8 (k) x 4 (m) block.
  static constexpr int A_BLOCKS = (BK / 8) * (BM / 4);
  static constexpr int A_ITERS = A_BLOCKS / NWARPS;
  // B copy: 16-byte chunks (aligned path) or single floats (unaligned path).
  static constexpr int B_CHUNKS = BK * BN / 4;
  static constexpr int B_ITERS_VEC = B_CHUNKS / NT;
  static constexpr int B_ITERS_SCALAR = BK * BN / NT;
  // XOR swizzle of the As and Bs chunk indices: low bits flipped by k.
  static constexpr int SWZ = (BM * AW / 4 >= 8) ? 7 : (BM * AW / 4 - 1);
  static constexpr int SWZB = (BN / 4 >= 8) ? 7 : (BN / 4 - 1);
  // Copies for transposed operands (op(A) = A_st^T with A_st K x M, op(B) = B_st^T with
  // B_st N x K, both row-major): A_st rows are already As rows (16- or 4-byte copies);
  // B_st is transposed into Bs by 4-byte copies, one 8 (k) x 4 (n) block per warp
  // instruction, like the A copy of the non-transposed path.
  static constexpr int AT_ITERS_VEC = BK * BM / 4 / NT;
  static constexpr int AT_ITERS_SCALAR = BK * BM / NT;
  static constexpr int BT_BLOCKS = (BK / 8) * (BN / 4);
  static constexpr int BT_ITERS = BT_BLOCKS / NWARPS;

  static_assert(BM % WM == 0 && BN % WN == 0, "warp tiles must divide the CTA tile");
  static_assert(LM * LN == 32, "a warp is 32 lanes");
  static_assert(TM % 4 == 0 && TN % 4 == 0, "thread tiles are made of 4x4 blocks");
  static_assert(WM % (LM * 4) == 0 && WN % (LN * 4) == 0, "lane layout must tile the warp");
  static_assert(BK % 8 == 0, "A copies move 8 k values per row");
  static_assert(A_BLOCKS % NWARPS == 0, "A copy blocks must split evenly over warps");
  static_assert(NWARPS % (BK / 8) == 0, "fixed k offset per thread for A copies");
  static_assert(B_CHUNKS % NT == 0 && NT % (BN / 4) == 0, "B 16-byte copies must tile");
  static_assert((BK * BN) % NT == 0, "B 4-byte copies must tile");
  static_assert(STAGES >= 2, "need at least double buffering");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA on sm_103a");
  static_assert(MODE >= 0 && MODE <= 2, "unknown MODE");
  static_assert(MODE != 2 || BM % 32 == 0, "duplicated A layout needs BM % 32 == 0");
};

// Physical float index, inside one As row (fixed k), of logical column `x`:
//   MODE 0/1: x = m, one float per A row m.
//   MODE 2:   every A row m occupies two floats. Rows (2p, 2p+1) share one 16-byte chunk
//             {a_2p, a_2p, a_2p+1, a_2p+1}; chunk (p & 1) * (BM / 4) + (p >> 1) holds them,
//             so the two chunks a thread needs for rows 4l..4l+3 sit at l and BM/4 + l and
//             the lanes of a warp read consecutive chunks.
// The chunk index is then XOR-swizzled with k.
template <class Cfg>
__device__ __forceinline__ int a_phys(int k, int m, int dup) {
  if constexpr (Cfg::MODE == 2) {
    const int pr = m >> 1;
    const int chunk = (pr & 1) * (Cfg::BM / 4) + (pr >> 1);
    return ((chunk ^ (k & Cfg::SWZ)) << 2) | ((m & 1) << 1) | dup;
  } else {
    return (((m >> 2) ^ (k & Cfg::SWZ)) << 2) | (m & 3);
  }
}

// Physical float index of column n inside one Bs row (fixed k): the 16-byte chunk index is
// XOR-swizzled with k, so both the row-wise 16-byte copies and the transposing 4-byte
// copies (8 k x 4 n per warp instruction) hit 32 distinct banks.
template <class Cfg>
__device__ __forceinline__ int b_phys(int k, int n) {
  return (((n >> 2) ^ (k & Cfg::SWZB)) << 2) | (n & 3);
}

// Operand copy paths of the GEMM kernel.
//   A: APATH_N   A is M x K row-major, transposed into As by 4-byte copies;
//      APATH_T16 op(A) = A_st^T, A_st K x M row-major, 16-byte copies (lda % 4 == 0);
//      APATH_T4  the same layout with 4-byte copies.
//   B: BPATH_N4  B is K x N row-major, 4-byte copies;
//      BPATH_N16 the same with 16-byte copies (ldb % 4 == 0);
//      BPATH_T   op(B) = B_st^T, B_st N x K row-major, transposed into Bs by 4-byte copies.
enum { APATH_N = 0, APATH_T16 = 1, APATH_T4 = 2 };
enum { BPATH_N4 = 0, BPATH_N16 = 1, BPATH_T = 2 };

// d = a * b + c on register pairs {lo, hi} (two independent FP32 FMAs, round to nearest).
__device__ __forceinline__ void ffma2(unsigned long long &d, unsigned long long a,
                                      unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;\n" : "+l"(d) : "l"(a), "l"(b));
}

__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ float2 unpack2(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

// ---- thread-block clusters (sm_90+): rank, barrier, distributed shared memory loads ----

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster; orders shared-memory writes before it with
// reads after it, across the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// 16 bytes of CTA `rank`'s shared memory at the offset of the local address `local`.
__device__ __forceinline__ float4 ld_cluster4(uint32_t local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(local), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}

// Split-K finish inside a cluster (GemmParams::cluster). Every CTA of the cluster holds its
// K slice's BM x BN partial tile at `part` in its own shared memory, row-major, 16-byte
// aligned (out-of-range rows and columns hold zeros). CTA rank r finishes float4 groups
// [r * per, (r + 1) * per) of the tile: the S partials added in rank (= slice) order, then
// C = alpha * sum + beta * C (beta == 0: C not read) with the usual masks. The call
// synchronises the cluster before and after; every thread of every CTA must make it.
template <int BM, int BN, int THREADS>
__device__ __forceinline__ void cluster_split_finish(const float *part, const GemmParams &p,
                                                     int m0, int n0) {
  constexpr int G = BM * BN / 4;  // float4 groups of the tile
  constexpr int QMAX = 8;         // largest cluster (portable size)
  const int S = p.split;
  cluster_sync_all();  // the cluster's partial tiles are complete
  const uint32_t rank = cluster_rank();
  const int per = (G + S - 1) / S;
  const int e_end = min(G, ((int)rank + 1) * per);
  const uint32_t base = (uint32_t)__cvta_generic_to_shared(part);
  for (int e = (int)rank * per + (int)threadIdx.x; e < e_end; e += THREADS) {
    float4 v[QMAX];
#pragma unroll
    for (int q = 0; q < QMAX; ++q)  // every load in flight before the adds
      if (q < S) v[q] = ld_cluster4(base + 16u * (uint32_t)e, (uint32_t)q);
    float4 s = v[0];
#pragma unroll
    for (int q = 1; q < QMAX; ++q)
      if (q < S) {
        s.x += v[q].x;
        s.y += v[q].y;
        s.z += v[q].z;
        s.w += v[q].w;
      }
    const int row = m0 + e / (BN / 4);
    const int col = n0 + (e % (BN / 4)) * 4;
    if (row >= p.M || col >= p.N) continue;
    const float r[4] = {s.x, s.y, s.z, s.w};
    float *dst = p.C + (long long)row * p.ldc + col;
    if (p.vec_c && col + 3 < p.N) {
      float4 out;
      if (p.beta != 0.0f) {
        const float4 old = *reinterpret_cast<const float4 *>(dst);
        out = make_float4(fmaf(p.alpha, r[0], p.beta * old.x), fmaf(p.alpha, r[1], p.beta * old.y),
                          fmaf(p.alpha, r[2], p.beta * old.z), fmaf(p.alpha, r[3], p.beta * old.w));
      } else {
        out = make_float4(p.alpha * r[0], p.alpha * r[1], p.alpha * r[2], p.alpha * r[3]);
      }
      *reinterpret_cast<float4 *>(dst) = out;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (col + q < p.N)
          dst[q] = (p.beta != 0.0f) ? fmaf(p.alpha, r[q], p.beta * dst[q]) : p.alpha * r[q];
    }
  }
  cluster_sync_all();  // no CTA leaves while another may still read its partial
}

// Grouped tile order: GROUP_M tile-rows are swept column by column before moving on.
// Tile index -> (tile row, tile column); shared by the GEMM and split-K reduce kernels.
__device__ __forceinline__ void tile_coords(int bid, int tiles_m, int tiles_n, int group_m,
                                            int &tm, int &tn) {
  const int group_size = group_m * tiles_n;
  const int group = bid / group_size;
  const int first_m = group * group_m;
  const int rows = min(tiles_m - first_m, group_m);
  const int in_group = bid - group * group_size;
  tm = first_m + in_group % rows;
  tn = in_group / rows;
}

template <class Cfg, int APATH, int BPATH>
__global__ void __launch_bounds__(Cfg::NT, Cfg::MIN_BLOCKS)
    sgemm_ffma_kernel(const GemmParams p) {
  griddep_wait();  // (launched with programmatic dependent launch: see launch_1d)
  static_assert(APATH == APATH_N || Cfg::MODE != 2, "duplicated-A layout needs A row-major");
  static_assert(APATH != APATH_T16 || (Cfg::BK * Cfg::BM / 4) % Cfg::NT == 0, "A^T 16B tiling");
  static_assert(APATH != APATH_T4 || (Cfg::BK * Cfg::BM) % Cfg::NT == 0, "A^T 4B tiling");
  static_assert(BPATH != BPATH_T || (Cfg::BT_BLOCKS % Cfg::NWARPS == 0 &&
                                     Cfg::NWARPS % (Cfg::BK / 8) == 0),
                "B^T copy blocks must split evenly over warps");
  constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
  constexpr int TM = Cfg::TM, TN = Cfg::TN, LM = Cfg::LM, LN = Cfg::LN;
  constexpr int FM = Cfg::FM, FN = Cfg::FN, NT = Cfg::NT, NWARPS = Cfg::NWARPS;
  constexpr int MODE = Cfg::MODE;
  constexpr int AROW = BM * Cfg::AW;  // floats per As row (one k)

  extern __shared__ __align__(128) float smem[];
  float *As = smem;                               // [STAGES][BK][AROW] swizzled
  float *Bs = smem + STAGES * Cfg::A_STAGE;       // [STAGES][BK][BN]

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int warp_m = warp / Cfg::WARPS_N;
  const int warp_n = warp % Cfg::WARPS_N;
  // Lane layout inside the warp tile. Shared-memory loads merge equal addresses only
  // within aligned groups of 4 lanes, and a 128-bit load costs max(2, distinct addresses
  // per 4-lane group) wavefronts (measured on sm_103a). Each 4-lane group is therefore a
  // 2 x 2 block of (lane_m, lane_n): both the A and the B fragment loads then take the
  // 2-wavefront minimum (a row-major lane order would cost 4 for one of them).
  static_assert(LM >= 2 && LN >= 2, "2 x 2 lane groups need LM, LN >= 2");
  const int lane_hi = lane >> 2;
  const int lane_n = (lane_hi % (LN / 2)) * 2 + (lane & 1);
  const int lane_m = (lane_hi / (LN / 2)) * 2 + ((lane >> 1) & 1);

  // which tile, which K range (see GemmParams)
  const int w = blockIdx.x;
  const bool partial = w >= p.main_tiles;
  int tile = w, k_begin = 0, k_end = p.K;
  if (partial) {
    const int u = w - p.main_tiles;
    tile = p.main_tiles + u / p.split;
    k_begin = (u % p.split) * p.k_per_split;
    k_end = min(p.K, k_begin + p.k_per_split);
  }
  int tm, tn;
  tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
  const int m0 = tm * BM;
  const int n0 = tn * BN;

  const int KT = (k_end - k_begin + BK - 1) / BK;

  // ---- per-thread copy coordinates -------------------------------------------------
  // A: warp instruction it moves block b = it * NWARPS + warp; kb = b % (BK/8) is fixed
  // per warp because NWARPS is a multiple of BK/8.
  constexpr int KB = BK / 8;
  const int a_k = (warp % KB) * 8 + (lane & 7);              // k within the tile
  const int a_m_base = (warp / KB) * 4 + (lane >> 3);        // m for it = 0
  constexpr int A_M_STEP = (NWARPS / KB) * 4;                // m advance per iteration
  // B (16-byte path): chunk q = it * NT + tid; fixed column per thread.
  const int bv_n = (tid % (BN / 4)) * 4;
  const int bv_k_base = tid / (BN / 4);
  constexpr int BV_K_STEP = NT / (BN / 4);

  auto load_tile = [&](int kt, int slot) {
    const int k0 = k_begin + kt * BK;
    float *as_stage = As + slot * Cfg::A_STAGE;
    if constexpr (APATH == APATH_N) {
      // A, transposed on the fly into As[slot][k][a_phys(m)]
      float *as = as_stage + a_k * AROW;
      const int kg = k0 + a_k;
      const bool k_ok = kg < k_end;
#pragma unroll
      for (int it = 0; it < Cfg::A_ITERS; ++it) {
        const int m = a_m_base + it * A_M_STEP;
        const int mg = m0 + m;
        const bool ok = k_ok && (mg < p.M);
        const float *src = ok ? p.A + (long long)mg * p.lda + kg : p.A;
        cp_async_4(smem_addr(as + a_phys<Cfg>(a_k, m, 0)), src, ok ? 4 : 0);
        if constexpr (MODE == 2)
          cp_async_4(smem_addr(as + a_phys<Cfg>(a_k, m, 1)), src, ok ? 4 : 0);
      }
    } else if constexpr (APATH == APATH_T16) {
      // rows of A_st (fixed k) are rows of As: 16-byte chunks of 4 consecutive m
#pragma unroll
      for (int it = 0; it < Cfg::AT_ITERS_VEC; ++it) {
        const int q = it * NT + tid;
        const int kk = q / (BM / 4);
        const int mc = (q % (BM / 4)) * 4;
        const int kg = k0 + kk, mg = m0 + mc;
        const int bytes = (kg < k_end) ? max(0, min(4, p.M - mg)) * 4 : 0;
        const float *src = bytes ? p.A + (long long)kg * p.lda + mg : p.A;
        cp_async_16(smem_addr(as_stage + kk * AROW + a_phys<Cfg>(kk, mc, 0)), src, bytes);
      }
    } else {
#pragma unroll
      for (int it = 0; it < Cfg::AT_ITERS_SCALAR; ++it) {
        const int q = it * NT + tid;
        const int kk = q / BM;
        const int mm = q % BM;
        const int kg = k0 + kk, mg = m0 + mm;
        const bool ok = (kg < k_end) && (mg < p.M);
        const float *src = ok ? p.A + (long long)kg * p.lda + mg : p.A;
        cp_async_4(smem_addr(as_stage + kk * AROW + a_phys<Cfg>(kk, mm, 0)), src, ok ? 4 : 0);
      }
    }
    float *bs = Bs + slot * Cfg::B_STAGE;
    if constexpr (BPATH == BPATH_N16) {
      const int ng = n0 + bv_n;
      const int n_bytes = max(0, min(4, p.N - ng)) * 4;
#pragma unroll
      for (int it = 0; it < Cfg::B_ITERS_VEC; ++it) {
        const int kk = bv_k_base + it * BV_K_STEP;
        const int kgb = k0 + kk;
        const int bytes = (kgb < k_end) ? n_bytes : 0;
        const float *src = bytes ? p.B + (long long)kgb * p.ldb + ng : p.B;
        cp_async_16(smem_addr(bs + kk * BN + b_phys<Cfg>(kk, bv_n)), src, bytes);
      }
    } else if constexpr (BPATH == BPATH_N4) {
#pragma unroll
      for (int it = 0; it < Cfg::B_ITERS_SCALAR; ++it) {
        const int q = it * NT + tid;
        const int kk = q / BN;
        const int nn = q % BN;
        const int kgb = k0 + kk;
        const int ng = n0 + nn;
        const bool ok = (kgb < k_end) && (ng < p.N);
        const float *src = ok ? p.B + (long long)kgb * p.ldb + ng : p.B;
        cp_async_4(smem_addr(bs + kk * BN + b_phys<Cfg>(kk, nn)), src, ok ? 4 : 0);
      }
    } else {
      // B_st (N x K) transposed into Bs[k][b_phys(n)]: 8 consecutive k of 4 rows n per
      // warp instruction (coalesced 32-byte row segments, conflict-free smem writes)
      const int kk = (warp % KB) * 8 + (lane & 7);
      const int kg = k0 + kk;
      const bool k_ok = kg < k_end;
#pragma unroll
      for (int it = 0; it < Cfg::BT_ITERS; ++it) {
        const int nn = (it * (NWARPS / KB) + warp / KB) * 4 + (lane >> 3);
        const int ng = n0 + nn;
        const bool ok = k_ok && (ng < p.N);
        const float *src = ok ? p.B + (long long)ng * p.ldb + kg : p.B;
        cp_async_4(smem_addr(bs + kk * BN + b_phys<Cfg>(kk, nn)), src, ok ? 4 : 0);
      }
    }
  };

  // Accumulators: scalar for MODE 0, register pairs along N for the FFMA2 modes.
  constexpr int ACC_W = (MODE == 0) ? TN : TN / 2;
  using acc_t = typename std::conditional<MODE == 0, float, unsigned long long>::type;
  acc_t acc[TM][ACC_W];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < ACC_W; ++j) acc[i][j] = 0;

  // ---- prologue: fill STAGES-1 slots ------------------------------------------------
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < KT) load_tile(s, s);
    cp_async_commit();
  }

  // fragment addressing inside a stage
  const int a_row0 = warp_m * Cfg::WM + lane_m * 4;  // first of the thread's rows (tile)
  const int b_col0 = warp_n * Cfg::WN + lane_n * 4;

  // A fragments: MODE 0/1 -> FM float4 = TM values; MODE 2 -> 2*FM float4 = TM pairs.
  constexpr int FA = (MODE == 2) ? 2 * FM : FM;
  float4 fa[2][FA], fb[2][FN];

  auto load_frags = [&](const float *as, const float *bs, int k, int buf) {
    const float *arow = as + k * AROW;
#pragma unroll
    for (int r = 0; r < FM; ++r) {
      const int m = a_row0 + r * LM * 4;  // multiple of 4
      if constexpr (MODE == 2) {
        fa[buf][2 * r] = *reinterpret_cast<const float4 *>(arow + a_phys<Cfg>(k, m, 0));
        fa[buf][2 * r + 1] =
            *reinterpret_cast<const float4 *>(arow + a_phys<Cfg>(k, m + 2, 0));
      } else {
        fa[buf][r] = *reinterpret_cast<const float4 *>(arow + a_phys<Cfg>(k, m, 0));
      }
    }
#pragma unroll
    for (int c = 0; c < FN; ++c)
      fb[buf][c] = *reinterpret_cast<const float4 *>(bs + k * BN +
                                                      b_phys<Cfg>(k, b_col0 + c * LN * 4));
  };

  // ---- main loop ----------------------------------------------------------------------
  for (int kt = 0; kt < KT; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();  // tile kt visible to all; every warp is done with tile kt-1's slot
    {
      const int next = kt + STAGES - 1;
      if (next < KT) load_tile(next, next % STAGES);
      cp_async_commit();
    }
    const int slot = kt % STAGES;
    const float *as = As + slot * Cfg::A_STAGE;
    const float *bs = Bs + slot * Cfg::B_STAGE;

    load_frags(as, bs, 0, 0);
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const int cur = k & 1;
      if (k + 1 < BK) load_frags(as, bs, k + 1, cur ^ 1);
      if constexpr (MODE == 0) {
        float a[TM], b[TN];
#pragma unroll
        for (int r = 0; r < FM; ++r) {
          a[r * 4 + 0] = fa[cur][r].x;
          a[r * 4 + 1] = fa[cur][r].y;
          a[r * 4 + 2] = fa[cur][r].z;
          a[r * 4 + 3] = fa[cur][r].w;
        }
#pragma unroll
        for (int c = 0; c < FN; ++c) {
          b[c * 4 + 0] = fb[cur][c].x;
          b[c * 4 + 1] = fb[cur][c].y;
          b[c * 4 + 2] = fb[cur][c].z;
          b[c * 4 + 3] = fb[cur][c].w;
        }
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
          for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      } else {
        // b pairs (b_j, b_j+1) straight from the float4 fragments
        unsigned long long b2[TN / 2];
#pragma unroll
        for (int c = 0; c < FN; ++c) {
          b2[2 * c] = pack2(fb[cur][c].x, fb[cur][c].y);
          b2[2 * c + 1] = pack2(fb[cur][c].z, fb[cur][c].w);
        }
        unsigned long long a2[TM];  // {a_i, a_i}
#pragma unroll
        for (int r = 0; r < FM; ++r) {
          if constexpr (MODE == 2) {
            a2[r * 4 + 0] = pack2(fa[cur][2 * r].x, fa[cur][2 * r].y);
            a2[r * 4 + 1] = pack2(fa[cur][2 * r].z, fa[cur][2 * r].w);
            a2[r * 4 + 2] = pack2(fa[cur][2 * r + 1].x, fa[cur][2 * r + 1].y);
            a2[r * 4 + 3] = pack2(fa[cur][2 * r + 1].z, fa[cur][2 * r + 1].w);
          } else {
            a2[r * 4 + 0] = pack2(fa[cur][r].x, fa[cur][r].x);
            a2[r * 4 + 1] = pack2(fa[cur][r].y, fa[cur][r].y);
            a2[r * 4 + 2] = pack2(fa[cur][r].z, fa[cur][r].z);
            a2[r * 4 + 3] = pack2(fa[cur][r].w, fa[cur][r].w);
          }
        }
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
          for (int j = 0; j < TN / 2; ++j) ffma2(acc[i][j], a2[i], b2[j]);
      }
    }
  }
  cp_async_wait<0>();
  griddep_launch_dependents();

  // ---- epilogue -----------------------------------------------------------------------
  // Thread element (i, j) of the tile sits at row warp_m*WM + (i/4)*LM*4 + lane_m*4 + i%4
  // and column warp_n*WN + (j/4)*LN*4 + lane_n*4 + j%4.
  auto acc4 = [&](int i, int c, float v[4]) {
    if constexpr (MODE == 0) {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = acc[i][c * 4 + e];
    } else {
      const float2 lo = unpack2(acc[i][c * 2]);
      const float2 hi = unpack2(acc[i][c * 2 + 1]);
      v[0] = lo.x;
      v[1] = lo.y;
      v[2] = hi.x;
      v[3] = hi.y;
    }
  };
  if (partial) {
    // Whole partial tile, in range or not (out-of-range rows and columns hold zeros,
    // since their loads were zero-filled); 16-byte stores, ws 16-byte aligned. In cluster
    // mode the tile goes to this CTA's shared memory (the ring is free once every warp is
    // past the K loop) and the cluster finishes it.
    if (p.cluster) __syncthreads();
    float *wt = p.cluster ? smem : p.ws + (long long)(w - p.main_tiles) * (BM * BN);
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int r = a_row0 + (i >> 2) * LM * 4 + (i & 3);
#pragma unroll
      for (int c = 0; c < FN; ++c) {
        float v[4];
        acc4(i, c, v);
        *reinterpret_cast<float4 *>(wt + r * BN + b_col0 + c * LN * 4) =
            make_float4(v[0], v[1], v[2], v[3]);
      }
    }
    if (p.cluster) cluster_split_finish<BM, BN, Cfg::NT>(smem, p, m0, n0);
    return;
  }
  const int row_base = m0 + a_row0;
  const int col_base = n0 + b_col0;
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int row = row_base + (i >> 2) * LM * 4 + (i & 3);
    if (row >= p.M) continue;
#pragma unroll
    for (int c = 0; c < FN; ++c) {
      const int col = col_base + c * LN * 4;
      if (col >= p.N) continue;
      float v[4];
      acc4(i, c, v);
      float *dst = p.C + (long long)row * p.ldc + col;
      if (p.vec_c && col + 3 < p.N) {
        float4 out;
        if (p.beta != 0.0f) {
          const float4 old = *reinterpret_cast<const float4 *>(dst);
          out.x = fmaf(p.alpha, v[0], p.beta * old.x);
          out.y = fmaf(p.alpha, v[1], p.beta * old.y);
          out.z = fmaf(p.alpha, v[2], p.beta * old.z);
          out.w = fmaf(p.alpha, v[3], p.beta * old.w);
        } else {
          out = make_float4(p.alpha * v[0], p.alpha * v[1], p.alpha * v[2], p.alpha * v[3]);
        }
        *reinterpret_cast<float4 *>(dst) = out;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (col + e < p.N) {
            dst[e] = (p.beta != 0.0f) ? fmaf(p.alpha, v[e], p.beta * dst[e]) : p.alpha * v[e];
          }
        }
      }
    }
  }
}

}  // namespace sgemm
