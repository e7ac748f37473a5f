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
  float *ws;          // split-K partials, [split][M][ldw]; unused when split == 1
  long long ldw;      // row stride of the partials (N rounded up to 4)
  int k_per_split;    // K elements per slice, a multiple of BK
  int tiles_m, tiles_n;
  int group_m;        // tile-rows per L2 group
  int vec_c;          // 1: C is 16-byte aligned with ldc % 4 == 0 (128-bit epilogue)
};

// ------------------------------------------------------------------------------------
// PTX wrappers (cp.async family, available sm_80+; compiled here for sm_103a).

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
template <int BM_, int BN_, int BK_, int WM_, int WN_, int TM_, int TN_, int STAGES_,
          int MIN_BLOCKS_>
struct TileConfig {
  static constexpr int BM = BM_, BN = BN_, BK = BK_;
  static constexpr int WM = WM_, WN = WN_, TM = TM_, TN = TN_;
  static constexpr int STAGES = STAGES_, MIN_BLOCKS = MIN_BLOCKS_;
  static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
  static constexpr int NWARPS = WARPS_M * WARPS_N;
  static constexpr int NT = NWARPS * 32;
  static constexpr int LM = WM / TM, LN = WN / TN;  // lanes along M and N in a warp
  static constexpr int FM = TM / 4, FN = TN / 4;    // float4 fragments per k step
  static constexpr int A_STAGE = BK * BM, B_STAGE = BK * BN;  // floats per stage
  static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
  // A copy: one warp instruction moves an 8 (k) x 4 (m) block.
  static constexpr int A_BLOCKS = (BK / 8) * (BM / 4);
  static constexpr int A_ITERS = A_BLOCKS / NWARPS;
  // B copy: 16-byte chunks (aligned path) or single floats (unaligned path).
  static constexpr int B_CHUNKS = BK * BN / 4;
  static constexpr int B_ITERS_VEC = B_CHUNKS / NT;
  static constexpr int B_ITERS_SCALAR = BK * BN / NT;
  // XOR swizzle of As chunk index: low bits flipped by k.
  static constexpr int SWZ = (BM / 4 >= 8) ? 7 : (BM / 4 - 1);

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
};

// Grouped tile order: GROUP_M tile-rows are swept column by column before moving on.
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

template <class Cfg, bool VEC_B, bool SPLIT>
__global__ void __launch_bounds__(Cfg::NT, Cfg::MIN_BLOCKS)
    sgemm_ffma_kernel(const GemmParams p) {
  constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
  constexpr int TM = Cfg::TM, TN = Cfg::TN, LM = Cfg::LM, LN = Cfg::LN;
  constexpr int FM = Cfg::FM, FN = Cfg::FN, NT = Cfg::NT, NWARPS = Cfg::NWARPS;
  constexpr int SWZ = Cfg::SWZ;

  extern __shared__ __align__(128) float smem[];
  float *As = smem;                               // [STAGES][BK][BM] swizzled
  float *Bs = smem + STAGES * Cfg::A_STAGE;       // [STAGES][BK][BN]

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int warp_m = warp / Cfg::WARPS_N;
  const int warp_n = warp % Cfg::WARPS_N;
  const int lane_m = lane / LN;
  const int lane_n = lane % LN;

  int tm, tn;
  tile_coords(blockIdx.x, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
  const int m0 = tm * BM;
  const int n0 = tn * BN;

  const int k_begin = SPLIT ? blockIdx.y * p.k_per_split : 0;
  const int k_end = SPLIT ? min(p.K, k_begin + p.k_per_split) : p.K;
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
    // A, transposed on the fly into As[slot][k][swizzled m]
    float *as = As + slot * Cfg::A_STAGE;
    const int kg = k0 + a_k;
    const bool k_ok = kg < k_end;
#pragma unroll
    for (int it = 0; it < Cfg::A_ITERS; ++it) {
      const int m = a_m_base + it * A_M_STEP;
      const int mg = m0 + m;
      const bool ok = k_ok && (mg < p.M);
      const float *src = ok ? p.A + (long long)mg * p.lda + kg : p.A;
      const int col = (((m >> 2) ^ (a_k & SWZ)) << 2) | (m & 3);
      cp_async_4(smem_addr(as + a_k * BM + col), src, ok ? 4 : 0);
    }
    float *bs = Bs + slot * Cfg::B_STAGE;
    if constexpr (VEC_B) {
      const int ng = n0 + bv_n;
      const int n_bytes = max(0, min(4, p.N - ng)) * 4;
#pragma unroll
      for (int it = 0; it < Cfg::B_ITERS_VEC; ++it) {
        const int kk = bv_k_base + it * BV_K_STEP;
        const int kgb = k0 + kk;
        const int bytes = (kgb < k_end) ? n_bytes : 0;
        const float *src = bytes ? p.B + (long long)kgb * p.ldb + ng : p.B;
        cp_async_16(smem_addr(bs + kk * BN + bv_n), src, bytes);
      }
    } else {
#pragma unroll
      for (int it = 0; it < Cfg::B_ITERS_SCALAR; ++it) {
        const int q = it * NT + tid;
        const int kk = q / BN;
        const int nn = q % BN;
        const int kgb = k0 + kk;
        const int ng = n0 + nn;
        const bool ok = (kgb < k_end) && (ng < p.N);
        const float *src = ok ? p.B + (long long)kgb * p.ldb + ng : p.B;
        cp_async_4(smem_addr(bs + kk * BN + nn), src, ok ? 4 : 0);
      }
    }
  };

  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

  // ---- prologue: fill STAGES-1 slots ------------------------------------------------
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < KT) load_tile(s, s);
    cp_async_commit();
  }

  // fragment addressing inside a stage
  const int a_chunk0 = (warp_m * Cfg::WM + lane_m * 4) >> 2;  // chunk of sub-block 0
  const int b_col0 = warp_n * Cfg::WN + lane_n * 4;

  float4 fa[2][FM], fb[2][FN];

  auto load_frags = [&](const float *as, const float *bs, int k, int buf) {
#pragma unroll
    for (int r = 0; r < FM; ++r) {
      const int chunk = a_chunk0 + r * LM;
      fa[buf][r] = *reinterpret_cast<const float4 *>(as + k * BM + ((chunk ^ (k & SWZ)) << 2));
    }
#pragma unroll
    for (int c = 0; c < FN; ++c)
      fb[buf][c] = *reinterpret_cast<const float4 *>(bs + k * BN + b_col0 + c * LN * 4);
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
    }
  }
  cp_async_wait<0>();

  // ---- epilogue -----------------------------------------------------------------------
  // Thread element (i, j) of acc sits at tile row warp_m*WM + (i/4)*LM*4 + lane_m*4 + i%4
  // and tile column warp_n*WN + (j/4)*LN*4 + lane_n*4 + j%4.
  const int row_base = m0 + warp_m * Cfg::WM + lane_m * 4;
  const int col_base = n0 + warp_n * Cfg::WN + lane_n * 4;
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int row = row_base + (i >> 2) * LM * 4 + (i & 3);
    if (row >= p.M) continue;
#pragma unroll
    for (int c = 0; c < FN; ++c) {
      const int col = col_base + c * LN * 4;
      if (col >= p.N) continue;
      const float *v = &acc[i][c * 4];
      if constexpr (SPLIT) {
        // partial sums of this K slice; ldw % 4 == 0 and ws 16-byte aligned
        float *dst = p.ws + ((long long)blockIdx.y * p.M + row) * p.ldw + col;
        if (col + 3 < p.N) {
          *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (col + e < p.N) dst[e] = v[e];
        }
      } else {
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
            out = make_float4(p.alpha * v[0], p.alpha * v[1], p.alpha * v[2],
                              p.alpha * v[3]);
          }
          *reinterpret_cast<float4 *>(dst) = out;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (col + e < p.N) {
              dst[e] = (p.beta != 0.0f) ? fmaf(p.alpha, v[e], p.beta * dst[e])
                                        : p.alpha * v[e];
            }
          }
        }
      }
    }
  }
}

}  // namespace sgemm
