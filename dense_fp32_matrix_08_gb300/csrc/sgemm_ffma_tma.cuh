// TMA-fed FP32 FFMA2 GEMM for sm_103a: C = alpha * A * B + beta * C, row-major, for
// 16-byte aligned A and B with lda, ldb multiples of 4 and no transposition.
//
// Same register outer product as sgemm_ffma.cuh (8 x TN FFMA2 thread tiles in 64 x 4 TN
// warp tiles, four warps per 128 x 8 TN CTA tile, MINB CTAs per SM), but the operand tiles
// reach shared memory by TMA instead of per-thread copies: one thread issues two
// cp.async.bulk.tensor copies per 32-wide K block into a STAGES-deep ring, and the math
// warps spend no issue slots on address arithmetic or copies (on this GPU those took about
// 18% of the slots of the copy-based kernel). Each stage has a "full" mbarrier (TMA bytes)
// and an "empty" mbarrier (one arrival per warp when it has finished reading the stage);
// the refill of a stage is issued at the start of the next K block, as soon as every warp
// has released it, so a 2-stage ring still overlaps each copy with a whole K block.
//
// Layouts in shared memory:
//  * A tile: 128 rows (m) x 32 k, as stored (k contiguous), written by TMA with the 128-byte
//    swizzle: the 16-byte chunk c of row r sits at chunk c ^ (r & 7). A thread's eight rows
//    are r = lane_m + 8 i, so the eight row groups of a warp hit eight different chunks:
//    every 128-bit fragment load is conflict-free. One float4 gives a row's values for 4
//    consecutive k, so A fragments are loaded once per 4 k steps.
//  * B tile: 32 k x BN n, as stored (n contiguous), no swizzle; a thread's TN columns are
//    TN / 4 float4 at stride 16 columns, as in the copy-based kernel.
// Ragged edges: TMA fills out-of-range rows / columns / k with zeros, so the main loop has
// no masks; the epilogue masks rows and columns. Every mbarrier wait is bounded; a wait
// that gives up sets a device status word and the CTA stops computing (the result is then
// invalid, which the status reports).
#pragma once

#include <cuda.h>

#include "sgemm_ffma.cuh"
#include "sgemm_ptx.cuh"

namespace sgemm {
namespace tma {

// BN_ = 8 TN_ columns per CTA; DBA_: double-buffer the A fragments (needs ~32 more
// registers per thread). AMODE_ says how the math reads A:
//   0  as stored, [128 m][32 k] 128-byte swizzled tiles, one float4 = 4 k of one row;
//   1  k-major: A is supplied as At = A^T (K x M row-major) and its tile arrives as
//      [32 k][128 m], like the B tile;
//   2  as stored by TMA (mode 0 tiles), then transposed by the CTA into a [32 k][128 m]
//      shared-memory buffer once per K block (two CTA barriers per K block).
// In modes 1 and 2 a thread's rows are lane_m * 4 + e + 32 r of its warp tile and both
// fragments are double-buffered per k step (8 + TN values per k, instead of mode 0's
// 8 float4 of A per 4 k). On this GPU that loop sustains ~9% more FFMA2 throughput.
template <int BN_, int TN_, int STAGES_, int MINB_, bool DBA_, int AMODE_ = 0>
struct TmaCfg {
  static constexpr int BM = 128, BN = BN_, BK = 32, STAGES = STAGES_, THREADS = 128;
  static constexpr int WM = 64, WN = BN / 2, TM = 8, TN = TN_, LM = 8, LN = 4, WARPS_N = 2;
  static constexpr int MINB = MINB_;
  static constexpr bool DBA = DBA_;
  static constexpr int AMODE = AMODE_;
  static constexpr bool AT = AMODE != 0;  // the math reads A as [k][m]
  static constexpr bool TX = AMODE == 2;  // ... from the CTA's transposed copy
  static constexpr int A_BYTES = BM * BK * 4, B_BYTES = BK * BN * 4;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int T_BYTES = TX ? BK * BM * 4 : 0;  // transposed A buffer
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + 1024 + 64 + T_BYTES;  // + alignment slack, barriers

  static_assert(LM * LN == 32 && WM == LM * TM && WN == LN * TN, "lane layout");
  static_assert((BM / WM) * (BN / WN) * 32 == THREADS, "four warps");
  static_assert(BK * 4 == 128, "A rows are one 128-byte swizzle span");
  static_assert(STAGE_BYTES % 1024 == 0, "every A stage 1024-byte aligned (swizzle atom)");
  static_assert(TN % 4 == 0 && BN <= 256, "B box: float4 columns, at most 256 wide");
  static_assert(STAGES >= 2, "a ring needs two stages");
  static_assert(AMODE >= 0 && AMODE <= 2, "A read mode");
  static_assert(!TX || BM == THREADS, "transpose: one A row per thread");
  static_assert(BM * BN * 4 <= STAGES * STAGE_BYTES, "a partial tile fits in the ring");
};

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MINB)
    sgemm_tma_kernel(const __grid_constant__ CUtensorMap map_a,
                     const __grid_constant__ CUtensorMap map_b, const GemmParams p,
                     int *status) {
  constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
  constexpr int THREADS = Cfg::THREADS, WM = Cfg::WM, WN = Cfg::WN, TM = Cfg::TM;
  constexpr int TN = Cfg::TN, LN = Cfg::LN, WARPS_N = Cfg::WARPS_N;
  constexpr int A_BYTES = Cfg::A_BYTES, STAGE_BYTES = Cfg::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle needs 1024-byte alignment
  const float *smem_f = reinterpret_cast<const float *>(smem_raw + (base - raw));
  const uint32_t bars = base + STAGES * STAGE_BYTES;  // full[s] at 8 s, empty[s] at 8 (S + s)
  // mode 2: the transposed A buffer follows the 64 bytes of barriers
  float *tbuf = reinterpret_cast<float *>(smem_raw + (base - raw) + STAGES * STAGE_BYTES + 64);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int warp_m = warp / WARPS_N;
  const int warp_n = warp % WARPS_N;
  // 2 x 2 lane groups (see sgemm_ffma.cuh): both fragment loads take 2 wavefronts
  const int lane_hi = lane >> 2;
  const int lane_n = (lane_hi % (LN / 2)) * 2 + (lane & 1);
  const int lane_m = (lane_hi / (LN / 2)) * 2 + ((lane >> 1) & 1);

  // work decomposition: whole tiles, then K slices of the remaining tiles (GemmParams)
  const int w = blockIdx.x;
  const bool partial = w >= p.main_tiles;
  int tile = w, k_begin = 0, k_end = p.K;
  if (partial) {
    const int u = w - p.main_tiles;
    tile = p.main_tiles + u / p.split;
    k_begin = (u % p.split) * p.k_per_split;  // a multiple of BK
    k_end = min(p.K, k_begin + p.k_per_split);
  }
  int tm, tn;
  tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
  const int m0 = tm * BM;
  const int n0 = tn * BN;
  const int KT = (k_end - k_begin + BK - 1) / BK;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bars + 8 * s, 1);
      mbar_init(bars + 8 * (STAGES + s), THREADS / 32);
    }
    mbar_init_fence();
    tma_prefetch_map(&map_a);
    tma_prefetch_map(&map_b);
  }
  __syncthreads();
  // The launch allows programmatic dependent launch (launch_1d): everything above touches
  // only shared memory and the kernel's parameters, so it may overlap the previous
  // kernel's last CTAs; from here on the previous kernel's writes are visible.
  griddep_wait();

  auto issue = [&](int kt) {  // thread 0 only
    const int s = kt % STAGES;
    const uint32_t full = bars + 8 * s;
    const uint32_t st = base + s * STAGE_BYTES;
    mbar_expect_tx(full, STAGE_BYTES);
    if constexpr (Cfg::AMODE == 1)
      tma_load_2d(st, &map_a, m0, k_begin + kt * BK, full);
    else
      tma_load_2d(st, &map_a, k_begin + kt * BK, m0, full);
    tma_load_2d(st + A_BYTES, &map_b, n0, k_begin + kt * BK, full);
  };
  int issued = 0;
  if (tid == 0) {
    for (int kt = 0; kt < STAGES - 1 && kt < KT; ++kt) issue(kt);
    issued = min(STAGES - 1, KT);
  }

  unsigned long long acc[TM][TN / 2];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN / 2; ++j) acc[i][j] = 0;

  const int a_row = warp_m * WM + lane_m;        // + 8 i (A as stored)
  const int a_col0 = warp_m * WM + lane_m * 4;    // + e + 32 r (AT: rows of As[k][.])
  const int swz = lane_m & 7;                    // == a_row & 7 for every i
  const int b_col0 = warp_n * WN + lane_n * 4;   // + 16 jj
  bool ok = true;

  for (int kt = 0; kt < KT; ++kt) {
    const int s = kt % STAGES;
    const bool got = mbar_wait(bars + 8 * s, (uint32_t)(kt / STAGES) & 1u);
    // Mode 2 has CTA barriers in this loop, so a wait that gave up must end the loop for
    // every warp at once: the vote is also the barrier that frees the transposed buffer.
    const bool give_up = Cfg::TX ? __syncthreads_or(!got) != 0 : !got;
    if (give_up) {
      ok = false;
      if (!got && lane == 0) atomicCAS(status, 0, 1);
      break;
    }
    if (tid == 0 && issued < KT) {
      // refill the stage that k tile kt - 1 used (kt + STAGES - 1 lands there) once every
      // warp has released it
      if (kt >= 1 && !mbar_wait(bars + 8 * (STAGES + (kt - 1) % STAGES),
                                (uint32_t)((kt - 1) / STAGES) & 1u)) {
        atomicCAS(status, 0, 2);
      } else {
        issue(issued);
        ++issued;
      }
    }
    const float *as = smem_f + s * (STAGE_BYTES / 4);
    const float *bs = as + A_BYTES / 4;
    if constexpr (Cfg::TX) {
      // Transpose this K block's A tile (row tid, 8 swizzled chunks of 4 k) into
      // tbuf[k][m]: lanes read 8 consecutive rows per wavefront (8 distinct chunks) and
      // write 32 consecutive floats per store. The vote above kept the buffer until every
      // warp had finished the previous K block; this barrier publishes it.
      const float *arow = as + tid * BK;
#pragma unroll
      for (int c = 0; c < BK / 4; ++c) {
        const float4 v = *reinterpret_cast<const float4 *>(arow + ((c ^ (tid & 7)) << 2));
        tbuf[(4 * c + 0) * BM + tid] = v.x;
        tbuf[(4 * c + 1) * BM + tid] = v.y;
        tbuf[(4 * c + 2) * BM + tid] = v.z;
        tbuf[(4 * c + 3) * BM + tid] = v.w;
      }
      __syncthreads();
      as = tbuf;
    }
    if constexpr (Cfg::AT) {
      // As[k][m], Bs[k][n]: per k step TM / 4 + TN / 4 float4, double-buffered across k
      float4 fa[2][TM / 4], fb[2][TN / 4];
      auto load = [&](int k, int buf) {
#pragma unroll
        for (int r = 0; r < TM / 4; ++r)
          fa[buf][r] = *reinterpret_cast<const float4 *>(as + k * BM + a_col0 + 32 * r);
#pragma unroll
        for (int jj = 0; jj < TN / 4; ++jj)
          fb[buf][jj] = *reinterpret_cast<const float4 *>(bs + k * BN + b_col0 + 16 * jj);
      };
      load(0, 0);
#pragma unroll
      for (int k = 0; k < BK; ++k) {
        if (k + 1 < BK) load(k + 1, (k + 1) & 1);
        const float4 *fac = fa[k & 1];
        const float4 *fbc = fb[k & 1];
        unsigned long long b2[TN / 2];
#pragma unroll
        for (int jj = 0; jj < TN / 4; ++jj) {
          b2[2 * jj] = pack2(fbc[jj].x, fbc[jj].y);
          b2[2 * jj + 1] = pack2(fbc[jj].z, fbc[jj].w);
        }
        unsigned long long a2[TM];
#pragma unroll
        for (int i = 0; i < TM; ++i) {
          const float4 &f = fac[i >> 2];
          const int e = i & 3;
          const float a = e == 0 ? f.x : e == 1 ? f.y : e == 2 ? f.z : f.w;
          a2[i] = pack2(a, a);
        }
        // j outer: each B pair feeds TM consecutive instructions
#pragma unroll
        for (int j = 0; j < TN / 2; ++j)
#pragma unroll
          for (int i = 0; i < TM; ++i) ffma2(acc[i][j], a2[i], b2[j]);
      }
    } else {
      // Fragments are double-buffered: the A float4s of chunk c + 1 (4 k each) load while
      // chunk c computes, and the B float4s of step k + 1 while step k computes.
      constexpr int NA = Cfg::DBA ? 2 : 1;
      float4 fa[NA][TM], fb[2][TN / 4];
      auto load_a = [&](int c, int buf) {
  #pragma unroll
        for (int i = 0; i < TM; ++i)
          fa[buf][i] =
              *reinterpret_cast<const float4 *>(as + (a_row + 8 * i) * BK + ((c ^ swz) << 2));
      };
      auto load_b = [&](int k, int buf) {
  #pragma unroll
        for (int jj = 0; jj < TN / 4; ++jj)
          fb[buf][jj] = *reinterpret_cast<const float4 *>(bs + k * BN + b_col0 + 16 * jj);
      };
      load_a(0, 0);
      load_b(0, 0);
  #pragma unroll
      for (int c = 0; c < BK / 4; ++c) {
  #pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int k = 4 * c + kk;
          if (Cfg::DBA && kk == 1 && c + 1 < BK / 4) load_a(c + 1, (c + 1) & (NA - 1));
          if (!Cfg::DBA && kk == 0 && c > 0) load_a(c, 0);
          if (k + 1 < BK) load_b(k + 1, (k + 1) & 1);
          const float4 *fac = fa[c & (NA - 1)];
          const float4 *fbc = fb[k & 1];
          unsigned long long b2[TN / 2];
  #pragma unroll
          for (int jj = 0; jj < TN / 4; ++jj) {
            b2[2 * jj] = pack2(fbc[jj].x, fbc[jj].y);
            b2[2 * jj + 1] = pack2(fbc[jj].z, fbc[jj].w);
          }
  #pragma unroll
          for (int i = 0; i < TM; ++i) {
            const float a = kk == 0 ? fac[i].x : kk == 1 ? fac[i].y : kk == 2 ? fac[i].z : fac[i].w;
            const unsigned long long a2 = pack2(a, a);
  #pragma unroll
            for (int j = 0; j < TN / 2; ++j) ffma2(acc[i][j], a2, b2[j]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (STAGES + s));  // this warp is done with stage s
  }
  griddep_launch_dependents();
  // Thread 0 may not leave while copies it issued are in flight: wait for the last ones.
  if (tid == 0) {
    for (int kt = issued - 1; kt >= 0 && kt >= issued - STAGES; --kt)
      mbar_wait(bars + 8 * (kt % STAGES), (uint32_t)(kt / STAGES) & 1u);
  }
  if (!ok && !p.cluster) return;  // (cluster mode: every CTA must reach the cluster barriers)

  // ---- epilogue: thread element (i, 4 jj + e) is row trow(i), column b_col0 + 16 jj + e
  auto trow = [&](int i) {
    return Cfg::AT ? a_col0 + (i & 3) + 32 * (i >> 2) : a_row + 8 * i;
  };
  if (partial) {
    // cluster mode: the partial tile goes to this CTA's shared memory (the ring, free once
    // every warp is past the K loop and the copies are drained) and the cluster finishes it
    if (p.cluster) __syncthreads();
    float *part = reinterpret_cast<float *>(smem_raw + (base - raw));
    float *wt = p.cluster ? part : p.ws + (long long)(w - p.main_tiles) * (BM * BN);
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int jj = 0; jj < TN / 4; ++jj) {
        const float2 lo = unpack2(acc[i][2 * jj]), hi = unpack2(acc[i][2 * jj + 1]);
        *reinterpret_cast<float4 *>(wt + trow(i) * BN + b_col0 + 16 * jj) =
            make_float4(lo.x, lo.y, hi.x, hi.y);
      }
    if (p.cluster) cluster_split_finish<BM, BN, THREADS>(part, p, m0, n0);
    return;
  }
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int row = m0 + trow(i);
    if (row >= p.M) continue;
#pragma unroll
    for (int jj = 0; jj < TN / 4; ++jj) {
      const int col = n0 + b_col0 + 16 * jj;
      if (col >= p.N) continue;
      const float2 lo = unpack2(acc[i][2 * jj]), hi = unpack2(acc[i][2 * jj + 1]);
      const float v[4] = {lo.x, lo.y, hi.x, hi.y};
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
        for (int e = 0; e < 4; ++e)
          if (col + e < p.N)
            dst[e] = (p.beta != 0.0f) ? fmaf(p.alpha, v[e], p.beta * dst[e]) : p.alpha * v[e];
      }
    }
  }
}

}  // namespace tma
}  // namespace sgemm
