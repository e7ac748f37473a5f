// K-paired TMA-fed FP32 GEMM for sm_103a: C = alpha * A * B + beta * C with A row-major
// (M x K) and B supplied K-major, i.e. as Bt = B^T (N x K, row-major), both 16-byte aligned
// with leading dimensions that are multiples of 4.
//
// The packed FFMA2 instruction (fma.rn.f32x2) does two independent FP32 FMAs on register
// pairs. The broadcast layout of sgemm_ffma.cuh / sgemm_ffma_tma.cuh pairs two output
// columns and has to build {a, a} from one A value with an extra move per A value and k
// step. Here the pair runs along k instead: the accumulator of output (i, j) is the pair
// {sum over even k, sum over odd k} and one FFMA2 adds {a_i(k), a_i(k+1)} * {b_j(k),
// b_j(k+1)}. Both operand pairs are two adjacent registers of a 128-bit fragment load (A
// and Bt tiles are k-contiguous), so the inner loop is fragment loads and FFMA2 only. The
// two halves are added once in the epilogue, which makes every output the sum of an
// even-k and an odd-k partial sum, each accumulated in k order: a fixed, deterministic
// order, with the same error bound as a single running sum (K/2 + 1 rounding steps per
// half, one more for the final add).
//
// Tiles: a CTA owns a 128 x 128 block of C; 8 warps (2 along m x 4 along n) own 64 x 32
// warp tiles; a thread owns 8 x 8 outputs (rows lane_m + 8 i, columns lane_n + 4 j of its
// warp tile), 128 accumulator registers. Lanes are grouped in 2 x 2 quads (lane_m, lane_n)
// so that each aligned group of four lanes reads two distinct 16-byte chunks per load.
// Operand tiles come by TMA into a STAGES-deep ring: [128 rows][32 k] for A and for Bt,
// 128-byte swizzled (chunk c of row r at chunk c ^ (r & 7)), so the eight rows a warp reads
// per load sit in eight different bank groups. One thread issues the copies; "full" and
// "empty" mbarriers hand stages between it and the eight warps; every wait is bounded and a
// wait that gives up sets the device status word (the result is then invalid).
// Epilogue: the 128 x 128 tile is staged through shared memory (row pitch 132 floats,
// conflict-free scalar stores) and written to C with coalesced 128-bit read-modify-writes.
#pragma once

#include <cuda.h>

#include "sgemm_ffma.cuh"
#include "sgemm_ptx.cuh"

namespace sgemm {
namespace kpair {

constexpr int BM = 128, BN = 128, BK = 32, THREADS = 256;
constexpr int WARPS_N = 4, WM = 64, WN = 32, TM = 8, TN = 8, LM = 8, LN = 4;
constexpr int A_BYTES = BM * BK * 4, B_BYTES = BN * BK * 4;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int CPITCH = BN + 4;  // staging row pitch (floats) of the epilogue
template <int STAGES>
constexpr int smem_bytes() {
  return STAGES * STAGE_BYTES + 1024 + 128;  // + alignment slack, barriers
}

static_assert(LM * LN == 32 && WM == LM * TM && WN == LN * TN, "lane layout");
static_assert((BM / WM) * (BN / WN) * 32 == THREADS, "eight warps");
static_assert(BK * 4 == 128, "operand rows are one 128-byte swizzle span");

template <int STAGES>
__global__ void __launch_bounds__(THREADS, 1)
    sgemm_kpair_kernel(const __grid_constant__ CUtensorMap map_a,
                       const __grid_constant__ CUtensorMap map_bt, const GemmParams p,
                       int *status) {
  static_assert(BM * CPITCH * 4 <= STAGES * STAGE_BYTES, "C staging fits in the ring");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle needs 1024-byte alignment
  float *smem_f = reinterpret_cast<float *>(smem_raw + (base - raw));
  const uint32_t bars = base + STAGES * STAGE_BYTES;  // full[s] at 8 s, empty[s] at 8 (S + s)

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int warp_m = warp / WARPS_N;
  const int warp_n = warp % WARPS_N;
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
  }
  __syncthreads();

  auto issue = [&](int kt) {  // thread 0 only
    const int s = kt % STAGES;
    const uint32_t full = bars + 8 * s;
    const uint32_t st = base + s * STAGE_BYTES;
    mbar_expect_tx(full, STAGE_BYTES);
    tma_load_2d(st, &map_a, k_begin + kt * BK, m0, full);
    tma_load_2d(st + A_BYTES, &map_bt, k_begin + kt * BK, n0, full);
  };
  int issued = 0;
  if (tid == 0) {
    tma_prefetch_map(&map_a);
    tma_prefetch_map(&map_bt);
    for (int kt = 0; kt < STAGES - 1 && kt < KT; ++kt) issue(kt);
    issued = min(STAGES - 1, KT);
  }

  unsigned long long acc[TM][TN];  // {even-k sum, odd-k sum}
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0;

  const int a_row = warp_m * WM + lane_m;  // + 8 i; a_row & 7 == lane_m
  const int b_row = warp_n * WN + lane_n;  // + 4 j; (b_row + 4 j) & 7 == lane_n + 4 (j & 1)
  bool ok = true;

  for (int kt = 0; kt < KT; ++kt) {
    const int s = kt % STAGES;
    if (!mbar_wait(bars + 8 * s, (uint32_t)(kt / STAGES) & 1u)) {
      ok = false;
      if (lane == 0) atomicCAS(status, 0, 1);
      break;
    }
    const float *as = smem_f + s * (STAGE_BYTES / 4);
    const float *bs = as + A_BYTES / 4;
#pragma unroll
    for (int c = 0; c < BK / 4; ++c) {
      float4 fa[TM], fb[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i)
        fa[i] = *reinterpret_cast<const float4 *>(as + (a_row + 8 * i) * BK +
                                                  ((c ^ lane_m) << 2));
#pragma unroll
      for (int j = 0; j < TN; ++j)
        fb[j] = *reinterpret_cast<const float4 *>(bs + (b_row + 4 * j) * BK +
                                                  ((c ^ (lane_n + 4 * (j & 1))) << 2));
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const unsigned long long a2 = pack2(fa[i].x, fa[i].y);
#pragma unroll
        for (int j = 0; j < TN; ++j) ffma2(acc[i][j], a2, pack2(fb[j].x, fb[j].y));
      }
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const unsigned long long a2 = pack2(fa[i].z, fa[i].w);
#pragma unroll
        for (int j = 0; j < TN; ++j) ffma2(acc[i][j], a2, pack2(fb[j].z, fb[j].w));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (STAGES + s));  // this warp is done with stage s
    if (tid == 0 && issued < KT) {
      // refill the stage that k tile kt - 1 used (kt + STAGES - 1 lands there)
      if (kt >= 1 && !mbar_wait(bars + 8 * (STAGES + (kt - 1) % STAGES),
                                (uint32_t)((kt - 1) / STAGES) & 1u)) {
        atomicCAS(status, 0, 2);
      } else {
        issue(issued);
        ++issued;
      }
    }
  }
  // Thread 0 may not leave, nor may the ring be reused for staging, while copies it issued
  // are in flight: wait for the last ones.
  if (tid == 0) {
    for (int kt = issued - 1; kt >= 0 && kt >= issued - STAGES; --kt)
      if (!mbar_wait(bars + 8 * (kt % STAGES), (uint32_t)(kt / STAGES) & 1u))
        atomicCAS(status, 0, 3);
  }
  // The whole block takes part in the staging below, so a warp whose wait gave up still
  // arrives here (its accumulators are incomplete; the status word already says so).
  (void)ok;
  __syncthreads();

  // ---- epilogue: stage the tile as [128][CPITCH] floats, then write rows coalesced
  float *stage = smem_f;
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const float2 h = unpack2(acc[i][j]);
      stage[(a_row + 8 * i) * CPITCH + b_row + 4 * j] = h.x + h.y;
    }
  __syncthreads();
  constexpr int VPR = BN / 4;  // float4 per tile row
  if (partial) {
    float *wt = p.ws + (long long)(w - p.main_tiles) * (BM * BN);
#pragma unroll 4
    for (int e = tid; e < BM * VPR; e += THREADS) {
      const int r = e / VPR, c4 = (e % VPR) * 4;
      *reinterpret_cast<float4 *>(wt + r * BN + c4) =
          *reinterpret_cast<const float4 *>(stage + r * CPITCH + c4);
    }
    return;
  }
#pragma unroll 4
  for (int e = tid; e < BM * VPR; e += THREADS) {
    const int r = e / VPR, c4 = (e % VPR) * 4;
    const int row = m0 + r, col = n0 + c4;
    if (row >= p.M || col >= p.N) continue;
    const float4 v = *reinterpret_cast<const float4 *>(stage + r * CPITCH + c4);
    float *dst = p.C + (long long)row * p.ldc + col;
    if (p.vec_c && col + 3 < p.N) {
      float4 out;
      if (p.beta != 0.0f) {
        const float4 old = *reinterpret_cast<const float4 *>(dst);
        out.x = fmaf(p.alpha, v.x, p.beta * old.x);
        out.y = fmaf(p.alpha, v.y, p.beta * old.y);
        out.z = fmaf(p.alpha, v.z, p.beta * old.z);
        out.w = fmaf(p.alpha, v.w, p.beta * old.w);
      } else {
        out = make_float4(p.alpha * v.x, p.alpha * v.y, p.alpha * v.z, p.alpha * v.w);
      }
      *reinterpret_cast<float4 *>(dst) = out;
    } else {
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (col + q < p.N)
          dst[q] = (p.beta != 0.0f) ? fmaf(p.alpha, vv[q], p.beta * dst[q]) : p.alpha * vv[q];
    }
  }
}

}  // namespace kpair
}  // namespace sgemm
