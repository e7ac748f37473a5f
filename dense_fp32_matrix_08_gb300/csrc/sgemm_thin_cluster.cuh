// Thin-product kernel with the K split reduced inside a thread-block cluster, for sm_103a.
// C (M x N) = alpha * A * B + beta * C where one side is thin: thin-M (16 rows per row block,
// B streamed) or thin-N (16 columns per column block, A streamed; the kernel then works on
// C^T = B^T A^T with the roles of the operands swapped).
//
// The streamed ("wide") operand is read once from HBM at 8 FLOP per byte, just under this
// GPU's FP32/HBM ridge, so the kernel's job is to keep HBM busy from the first cycle to the
// last. Compared with the split-K kernel in sgemm_thin_tma.cuh:
//  * Both operands arrive by TMA, chunk by chunk: a chunk is 8 k of the wide operand for the
//    CTA's 128 wide indices (4 KB) plus the same 8 k of the thin ("small") operand for its 16
//    indices (512 B). No staging prologue holds back the first FMA.
//  * The K slices of one C tile are the CTAs of one cluster (1 x S x 1, S = 1, 2, 4 or 8).
//    Each CTA adds its 16 warps' partial tiles in warp order, then the cluster adds the S
//    CTA partials through distributed shared memory in rank order, each CTA finishing 1/S
//    of the tile with the alpha / beta epilogue. No workspace, no second launch; every
//    output is a fixed-order sum.
//  * The tile is 16 x 128 so that clusters of 4 fill the GPU on 16 x 4096 and 4096 x 16
//    products (32 tiles x 4 slices = 128 CTAs, one per SM).
//
// Warps: 16, each with two private ring stages and the chunks c = w, w + 16, ... of the
// CTA's K slice (lane 0 issues, the warp waits on the stage's mbarrier with a bounded poll,
// computes, and refills the stage two chunks ahead). 16 warps of two stages measured 2-7%
// faster than 8 or 12 warps with the same bytes in flight. A lane owns all 16 small indices times
// 4 wide indices. FFMA2 pairs run along the small dimension, {s_2p, s_2p+1} straight from
// a 128-bit broadcast load of the small operand's k row, times the wide value duplicated
// into both halves, {w, w}: 32 FFMA2 per k against 4 duplications and 5 shared loads. On
// shared-memory-resident data this mix sustained 80-85% of the FP32 pipe (8 x 8 lane blocks
// with the duplication on the small side: 72-75%); 16 x 8 blocks with the two half-warps on
// alternate k reached more there but ran slower in this kernel. For thin-M the small chunk
// arrives as A[16 m][8 k] and each warp transposes it to [8 k][16 m] (one 128-bit load and
// four stores per lane) before use; for thin-N the B chunk [8 k][16 n] is already in that
// layout.
#pragma once

#include <cuda.h>

#include "sgemm_ffma.cuh"
#include "sgemm_ptx.cuh"
#include "sgemm_thin.cuh"

namespace sgemm {
namespace thin {
namespace cl {

constexpr int MT = 16;             // small extent of a tile
constexpr int BW = 128;            // wide extent of a tile
constexpr int KC = 8;              // k per chunk (one pair of TMA copies)
constexpr int WARPS = 16;
constexpr int SPW = 2;             // private ring stages per warp
constexpr int THREADS = WARPS * 32;
constexpr int STAGES = WARPS * SPW;
constexpr int BIG_BYTES = KC * BW * 4;      // wide-operand part of a chunk
constexpr int SMALL_BYTES = KC * MT * 4;    // small-operand part of a chunk
constexpr int BIG_RING = STAGES * BIG_BYTES;
constexpr int SMALL_RING = STAGES * SMALL_BYTES;
constexpr int TILE_FLOATS = MT * BW;
constexpr int RED_BYTES = WARPS * TILE_FLOATS * 4;  // warp partials (reuse the wide ring)
constexpr int PART_BYTES = TILE_FLOATS * 4;         // the CTA partial (reuses the small ring)
constexpr int TP = 20;             // row pitch (floats) of a warp's transposed small chunk
constexpr int TBUF_BYTES = WARPS * KC * TP * 4;
constexpr int MAX_CLUSTER = 8;
constexpr size_t SMEM_BYTES = 1024 + BIG_RING + SMALL_RING + TBUF_BYTES + 8 * STAGES;
static_assert(RED_BYTES <= BIG_RING, "warp partials fit in the wide ring");
static_assert(PART_BYTES <= SMALL_RING, "the CTA partial fits in the small ring");
static_assert((TILE_FLOATS / 4) % MAX_CLUSTER == 0, "the tile splits over a cluster");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");

}  // namespace cl

// grid = (wide tiles, S, small tiles) launched in clusters of (1, S, 1), S = p.split; the CTA
// of cluster rank s takes K range [s * p.k_per_split, (s + 1) * p.k_per_split) (a multiple
// of KC; a range past K is empty and contributes zeros).
//  * TN = false (thin-M): map_big is B (K x N) in [8 k][128 n] boxes, map_small is A (M x K)
//    in [16 m][8 k] boxes. Lane l owns C columns 4l .. 4l + 3 of the tile.
//  * TN = true (thin-N): map_big is A (M x K) in [128 m][8 k] boxes with the 32-byte swizzle
//    (16-byte half hh of row r lands at hh ^ ((r >> 2) & 1)), map_small is B (K x N) in
//    [8 k][16 n] boxes. Lane l owns C rows l + 32 c, c = 0..3, of the tile.
// Out-of-range rows and columns of a box read as zero, so a ragged last chunk adds zeros.
template <bool TN>
__global__ void __launch_bounds__(cl::THREADS, 1)
    thin_cluster_kernel(const __grid_constant__ CUtensorMap map_big,
                        const __grid_constant__ CUtensorMap map_small, const ThinParams p,
                        int *status) {
  griddep_wait();  // (launched with programmatic dependent launch: see launch_thin_cluster)
  using namespace cl;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sbase = smem_raw + (base - raw);
  const float *big = reinterpret_cast<const float *>(sbase);
  const float *sml = reinterpret_cast<const float *>(sbase + BIG_RING);
  float *tbuf = reinterpret_cast<float *>(sbase + BIG_RING + SMALL_RING);
  const uint32_t sml_base = base + BIG_RING;
  const uint32_t bars = base + BIG_RING + SMALL_RING + TBUF_BYTES;  // full[stage]

  const int wblk = blockIdx.x, slice = blockIdx.y, sblk = blockIdx.z;
  const int w0 = wblk * BW, s0 = sblk * MT;
  const int k0 = slice * p.k_per_split;
  const int KS = max(0, min(p.K - k0, p.k_per_split));
  const int NCH = (KS + KC - 1) / KC;  // chunks in the slice
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int my_chunks = NCH > warp ? (NCH - warp + WARPS - 1) / WARPS : 0;

  // C elements this thread finishes (float4 groups e = rank * per + t, t = tid, tid + THREADS)
  // and, with beta != 0, their old values, loaded now so that the read is off the tail.
  const int S = p.split;
  const int per = (TILE_FLOATS / 4) / S;
  constexpr int R = TN ? BW : MT, CC = TN ? MT : BW;  // the tile in C orientation
  static_assert(R * CC == TILE_FLOATS, "tile");
  constexpr int FIN = (TILE_FLOATS / 4 + THREADS - 1) / THREADS;  // groups per thread, at most
  const uint32_t rank = S > 1 ? cluster_rank() : 0u;
  float4 cold[FIN];
#pragma unroll
  for (int f = 0; f < FIN; ++f) {
    cold[f] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int t = tid + f * THREADS;
    const int e = (int)rank * per + t;
    const int row = (TN ? w0 : s0) + e / (CC / 4);
    const int col = (TN ? s0 : w0) + (e % (CC / 4)) * 4;
    if (t < per && p.beta != 0.0f && p.vec_c && row < p.M && col + 3 < p.N)
      cold[f] = *reinterpret_cast<const float4 *>(p.C + (long long)row * p.ldc + col);
  }

  auto stage_of = [&](int j) { return warp * SPW + (j % SPW); };
  auto issue = [&](int j) {  // lane 0: both parts of chunk warp + WARPS j into its stage
    const int st = stage_of(j);
    const int kc = k0 + (warp + WARPS * j) * KC;
    const uint32_t bar = bars + 8 * st;
    mbar_expect_tx(bar, BIG_BYTES + SMALL_BYTES);
    if constexpr (TN) {
      tma_load_2d(base + st * BIG_BYTES, &map_big, kc, w0, bar);
      tma_load_2d(sml_base + st * SMALL_BYTES, &map_small, s0, kc, bar);
    } else {
      tma_load_2d(base + st * BIG_BYTES, &map_big, w0, kc, bar);
      tma_load_2d(sml_base + st * SMALL_BYTES, &map_small, kc, s0, bar);
    }
  };
  if (lane == 0) {
    for (int q = 0; q < SPW; ++q) mbar_init(bars + 8 * (warp * SPW + q), 1);
    mbar_init_fence();
    if (warp == 0) {
      tma_prefetch_map(&map_big);
      tma_prefetch_map(&map_small);
    }
    for (int j = 0; j < SPW && j < my_chunks; ++j) issue(j);
  }
  __syncwarp();  // the warp's barriers are initialised before any lane polls them

  // acc[sp][c] = {v(small 2sp, wide c), v(small 2sp + 1, wide c)} for the lane's wide c
  unsigned long long acc[MT / 2][4];
#pragma unroll
  for (int sp = 0; sp < MT / 2; ++sp)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[sp][c] = 0;

  // one k: the 16 small values (4 broadcast float4 of a [k][16] row) times 4 wide values
  auto step = [&](const float *srow, const float (&wv)[4]) {
    unsigned long long sp2[MT / 2];
#pragma unroll
    for (int r = 0; r < MT / 4; ++r) {
      const float4 f = *reinterpret_cast<const float4 *>(srow + 4 * r);
      sp2[2 * r] = pack2(f.x, f.y);
      sp2[2 * r + 1] = pack2(f.z, f.w);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const unsigned long long wd = pack2(wv[c], wv[c]);
#pragma unroll
      for (int sp = 0; sp < MT / 2; ++sp) ffma2(acc[sp][c], sp2[sp], wd);
    }
  };

  float *tb = tbuf + warp * (KC * TP);
  int waited = 0;  // chunks whose copies this warp has seen complete
  for (int j = 0; j < my_chunks; ++j) {
    const int st = stage_of(j);
    if (!mbar_wait(bars + 8 * st, (uint32_t)(j / SPW) & 1u)) {
      if (lane == 0) atomicCAS(status, 0, 1);
      break;
    }
    waited = j + 1;
    const float *bs = big + st * (BIG_BYTES / 4);
    const float *ss = sml + st * (SMALL_BYTES / 4);
    if constexpr (TN) {
      const int swz = (lane >> 2) & 1;  // == ((lane + 32 c) >> 2) & 1 for every c
#pragma unroll
      for (int hq = 0; hq < KC / 4; ++hq) {
        float4 wq[4];  // rows lane + 32 c, k = 4 hq .. 4 hq + 3
#pragma unroll
        for (int c = 0; c < 4; ++c)
          wq[c] = *reinterpret_cast<const float4 *>(bs + (lane + 32 * c) * KC + ((hq ^ swz) << 2));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          float wv[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            wv[c] = kk == 0 ? wq[c].x : kk == 1 ? wq[c].y : kk == 2 ? wq[c].z : wq[c].w;
          step(ss + (4 * hq + kk) * MT, wv);
        }
      }
    } else {
      // A[16 m][8 k] -> tb[8 k][16 m] (row pitch TP keeps the two k halves in other banks)
      {
        const float4 v = *reinterpret_cast<const float4 *>(ss + (lane >> 1) * KC + 4 * (lane & 1));
        float *d = tb + 4 * (lane & 1) * TP + (lane >> 1);
        d[0] = v.x;
        d[TP] = v.y;
        d[2 * TP] = v.z;
        d[3 * TP] = v.w;
      }
      __syncwarp();
#pragma unroll
      for (int k = 0; k < KC; ++k) {
        const float4 b = *reinterpret_cast<const float4 *>(bs + k * BW + 4 * lane);
        const float wv[4] = {b.x, b.y, b.z, b.w};
        step(tb + k * TP, wv);
      }
    }
    __syncwarp();  // every lane has read the stage (and tb) before they are refilled
    if (lane == 0 && j + SPW < my_chunks) issue(j + SPW);
  }
  griddep_launch_dependents();
  // No copy may still be writing the rings when they are reused below: a warp that stopped
  // early waits (bounded) for the copies it issued and has not seen complete.
  if (lane == 0) {
    const int issued = min(my_chunks, waited + SPW);
    for (int j = waited; j < issued; ++j)
      if (!mbar_wait(bars + 8 * stage_of(j), (uint32_t)(j / SPW) & 1u)) atomicCAS(status, 0, 3);
  }
  __syncthreads();

  // Warp partials -> red[warp] in C orientation (R rows of CC floats); thin-N rows hold their
  // four 16-byte groups j at j ^ ((row >> 1) & 3), which spreads a warp's stores over all
  // banks. Then the CTA partial part = their sum in warp order.
  float *red = reinterpret_cast<float *>(sbase);
  float *wred = red + warp * TILE_FLOATS;
  if constexpr (TN) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int row = lane + 32 * c;
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // columns 4j .. 4j + 3 = small pairs 2j, 2j + 1
        const float2 lo = unpack2(acc[2 * j][c]), hi = unpack2(acc[2 * j + 1][c]);
        *reinterpret_cast<float4 *>(wred + row * CC + 4 * (j ^ ((row >> 1) & 3))) =
            make_float4(lo.x, lo.y, hi.x, hi.y);
      }
    }
  } else {
#pragma unroll
    for (int sp = 0; sp < MT / 2; ++sp) {
      float2 v[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) v[c] = unpack2(acc[sp][c]);
      *reinterpret_cast<float4 *>(wred + (2 * sp) * CC + 4 * lane) =
          make_float4(v[0].x, v[1].x, v[2].x, v[3].x);
      *reinterpret_cast<float4 *>(wred + (2 * sp + 1) * CC + 4 * lane) =
          make_float4(v[0].y, v[1].y, v[2].y, v[3].y);
    }
  }
  __syncthreads();
  float4 *part = reinterpret_cast<float4 *>(sbase + BIG_RING);
  const float4 *r4 = reinterpret_cast<const float4 *>(red);
  for (int e = tid; e < TILE_FLOATS / 4; e += THREADS) {
    int off = e;  // float4 index of group e inside one warp's partial
    if constexpr (TN) {
      const int row = e / (CC / 4), j = e % (CC / 4);
      off = row * (CC / 4) + (j ^ ((row >> 1) & 3));
    }
    float4 s = r4[off];
#pragma unroll
    for (int w = 1; w < WARPS; ++w) {  // in warp order
      const float4 v = r4[w * (TILE_FLOATS / 4) + off];
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    part[e] = s;
  }
  // The cluster's CTA partials are complete: CTA rank r finishes float4 groups
  // [r * per, (r + 1) * per) of the tile, adding the S partials in rank order.
  if (S > 1)
    cluster_sync_all();
  else
    __syncthreads();
#pragma unroll
  for (int f = 0; f < FIN; ++f) {
    const int t = tid + f * THREADS;
    if (t >= per) break;
    const int e = (int)rank * per + t;
    float4 s;
    if (S > 1) {
      const uint32_t local = saddr(part + e);
      float4 v[MAX_CLUSTER];
#pragma unroll
      for (int q = 0; q < MAX_CLUSTER; ++q)  // all loads in flight before the adds
        if (q < S) v[q] = ld_cluster4(local, (uint32_t)q);
      s = v[0];
#pragma unroll
      for (int q = 1; q < MAX_CLUSTER; ++q)
        if (q < S) {
          s.x += v[q].x;
          s.y += v[q].y;
          s.z += v[q].z;
          s.w += v[q].w;
        }
    } else {
      s = part[e];
    }
    const int row = (TN ? w0 : s0) + e / (CC / 4);
    const int col = (TN ? s0 : w0) + (e % (CC / 4)) * 4;
    if (row < p.M && col < p.N) {
      float *dst = p.C + (long long)row * p.ldc + col;
      const float v[4] = {s.x, s.y, s.z, s.w};
      if (p.vec_c && col + 3 < p.N) {
        float4 out;
        if (p.beta != 0.0f) {
          const float4 old = cold[f];
          out = make_float4(fmaf(p.alpha, v[0], p.beta * old.x),
                            fmaf(p.alpha, v[1], p.beta * old.y),
                            fmaf(p.alpha, v[2], p.beta * old.z),
                            fmaf(p.alpha, v[3], p.beta * old.w));
        } else {
          out = make_float4(p.alpha * v[0], p.alpha * v[1], p.alpha * v[2], p.alpha * v[3]);
        }
        *reinterpret_cast<float4 *>(dst) = out;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (col + q < p.N)
            dst[q] = (p.beta != 0.0f) ? fmaf(p.alpha, v[q], p.beta * dst[q]) : p.alpha * v[q];
      }
    }
  }
  // No CTA leaves while another may still read its partial.
  if (S > 1) cluster_sync_all();
}

}  // namespace thin
}  // namespace sgemm
