// 3xTF32 SGEMM on the 5th-generation tensor cores (tcgen05, TMEM, TMA) of sm_103a.
//
// C = alpha * A * B + beta * C with FP32 inputs and FP32 accumulation, computed as
//   A * B ~= A_hi * B_hi + A_hi * B_lo + A_lo * B_hi,
// where x_hi = tf32(x) (round to nearest, ties away) and x_lo = tf32(x - x_hi). x - x_hi is
// exact in FP32, so each product misses only the lo * lo term and the rounding of x_lo,
// about 2^-21 of |a * b|: far inside the 1e-4 * sum |a b| bound of the FP32 contract.
// This is the tensor-core path the SGEMM study lists as the next step after the FFMA path
// ("Lecture 4 - GPU Acceleration", section 5.5: for large tiles FP32 GEMM becomes compute
// bound, and tensor cores raise the ceiling); the pages themselves stop at FFMA.
//
// Data flow (three launches on the caller's stream):
//  1. split_rows_kernel:  A (M x K, lda) -> A_hi, A_lo (Mp x Kp, K-major, zero padded)
//  2. split_cols_kernel:  B (K x N, ldb) -> B_hi, B_lo (Np x Kp, K-major = B transposed)
//  3. tc3_kernel:         persistent (one CTA per SM, 128 x 128 C tiles in grouped order,
//     tile t, t + grid, ...), warp-specialised:
//       warp 0 lane 0   streams the four operand tiles of each 32-wide K block (A_hi, A_lo,
//                       B_hi, B_lo, 128 x 32 each) into a 3-stage shared-memory ring with
//                       TMA (128-byte swizzle);
//       warp 1 lane 0   issues 12 tcgen05.mma (kind::tf32, M=128 N=128 K=8) per K block
//                       into one of two TMEM accumulators (128 lanes x 128 FP32 columns
//                       each), alternating per tile;
//       warps 2 - 5     drain the other accumulator meanwhile: tcgen05.ld, a per-warp
//                       transpose in shared memory, and coalesced alpha / beta row stores.
//     The epilogue of tile i thus overlaps the MMAs of tile i + 1. (A 128 x 256 tile, all
//     512 TMEM columns, measured the same at 8192^3 and slower at 4096^3: fewer tiles.)
// Every wait on an mbarrier is bounded: a wait that gives up records an error in a device
// status word (read with sgemm_f32_3xtf32_status) and the CTA still frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/sgemm_f32.h"
#include "sgemm_ffma.cuh"
#include "sgemm_internal.h"
#include "sgemm_plan.h"
#include "sgemm_ptx.cuh"

namespace sgemm {
namespace tc {

constexpr int BM = 128, BN = 128, BK = 32, STAGES = 3;
constexpr int EPI_WARPS = 4, THREADS = 32 * (2 + EPI_WARPS);  // producer, MMA, epilogue
constexpr int A_TILE = BM * BK * 4;          // one 128 x 32 FP32 operand tile of A
constexpr int B_TILE = BN * BK * 4;          // one 256 x 32 FP32 operand tile of B^T
constexpr int STAGE_BYTES = 2 * A_TILE + 2 * B_TILE;  // A_hi, A_lo, B_hi, B_lo
constexpr int EPI_PITCH = 33;                // transpose buffer row pitch (floats)
constexpr int EPI_BYTES = EPI_WARPS * 32 * EPI_PITCH * 4;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + 128;
constexpr uint32_t ACC_COLS = BN;            // one accumulator: BN FP32 columns
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;

static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA on sm_103a");
static_assert(TMEM_COLS <= 512, "two accumulators fit in TMEM");
static_assert(BN % 16 == 0 && BN <= 256, "tcgen05.mma N for M = 128");

// Instruction descriptor of tcgen05.mma kind::tf32: D in FP32 (bits 4-5 = 1), A and B in
// TF32 (bits 7-9 and 10-12 = 2), both K-major (bits 15, 16 = 0), N / 8 in bits 17-22,
// M / 16 in bits 24-28.
constexpr uint32_t IDESC = (1u << 4) | (2u << 7) | (2u << 10) |
                           ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct Params {
  int M, N, KT;  // KT: number of 32-wide K blocks (Kp / BK)
  int tiles_m, tiles_n, group_m;
  float alpha, beta;
  float *C;
  long long ldc;
};

// Device status word: 0 = fine; otherwise the first failing condition (1 = a producer
// wait, 2 = an MMA wait, 3 = an epilogue wait gave up).
__device__ int g_tc_status;

// ------------------------------------------------------------------------------------
// PTX wrappers

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, 128 x BN x 8, TF32 inputs, FP32 accumulation.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
      : "memory");
}

// 32 consecutive FP32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile laid out by TMA with the
// 128-byte swizzle: rows of 128 bytes (32 FP32), 8-row groups 1024 bytes apart. Fields:
// start address >> 4 (bits 0-13), leading byte offset >> 4 (bits 16-29, not used by
// swizzled K-major layouts, set to 1), stride byte offset >> 4 (bits 32-45: 1024 B),
// descriptor version 1 (bits 46-47), swizzle mode 2 = 128 B (bits 61-63). Advancing K by 8
// TF32 within the 128-byte swizzle atom adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// ------------------------------------------------------------------------------------
// Split passes (HBM bound).

// hi, lo: R_pad x C_pad row-major (ld = C_pad, a multiple of 32); X: R x C with ld ldx.
__global__ void split_rows_kernel(const float *__restrict__ X, long long ldx, int R, int Cc,
                                  float *__restrict__ hi, float *__restrict__ lo, int R_pad,
                                  int C_pad) {
  constexpr int U = 4;  // 4-column groups per thread and round, all reads issued first
  const long long quads = C_pad / 4;
  const long long total = (long long)R_pad * quads;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long g0 = blockIdx.x * (long long)blockDim.x + threadIdx.x; g0 < total;
       g0 += U * stride) {
    float x[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long g = g0 + u * stride;
      const long long r = g / quads;
      const int c = (int)(g - r * quads) * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        x[u][e] = (g < total && r < R && c + e < Cc) ? X[r * ldx + c + e] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long g = g0 + u * stride;
      if (g >= total) break;
      const long long r = g / quads;
      const int c = (int)(g - r * quads) * 4;
      float h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h[e] = tf32_rna(x[u][e]);
        l[e] = tf32_rna(x[u][e] - h[e]);
      }
      *reinterpret_cast<float4 *>(hi + r * C_pad + c) = make_float4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<float4 *>(lo + r * C_pad + c) = make_float4(l[0], l[1], l[2], l[3]);
    }
  }
}

// Transposing split: out[n][k] = split(X[k][n]); X: R (=K) x Cc (=N) with ld ldx;
// hi, lo: Cc_pad x R_pad row-major (ld = R_pad, a multiple of 4: 128-bit stores), zero
// beyond R and Cc. 64 x 64 tiles through shared memory, grid-stride; each of the 256
// threads has its 16 reads of a tile in flight at once (128-bit when VEC: ldx % 4 == 0 and
// X 16-byte aligned).
template <bool VEC>
__global__ void __launch_bounds__(256) split_cols_kernel(const float *__restrict__ X,
                                                         long long ldx, int R, int Cc,
                                                         float *__restrict__ hi,
                                                         float *__restrict__ lo, int R_pad,
                                                         int Cc_pad) {
  __shared__ float t[64][65];
  const long long tiles_n = (Cc_pad + 63) / 64;
  const long long tiles = tiles_n * ((R_pad + 63) / 64);
  const int tid = threadIdx.x, cg = tid & 15, ro = tid >> 4;
  for (long long tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int k0 = (int)(tile / tiles_n) * 64;
    const int n0 = (int)(tile % tiles_n) * 64;
    float v[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = k0 + ro + 16 * i, n = n0 + 4 * cg;
      const float *src = X + (long long)k * ldx + n;
      if (VEC && k < R && n + 3 < Cc) {
        const float4 f = __ldcs(reinterpret_cast<const float4 *>(src));
        v[i][0] = f.x;
        v[i][1] = f.y;
        v[i][2] = f.z;
        v[i][3] = f.w;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[i][j] = (k < R && n + j < Cc) ? src[j] : 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) t[ro + 16 * i][4 * cg + j] = v[i][j];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int nl = ro + 16 * i, kl = 4 * cg;
      const int n = n0 + nl, k = k0 + kl;
      if (n >= Cc_pad || k >= R_pad) continue;  // R_pad is a multiple of 4: whole groups
      float h[4], l[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x = t[kl + j][nl];
        h[j] = tf32_rna(x);
        l[j] = tf32_rna(x - h[j]);
      }
      const long long o = (long long)n * R_pad + k;
      *reinterpret_cast<float4 *>(hi + o) = make_float4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<float4 *>(lo + o) = make_float4(l[0], l[1], l[2], l[3]);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------------------------
// The tensor-core GEMM kernel.

__global__ void __launch_bounds__(THREADS, 1)
    tc3_kernel(const __grid_constant__ CUtensorMap map_ah, const __grid_constant__ CUtensorMap map_al,
               const __grid_constant__ CUtensorMap map_bh, const __grid_constant__ CUtensorMap map_bl,
               const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
  float *epi = reinterpret_cast<float *>(smem_raw + (base - raw) + STAGES * STAGE_BYTES);
  const uint32_t bars = base + STAGES * STAGE_BYTES + EPI_BYTES;
  // full[s] at bars + 8 s, empty[s] at bars + 8 (STAGES + s), acc_full[b] and acc_empty[b]
  // after them, then the TMEM address slot
  const uint32_t acc_full = bars + 8 * (2 * STAGES);
  const uint32_t acc_empty = acc_full + 16;
  const uint32_t tmem_slot = acc_empty + 16;
  volatile uint32_t *tmem_slot_ptr =
      reinterpret_cast<volatile uint32_t *>(smem_raw + (tmem_slot - raw));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles = p.tiles_m * p.tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bars + 8 * s, 1);
      mbar_init(bars + 8 * (STAGES + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + 8 * b, 1);
      mbar_init(acc_empty + 8 * b, EPI_WARPS);
    }
    mbar_init_fence();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot_ptr;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer: every K block of every tile of this CTA, in order
    tma_prefetch_map(&map_ah);
    tma_prefetch_map(&map_al);
    tma_prefetch_map(&map_bh);
    tma_prefetch_map(&map_bl);
    long long g = 0;  // K blocks issued by this CTA
    bool ok = true;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      int tm, tn;
      tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
      for (int kt = 0; kt < p.KT; ++kt, ++g) {
        const int s = (int)(g % STAGES);
        const uint32_t ph = (uint32_t)(g / STAGES) & 1u;
        if (g >= STAGES && !mbar_wait(bars + 8 * (STAGES + s), ph ^ 1u)) {
          atomicCAS(&g_tc_status, 0, 1);
          ok = false;
          break;
        }
        const uint32_t st = base + s * STAGE_BYTES;
        const uint32_t full = bars + 8 * s;
        mbar_expect_tx(full, STAGE_BYTES);
        tma_load_2d(st, &map_ah, kt * BK, tm * BM, full);
        tma_load_2d(st + A_TILE, &map_al, kt * BK, tm * BM, full);
        tma_load_2d(st + 2 * A_TILE, &map_bh, kt * BK, tn * BN, full);
        tma_load_2d(st + 2 * A_TILE + B_TILE, &map_bl, kt * BK, tn * BN, full);
      }
    }
    // Before this thread may leave, the last loads it issued into each stage must have
    // landed (normally long done: the MMA thread consumed them).
    for (long long k = g - 1; k >= 0 && k >= g - STAGES; --k)
      mbar_wait(bars + 8 * (int)(k % STAGES), (uint32_t)(k / STAGES) & 1u);
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: tile i accumulates into TMEM columns (i & 1) * ACC_COLS
    long long g = 0;
    bool ok = true;
    int i = 0;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++i) {
      const int b = i & 1;
      if (i >= 2 && !mbar_wait(acc_empty + 8 * b, ((uint32_t)(i >> 1) & 1u) ^ 1u)) {
        atomicCAS(&g_tc_status, 0, 2);
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)b * ACC_COLS;
      for (int kt = 0; kt < p.KT; ++kt, ++g) {
        const int s = (int)(g % STAGES);
        if (!mbar_wait(bars + 8 * s, (uint32_t)(g / STAGES) & 1u)) {
          atomicCAS(&g_tc_status, 0, 2);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = base + s * STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 8; ++kk) {
          const uint64_t ah = sw128_desc(st + kk * 32);
          const uint64_t al = sw128_desc(st + A_TILE + kk * 32);
          const uint64_t bh = sw128_desc(st + 2 * A_TILE + kk * 32);
          const uint64_t bl = sw128_desc(st + 2 * A_TILE + B_TILE + kk * 32);
          // small correction terms first, then the main product
          mma_tf32(acc, al, bh, (kt | kk) != 0 ? 1u : 0u);
          mma_tf32(acc, ah, bl, 1u);
          mma_tf32(acc, ah, bh, 1u);
        }
        mma_commit(bars + 8 * (STAGES + s));  // stage s free once these MMAs complete
      }
      if (ok) mma_commit(acc_full + 8 * b);  // accumulator b complete
    }
  } else if (warp >= 2) {
    // ---- epilogue: warp w reads TMEM lane quadrant w % 4 = tile rows 32 (w % 4) .. + 31
    const int q = warp & 3;
    float *buf = epi + (warp - 2) * 32 * EPI_PITCH;
    int i = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
      const int b = i & 1;
      const bool ready =
          __all_sync(0xffffffffu, mbar_wait(acc_full + 8 * b, (uint32_t)(i >> 1) & 1u));
      if (!ready) {
        if (lane == 0) atomicCAS(&g_tc_status, 0, 3);
        break;
      }
      tc_fence_after();
      int tm, tn;
      tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
      const int row0 = tm * BM + q * 32;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + (uint32_t)b * ACC_COLS + ((uint32_t)(q * 32) << 16) + (uint32_t)c, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) buf[lane * EPI_PITCH + j] = __uint_as_float(v[j]);
        __syncwarp();
        // lane l now writes column c + l of the warp's 32 rows: 128-byte row segments
        const int col = tn * BN + c + lane;
        if (col < p.N) {
#pragma unroll 4
          for (int r = 0; r < 32; ++r) {
            const int row = row0 + r;
            if (row < p.M) {
              float *dst = p.C + (long long)row * p.ldc + col;
              const float accv = buf[r * EPI_PITCH + lane];
              *dst = (p.beta != 0.0f) ? fmaf(p.alpha, accv, p.beta * *dst) : p.alpha * accv;
            }
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + 8 * b);  // accumulator b may be reused
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------------------------
// Host side

// Tensor map of a rows x cols row-major FP32 matrix (ld = cols, cols % 32 == 0), boxes of
// 32 (along the contiguous dimension) x box_rows, 128-byte swizzle.
static bool make_map(CUtensorMap *map, const float *ptr, long long rows, long long cols,
                     int box_rows) {
  return encode_map_2d(map, ptr, rows, cols, cols, BK, box_rows, true);
}

struct Shape {
  long long Mp, Np, Kp;
  size_t ws_bytes;
};

static Shape padded(int M, int N, int K) {
  Shape s;
  s.Mp = ceil_div(M, BM) * BM;
  s.Np = ceil_div(N, BN) * BN;
  s.Kp = ceil_div(K, BK) * BK;
  s.ws_bytes = (size_t)4 * 2 * (size_t)(s.Mp * s.Kp + s.Np * s.Kp);
  return s;
}

static std::once_flag g_attr_once[64];
static cudaError_t g_attr_err[64];

static cudaError_t kernel_setup() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(g_attr_once[dev], [dev]() {
    g_attr_err[dev] =
        cudaFuncSetAttribute(tc3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  return g_attr_err[dev];
}

}  // namespace tc

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

bool encode_map_2d(CUtensorMap *map, const float *ptr, long long rows, long long cols,
                   long long ld, int box_cols, int box_rows, bool swizzle128) {
  return encode_map_2d_swizzle(map, ptr, rows, cols, ld, box_cols, box_rows,
                               swizzle128 ? 128 : 0);
}

bool encode_map_2d_swizzle(CUtensorMap *map, const float *ptr, long long rows, long long cols,
                           long long ld, int box_cols, int box_rows, int swizzle_bytes) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle_bytes == 32) swz = CU_TENSOR_MAP_SWIZZLE_32B;
  else if (swizzle_bytes == 64) swz = CU_TENSOR_MAP_SWIZZLE_64B;
  else if (swizzle_bytes == 128) swz = CU_TENSOR_MAP_SWIZZLE_128B;
  else if (swizzle_bytes != 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace sgemm

using namespace sgemm;

extern "C" int sgemm_f32_3xtf32_workspace_size(int M, int N, int K, size_t *bytes) {
  if (M < 0) return -1;
  if (N < 0) return -2;
  if (K < 0) return -3;
  if (bytes) *bytes = (M == 0 || N == 0 || K == 0) ? 0 : tc::padded(M, N, K).ws_bytes;
  return 0;
}

extern "C" int sgemm_f32_3xtf32(int M, int N, int K, float alpha, const float *A, int lda,
                                const float *B, int ldb, float beta, float *C, int ldc,
                                cudaStream_t stream) {
  Problem pr{M, N, K, lda, ldb, ldc};
  int rc = validate(pr, alpha, A != nullptr, B != nullptr, C != nullptr);
  if (rc != 0) return rc;
  if (M == 0 || N == 0) return 0;
  if (alpha == 0.0f || K == 0)  // beta-scale quick return: no product to compute
    return sgemm_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
  int num_sms = 0;
  cudaError_t e = device_setup(&num_sms);
  if (e != cudaSuccess) return (int)e;
  e = tc::kernel_setup();
  if (e != cudaSuccess) return (int)e;
  const tc::Shape sh = tc::padded(M, N, K);
  const long long tiles_m = sh.Mp / tc::BM, tiles_n = sh.Np / tc::BN;
  if (tiles_m * tiles_n > 0x7fffffffLL) return (int)cudaErrorInvalidConfiguration;
  float *ws = nullptr;
  e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws), sh.ws_bytes, workspace_pool(),
                              stream);
  if (e != cudaSuccess) return (int)e;
  float *ah = ws, *al = ah + sh.Mp * sh.Kp, *bh = al + sh.Mp * sh.Kp, *bl = bh + sh.Np * sh.Kp;

  {
    const long long work = sh.Mp * (sh.Kp / 4);
    const int blocks = (int)std::max<long long>(1, std::min<long long>((work + 255) / 256,
                                                                        (long long)num_sms * 8));
    tc::split_rows_kernel<<<blocks, 256, 0, stream>>>(A, lda, M, K, ah, al, (int)sh.Mp,
                                                      (int)sh.Kp);
  }
  {
    const long long tiles = ((sh.Np + 63) / 64) * ((sh.Kp + 63) / 64);
    const int blocks = (int)std::max<long long>(1, std::min<long long>(tiles, (long long)num_sms * 8));
    if (ldb % 4 == 0 && (reinterpret_cast<uintptr_t>(B) & 15u) == 0)
      tc::split_cols_kernel<true><<<blocks, 256, 0, stream>>>(B, ldb, K, N, bh, bl, (int)sh.Kp,
                                                              (int)sh.Np);
    else
      tc::split_cols_kernel<false><<<blocks, 256, 0, stream>>>(B, ldb, K, N, bh, bl,
                                                               (int)sh.Kp, (int)sh.Np);
  }
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    CUtensorMap m_ah, m_al, m_bh, m_bl;
    if (!tc::make_map(&m_ah, ah, sh.Mp, sh.Kp, tc::BM) ||
        !tc::make_map(&m_al, al, sh.Mp, sh.Kp, tc::BM) ||
        !tc::make_map(&m_bh, bh, sh.Np, sh.Kp, tc::BN) ||
        !tc::make_map(&m_bl, bl, sh.Np, sh.Kp, tc::BN)) {
      e = cudaErrorInvalidValue;
    } else {
      tc::Params p;
      p.M = M;
      p.N = N;
      p.KT = (int)(sh.Kp / tc::BK);
      p.tiles_m = (int)tiles_m;
      p.tiles_n = (int)tiles_n;
      p.group_m = (int)std::min<long long>(16, tiles_m);
      p.alpha = alpha;
      p.beta = beta;
      p.C = C;
      p.ldc = ldc;
      // persistent: one CTA per SM (or per tile when there are fewer tiles)
      const long long grid = std::min<long long>(tiles_m * tiles_n, num_sms);
      tc::tc3_kernel<<<(unsigned)grid, tc::THREADS, tc::SMEM_BYTES, stream>>>(m_ah, m_al,
                                                                            m_bh, m_bl, p);
      e = cudaGetLastError();
    }
  }
  const cudaError_t ef = cudaFreeAsync(ws, stream);
  if (e == cudaSuccess) e = ef;
  return (int)e;
}

extern "C" int sgemm_f32_3xtf32_status(int *status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, tc::g_tc_status, sizeof(int));
  if (e != cudaSuccess) return (int)e;
  const int zero = 0;
  e = cudaMemcpyToSymbol(tc::g_tc_status, &zero, sizeof(int));
  if (status) *status = v;
  return (int)e;
}
