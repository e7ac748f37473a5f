// sgemm_f32_host: C = alpha * A * B + beta * C with A, B and C in host memory. The product
// runs on the GPU in row blocks; the host <-> device copies of one block overlap the
// computation of its neighbours:
//
//   copy-in stream   B/A0 chunk 0, 1, ... C0   A1 C1   .......  A2 C2 (after D2H 0) ...
//   compute stream     GEMM 0 chunk 0, 1, ...  +C0   GEMM 1    GEMM 2 ...
//   copy-out stream                               C0 out    C1 out   ...
//
// With a large B the first block is computed in K chunks as B and A0 arrive (see below), so
// the GEMMs start after one chunk instead of all of B. The last block is computed in two row
// parts, so that only the second part's copy out follows the last GEMM.
//
// Device buffers (B whole; A and C blocks, double-buffered) come from the library's
// workspace pool on the caller's stream and go back to it when the work is done.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/sgemm_f32.h"
#include "sgemm_internal.h"
#include "sgemm_plan.h"

namespace sgemm {
namespace {

struct CopyStreams {
  std::mutex mu;
  cudaStream_t in = nullptr, out = nullptr;  // set together, once both exist
};
CopyStreams g_copy[64];

// The current device's two copy streams, created by the first call on the device that
// succeeds and kept until exit. A failed creation is returned and tried again by the next
// call, not kept for the process.
cudaError_t copy_streams(cudaStream_t *in, cudaStream_t *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  CopyStreams &c = g_copy[dev];
  std::lock_guard<std::mutex> lock(c.mu);
  if (c.in == nullptr) {
    cudaStream_t si = nullptr, so = nullptr;
    e = cudaStreamCreateWithFlags(&si, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&so, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
      if (si != nullptr) cudaStreamDestroy(si);
      return e;
    }
    c.in = si;
    c.out = so;
  }
  *in = c.in;
  *out = c.out;
  return cudaSuccess;
}

// Events of one call; destroyed after enqueueing (CUDA releases them once complete).
struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  cudaError_t make(cudaEvent_t *out) {
    cudaError_t e = cudaEventCreateWithFlags(out, cudaEventDisableTiming);
    if (e == cudaSuccess) ev.push_back(*out);
    return e;
  }
};

// y += beta * x over n contiguous floats (both pool buffers, 256-byte aligned): the first
// block's beta * C0 when that block is computed in K chunks.
__global__ void add_scaled_kernel(float *__restrict__ y, const float *__restrict__ x,
                                  long long n, float beta) {
  const long long n4 = n / 4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  float4 *y4 = reinterpret_cast<float4 *>(y);
  const float4 *x4 = reinterpret_cast<const float4 *>(x);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 a = x4[i];
    float4 b = y4[i];
    b.x = fmaf(beta, a.x, b.x);
    b.y = fmaf(beta, a.y, b.y);
    b.z = fmaf(beta, a.z, b.z);
    b.w = fmaf(beta, a.w, b.w);
    y4[i] = b;
  }
  if (blockIdx.x == 0)
    for (long long i = 4 * n4 + threadIdx.x; i < n; i += blockDim.x) y[i] = fmaf(beta, x[i], y[i]);
}

}  // namespace
}  // namespace sgemm

using namespace sgemm;

extern "C" int sgemm_f32_host(int M, int N, int K, float alpha, const float *A, int lda,
                              const float *B, int ldb, float beta, float *C, int ldc,
                              cudaStream_t stream) {
  Problem pr{M, N, K, lda, ldb, ldc};
  int rc = validate(pr, alpha, A != nullptr, B != nullptr, C != nullptr);
  if (rc != 0) return rc;
  if (M == 0 || N == 0) return 0;
  const bool reads_ab = K > 0 && alpha != 0.0f;
  if (!reads_ab && beta == 1.0f) return 0;  // C unchanged
  int num_sms = 0;
  cudaError_t e = device_setup(&num_sms);
  if (e != cudaSuccess) return (int)e;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  e = copy_streams(&s_in, &s_out);
  if (e != cudaSuccess) return (int)e;

  // Row blocks: about 2048 rows (enough tiles for several waves of the GEMM kernel),
  // at most 8 blocks, a multiple of 128 rows.
  const int nb = std::max(1, std::min(8, M / 2048));
  const int mb = (int)std::min<long long>(M, ceil_div(ceil_div(M, nb), 128) * 128);
  const int blocks = (int)ceil_div(M, mb);
  const bool need_c_in = beta != 0.0f;

  const size_t b_bytes = reads_ab ? (size_t)K * N * 4 : 0;
  const size_t a_bytes = reads_ab ? (size_t)mb * K * 4 : 0;
  const size_t c_bytes = (size_t)mb * N * 4;
  float *dB = nullptr, *dA[2] = {nullptr, nullptr}, *dC[2] = {nullptr, nullptr};
  cudaMemPool_t pool = workspace_pool();
  auto alloc = [&](float **p, size_t bytes) {
    if (bytes == 0 || e != cudaSuccess) return;
    e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(p), bytes, pool, stream);
  };
  // Head: with several blocks and a large B, block 0 is computed in K chunks as B arrives,
  // C0 = alpha A0[:, k0:k1) B[k0:k1, :] + C0 chunk by chunk (the first chunk with beta 0),
  // then C0 += beta * C0_old from a staging copy, so the GEMMs start after one small chunk
  // of B and A0 instead of all of B and the C0 rows. The chunk boundaries round the running
  // sum to FP32 once per chunk; the result stays within the library's bound, but is not
  // bitwise the single-call result.
  const bool chunk_head = reads_ab && blocks >= 2 && K >= 1024 && b_bytes >= ((size_t)32 << 20);
  float *dCs = nullptr;  // staged C0 rows (chunked head with beta != 0)
  alloc(&dB, b_bytes);
  for (int q = 0; q < std::min(2, blocks); ++q) {
    alloc(&dA[q], a_bytes);
    alloc(&dC[q], c_bytes);
  }
  if (chunk_head && need_c_in) alloc(&dCs, c_bytes);
  Events evs;
  cudaEvent_t ev_start = nullptr;
  if (e == cudaSuccess) e = evs.make(&ev_start);
  if (e == cudaSuccess) e = cudaEventRecord(ev_start, stream);  // buffers are allocated
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_in, ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, ev_start, 0);

  auto rows_of = [&](int i) { return std::min(mb, M - i * mb); };
  // Tail: when there are two or more blocks, the last one (if 1024 rows or more) is computed
  // in two parts, its last 3/8 (rounded up to 128 rows) apart, so that only their copy out
  // follows the last GEMM. 2048 rows split as 1280 + 768.
  auto tail_rows = [&](int rows) -> int {
    if (blocks < 2 || rows < 1024) return 0;
    const long long t = ceil_div(3LL * rows, 8 * 128) * 128;
    return t < rows ? (int)t : 0;
  };
  std::vector<cudaEvent_t> ev_in(blocks, nullptr), ev_done(blocks, nullptr),
      ev_out(blocks, nullptr);
  auto copy_in = [&](int i) {  // on s_in: A and C rows of block i into buffer i % 2
    const int r0 = i * mb, rows = rows_of(i);
    if (e == cudaSuccess && reads_ab)
      e = cudaMemcpy2DAsync(dA[i % 2], (size_t)K * 4, A + (long long)r0 * lda, (size_t)lda * 4,
                            (size_t)K * 4, rows, cudaMemcpyHostToDevice, s_in);
    if (e == cudaSuccess && need_c_in)
      e = cudaMemcpy2DAsync(dC[i % 2], (size_t)N * 4, C + (long long)r0 * ldc, (size_t)ldc * 4,
                            (size_t)N * 4, rows, cudaMemcpyHostToDevice, s_in);
    if (e == cudaSuccess) e = evs.make(&ev_in[i]);
    if (e == cudaSuccess) e = cudaEventRecord(ev_in[i], s_in);
  };

  // Chunk boundaries: a first chunk of 256, then each chunk twice as long as the one before
  // (from the second chunk on, the copies run ahead of the GEMMs); a rest shorter than half
  // a chunk joins that chunk. K = 8192 gives 256, 512, 1024, 2048 and 4352.
  std::vector<int> kb{0};
  if (chunk_head) {
    kb.push_back(std::min(K, 256));
    long long len = 256;
    while (kb.back() < K) {
      len *= 2;
      long long next = kb.back() + len;
      if (K - next < len / 2) next = K;
      kb.push_back((int)std::min<long long>(K, next));
    }
  } else {
    kb.push_back(K);
  }
  const int nchunks = (int)kb.size() - 1;
  std::vector<cudaEvent_t> ev_chunk(chunk_head ? nchunks : 0, nullptr);
  cudaEvent_t ev_c0 = nullptr;
  if (chunk_head) {
    const int rows0 = rows_of(0);
    for (int c = 0; c < nchunks && e == cudaSuccess; ++c) {
      const int k0 = kb[c], kn = kb[c + 1] - kb[c];
      e = cudaMemcpy2DAsync(dB + (size_t)k0 * N, (size_t)N * 4, B + (long long)k0 * ldb,
                            (size_t)ldb * 4, (size_t)N * 4, kn, cudaMemcpyHostToDevice, s_in);
      if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(dA[0] + k0, (size_t)K * 4, A + k0, (size_t)lda * 4,
                              (size_t)kn * 4, rows0, cudaMemcpyHostToDevice, s_in);
      if (e == cudaSuccess) e = evs.make(&ev_chunk[c]);
      if (e == cudaSuccess) e = cudaEventRecord(ev_chunk[c], s_in);
    }
    if (need_c_in) {
      if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(dCs, (size_t)N * 4, C, (size_t)ldc * 4, (size_t)N * 4, rows0,
                              cudaMemcpyHostToDevice, s_in);
      if (e == cudaSuccess) e = evs.make(&ev_c0);
      if (e == cudaSuccess) e = cudaEventRecord(ev_c0, s_in);
    }
    if (e == cudaSuccess) ev_in[0] = ev_chunk[nchunks - 1];
  } else {
    if (e == cudaSuccess && reads_ab)
      e = cudaMemcpy2DAsync(dB, (size_t)N * 4, B, (size_t)ldb * 4, (size_t)N * 4, K,
                            cudaMemcpyHostToDevice, s_in);
    copy_in(0);
  }
  if (blocks > 1) copy_in(1);
  // on s_out, once `ready` has completed: rows [p0, p0 + n) of block i back to the host
  auto copy_out = [&](int i, int p0, int n, cudaEvent_t ready) {
    cudaError_t r = cudaStreamWaitEvent(s_out, ready, 0);
    if (r == cudaSuccess)
      r = cudaMemcpy2DAsync(C + (long long)(i * mb + p0) * ldc, (size_t)ldc * 4,
                            dC[i % 2] + (size_t)p0 * N, (size_t)N * 4, (size_t)N * 4, n,
                            cudaMemcpyDeviceToHost, s_out);
    return r;
  };
  for (int i = 0; i < blocks && e == cudaSuccess; ++i) {
    const int rows = rows_of(i);
    int out0 = 0;  // first row of the block still to be copied out after its GEMMs
    if (i == 0 && chunk_head) {
      for (int c = 0; c < nchunks && e == cudaSuccess && rc == 0; ++c) {
        const int k0 = kb[c], kn = kb[c + 1] - kb[c];
        e = cudaStreamWaitEvent(stream, ev_chunk[c], 0);
        if (e == cudaSuccess)
          rc = sgemm_f32(rows, N, kn, alpha, dA[0] + k0, K, dB + (size_t)k0 * N, N,
                         c == 0 ? 0.0f : 1.0f, dC[0], N, stream);
      }
      if (e == cudaSuccess && rc == 0 && need_c_in) {
        e = cudaStreamWaitEvent(stream, ev_c0, 0);
        if (e == cudaSuccess) {
          add_scaled_kernel<<<num_sms * 4, 256, 0, stream>>>(dC[0], dCs, (long long)rows * N,
                                                              beta);
          e = cudaGetLastError();
        }
      }
      if (e != cudaSuccess || rc != 0) break;
    } else {
      e = cudaStreamWaitEvent(stream, ev_in[i], 0);
      if (e != cudaSuccess) break;
      // The block's product on the caller's stream, through the library's own entry point.
      // The last block's first rows go out while the GEMM of its tail runs.
      const int part = i == blocks - 1 ? rows - tail_rows(rows) : rows;
      for (int p0 = 0; p0 < rows && e == cudaSuccess && rc == 0; p0 += part) {
        const int n = std::min(part, rows - p0);
        rc = sgemm_f32(n, N, K, alpha, reads_ab ? dA[i % 2] + (size_t)p0 * K : nullptr,
                       std::max(1, K), reads_ab ? dB : nullptr, N, beta,
                       dC[i % 2] + (size_t)p0 * N, N, stream);
        if (rc == 0 && p0 + n < rows) {
          cudaEvent_t ev_part = nullptr;
          e = evs.make(&ev_part);
          if (e == cudaSuccess) e = cudaEventRecord(ev_part, stream);
          if (e == cudaSuccess) e = copy_out(i, p0, n, ev_part);
        }
        out0 = p0;
      }
      if (e != cudaSuccess || rc != 0) break;
    }
    e = evs.make(&ev_done[i]);
    if (e == cudaSuccess) e = cudaEventRecord(ev_done[i], stream);
    if (e == cudaSuccess) e = copy_out(i, out0, rows - out0, ev_done[i]);
    if (e == cudaSuccess) e = evs.make(&ev_out[i]);
    if (e == cudaSuccess) e = cudaEventRecord(ev_out[i], s_out);
    // block i + 2 reuses buffer i % 2 once block i's result has left it
    if (e == cudaSuccess && i + 2 < blocks) {
      e = cudaStreamWaitEvent(s_in, ev_out[i], 0);
      copy_in(i + 2);
    }
  }
  // The caller's stream owns the result: it waits for the last copies out, then frees.
  for (int i = 0; i < blocks; ++i)
    if (ev_out[i] != nullptr) {
      const cudaError_t w = cudaStreamWaitEvent(stream, ev_out[i], 0);
      if (e == cudaSuccess) e = w;
    }
  if (ev_start != nullptr && (e != cudaSuccess || rc != 0)) {
    // on an error the copy streams may still reference the buffers: join them first
    cudaEvent_t j1 = nullptr, j2 = nullptr;
    if (evs.make(&j1) == cudaSuccess && cudaEventRecord(j1, s_in) == cudaSuccess)
      cudaStreamWaitEvent(stream, j1, 0);
    if (evs.make(&j2) == cudaSuccess && cudaEventRecord(j2, s_out) == cudaSuccess)
      cudaStreamWaitEvent(stream, j2, 0);
  }
  for (float *p : {dB, dA[0], dA[1], dC[0], dC[1], dCs})
    if (p != nullptr) {
      const cudaError_t f = cudaFreeAsync(p, stream);
      if (e == cudaSuccess) e = f;
    }
  if (rc != 0) return rc;
  return (int)e;
}
