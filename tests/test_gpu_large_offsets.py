"""GPU parity at sizes where an operand holds more than 2^31 elements, so element offsets
(row x leading dimension + column) only fit in 64 bits.

Each case fills its operands on the device from a seeded generator (uniform [-1, 1)),
runs one call through the C ABI, and checks a sample of C against the FP64 oracle with
the usual bound |C - R| <= 1e-4 (S + |beta c|). The sample takes rows and columns at both
ends, on either side of the row where the offset of the large operand passes 2^31, and at
random. The oracle computes the sampled block as the plain product of the sampled rows of
A and the sampled columns of B.

The shapes reach the kernels the automatic plan picks for large problems: the k-major
128x96 TMA kernel (with its A^T copy), the copy-fed kernel on unaligned operands, the
A-as-stored TMA kernel with a split tail, the thin cluster kernels, the generic split-K
kernel, and the 3xTF32 tensor-core variant.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_bound

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dense_fp32_matrix_08_gb300 as sg

LIMIT = 2 ** 31
ALPHA, BETA = 0.75, -1.25


def _uniform(rows, cols, gen):
    return torch.rand((rows, cols), generator=gen, device="cuda", dtype=torch.float32) * 2 - 1


def _sample(n, lds, rng, count=24):
    """Indices 0..3, the last 8, for each leading dimension ld in `lds` the three around
    the index where index * ld passes 2^31, and `count` random ones."""
    idx = list(range(min(n, 4))) + list(range(max(0, n - 8), n))
    for ld in lds:
        edge = LIMIT // ld
        idx += [i for i in (edge - 1, edge, edge + 1) if 0 <= i < n]
    idx += list(rng.integers(0, n, count))
    return np.unique(np.array(idx, dtype=np.int64))


def _check_case(M, N, K, fn, seed, what):
    need = 4 * (M * K + K * N + M * N) * 3  # operands, plus copies and split buffers
    free, _ = torch.cuda.mem_get_info()
    if free < need + (4 << 30):
        pytest.skip(f"needs {need / 2**30:.1f} GiB of free device memory")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    A = _uniform(M, K, gen)
    B = _uniform(K, N, gen)
    C = _uniform(M, N, gen)
    rng = np.random.default_rng(seed)
    # rows where A's offsets (ld K) or C's (ld N) pass 2^31; every output element reads
    # all K rows of B, so B's far rows need no sampling
    rows = _sample(M, [ld for ld, big in ((K, M * K > LIMIT), (N, M * N > LIMIT)) if big], rng)
    cols = _sample(N, [], rng)
    ri = torch.from_numpy(rows).cuda()
    ci = torch.from_numpy(cols).cuda()
    A_s = A.index_select(0, ri).cpu()
    B_s = B.index_select(1, ci).cpu().contiguous()
    C_s = C.index_select(0, ri).index_select(1, ci).cpu().contiguous()
    rc = fn(M, N, K, ALPHA, A.data_ptr(), K, B.data_ptr(), N, BETA, C.data_ptr(), N)
    assert rc == 0, f"{what}: returned {rc}"
    torch.cuda.synchronize()
    out = C.index_select(0, ri).index_select(1, ci).cpu().numpy()
    del A, B, C
    torch.cuda.empty_cache()
    R, S = oracle.sgemm_f64(A_s, B_s, C_s, ALPHA, BETA)
    assert_bound(out, R, S, BETA, C_s.numpy(), f"{what} {M}x{N}x{K}")


# (M, N, K): which operand passes 2^31 elements, and the plan the shape gets
CASES = [
    (4096, 524400, 4096),   # B and C; k-major 128x96 TMA kernel after the A^T copy
    (4096, 524401, 4096),   # B and C, odd N (no TMA for B or C); copy-fed kernel
    (65539, 96, 32772),     # A; TMA kernel reading A as stored, split tail + reduce
    (65539, 32772, 8),      # C; short K, whole tiles only
    (16, 32772, 65540),     # B; thin-M cluster kernel
    (16, 32772, 65539),     # B, odd K; generic split-K kernel with the reduce
    (65539, 16, 32772),     # A; thin-N cluster kernel
]


@pytest.mark.parametrize("shape", CASES)
def test_offsets_past_2e31(shape):
    M, N, K = shape
    assert max(M * K, K * N, M * N) > LIMIT
    plan = sg.sgemm_f32_plan(M, N, K, K, N, N, ALPHA, BETA)
    assert plan["status"] == 0
    _check_case(M, N, K, sg.sgemm_f32, seed=M + 3 * N + 7 * K,
                what=f"sgemm_f32 (configuration {plan['variant']}, split {plan['split']})")
    assert sg.sgemm_f32_status() == (0, 0)


def test_offsets_past_2e31_3xtf32():
    M, N, K = 65539, 128, 32772
    _check_case(M, N, K, sg.sgemm_f32_3xtf32, seed=11, what="sgemm_f32_3xtf32")
    assert sg.sgemm_f32_3xtf32_status() == (0, 0)
