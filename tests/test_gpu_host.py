"""sgemm_f32_host: A, B, C in host memory, computed on the GPU in row blocks whose copies
overlap the neighbouring blocks' GEMMs. Parity against the CPU oracle with the usual bound
|C - R| <= 1e-4 (S + |beta c|), on shapes with one, two and four row blocks (the last reuses
the first block's buffers), padded leading dimensions, pinned and pageable memory, and the
quick-return cases."""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_inputs
from parity_util import assert_bound

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dense_fp32_matrix_08_gb300 as sg


def _host_view(x: torch.Tensor, ld: int, pinned: bool) -> torch.Tensor:
    rows, cols = x.shape
    buf = torch.full((max(rows, 1), ld), float("nan"))
    if pinned:
        buf = buf.pin_memory()
    view = buf[:rows, :cols]
    view.copy_(x)
    return buf, view


def _block_edges(M):
    """First rows of the row blocks and of the last block's separately computed tail, by the
    rule sgemm_f32_host documents: about 2048 rows a block (a multiple of 128, at most 8
    blocks); with two or more blocks, the last block's last 3/8 (rounded up to 128 rows) is
    computed and copied out apart when that block has 1024 rows or more."""
    nb = max(1, min(8, M // 2048))
    mb = min(M, -(-(-(-M // nb)) // 128) * 128)
    blocks = -(-M // mb)
    edges = [i * mb for i in range(blocks)]
    last = M - edges[-1]
    if blocks >= 2 and last >= 1024:
        tail = -(-3 * last // 1024) * 128
        if tail < last:
            edges.append(M - tail)
    return edges


# (4200, 2048, 4100): two row blocks and a 33.6 MB B, so the first block runs in K chunks
# of 256, 512, 1024 and 2308 as B arrives; the second block (2024 rows) is computed as
# 1256 + 768 rows
@pytest.mark.parametrize("shape", [(300, 200, 100), (5000, 700, 300), (9000, 64, 50),
                                   (4200, 2048, 4100)])
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("alpha,beta", [(0.75, -1.25), (1.0, 0.0)])
def test_host_entry_against_oracle(shape, pinned, alpha, beta):
    M, N, K = shape
    A, B, C = make_inputs(M, N, K, seed=M + N + K)
    bufA, hA = _host_view(A, K + 3, pinned)
    bufB, hB = _host_view(B, N + 1, pinned)
    bufC, hC = _host_view(C, N + 5, pinned)
    stream = torch.cuda.Stream()
    rc = sg.sgemm_f32_host(M, N, K, alpha, bufA, K + 3, bufB, N + 1, beta, bufC, N + 5, stream)
    assert rc == 0
    stream.synchronize()
    if M * N * K > 10**9:  # oracle on sampled rows: both sides of every block and part edge
        edges = [r for e in _block_edges(M) for r in range(max(0, e - 4), min(M, e + 4))]
        rows = np.unique(np.concatenate([np.arange(0, 8), np.array(edges, dtype=np.int64),
                                         np.random.default_rng(M).integers(0, M, 40), [M - 1]]))
        R, S = oracle.sgemm_f64_rows(A, B, C, alpha, beta, rows)
        assert_bound(hC.numpy()[rows], R, S, beta, C.numpy()[rows], f"host {shape} pinned={pinned}")
        return
    R, S = oracle.sgemm_f64(A, B, C, alpha, beta)
    assert_bound(hC.numpy(), R, S, beta, C.numpy(), f"host {shape} pinned={pinned}")
    assert torch.isnan(bufC[:, N:]).all(), "padding columns of C must be untouched"


def test_host_quick_returns():
    M, N, K = 70, 50, 30
    A, B, C = make_inputs(M, N, K, seed=5)
    hC = C.clone()
    nanA = torch.full((M, K), float("nan"))
    assert sg.sgemm_f32_host(M, N, K, 0.0, nanA, K, nanA, N, 2.0, hC, N) == 0
    torch.cuda.synchronize()
    assert torch.equal(hC, C * 2.0)
    hC = C.clone()
    assert sg.sgemm_f32_host(M, N, 0, 1.0, None, 1, None, N, 0.0, hC, N) == 0
    torch.cuda.synchronize()
    assert torch.equal(hC, torch.zeros_like(C))
    hC = C.clone()
    assert sg.sgemm_f32_host(M, N, K, 0.0, None, K, None, N, 1.0, hC, N) == 0
    assert torch.equal(hC, C)
    assert sg.sgemm_f32_host(-1, N, K, 1.0, A, K, B, N, 1.0, hC, N) == -1
    assert sg.sgemm_f32_host(M, N, K, 1.0, A, K - 1, B, N, 1.0, hC, N) == -6
