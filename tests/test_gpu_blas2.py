"""GPU parity of SGEMV and SDOT (sgemv_f32, sdot_f32) against the CPU oracle.

Both are special cases of the oracle's GEMM: y = alpha op(A) x + beta y is a GEMM with one
column (B = x as a K x 1 matrix, C = y as M x 1), and x . y is a 1 x 1 GEMM. Strided vectors
are gathered on the host (a copy, not arithmetic) before the oracle sees them. The bound is
the usual |r - R| <= 1e-4 (S + |beta c|).
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_bound

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dense_fp32_matrix_08_gb300 as sg


def _strided(v: np.ndarray, inc: int, fill=np.nan):
    """Device buffer holding v with element stride inc (BLAS order for negative inc)."""
    n = v.size
    buf = np.full(max(1, 1 + (n - 1) * abs(inc)) + 3, fill, np.float32)
    idx = np.arange(n) * abs(inc)
    buf[idx if inc > 0 else idx[::-1]] = v
    return torch.from_numpy(buf).cuda(), idx if inc > 0 else idx[::-1]


GEMV = [(1, 1), (7, 13), (1000, 37), (37, 1000), (513, 1031), (16, 8195), (4096, 16)]


@pytest.mark.parametrize("trans", [0, 1])
@pytest.mark.parametrize("incs", [(1, 1), (2, -3), (-1, 2)])
@pytest.mark.parametrize("aligned", [True, False])
def test_sgemv(trans, incs, aligned):
    incx, incy = incs
    rng = np.random.default_rng(7 + trans)
    for (M, N) in GEMV:
        A = rng.standard_normal((M, N)).astype(np.float32)
        xlen, ylen = (M, N) if trans else (N, M)
        x = rng.standard_normal(xlen).astype(np.float32)
        y = rng.standard_normal(ylen).astype(np.float32)
        lda = N if aligned else N + 1
        off = 0 if aligned else 1
        bufA = torch.full((M * lda + off + 4,), float("nan"), device="cuda")
        dA = bufA.as_strided((M, N), (lda, 1), off)
        dA.copy_(torch.from_numpy(A).cuda())
        dx, _ = _strided(x, incx)
        dy, yidx = _strided(y, incy)
        rc = sg.sgemv_f32(trans, M, N, 0.5, dA, lda, dx, incx, -2.0, dy, incy)
        assert rc == 0
        torch.cuda.synchronize()
        out = dy.cpu().numpy()[yidx]
        opA = A.T.copy() if trans else A
        R, S = oracle.sgemm_f64(opA, x.reshape(-1, 1), y.reshape(-1, 1), 0.5, -2.0)
        assert_bound(out.reshape(-1, 1), R, S, -2.0, y.reshape(-1, 1),
                     f"sgemv T{trans} {M}x{N} inc{incs}")
        # untouched gaps between strided y elements
        rest = np.delete(dy.cpu().numpy(), yidx)
        assert np.all(np.isnan(rest))


def test_sgemv_alpha_zero_does_not_read():
    M, N = 50, 40
    dA = torch.full((M, N), float("nan"), device="cuda")
    dx = torch.full((N,), float("nan"), device="cuda")
    y = torch.arange(M, dtype=torch.float32, device="cuda")
    assert sg.sgemv_f32(0, M, N, 0.0, dA, N, dx, 1, 3.0, y, 1) == 0
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), torch.arange(M, dtype=torch.float32) * 3.0)


@pytest.mark.parametrize("n", [0, 1, 5, 1000, 1 << 20, (1 << 22) + 3])
@pytest.mark.parametrize("incs", [(1, 1), (3, -2)])
def test_sdot(n, incs):
    incx, incy = incs
    rng = np.random.default_rng(n + 11)
    x = rng.standard_normal(n).astype(np.float32)
    y = rng.standard_normal(n).astype(np.float32)
    dx, _ = _strided(x, incx)
    dy, _ = _strided(y, incy)
    res = torch.full((1,), float("nan"), device="cuda")
    assert sg.sdot_f32(n, dx, incx, dy, incy, res) == 0
    torch.cuda.synchronize()
    if n == 0:
        assert res.item() == 0.0
        return
    R, S = oracle.sgemm_f64(x.reshape(1, -1), y.reshape(-1, 1), None, 1.0, 0.0)
    assert_bound(res.cpu().numpy().reshape(1, 1), R, S, 0.0, None, f"sdot n={n} {incs}")


def test_sdot_deterministic():
    n = (1 << 24) + 7
    x = torch.randn(n, device="cuda")
    y = torch.randn(n, device="cuda")
    r1 = torch.empty(1, device="cuda")
    r2 = torch.empty(1, device="cuda")
    assert sg.sdot_f32(n, x, 1, y, 1, r1) == 0
    assert sg.sdot_f32(n, x, 1, y, 1, r2) == 0
    torch.cuda.synchronize()
    assert torch.equal(r1, r2)
