"""GPU parity of the transposed-operand (sgemm_f32_ex) and column-major (sgemm_f32_colmajor)
entry points against the CPU oracle.

The oracle computes the plain row-major product; the tests materialise op(A) and op(B) on
the host (a transpose is a copy, not arithmetic) and compare elementwise with the bound
|C - R| <= 1e-4 (S + |beta c|).
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_inputs
from parity_util import assert_bound, guard_intact, to_device_view

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dense_fp32_matrix_08_gb300 as sg

# (M, N, K): thin M, thin N, small, larger than one tile in every dimension
SHAPES = [(16, 300, 257), (300, 16, 129), (61, 70, 50), (700, 900, 300), (1, 1, 1),
          (129, 257, 33)]


def _stored(x: torch.Tensor, trans: int) -> torch.Tensor:
    """The stored matrix whose op() is x."""
    return x.t().contiguous() if trans else x


@pytest.mark.parametrize("transa", [0, 1])
@pytest.mark.parametrize("transb", [0, 1])
@pytest.mark.parametrize("aligned", [True, False])
def test_ex_against_oracle(transa, transb, aligned):
    for (M, N, K) in SHAPES:
        opA, opB, C = make_inputs(M, N, K, seed=M + 5 * N + 11 * K + 3 * transa + transb)
        As, Bs = _stored(opA, transa), _stored(opB, transb)
        if aligned:
            lds, offs = (None, None, None), (0, 0, 0)
        else:  # odd leading dimensions and element offsets: 4-byte copy paths
            lds = (As.shape[1] + 1, Bs.shape[1] + 3, N + 5)
            offs = (1, 3, 5)
        dA, _ = to_device_view(As, lds[0], offs[0])
        dB, _ = to_device_view(Bs, lds[1], offs[1])
        dC, bufC = to_device_view(C, lds[2], offs[2])
        rc = sg.sgemm_f32_ex(transa, transb, M, N, K, 0.75, dA, dA.stride(0), dB, dB.stride(0),
                             -1.5, dC, dC.stride(0))
        assert rc == 0
        torch.cuda.synchronize()
        assert guard_intact(bufC, dC)
        R, S = oracle.sgemm_f64(opA, opB, C, 0.75, -1.5)
        assert_bound(dC.cpu().numpy(), R, S, -1.5, C.numpy(),
                     f"ex T{transa}{transb} {M, N, K} aligned={aligned}")


def test_ex_no_transpose_is_sgemm_f32():
    M, N, K = 333, 444, 555
    A, B, C = make_inputs(M, N, K, seed=31)
    dA, dB = A.cuda(), B.cuda()
    c1, c2 = C.cuda(), C.cuda()
    assert sg.sgemm_f32(M, N, K, 1.0, dA, K, dB, N, 0.5, c1, N) == 0
    assert sg.sgemm_f32_ex(0, 0, M, N, K, 1.0, dA, K, dB, N, 0.5, c2, N) == 0
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


def test_colmajor_swap_trick_golden():
    """The swap trick of "Lecture 4 - GPU Acceleration", section 5.4: for row-major A
    (M x K), B (K x N), the column-major call sgemm('N','N', m=N, n=M, k=K, B, ldb=N, A,
    lda=K, C, ldc=N) leaves the row-major A B in C. Our column-major entry point must give
    exactly what the row-major entry point gives; the call without the swap computes a
    different product."""
    M, N, K = 96, 80, 64
    A, B, C0 = make_inputs(M, N, K, seed=32)
    dA, dB = A.cuda(), B.cuda()
    row = torch.zeros((M, N), device="cuda")
    assert sg.sgemm_f32(M, N, K, 1.0, dA, K, dB, N, 0.0, row, N) == 0
    swapped = torch.zeros((M, N), device="cuda")
    assert sg.sgemm_f32_colmajor(0, 0, N, M, K, 1.0, dB, N, dA, K, 0.0, swapped, N) == 0
    torch.cuda.synchronize()
    assert torch.equal(row, swapped)
    R, S = oracle.sgemm_f64(A, B, None, 1.0, 0.0)
    assert_bound(swapped.cpu().numpy(), R, S, 0.0, None, "swap trick")
    # without the swap (square case so that the call is legal): a different matrix
    Aq, Bq, _ = make_inputs(64, 64, 64, seed=33)
    wrong = torch.zeros((64, 64), device="cuda")
    assert sg.sgemm_f32_colmajor(0, 0, 64, 64, 64, 1.0, Aq.cuda(), 64, Bq.cuda(), 64, 0.0,
                                 wrong, 64) == 0
    torch.cuda.synchronize()
    Rq, _ = oracle.sgemm_f64(Aq, Bq, None, 1.0, 0.0)
    assert np.max(np.abs(wrong.cpu().numpy() - Rq)) > 1.0


@pytest.mark.parametrize("transa", [0, 1])
@pytest.mark.parametrize("transb", [0, 1])
def test_colmajor_against_oracle(transa, transb):
    """Column-major operands (Fortran order): A_cm is m x k (or k x m), B_cm k x n (or
    n x k), C_cm m x n, each stored column by column with ld = its row count + padding."""
    m, n, k = 150, 130, 70
    opA, opB, C = make_inputs(m, n, k, seed=34 + 2 * transa + transb)
    A_cm = opA.numpy().T if transa else opA.numpy()   # the column-major matrix as 2-D
    B_cm = opB.numpy().T if transb else opB.numpy()

    def colmajor_buffer(x, pad):
        rows, cols = x.shape
        ld = rows + pad
        buf = np.full((cols, ld), np.nan, np.float32)  # row c of buf = column c of x
        buf[:, :rows] = x.T
        return torch.from_numpy(buf).cuda(), ld

    dA, lda = colmajor_buffer(A_cm, 3)
    dB, ldb = colmajor_buffer(B_cm, 1)
    dC, ldc = colmajor_buffer(C.numpy(), 2)
    rc = sg.sgemm_f32_colmajor(transa, transb, m, n, k, 2.0, dA, lda, dB, ldb, 0.25, dC, ldc)
    assert rc == 0
    torch.cuda.synchronize()
    out = dC.cpu().numpy()[:, :m].T  # back to m x n
    assert np.all(np.isnan(dC.cpu().numpy()[:, m:]))  # padding rows untouched
    R, S = oracle.sgemm_f64(opA, opB, C, 2.0, 0.25)
    assert_bound(out, R, S, 0.25, C.numpy(), f"colmajor T{transa}{transb}")


@pytest.mark.parametrize("variant", [35, 36])
def test_k_major_tma_reads_transposed_a_directly(variant):
    """With op(A) = A_st^T and A_st aligned, the k-major TMA-fed configurations read A_st as
    the A^T they need (no copy): parity, and the same result bits as their row-major run."""
    M, N, K = 700, 520, 300
    opA, opB, C = make_inputs(M, N, K, seed=variant)
    At = opA.t().contiguous()
    dC1, dC2 = C.cuda(), C.cuda()
    assert sg.sgemm_f32_ex_forced(1, 0, M, N, K, 1.0, At.cuda(), M, opB.cuda(), N, 0.5, dC1, N,
                                  variant, 0) == 0
    assert sg.sgemm_f32_forced(M, N, K, 1.0, opA.cuda(), K, opB.cuda(), N, 0.5, dC2, N,
                               variant, 0) == 0
    torch.cuda.synchronize()
    assert torch.equal(dC1, dC2)
    R, S = oracle.sgemm_f64(opA, opB, C, 1.0, 0.5)
    assert_bound(dC1.cpu().numpy(), R, S, 0.5, C.numpy(), f"A^T direct v{variant}")
    # no path for a transposed B
    assert sg.sgemm_f32_ex_forced(1, 1, M, N, K, 1.0, At.cuda(), M, opB.t().contiguous().cuda(),
                                  K, 0.5, dC1, N, variant, 0) == -14
