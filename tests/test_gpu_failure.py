"""Failure detection without a GPU fault: every mbarrier wait in the library's kernels is
bounded in time. The self-test waits, with the kernels' own wait, on a barrier phase that
nothing completes. The wait must give up after about a second, the kernel must end
normally, and the context must stay usable (a GEMM right after it meets the oracle bound
and leaves the status words clear)."""
import pytest
import torch

import oracle
from parity_util import assert_bound
from workloads import make_inputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dense_fp32_matrix_08_gb300 as sg


def test_bounded_wait_gives_up_and_context_survives():
    r = sg.sgemm_f32_wait_selftest()
    assert r["status"] == 0, r
    assert r["timed_out"] == 1, r
    assert 0.9 <= r["seconds"] <= 10.0, r
    M, N, K = 300, 260, 200
    A, B, C = make_inputs(M, N, K, seed=5)
    dC = C.cuda()
    assert sg.sgemm_f32(M, N, K, 1.0, A.cuda(), K, B.cuda(), N, 0.5, dC, N) == 0
    torch.cuda.synchronize()
    R, S = oracle.sgemm_f64(A, B, C, 1.0, 0.5)
    assert_bound(dC.cpu().numpy(), R, S, 0.5, C.numpy(), "after the self-test")
    assert sg.sgemm_f32_status() == (0, 0)
