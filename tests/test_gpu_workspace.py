"""The library's workspace pool: what a call keeps, and sgemm_f32_release_workspace.

sgemm_f32 takes its workspace (the transposed copy of A that the k-major plans read, aligned
operand copies, split-K partial tiles) from a stream-ordered pool of the library's own,
which keeps freed memory for reuse. These tests check that the pool really holds a large
plan's workspace after the call, that the release entry point hands it back (and reports
how much), that a second release finds nothing, and that calls after a release still give
the same, correct result.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_bound
from workloads import make_inputs

pytestmark = pytest.mark.gpu


def test_release_returns_the_pool_memory():
    import dense_fp32_matrix_08_gb300 as sg

    M = N = K = 4096
    plan = sg.sgemm_f32_plan(M, N, K, K, N, N, 1.0, 0.5, 0)
    assert plan["status"] == 0
    assert plan["ws_bytes"] >= 4 * M * K, "the automatic plan reads a transposed copy of A"
    A, B, C = make_inputs(M, N, K, seed=61)
    dA, dB = A.cuda(), B.cuda()
    first = C.cuda()
    assert sg.sgemm_f32(M, N, K, 1.0, dA, K, dB, N, 0.5, first, N) == 0
    torch.cuda.synchronize()

    rc, released = sg.sgemm_f32_release_workspace()
    assert rc == 0
    assert released >= plan["ws_bytes"], (released, plan["ws_bytes"])
    rc, again = sg.sgemm_f32_release_workspace()
    assert rc == 0 and again == 0

    # the pool grows again for the next call; the result is bitwise the first call's
    second = C.cuda()
    assert sg.sgemm_f32(M, N, K, 1.0, dA, K, dB, N, 0.5, second, N) == 0
    torch.cuda.synchronize()
    assert torch.equal(first, second)
    rows = np.array([0, 1, 2047, M - 1])
    R, S = oracle.sgemm_f64_rows(A, B, C, 1.0, 0.5, rows)
    assert_bound(second.cpu().numpy()[rows], R, S, 0.5, C.numpy()[rows], "after release")
    rc, released = sg.sgemm_f32_release_workspace()
    assert rc == 0 and released >= plan["ws_bytes"]
    assert sg.sgemm_f32_status() == (0, 0)


def test_release_with_nothing_held():
    import dense_fp32_matrix_08_gb300 as sg

    assert sg.sgemm_f32_release_workspace()[0] == 0
    rc, released = sg.sgemm_f32_release_workspace()
    assert rc == 0 and released == 0


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (2100, 2600, 300), (16, 4096, 4096)])
def test_minimal_workspace_runs_the_twin(M, N, K):
    """sgemm_f32_ws with the workspace sgemm_f32_workspace_size_min reports: the plan
    without its A^T copy (split-K partial tiles only), run by the twin configuration that
    transposes A in shared memory, bitwise the same as sgemm_f32; one byte less is refused
    (-13) without touching C. Plans without an A^T copy need the same size either way."""
    import dense_fp32_matrix_08_gb300 as sg

    rc, full = sg.sgemm_f32_workspace_size(M, N, K, K, N, N)
    assert rc == 0
    rc, small = sg.sgemm_f32_workspace_size_min(M, N, K, K, N, N)
    assert rc == 0 and small <= full
    plan = sg.sgemm_f32_plan(M, N, K, K, N, N, 1.0, 1.0, 0)
    if plan["variant"] in (35, 36, 39, 40):
        at_copy = -(-4 * K * (-(-M // 4) * 4) // 256) * 256
        assert full - small == at_copy
    else:
        assert small == full
    A, B, C = make_inputs(M, N, K, seed=M + 7)
    dA, dB = A.cuda(), B.cuda()
    ref = C.cuda()
    assert sg.sgemm_f32(M, N, K, 1.0, dA, K, dB, N, 1.0, ref, N) == 0
    ws = torch.empty(max(small, 16), dtype=torch.uint8, device="cuda")
    out = C.cuda()
    assert sg.sgemm_f32_ws(M, N, K, 1.0, dA, K, dB, N, 1.0, out, N, ws.data_ptr(), small) == 0
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    if small > 0:
        before = C.cuda()
        rc = sg.sgemm_f32_ws(M, N, K, 1.0, dA, K, dB, N, 1.0, before, N, ws.data_ptr(),
                             small - 1)
        torch.cuda.synchronize()
        assert rc == -13
        assert torch.equal(before.cpu(), C)
    rows = np.array([0, M // 2, M - 1])
    R, S = oracle.sgemm_f64_rows(A, B, C, 1.0, 1.0, rows)
    assert_bound(out.cpu().numpy()[rows], R, S, 1.0, C.numpy()[rows], "minimal workspace")
