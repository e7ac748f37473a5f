"""sgemm_f32_noalloc: the entry point for callers that may not allocate device memory.

Some callers cannot call cudaMalloc: code inside a host framework that owns all device
memory (a plugin of an inference runtime, for example) and loops that forbid allocation
after start-up. For them the library's split-K workspace lives in a fixed per-device scratch
array instead. These tests call that entry point through the C ABI on problems whose plan
really uses the scratch, twice in a row (the second call finds the first call's leftovers in
the array), and compare each result with sgemm_f32's, within the same elementwise bound the
parity tests use. They also check that a problem needing more scratch than the array holds
is refused with the documented error, without touching C.

This file is named to be collected last, so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import os
import re

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_bound
from workloads import make_inputs

pytestmark = pytest.mark.gpu

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "sgemm_f32.h")


def _header_int(name):
    text = open(HEADER).read()
    m = re.search(rf"#define\s+{name}\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    if m:
        return int(m.group(1)) << int(m.group(2))
    m = re.search(rf"#define\s+{name}\s+\((-?\d+)\)", text)
    return int(m.group(1))


SCRATCH_BYTES = _header_int("SGEMM_F32_NOALLOC_SCRATCH_BYTES")
ERR_TOO_SMALL = _header_int("SGEMM_F32_ERR_SCRATCH_TOO_SMALL")


@pytest.mark.parametrize("M,N,K,alpha,beta,seed", [
    # thin M with an A that TMA cannot address (lda = 4099): the cluster kernel reads an
    # aligned copy of A made in the scratch
    (16, 4096, 4099, 1.0, 1.0, 41),
    (2100, 2600, 300, 1.5, 0.5, 42),    # whole waves plus a split last wave
    (4096, 18, 2048, -0.75, 0.0, 43),   # thin N, ldb = 18: an aligned copy of B; beta = 0
])
def test_noalloc_matches_sgemm_f32_twice(M, N, K, alpha, beta, seed):
    import dense_fp32_matrix_08_gb300 as sg

    plan = sg.sgemm_f32_plan(M, N, K, K, N, N, alpha, beta, 0)
    assert plan["status"] == 0
    assert 0 < plan["ws_bytes"] <= SCRATCH_BYTES, "case must use, and fit, the scratch"
    A, B, C = make_inputs(M, N, K, seed=seed)
    dA, dB = A.cuda(), B.cuda()
    ref = C.cuda()
    assert sg.sgemm_f32(M, N, K, alpha, dA, K, dB, N, beta, ref, N) == 0
    torch.cuda.synchronize()
    ref = ref.cpu()
    R, S = oracle.sgemm_f64(A, B, C, alpha, beta)
    tol_S = S
    for call in range(2):
        dC = C.cuda()
        assert sg.sgemm_f32_noalloc(M, N, K, alpha, dA, K, dB, N, beta, dC, N) == 0
        torch.cuda.synchronize()
        out = dC.cpu()
        # the same plan and kernels as sgemm_f32, whatever the scratch held before ...
        assert torch.equal(out, ref), f"noalloc call {call} is not bitwise sgemm_f32's"
        # ... within the parity tests' bound of the existing entry point ...
        assert_bound(out.numpy(), ref.numpy().astype(np.float64), tol_S, beta, C.numpy(),
                     f"noalloc call {call} vs sgemm_f32")
        # ... and against the oracle
        assert_bound(out.numpy(), R, S, beta, C.numpy(), f"noalloc call {call} vs oracle")


def test_noalloc_refuses_problems_beyond_the_scratch():
    import dense_fp32_matrix_08_gb300 as sg

    # Odd leading dimensions: the plan's aligned operand copies cannot be dropped (only an
    # A^T copy has a shared-memory twin), so a large enough problem exceeds the scratch.
    big = None
    for n in (3001, 3201, 3601, 4001, 6001):
        p = sg.sgemm_f32_plan(n, n, n, n, n, n, 1.0, 1.0, 0)
        if p["ws_bytes"] > SCRATCH_BYTES:
            big = n
            break
    if big is None:
        pytest.skip("no candidate shape needs more scratch than the array on this device")
    n = big
    A = torch.zeros((n, n), device="cuda")
    B = torch.zeros((n, n), device="cuda")
    C = torch.full((n, n), 7.0, device="cuda")
    assert sg.sgemm_f32_noalloc(n, n, n, 1.0, A, n, B, n, 1.0, C, n) == ERR_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((C == 7.0).all())


def test_noalloc_without_scratch_need():
    """A plan without split-K runs without touching the scratch at all."""
    import dense_fp32_matrix_08_gb300 as sg

    M, N, K = 2432, 2432, 64  # short K: whole tiles, no split-K, no pre-pass copy
    p = sg.sgemm_f32_plan(M, N, K, K, N, N, 1.0, 0.0, 0)
    if p["ws_bytes"] != 0:
        pytest.skip("plan on this device uses split-K for this shape")
    A, B, C = make_inputs(M, N, K, seed=44)
    dC = C.cuda()
    assert sg.sgemm_f32_noalloc(M, N, K, 1.0, A.cuda(), K, B.cuda(), N, 0.0, dC, N) == 0
    torch.cuda.synchronize()
    R, S = oracle.sgemm_f64(A, B, None, 1.0, 0.0)
    assert_bound(dC.cpu().numpy(), R, S, 0.0, None, "noalloc small")


def test_noalloc_twin_is_bitwise_sgemm_f32():
    """A large aligned problem whose plan reads a transposed copy of A (more workspace than
    the scratch) runs through the twin configuration that transposes A in shared memory:
    the same tiles, slices and k order, so the result is bitwise sgemm_f32's."""
    import dense_fp32_matrix_08_gb300 as sg

    n = 3072
    p = sg.sgemm_f32_plan(n, n, n, n, n, n, 1.0, 0.5, 0)
    if p["ws_bytes"] <= SCRATCH_BYTES:
        pytest.skip("the plan for this shape fits the scratch on this device")
    A, B, C = make_inputs(n, n, n, seed=45)
    dA, dB = A.cuda(), B.cuda()
    ref = C.cuda()
    out = C.cuda()
    assert sg.sgemm_f32(n, n, n, 1.0, dA, n, dB, n, 0.5, ref, n) == 0
    assert sg.sgemm_f32_noalloc(n, n, n, 1.0, dA, n, dB, n, 0.5, out, n) == 0
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    rows = np.array([0, 1, 1535, n - 1])
    R, S = oracle.sgemm_f64_rows(A, B, C, 1.0, 0.5, rows)
    assert_bound(out.cpu().numpy()[rows], R, S, 0.5, C.numpy()[rows], "noalloc twin")
