"""GPU parity of the tensor-core 3xTF32 variant (sgemm_f32_3xtf32) against the CPU oracle,
with the same elementwise bound as the FFMA path: |C - R| <= 1e-4 (S + |beta c|).

The variant is reported separately; it must still meet the FP32 contract on every
configuration, and its device status word must stay 0 (no bounded wait gave up).
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import BY_NAME, make_inputs, workload_inputs
from parity_util import assert_bound, guard_intact, to_device_view

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dense_fp32_matrix_08_gb300 as sg


def _run_tc(A, B, C, alpha, beta, lda=None, ldb=None, ldc=None, offs=(0, 0, 0),
            fill_c=float("nan")):
    M, K = A.shape
    N = B.shape[1]
    dA, _ = to_device_view(A, lda, offs[0])
    dB, _ = to_device_view(B, ldb, offs[1])
    dC, bufC = to_device_view(C, ldc, offs[2], fill=fill_c)
    rc = sg.sgemm_f32_3xtf32(M, N, K, alpha, dA.data_ptr() if dA.numel() else 0,
                             max(dA.stride(0), 1), dB.data_ptr() if dB.numel() else 0,
                             max(dB.stride(0), 1), beta, dC.data_ptr() if dC.numel() else 0,
                             max(dC.stride(0), 1))
    assert rc == 0, f"sgemm_f32_3xtf32 returned {rc}"
    torch.cuda.synchronize()
    st = sg.sgemm_f32_3xtf32_status()
    assert st == (0, 0), f"device status {st}"
    return dC.cpu(), guard_intact(bufC, dC, fill_c)


SMALL = [(1, 1, 1), (5, 7, 9), (127, 129, 33), (128, 128, 32), (300, 260, 200),
         (129, 257, 1031), (16, 300, 96), (333, 16, 64)]


@pytest.mark.parametrize("shape", SMALL, ids=[f"{m}x{n}x{k}" for m, n, k in SMALL])
def test_tc_small(shape):
    M, N, K = shape
    A, B, C = make_inputs(M, N, K, seed=M + 3 * N + 7 * K)
    out, guard = _run_tc(A, B, C, 0.75, -1.25)
    assert guard
    R, S = oracle.sgemm_f64(A, B, C, 0.75, -1.25)
    assert_bound(out.numpy(), R, S, -1.25, C.numpy(), f"3xtf32 {shape}")


def test_tc_unaligned_views():
    M, N, K = 200, 150, 130
    A, B, C = make_inputs(M, N, K, seed=21)
    out, guard = _run_tc(A, B, C, 1.0, 0.5, K + 1, N + 3, N + 5, offs=(1, 3, 5))
    assert guard
    R, S = oracle.sgemm_f64(A, B, C, 1.0, 0.5)
    assert_bound(out.numpy(), R, S, 0.5, C.numpy(), "3xtf32 unaligned")


def test_tc_fp32_fidelity_exact():
    """A = 1 + 2^-15 is not a TF32 value: the hi/lo split must carry the 2^-15 part, so
    the exact FP32 result 256 + 2^-7 comes out (plain TF32 would give 256)."""
    M, N, K = 128, 128, 256
    A = torch.full((M, K), 1.0 + 2.0 ** -15)
    B = torch.ones((K, N))
    out, _ = _run_tc(A, B, torch.zeros((M, N)), 1.0, 0.0)
    assert torch.all(out == 256.0 + 2.0 ** -7)


def test_tc_beta_zero_and_quick_returns():
    A, B, _ = make_inputs(96, 80, 64, seed=22)
    out, _ = _run_tc(A, B, torch.full((96, 80), float("nan")), 2.0, 0.0)
    R, S = oracle.sgemm_f64(A, B, None, 2.0, 0.0)
    assert torch.isfinite(out).all()
    assert_bound(out.numpy(), R, S, 0.0, None, "3xtf32 beta=0")
    _, _, C = make_inputs(96, 80, 64, seed=23)
    out0, _ = _run_tc(torch.full((96, 64), float("nan")), torch.full((64, 80), float("nan")),
                      C, 0.0, 3.0)
    assert torch.equal(out0, C * 3.0)


@pytest.mark.parametrize("name", ["sgemm_256cube", "sgemm_1024cube",
                                  "sgemm_4099x3001x777_ragged", "sgemm_16x4096x4096_thin_m",
                                  "sgemm_4096x16x8192_thin_n"])
def test_tc_config_full(name):
    w = BY_NAME[name]
    A, B, C = workload_inputs(w)
    out, guard = _run_tc(A, B, C, w.alpha, w.beta)
    assert guard
    R, S = oracle.sgemm_f64(A, B, C, w.alpha, w.beta)
    assert_bound(out.numpy(), R, S, w.beta, C.numpy(), name)


@pytest.mark.parametrize("name", ["sgemm_4096cube", "sgemm_4097cube_unaligned",
                                  "sgemm_8192cube", "sgemm_8192x14336x4096"])
def test_tc_config_sampled(name):
    w = BY_NAME[name]
    A, B, C = workload_inputs(w)
    out, guard = _run_tc(A, B, C, w.alpha, w.beta, fill_c=0.0)
    assert guard
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([[0, w.M - 1, (w.M // 128) * 128 - 1],
                                     rng.integers(0, w.M, 24)]))
    rows = rows[(rows >= 0) & (rows < w.M)]
    R, S = oracle.sgemm_f64_rows(A, B, C, w.alpha, w.beta, rows)
    assert_bound(out.numpy()[rows], R, S, w.beta, C.numpy()[rows], name + " rows")
