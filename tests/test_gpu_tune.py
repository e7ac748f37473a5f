"""sgemm_f32_autotune on the GPU: it only reads C, records the fastest measured plan, and
later calls of sgemm_f32 / sgemm_f32_ex use that plan (bitwise the same result as forcing
it) and still meet the oracle bound."""
import pytest
import torch

import oracle
from workloads import make_inputs
from parity_util import assert_bound

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dense_fp32_matrix_08_gb300 as sg


@pytest.fixture(autouse=True)
def _empty_table():
    sg.sgemm_f32_tune_clear()
    yield
    sg.sgemm_f32_tune_clear()


@pytest.mark.parametrize("shape", [(700, 900, 300), (2048, 1536, 1024), (16, 2048, 2048)])
def test_autotune_records_and_is_used(shape, tmp_path):
    M, N, K = shape
    A, B, C = make_inputs(M, N, K, seed=M + N + K)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    res = sg.sgemm_f32_autotune(0, 0, M, N, K, 0.5, dA, K, dB, N, 2.0, dC, N, reps=2)
    torch.cuda.synchronize()
    assert res["status"] == 0 and 0 <= res["variant"] < sg.sgemm_f32_num_variants()
    assert res["ms"] > 0.0
    assert torch.equal(dC.cpu(), C), "autotune must not modify C"
    assert sg.sgemm_f32_tune_count() == 1
    plan = sg.sgemm_f32_plan(M, N, K, K, N, N, 0.5, 2.0, 0)
    assert plan["variant"] == res["variant"]  # the planner now reports the tuned plan

    out_auto = C.cuda()
    assert sg.sgemm_f32(M, N, K, 0.5, dA, K, dB, N, 2.0, out_auto, N) == 0
    out_forced = C.cuda()
    assert sg.sgemm_f32_forced(M, N, K, 0.5, dA, K, dB, N, 2.0, out_forced, N,
                               res["variant"], res["split"]) == 0
    torch.cuda.synchronize()
    assert torch.equal(out_auto, out_forced)
    R, S = oracle.sgemm_f64(A, B, C, 0.5, 2.0)
    assert_bound(out_auto.cpu().numpy(), R, S, 2.0, C.numpy(), f"tuned {shape}")

    # the file round trip reproduces the same plan
    path = tmp_path / "tuned.txt"
    assert sg.sgemm_f32_tune_save(path) == 1
    sg.sgemm_f32_tune_clear()
    assert sg.sgemm_f32_tune_load(path) == 1
    assert sg.sgemm_f32_plan(M, N, K, K, N, N, 0.5, 2.0, 0)["variant"] == res["variant"]


def test_autotune_transposed_operands():
    M, N, K = 640, 768, 512
    opA, opB, C = make_inputs(M, N, K, seed=77)
    At, Bt = opA.t().contiguous().cuda(), opB.t().contiguous().cuda()  # stored K x M, N x K
    dC = C.cuda()
    res = sg.sgemm_f32_autotune(1, 1, M, N, K, 1.0, At, M, Bt, K, -1.0, dC, N)
    assert res["status"] == 0 and res["variant"] >= 0
    out = C.cuda()
    assert sg.sgemm_f32_ex(1, 1, M, N, K, 1.0, At, M, Bt, K, -1.0, out, N) == 0
    torch.cuda.synchronize()
    R, S = oracle.sgemm_f64(opA, opB, C, 1.0, -1.0)
    assert_bound(out.cpu().numpy(), R, S, -1.0, C.numpy(), "tuned transposed")


def test_autotune_quick_returns_and_errors():
    dA = torch.zeros((8, 8), device="cuda")
    r = sg.sgemm_f32_autotune(0, 0, 8, 8, 8, 0.0, dA, 8, dA, 8, 1.0, dA, 8)
    assert r == {"status": 0, "variant": -1, "split": 0, "ms": 0.0}
    # sgemm_f32_ex numbering: M is argument 3
    assert sg.sgemm_f32_autotune(0, 0, -1, 8, 8, 1.0, dA, 8, dA, 8, 1.0, dA, 8)["status"] == -3
    assert sg.sgemm_f32_tune_count() == 0
