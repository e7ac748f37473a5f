"""CUDA-graph capture: sgemm_f32 (TMA-fed with an A^T copy and a split last wave, the thin-M
kernel with its reduce, an unaligned problem with aligned copies) and sgemm_f32_host (two
copy streams joined by events) are captured with stream capture and replayed; every replay
must give the oracle's result (the captured workspace allocations are graph memory nodes)."""
import pytest
import torch

import oracle
from workloads import make_inputs
from parity_util import assert_bound

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dense_fp32_matrix_08_gb300 as sg


@pytest.mark.parametrize("shape", [(2048, 1536, 1024), (16, 4096, 4096), (1001, 999, 997)])
def test_capture_and_replay_sgemm_f32(shape):
    M, N, K = shape
    A, B, C = make_inputs(M, N, K, seed=M + K)
    dA, dB = A.cuda(), B.cuda()
    dC = torch.empty((M, N), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # first call outside capture: one-time setup
        assert sg.sgemm_f32(M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N, stream=s) == 0
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rc = sg.sgemm_f32(M, N, K, 0.5, dA, K, dB, N, 0.0, dC, N, stream=s)
    assert rc == 0
    R, S = oracle.sgemm_f64(A, B, None, 0.5, 0.0)
    for it in range(3):
        dC.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_bound(dC.cpu().numpy(), R, S, 0.0, None, f"graph replay {it} {shape}")
    dB.mul_(2.0)  # replays read the current operands
    g.replay()
    torch.cuda.synchronize()
    R2, S2 = oracle.sgemm_f64(A, B * 2.0, None, 0.5, 0.0)
    assert_bound(dC.cpu().numpy(), R2, S2, 0.0, None, f"graph replay, new B {shape}")


def test_capture_and_replay_host_entry():
    M, N, K = 4500, 300, 200  # two row blocks: both copy streams take part
    A, B, C = make_inputs(M, N, K, seed=91)
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.zeros((M, N)).pin_memory()
    s = torch.cuda.Stream()
    assert sg.sgemm_f32_host(M, N, K, 1.0, hA, K, hB, N, 0.0, hC, N, s) == 0
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rc = sg.sgemm_f32_host(M, N, K, 2.0, hA, K, hB, N, 0.0, hC, N, s)
    assert rc == 0
    R, S = oracle.sgemm_f64(A, B, None, 2.0, 0.0)
    for it in range(2):
        hC.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_bound(hC.numpy(), R, S, 0.0, None, f"host graph replay {it}")
