"""Concurrent calls: several host threads, each on its own stream, call sgemm_f32 at once
(TMA-fed, split-K and thin plans: the shared workspace pool, the per-thread plan cache and
the device status word). Every result must meet the oracle bound, and the status word must
stay 0."""
import threading

import pytest
import torch

import oracle
from workloads import make_inputs
from parity_util import assert_bound

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dense_fp32_matrix_08_gb300 as sg

SHAPES = [(1024, 1024, 1024), (16, 2048, 2048), (2048, 768, 512), (777, 555, 333),
          (3000, 16, 2000), (4097, 300, 129)]


def test_threads_on_separate_streams():
    sg.sgemm_f32_status()  # clear
    inputs = [make_inputs(M, N, K, seed=i + 50) for i, (M, N, K) in enumerate(SHAPES)]
    outs = [None] * len(SHAPES)
    errors = []

    def worker(i):
        try:
            M, N, K = SHAPES[i]
            A, B, C = inputs[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
                s.synchronize()
                for _ in range(4):  # C = 0.5 A B + 0 C, idempotent
                    rc = sg.sgemm_f32(M, N, K, 0.5, dA, K, dB, N, 0.0, dC, N, stream=s)
                    if rc != 0:
                        errors.append((i, rc))
                s.synchronize()
                outs[i] = dC.cpu()
        except Exception as e:  # surfaced below
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(SHAPES))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, (M, N, K) in enumerate(SHAPES):
        A, B, _ = inputs[i]
        R, S = oracle.sgemm_f64(A, B, None, 0.5, 0.0)
        assert_bound(outs[i].numpy(), R, S, 0.0, None, f"thread {i} {SHAPES[i]}")
    assert sg.sgemm_f32_status() == (0, 0)
