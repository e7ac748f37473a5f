"""Stream order under programmatic dependent launch.

The GEMM and thin cluster kernels are launched so that a kernel's CTAs may start while the
previous kernel on the stream is still finishing; each waits for that kernel before it
touches global memory. These tests make every kind of dependence between consecutive calls
happen with no synchronisation in between, and require the results to be bitwise those of
the same calls run one at a time with the stream synchronised after each:
- read after write: each call's A is the previous call's C (a chain of products);
- write after read: a call overwrites, as its C, the B the previous call read;
- write after write: consecutive calls accumulate into the same C (beta != 0);
- the same chain captured into a CUDA graph and replayed.
Shapes cover the thin cluster kernel (16 rows), the mid-size plan (A^T copy, then the
GEMM with a split finished inside a cluster) and the large plan (A^T copy, GEMM with a
split tail, reduce kernel).
"""
import pytest
import torch

import dense_fp32_matrix_08_gb300 as sg

pytestmark = pytest.mark.gpu

# (M, N): chains need K == N so that an M x N result can be the next M x K operand
SHAPES = [(16, 1024), (1024, 1024), (2048, 2048)]


def _operands(M, N, steps, seed):
    g = torch.Generator().manual_seed(seed)
    A0 = torch.rand(M, N, generator=g) * 2 - 1
    Bs = [(torch.rand(N, N, generator=g) * 2 - 1) / N ** 0.5 for _ in range(steps)]
    Cs = [torch.randn(M, N, generator=g) for _ in range(steps)]
    return A0.cuda(), [b.cuda() for b in Bs], [c.cuda() for c in Cs]


def _chain(M, N, A0, Bs, C0s, beta, sync_each, stream):
    """C_i = X_i B_i + beta C0_i with X_0 = A0 and X_{i+1} = C_i; returns the C_i."""
    Cs = [c.clone() for c in C0s]
    torch.cuda.synchronize()
    x = A0
    with torch.cuda.stream(stream):
        for b, c in zip(Bs, Cs):
            rc = sg.sgemm_f32(M, N, N, 1.0, x, N, b, N, beta, c, N, stream=stream)
            assert rc == 0, rc
            if sync_each:
                stream.synchronize()
            x = c
    stream.synchronize()
    return Cs


@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_chain_reads_previous_output(M, N, beta):
    A0, Bs, C0s = _operands(M, N, 4, seed=M + N)
    st = torch.cuda.Stream()
    ref = _chain(M, N, A0, Bs, C0s, beta, True, st)
    got = _chain(M, N, A0, Bs, C0s, beta, False, st)
    for i, (r, g) in enumerate(zip(ref, got)):
        assert torch.isfinite(r).all()
        assert torch.equal(r, g), f"step {i}"
    assert sg.sgemm_f32_status() == (0, 0)


@pytest.mark.parametrize("M,N", SHAPES)
def test_overwrite_operand_of_previous_call(M, N):
    # call 1: C1 = A X; call 2: X = A2 B2 (writes the B that call 1 read); call 3: C3 = A X
    A0, Bs, C0s = _operands(M, N, 3, seed=7 * M + N)
    A2 = torch.rand(M, N, generator=torch.Generator().manual_seed(M)).cuda()
    st = torch.cuda.Stream()

    def run(sync_each):
        X = Bs[0].clone()
        C1, C3 = C0s[0].clone(), C0s[2].clone()
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            assert sg.sgemm_f32(M, N, N, 1.0, A0, N, X, N, 0.0, C1, N, stream=st) == 0
            if sync_each:
                st.synchronize()
            # X (N x N) is overwritten: its first M rows by an M x N product
            assert sg.sgemm_f32(M, N, N, 1.0, A2, N, Bs[1], N, 0.0, X, N, stream=st) == 0
            if sync_each:
                st.synchronize()
            assert sg.sgemm_f32(M, N, N, 1.0, A0, N, X, N, 0.5, C3, N, stream=st) == 0
        st.synchronize()
        return C1, C3, X

    ref = run(True)
    got = run(False)
    for name, r, g in zip(("C1", "C3", "X"), ref, got):
        assert torch.equal(r, g), name


@pytest.mark.parametrize("M,N", SHAPES)
def test_accumulate_into_same_output(M, N):
    A0, Bs, C0s = _operands(M, N, 4, seed=11 * M + N)
    st = torch.cuda.Stream()

    def run(sync_each):
        C = C0s[0].clone()
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            for b in Bs:
                assert sg.sgemm_f32(M, N, N, 0.25, A0, N, b, N, 1.0, C, N, stream=st) == 0
                if sync_each:
                    st.synchronize()
        st.synchronize()
        return C

    assert torch.equal(run(True), run(False))


@pytest.mark.parametrize("M,N", SHAPES)
def test_chain_in_graph(M, N):
    A0, Bs, C0s = _operands(M, N, 4, seed=13 * M + N)
    st = torch.cuda.Stream()
    ref = _chain(M, N, A0, Bs, C0s, 0.0, True, st)
    Cs = [torch.full_like(c, float("nan")) for c in C0s]
    with torch.cuda.stream(st):
        x = A0  # one eager pass first: the pool and the device set-up exist before capture
        for b, c in zip(Bs, Cs):
            assert sg.sgemm_f32(M, N, N, 1.0, x, N, b, N, 0.0, c, N, stream=st) == 0
            x = c
    st.synchronize()
    for c in Cs:
        c.fill_(float("nan"))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        x = A0
        for b, c in zip(Bs, Cs):
            assert sg.sgemm_f32(M, N, N, 1.0, x, N, b, N, 0.0, c, N, stream=st) == 0
            x = c
    for _ in range(2):
        for c in Cs:
            c.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for i, (r, c) in enumerate(zip(ref, Cs)):
            assert torch.equal(r, c), f"step {i}"
