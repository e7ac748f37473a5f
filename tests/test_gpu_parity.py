"""GPU parity: the CUDA path (through the C ABI) against the CPU FP64 oracle.

Every comparison is elementwise with the bound |C_gpu - R| <= 1e-4 (S + |beta c|) (see
parity_util). Problems the oracle finishes in seconds are checked on every element; the
full-size configurations are checked on sampled rows (first, last and random ones, so
every ragged tile edge is included) plus random single elements, in the same launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import BY_NAME, CONFIGS, make_inputs, workload_inputs
from parity_util import assert_bound, guard_intact, to_device_view

pytestmark = pytest.mark.gpu
NUM_VARIANTS = 46  # tile configurations in the table; checked against the library below
# configurations kept in the table but not compiled (forcing one returns -14)
RETIRED = (6, 7, 9, 10, 11, 12, 14, 15, 17, 18, 19, 20, 22, 23, 24, 25)
BUILT = tuple(v for v in range(NUM_VARIANTS) if v not in RETIRED)
TMA_VARIANTS = (26, 30, 31, 32, 35, 36, 37, 38, 39, 40, 45)  # every TMA-fed instance
KPAIR_VARIANTS = (27, 28, 29)  # K-paired TMA-fed kernel: aligned A, any B (copied to B^T)
THIN_M, THIN_N = 33, 34  # streaming kernels for thin products
THIN_M_TMA = 41  # TMA-fed thin-M: B must be TMA-addressable
THIN_N_TMA = 42  # TMA-fed thin-N: A must be TMA-addressable
THIN_M_CL, THIN_N_CL = 43, 44  # cluster thin kernels: the streamed operand TMA-addressable
TMA_THIN = (THIN_M_TMA, THIN_N_TMA, THIN_M_CL, THIN_N_CL)

if torch.cuda.is_available():
    import dense_fp32_matrix_08_gb300 as sg


def _run(A, B, C, alpha, beta, lda=None, ldb=None, ldc=None, offs=(0, 0, 0), variant=-1,
         split=0, fill_c=float("nan")):
    """Upload, run sgemm_f32 (or the forced plan), download. Returns (C_out, guard_ok)."""
    M, K = A.shape
    N = B.shape[1]
    dA, _ = to_device_view(A, lda, offs[0])
    dB, _ = to_device_view(B, ldb, offs[1])
    dC, bufC = to_device_view(C, ldc, offs[2], fill=fill_c)
    if variant >= 0 or split > 0:
        rc = sg.sgemm_f32_forced(M, N, K, alpha, dA.data_ptr() if dA.numel() else 0,
                                 max(dA.stride(0), 1), dB.data_ptr() if dB.numel() else 0,
                                 max(dB.stride(0), 1), beta,
                                 dC.data_ptr() if dC.numel() else 0, max(dC.stride(0), 1),
                                 variant, split)
    else:
        rc = sg.sgemm_f32(M, N, K, alpha, dA.data_ptr() if dA.numel() else 0,
                          max(dA.stride(0), 1), dB.data_ptr() if dB.numel() else 0,
                          max(dB.stride(0), 1), beta, dC.data_ptr() if dC.numel() else 0,
                          max(dC.stride(0), 1))
    assert rc == 0, f"sgemm returned {rc}"
    torch.cuda.synchronize()
    return dC.cpu(), guard_intact(bufC, dC, fill_c)


# --------------------------------------------------------------------------------------
# The benchmark configurations.

SMALL = ["sgemm_256cube", "sgemm_1024cube", "sgemm_4099x3001x777_ragged",
         "sgemm_16x4096x4096_thin_m", "sgemm_4096x16x8192_thin_n"]
LARGE = ["sgemm_4096cube", "sgemm_4097cube_unaligned", "sgemm_8192cube",
         "sgemm_8192x14336x4096"]


@pytest.mark.parametrize("name", SMALL)
def test_config_full(name):
    w = BY_NAME[name]
    A, B, C = workload_inputs(w)
    out, guard = _run(A, B, C, w.alpha, w.beta)
    assert guard, "wrote outside the C view"
    R, S = oracle.sgemm_f64(A, B, C, w.alpha, w.beta)
    assert_bound(out.numpy(), R, S, w.beta, C.numpy(), name)


def _sample_rows(M, BMs=(16, 64, 128, 256), n_random=24, seed=0):
    rows = {0, 1, M - 2, M - 1}
    for bm in BMs:  # last full tile row and the ragged tail of every tile height
        t = (M // bm) * bm
        rows.update(r for r in (t - 1, t, t + 1) if 0 <= r < M)
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, M, n_random).tolist())
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", LARGE)
def test_config_sampled(name):
    w = BY_NAME[name]
    A, B, C = workload_inputs(w)
    out, guard = _run(A, B, C, w.alpha, w.beta, fill_c=0.0)
    assert guard
    rows = _sample_rows(w.M)
    R, S = oracle.sgemm_f64_rows(A, B, C, w.alpha, w.beta, rows)
    assert_bound(out.numpy()[rows], R, S, w.beta, C.numpy()[rows], name + " rows")
    rng = np.random.default_rng(1)
    ii = rng.integers(0, w.M, 4000)
    jj = rng.integers(0, w.N, 4000)
    Re, Se = oracle.sgemm_f64_entries(A, B, C, w.alpha, w.beta, ii, jj)
    assert_bound(out.numpy()[ii, jj], Re, Se, w.beta, C.numpy()[ii, jj], name + " entries")


# --------------------------------------------------------------------------------------
# Every variant, aligned and unaligned, with and without split-K, across ragged tiles.

def _variants():
    """Every compiled configuration (retired ones are refused, see test_retired_variant_is_refused)."""
    return [v for v in range(sg.sgemm_f32_num_variants()) if v not in RETIRED] \
        if torch.cuda.is_available() else []


RAGGED = [(1, 1, 1), (3, 5, 7), (17, 13, 9), (127, 129, 33), (129, 257, 65),
          (255, 31, 100), (16, 300, 257), (300, 16, 129), (257, 255, 1)]


@pytest.mark.parametrize("variant", BUILT)
@pytest.mark.parametrize("split", [1, 3, -1])
@pytest.mark.parametrize("aligned", [True, False])
def test_variant_ragged(variant, split, aligned):
    if not aligned and variant in TMA_THIN:
        pytest.skip("the TMA-fed thin kernels read their operands by TMA: aligned only")
    for (M, N, K) in RAGGED:
        A, B, C = make_inputs(M, N, K, seed=M * 7 + N * 3 + K)
        if aligned and variant in TMA_VARIANTS + KPAIR_VARIANTS + TMA_THIN:
            # TMA needs ld % 4 == 0: pad the rows
            lds, offs = (-(-K // 4) * 4, -(-N // 4) * 4, None), (0, 0, 0)
        elif variant in KPAIR_VARIANTS:  # aligned A; B and C with odd ld and offsets
            lds, offs = (-(-K // 4) * 4, N + 3, N + 5), (0, 3, 5)
        elif aligned:
            lds, offs = (None, None, None), (0, 0, 0)
        else:  # odd leading dimensions and odd element offsets: 32-bit paths everywhere
            lds, offs = (K + 1, N + 3, N + 5), (1, 3, 5)
        out, guard = _run(A, B, C, 0.75, -1.25, *lds, offs=offs, variant=variant,
                          split=split)
        assert guard, (M, N, K)
        R, S = oracle.sgemm_f64(A, B, C, 0.75, -1.25)
        assert_bound(out.numpy(), R, S, -1.25, C.numpy(), f"v{variant} s{split} {M,N,K}")


@pytest.mark.parametrize("variant", [0, 5, 8])
@pytest.mark.parametrize("split", [-1, -3])
def test_whole_waves_plus_split_tail(variant, split):
    """More tiles than fit in one wave: the full waves run whole, the tiles of the last
    wave are split along K and finished by the reduce kernel."""
    M, N, K = 2100, 2600, 300  # 17 x 11 = 187 tiles of 128 x 256; 289 of 128 x 128
    A, B, C = make_inputs(M, N, K, seed=77)
    out, guard = _run(A, B, C, 1.5, 0.5, variant=variant, split=split)
    assert guard
    R, S = oracle.sgemm_f64(A, B, C, 1.5, 0.5)
    assert_bound(out.numpy(), R, S, 0.5, C.numpy(), f"v{variant} tail split {split}")


def test_mid_size_sweep_auto_plan():
    """Random mid-size shapes under the automatic plan, which there chooses among the
    128 x 96 and 128 x 64 k-major tiles, cluster-finished splits and split tails. Checked
    on sampled rows (the first and last rows, rows at tile edges, random rows) against the
    oracle; guard bands must stay intact."""
    rng = np.random.default_rng(11)
    for t in range(12):
        M, N, K = (int(rng.integers(200, 3000)) for _ in range(3))
        A, B, C = make_inputs(M, N, K, seed=300 + t)
        out, guard = _run(A, B, C, 1.25, -0.5)
        assert guard, (M, N, K)
        rows = np.unique(np.concatenate([[0, 1, M - 1], np.arange(127, M, 128)[:4],
                                         rng.integers(0, M, 12)]))
        R, S = oracle.sgemm_f64_rows(A, B, C, 1.25, -0.5, rows)
        assert_bound(out.numpy()[rows], R, S, -0.5, C.numpy()[rows], f"auto {M,N,K}")


def test_ragged_sweep_auto_plan():
    """Small M, N, K around tile edges under the automatic plan."""
    edges = [1, 2, 3, 5, 8, 15, 16, 17, 127, 128, 129, 255, 256, 257]
    rng = np.random.default_rng(3)
    for t in range(60):
        M, N, K = (int(rng.choice(edges)) for _ in range(3))
        A, B, C = make_inputs(M, N, K, seed=100 + t)
        out, guard = _run(A, B, C, 1.0, 0.5)
        assert guard, (M, N, K)
        R, S = oracle.sgemm_f64(A, B, C, 1.0, 0.5)
        assert_bound(out.numpy(), R, S, 0.5, C.numpy(), f"auto {M,N,K}")


THIN_M_SHAPES = [(1, 1, 1), (5, 255, 7), (16, 256, 513), (16, 1000, 2049), (13, 4100, 64),
                 (16, 4096, 1100)]
THIN_N_SHAPES = [(1, 1, 1), (255, 5, 7), (1024, 16, 2049), (1000, 16, 4100), (4100, 13, 64),
                 (3000, 16, 1100)]


@pytest.mark.parametrize("kind", ["m", "n", "mt", "nt", "mc", "nc"])
@pytest.mark.parametrize("split", [0, 1, 5, 17])
@pytest.mark.parametrize("aligned", [True, False])
def test_thin_kernels(kind, split, aligned):
    """The thin-M / thin-N streaming kernels, forced, on ragged and slice-boundary shapes:
    K slices that are not a multiple of the 8-deep load batch, column quads and rows that
    cross N and M, one slice (alpha / beta in the kernel) and several (reduce kernel).
    The TMA-fed thin-M kernel ("mt") needs an aligned B; split 17 on K = 2049 / 1100 gives
    slices that end inside a 32-row B tile. The cluster kernels ("mc", "nc") take the split
    as their cluster size, rounded up to 1, 2, 4 or 8 (5 and 17 give 8: on K = 1 and 7 most
    of the cluster's K slices are empty)."""
    if kind in ("mt", "nt", "mc", "nc") and not aligned:
        pytest.skip("the TMA-fed thin kernels read their operands by TMA: aligned only")
    variant = {"m": THIN_M, "n": THIN_N, "mt": THIN_M_TMA, "nt": THIN_N_TMA,
               "mc": THIN_M_CL, "nc": THIN_N_CL}[kind]
    for (M, N, K) in (THIN_N_SHAPES if kind in ("n", "nt", "nc") else THIN_M_SHAPES):
        A, B, C = make_inputs(M, N, K, seed=M + 3 * N + 5 * K + split)
        if aligned:
            lds, offs = (-(-K // 4) * 4, -(-N // 4) * 4, None), (0, 0, 0)
        else:
            lds, offs = (K + 1, N + 3, N + 5), (1, 3, 5)
        out, guard = _run(A, B, C, 0.75, -1.25, *lds, offs=offs, variant=variant, split=split)
        assert guard, (M, N, K)
        R, S = oracle.sgemm_f64(A, B, C, 0.75, -1.25)
        assert_bound(out.numpy(), R, S, -1.25, C.numpy(), f"thin-{kind} s{split} {M,N,K}")


CLUSTER_SHAPES = [(16, 4096, 1000), (40, 1000, 777), (16, 129, 4104), (3, 4100, 4096)]


@pytest.mark.parametrize("thin_n", [False, True])
@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
@pytest.mark.parametrize("beta", [0.0, 2.0])
def test_thin_cluster_sizes(thin_n, cluster, beta):
    """The cluster thin kernels at every cluster size: several small blocks (M = 40 is 3 row
    blocks), wide extents that end inside a 128-wide tile, K slices that end inside an 8-k
    chunk, beta = 0 and beta != 0, and no write outside the C view. The result is
    bitwise the same on a second run (fixed-order sums within and across the cluster)."""
    for (M, N, K) in CLUSTER_SHAPES:
        if thin_n:
            M, N = N, M
        A, B, C = make_inputs(M, N, K, seed=M + 7 * N + 11 * K + cluster)
        lds = (-(-K // 4) * 4, -(-N // 4) * 4, None)
        v = THIN_N_CL if thin_n else THIN_M_CL
        out, guard = _run(A, B, C, 1.5, beta, *lds, variant=v, split=cluster)
        assert guard, (M, N, K)
        R, S = oracle.sgemm_f64(A, B, C, 1.5, beta)
        assert_bound(out.numpy(), R, S, beta, C.numpy(), f"v{v} S{cluster} {M,N,K}")
        again, _ = _run(A, B, C, 1.5, beta, *lds, variant=v, split=cluster)
        assert torch.equal(out, again), (M, N, K)


def _odd_ld(x):
    """A row stride of at least x elements that is not a multiple of 4 (16 bytes)."""
    return x + 1 if (x + 1) % 4 else x + 2


@pytest.mark.parametrize("thin_n", [False, True])
@pytest.mark.parametrize("cluster", [0, 1, 4, 8])
def test_thin_cluster_small_operand_copied(thin_n, cluster):
    """The cluster thin kernels when the small operand cannot be read by TMA as stored (a
    row stride that is not a multiple of 16 bytes and a misaligned base): it is first
    copied to aligned rows in the workspace, and the streamed operand is read as stored.
    Cluster 0 is the automatic plan, checked when the model takes the cluster kernel."""
    for (M, N, K) in [(16, 4096, 4099), (5, 1000, 777), (33, 4100, 2051)]:
        if thin_n:
            M, N = N, M
        A, B, C = make_inputs(M, N, K, seed=M + 5 * N + 3 * K + cluster)
        if thin_n:  # streamed A aligned; small B (N wide) at an odd stride and offset
            lds, offs = (-(-K // 4) * 4, _odd_ld(N), N + 1), (0, 1, 2)
        else:       # streamed B aligned; small A (K wide) at an odd stride and offset
            lds, offs = (_odd_ld(K), -(-N // 4) * 4, N + 1), (3, 0, 2)
        v = THIN_N_CL if thin_n else THIN_M_CL
        if cluster == 0:
            plan = sg.sgemm_f32_plan(M, N, K, *lds, 0.75, -1.25)
            if plan["variant"] != v:
                continue  # the model prefers another kernel for this shape
            assert plan["ws_bytes"] > 0 and plan["launches"] == 2, plan
            out, guard = _run(A, B, C, 0.75, -1.25, *lds, offs=offs)
        else:
            out, guard = _run(A, B, C, 0.75, -1.25, *lds, offs=offs, variant=v, split=cluster)
        assert guard, (M, N, K)
        R, S = oracle.sgemm_f64(A, B, C, 0.75, -1.25)
        assert_bound(out.numpy(), R, S, -1.25, C.numpy(), f"v{v} S{cluster} copied {M,N,K}")


CLUSTER_SPLIT_VARIANTS = (2, 13, 32, 35, 37)  # copy-fed and TMA-fed (A as stored / k-major)


@pytest.mark.parametrize("variant", CLUSTER_SPLIT_VARIANTS)
@pytest.mark.parametrize("split", [2, 5, 8])
@pytest.mark.parametrize("beta", [0.0, -1.25])
def test_cluster_split_finish(variant, split, beta):
    """Every tile split into 2 .. 8 K slices that run as one thread-block cluster and add
    their partial tiles through distributed shared memory (no workspace, no reduce
    launch): ragged tiles, K slices ending inside a K block, beta = 0 and beta != 0, and a
    bitwise-equal second run (the slices are added in rank order)."""
    for (M, N, K) in [(257, 255, 1000), (130, 100, 777), (1024, 1024, 1024)]:
        A, B, C = make_inputs(M, N, K, seed=M + N + K + split)
        lds = (-(-K // 4) * 4, -(-N // 4) * 4, None)
        out, guard = _run(A, B, C, 0.75, beta, *lds, variant=variant, split=split)
        assert guard, (M, N, K)
        R, S = oracle.sgemm_f64(A, B, C, 0.75, beta)
        assert_bound(out.numpy(), R, S, beta, C.numpy(), f"v{variant} cluster {split} {M,N,K}")
        again, _ = _run(A, B, C, 0.75, beta, *lds, variant=variant, split=split)
        assert torch.equal(out, again), (variant, split, M, N, K)


# --------------------------------------------------------------------------------------
# BLAS special cases and contract details.

def test_variant_count():
    assert sg.sgemm_f32_num_variants() == NUM_VARIANTS


@pytest.mark.parametrize("variant", RETIRED)
def test_retired_variant_is_refused(variant):
    """A configuration kept in the table but not compiled is refused without a launch."""
    A = torch.ones((64, 64), device="cuda")
    C = torch.full((64, 64), 3.0, device="cuda")
    assert sg.sgemm_f32_forced(64, 64, 64, 1.0, A, 64, A, 64, 1.0, C, 64, variant, 1) == -14
    torch.cuda.synchronize()
    assert bool((C == 3.0).all())


def test_tma_variants_on_unaligned_and_transposed_operands():
    """A TMA-fed configuration packs row-major operands that TMA cannot address (odd ld,
    misaligned pointer) into aligned copies and still meets the bound; it has no path for
    transposed operands (-14). The K-paired configurations need an addressable A (-14)."""
    A, B, C = make_inputs(64, 64, 64, seed=12)
    dA, _ = to_device_view(A, 65, 1)
    dB, _ = to_device_view(B, 67, 3)
    R, S = oracle.sgemm_f64(A, B, None, 1.0, 0.0)
    for v in TMA_VARIANTS:
        dC, _ = to_device_view(C)
        assert sg.sgemm_f32_forced(64, 64, 64, 1.0, dA, 65, dB, 67, 0.0, dC, 64, v, 1) == 0
        torch.cuda.synchronize()
        assert_bound(dC.cpu().numpy(), R, S, 0.0, None, f"packed v{v}")
        assert sg.sgemm_f32_ex_forced(1, 0, 64, 64, 64, 1.0, dA, 65, dB, 67, 0.0, dC, 64,
                                      v, 1) == -14
    dC, _ = to_device_view(C)
    for v in KPAIR_VARIANTS:
        assert sg.sgemm_f32_forced(64, 64, 64, 1.0, dA, 65, dB, 67, 0.0, dC, 64, v, 1) == -14


def test_status_words_clear():
    A, B, C = make_inputs(300, 300, 300, seed=13)
    for v in TMA_VARIANTS + KPAIR_VARIANTS:
        out, _ = _run(A, B, C, 1.0, 0.5, variant=v, split=1)
    assert sg.sgemm_f32_status() == (0, 0)


def test_beta_zero_does_not_read_c():
    A, B, _ = make_inputs(70, 90, 33, seed=5)
    C = torch.full((70, 90), float("nan"))
    out, _ = _run(A, B, C, 1.5, 0.0)
    R, S = oracle.sgemm_f64(A, B, None, 1.5, 0.0)
    assert torch.isfinite(out).all()
    assert_bound(out.numpy(), R, S, 0.0, None, "beta=0")


def test_alpha_zero_does_not_read_ab():
    A = torch.full((40, 30), float("nan"))
    B = torch.full((30, 50), float("nan"))
    _, _, C = make_inputs(40, 50, 30, seed=6)
    out, _ = _run(A, B, C, 0.0, -2.0)
    assert torch.equal(out, C * -2.0)
    out0, _ = _run(A, B, C, 0.0, 0.0)
    assert torch.equal(out0, torch.zeros_like(C))
    out1, _ = _run(A, B, C, 0.0, 1.0)
    assert torch.equal(out1, C)


def test_k_zero():
    A = torch.zeros((20, 0))
    B = torch.zeros((0, 24))
    _, _, C = make_inputs(20, 24, 1, seed=7)
    out, _ = _run(A, B, C, 1.0, 3.0)
    assert torch.equal(out, C * 3.0)


def test_empty_m_n_is_noop():
    for M, N in ((0, 5), (5, 0), (0, 0)):
        assert sg.sgemm_f32(M, N, 4, 1.0, 0, 4, 0, max(N, 1), 0.0, 0, max(N, 1)) == 0


def test_fp32_fidelity_exact():
    """A = 1 + 2^-15 (not representable in TF32), B = 1, K = 256: the exact sum is
    256 + 2^-7, which FP32 FFMA reaches exactly; a TF32 path would give 256."""
    M, N, K = 64, 64, 256
    A = torch.full((M, K), 1.0 + 2.0 ** -15)
    B = torch.ones((K, N))
    C = torch.zeros((M, N))
    for v in _variants():  # packed 64 x 256 and 256 x 64 operands: TMA-able as well
        out, _ = _run(A, B, C, 1.0, 0.0, variant=v, split=1)
        assert torch.all(out == 256.0 + 2.0 ** -7), f"variant {v}"


def test_deterministic_and_ws_entry_match():
    A, B, C = make_inputs(1000, 1000, 1000, seed=8)
    o1, _ = _run(A, B, C, 1.0, 1.0)
    o2, _ = _run(A, B, C, 1.0, 1.0)
    assert torch.equal(o1, o2)
    M = N = K = 1000
    dA, _ = to_device_view(A)
    dB, _ = to_device_view(B)
    dC, _ = to_device_view(C)
    rc, nbytes = sg.sgemm_f32_workspace_size(M, N, K, K, N, N)
    assert rc == 0
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    assert sg.sgemm_f32_ws(M, N, K, 1.0, dA, K, dB, N, 1.0, dC, N, ws.data_ptr(),
                           ws.numel()) == 0
    torch.cuda.synchronize()
    assert torch.equal(dC.cpu(), o1)
    if nbytes:
        # one byte short: refused (-13), unless the plan's only workspace is an A^T copy
        # that the twin configuration (A transposed in shared memory) does without, in
        # which case the result is bitwise the same
        dC2, _ = to_device_view(C)
        rc = sg.sgemm_f32_ws(M, N, K, 1.0, dA, K, dB, N, 1.0, dC2, N, ws.data_ptr(), nbytes - 1)
        assert rc in (0, -13)
        if rc == 0:
            torch.cuda.synchronize()
            assert torch.equal(dC2.cpu(), o1)
    # a plan whose split-K partial tiles need the workspace is refused when it is too small
    M, N, K = 2100, 2600, 300
    p = sg.sgemm_f32_plan(M, N, K, K, N, N, 1.0, 1.0, 0)
    if p["split"] > 1 and p["ws_bytes"] > 0:
        A, B, C = make_inputs(M, N, K, seed=9)
        dA, _ = to_device_view(A)
        dB, _ = to_device_view(B)
        dC, _ = to_device_view(C)
        # too small for the partial tiles alone (an A^T copy in the plan has a twin that
        # does without it; the partials have none)
        at_copy = 0
        if p["variant"] in (35, 36, 39, 40):
            at_copy = -(-4 * K * (-(-M // 4) * 4) // 256) * 256
        short = p["ws_bytes"] - at_copy - 1
        ws = torch.empty(p["ws_bytes"], dtype=torch.uint8, device="cuda")
        before = dC.clone()
        assert sg.sgemm_f32_ws(M, N, K, 1.0, dA, K, dB, N, 1.0, dC, N, ws.data_ptr(),
                               short) == -13
        torch.cuda.synchronize()
        assert torch.equal(dC, before)


def test_illegal_arguments_launch_nothing():
    A, B, C = make_inputs(8, 8, 8, seed=9)
    dA, _ = to_device_view(A)
    dB, _ = to_device_view(B)
    dC, _ = to_device_view(C)
    before = dC.clone()
    assert sg.sgemm_f32(8, 8, 8, 1.0, dA, 7, dB, 8, 0.0, dC, 8) == -6
    assert sg.sgemm_f32(8, 8, 8, 1.0, dA, 8, dB, 7, 0.0, dC, 8) == -8
    assert sg.sgemm_f32(8, 8, 8, 1.0, dA, 8, dB, 8, 0.0, dC, 7) == -11
    assert sg.sgemm_f32(8, 8, 8, 1.0, None, 8, dB, 8, 0.0, dC, 8) == -5
    torch.cuda.synchronize()
    assert torch.equal(dC, before)


def test_torch_tensor_helper_and_streams():
    A, B, C = make_inputs(300, 200, 100, seed=10)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
        sg.sgemm(dA, dB, dC, 2.0, 0.5)
    s.synchronize()
    R, S = oracle.sgemm_f64(A, B, C, 2.0, 0.5)
    assert_bound(dC.cpu().numpy(), R, S, 0.5, C.numpy(), "stream")
