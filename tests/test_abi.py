"""CPU-only checks of the C ABI: the library loads, exports every symbol its header
declares, rejects illegal arguments before touching the GPU, and plans launches as
intended. No compute call is made here (there may be no GPU)."""
import ctypes
import os
import re

import pytest

import dense_fp32_matrix_08_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMS = 152  # SM count planned for (GB300)


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = _declared_functions()
    assert "sgemm_f32" in names and len(names) >= 8
    lib = ctypes.CDLL(sg.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(sg.EXPORTED) <= set(names)


def test_version():
    assert sg.sgemm_f32_version().startswith("sgemm_f32 ")


@pytest.mark.parametrize("args,code", [
    ((-1, 4, 4, 1.0, 8, 4, 8, 4, 0.0, 8, 4), -1),
    ((4, -1, 4, 1.0, 8, 4, 8, 4, 0.0, 8, 4), -2),
    ((4, 4, -1, 1.0, 8, 4, 8, 4, 0.0, 8, 4), -3),
    ((4, 4, 4, 1.0, None, 4, 8, 4, 0.0, 8, 4), -5),
    ((4, 4, 4, 1.0, 8, 3, 8, 4, 0.0, 8, 4), -6),
    ((4, 4, 4, 1.0, 8, 4, None, 4, 0.0, 8, 4), -7),
    ((4, 4, 4, 1.0, 8, 4, 8, 3, 0.0, 8, 4), -8),
    ((4, 4, 4, 1.0, 8, 4, 8, 4, 0.0, None, 4), -10),
    ((4, 4, 4, 1.0, 8, 4, 8, 4, 0.0, 8, 3), -11),
    ((4, 4, 0, 1.0, 8, 0, 8, 4, 0.0, 8, 4), -6),     # lda >= max(1, K)
    ((-1, -1, -1, 1.0, None, 0, None, 0, 0.0, None, 0), -1),  # first illegal one wins
])
def test_illegal_arguments(args, code):
    # pointer 8 is never dereferenced: validation fails before any CUDA call
    assert sg.sgemm_f32(*args, stream=0) == code
    assert sg.sgemm_f32_ws(*args, 0, 0, stream=0) == code
    assert sg.sgemm_f32_forced(*args, -1, 0, stream=0) == code


def test_null_ab_allowed_when_not_read():
    # M == 0 or N == 0 returns 0 before any CUDA call
    assert sg.sgemm_f32(0, 4, 4, 1.0, None, 4, None, 4, 0.0, None, 4, stream=0) == 0
    assert sg.sgemm_f32(4, 0, 4, 1.0, None, 4, None, 1, 0.0, None, 1, stream=0) == 0
    # alpha == 0: A and B may be NULL (validation passes; plan says beta-scale only)
    p = sg.sgemm_f32_plan(4, 4, 4, 4, 4, 4, alpha=0.0, beta=2.0, num_sms=SMS)
    assert p["status"] == 0 and p["variant"] == -1 and p["launches"] == 1
    p = sg.sgemm_f32_plan(4, 4, 4, 4, 4, 4, alpha=0.0, beta=1.0, num_sms=SMS)
    assert p["launches"] == 0


def test_query_entry_points_reject_illegal_arguments_before_cuda():
    # the workspace queries return sgemm_f32's codes (argument positions of sgemm_f32)
    for f in (sg.sgemm_f32_workspace_size, sg.sgemm_f32_workspace_size_min):
        assert f(-1, 4, 4, 4, 4, 4) == (-1, 0)
        assert f(4, 4, 4, 3, 4, 4) == (-6, 0)   # lda < K
        assert f(4, 4, 4, 4, 3, 4) == (-8, 0)   # ldb < N
        assert f(4, 4, 4, 4, 4, 3) == (-11, 0)  # ldc < N
    # an empty problem needs no workspace; this query answers before any device set-up
    assert sg.sgemm_f32_workspace_size_min(0, 4, 4, 4, 4, 4) == (0, 0)
    # FP32 pipe probe: iters in 1 .. 2^24, reps in 1 .. 100, tflops not NULL
    for iters, reps, code in ((0, 5, -1), ((1 << 24) + 1, 5, -1), (16, 0, -2), (16, 101, -2)):
        r = sg.sgemm_f32_fma_probe(iters, reps)
        assert r == {"status": code, "tflops": 0.0, "ms": 0.0}
    lib = ctypes.CDLL(sg.LIB_PATH)
    assert lib.sgemm_f32_fma_probe(16, 5, None, None) == -3
    # cluster capacity: variant in range, cluster in 1 .. 8, ctas not NULL
    n = sg.sgemm_f32_num_variants()
    assert sg.sgemm_f32_cluster_capacity(-1, 2) == (-1, 0)
    assert sg.sgemm_f32_cluster_capacity(n, 2) == (-1, 0)
    assert sg.sgemm_f32_cluster_capacity(0, 0) == (-2, 0)
    assert sg.sgemm_f32_cluster_capacity(0, 9) == (-2, 0)
    assert lib.sgemm_f32_cluster_capacity(0, 2, None) == -3


def test_forced_variant_out_of_range():
    n = sg.sgemm_f32_num_variants()
    assert sg.sgemm_f32_forced(4, 4, 4, 1.0, 8, 4, 8, 4, 0.0, 8, 4, n, 1, stream=0) == -14
    assert sg.sgemm_f32_forced(4, 4, 4, 1.0, 8, 4, 8, 4, 0.0, 8, 4, -2, 1, stream=0) == -14


def test_variant_table():
    n = sg.sgemm_f32_num_variants()
    assert n >= 5
    for v in range(n):
        info = sg.sgemm_f32_variant_info(v)
        assert info["BM"] % 16 == 0 and info["BN"] % 16 == 0 and info["BK"] % 8 == 0
        assert info["TM"] * info["TN"] >= 16 and info["threads"] % 32 == 0
        # the CTA tile is exactly covered by its threads' accumulator tiles, once, or once
        # per k-group where several thread groups split the CTA's K range (thin-M: 4 groups,
        # or 8 warps that each take 4 of every stage's 32 k rows, or 16 warps that each take
        # every 16th 8-k chunk)
        covered = info["threads"] * info["TM"] * info["TN"]
        assert covered % (info["BM"] * info["BN"]) == 0
        assert covered // (info["BM"] * info["BN"]) in (1, 4, 8, 16)
    assert sg.sgemm_f32_variant_info(n) is None
    big = sg.sgemm_f32_variant_info(0)
    assert big["TM"] * big["TN"] >= 64  # at least an 8x8 register outer product


RETIRED = (6, 7, 9, 10, 11, 12, 14, 15, 17, 18, 19, 20, 22, 23, 24, 25)


def test_retired_variants_are_described_not_built():
    for v in range(sg.sgemm_f32_num_variants()):
        assert sg.sgemm_f32_variant_info(v)["built"] == (v not in RETIRED), v


def test_shared_memory_transpose_twins_are_not_automatic():
    """Configurations 37 and 38 (A transposed in the CTA) were measured slower than the
    automatic choice without them at 768^3 and 1536^3 (and 3-5% behind their k-major
    counterparts at 8192^3): the automatic plan never takes them."""
    for n in (512, 768, 1024, 1280, 1536, 1792, 2048, 3000, 4096, 8192):
        assert _plan(n, n, n, beta=0.5)["variant"] not in (37, 38), n
    for shp in [(1500, 1500, 4000), (4096, 1024, 2048), (4099, 3001, 777)]:
        assert _plan(*shp, beta=0.5)["variant"] not in (37, 38), shp


def test_plan_transpose_twin_45_for_long_k():
    """Configuration 45 (configuration 39's tiles with A transposed in the CTA, so no A^T
    copy) is automatic for K loops of 8 or more K blocks, where it measured fastest on GB300
    (4096 x 256 x 4096: 147.9 against 174.4 us per call; 2048^3: 264.7 against 273.3).
    Below that its per-block transpose and its 3 CTAs per SM do not pay (2432 x 2432 x 64:
    30.8 against 27.6 us), and the plan takes another configuration."""
    for shp in [(4096, 256, 4096), (2048, 2048, 2048), (256, 256, 8192)]:
        assert _plan(*shp, beta=0.5)["variant"] == 45, shp
    for shp in [(2432, 2432, 64), (4096, 4096, 128)]:
        assert _plan(*shp, beta=0.5)["variant"] != 45, shp


def _plan(M, N, K, beta=1.0):
    p = sg.sgemm_f32_plan(M, N, K, K, N, N, 1.0, beta, SMS)
    assert p["status"] == 0
    return p


def test_plan_headline_uses_large_tiles():
    p = _plan(8192, 8192, 8192)
    info = sg.sgemm_f32_variant_info(p["variant"])
    assert info["TM"] * info["TN"] >= 64
    pre = 1 if p["variant"] in AT_VARIANTS else 0  # the A^T copy
    assert p["launches"] == pre + (2 if p["split"] > 1 else 1)


THIN_CLUSTER = (43, 44)  # K slices reduced inside a cluster: no workspace, one launch


def test_plan_thin_shapes_use_thin_tiles_and_split_k():
    for M, N, K in ((16, 4096, 4096), (4096, 16, 8192)):
        p = _plan(M, N, K)
        info = sg.sgemm_f32_variant_info(p["variant"])
        assert min(info["BM"], info["BN"]) <= 16 and p["split"] > 1
        if p["variant"] in THIN_CLUSTER:
            assert p["split"] in (2, 4, 8) and p["ws_bytes"] == 0 and p["launches"] == 1
        else:
            assert p["ws_bytes"] > 0


def test_plan_thin_cluster_copies_an_unaligned_small_operand():
    """A thin problem whose small operand TMA cannot read as stored (odd K for thin-M's A,
    odd N for thin-N's B) still takes the cluster kernel: the small operand is copied to
    aligned rows first (one more launch, a workspace of that copy's size). An unaligned
    streamed operand rules the cluster kernels out, since copying it would double the
    traffic of an HBM-bound kernel."""
    M, N, K = 16, 4096, 4099
    p = sg.sgemm_f32_plan(M, N, K, K, N, N, 1.0, 1.0, SMS)
    assert p["variant"] == 43 and p["launches"] == 2
    assert p["ws_bytes"] == -(-M * (-(-K // 4) * 4) * 4 // 256) * 256  # the copy of A only
    M, N, K = 4096, 18, 2048
    p = sg.sgemm_f32_plan(M, N, K, K, N, N, 1.0, 0.0, SMS)
    assert p["variant"] == 44 and p["launches"] == 2
    assert p["ws_bytes"] == -(-K * (-(-N // 4) * 4) * 4 // 256) * 256  # the copy of B only
    for (M, N, K, lda, ldb) in ((16, 4097, 4096, 4096, 4097), (4096, 16, 8193, 8193, 16)):
        p = sg.sgemm_f32_plan(M, N, K, lda, ldb, N, 1.0, 1.0, SMS)
        assert p["variant"] not in THIN_CLUSTER, (M, N, K, p)


def test_plan_small_cube_finishes_split_in_a_cluster():
    """256^3 runs on the cluster thin kernel with every tile split along K: the slices run
    as one cluster and add their partial tiles in shared memory, so the call is one launch
    with no workspace (measured 5.15 us per call on GB300, against 6.1 for the tiled
    kernel's cluster split)."""
    p = _plan(256, 256, 256, beta=0.0)
    assert p["variant"] in THIN_CLUSTER
    assert p["split"] > 1 and p["main_tiles"] == 0
    assert p["launches"] == 1 and p["ws_bytes"] == 0


def test_plan_recalibrated_choices():
    """Choices of the model after its fixed costs were fitted to per-call times measured on
    GB300 (48 shapes, every automatic configuration and split): small cubes and flat
    products whose streamed operand stays in L2 take the cluster thin kernel, well past 64
    rows (measured 6.55 against 10.1 us at 384^3, 10.0 against 13.3 at 128 x 1024 x 1024,
    31.6 against 38.7 at 64 x 8192 x 1023); 128 x 4096 x 4096 splits 128 x 96 tiles 10 ways
    with the reduce kernel (81 against 103 us for a 7-way cluster split); configuration 36
    is never chosen."""
    for shp in [(200, 200, 200), (384, 384, 384), (512, 512, 512), (128, 1024, 1024),
                (64, 8192, 1023)]:
        assert _plan(*shp, beta=0.5)["variant"] == 43, shp
    p = _plan(128, 4096, 4096, beta=0.5)
    assert p["variant"] == 35 and p["split"] == 10 and p["launches"] == 3
    for n in (256, 512, 768, 1024, 1536, 2048, 3072, 4096, 8192):
        assert _plan(n, n, n, beta=0.5)["variant"] != 36, n
    for shp in [(2048, 2048, 256), (4096, 4096, 128), (1024, 8192, 1024)]:
        assert _plan(*shp, beta=0.5)["variant"] != 36, shp


def test_plan_calibration_points():
    """The model's choices at the shapes it was calibrated on (measured on GB300): 128 x 96
    k-major tiles for the large shapes, with a split last wave at 4099 x 3001 x 777;
    128 x 64 k-major tiles at 3000^3, where 4 CTAs per SM round the waves better."""
    assert _plan(8192, 8192, 8192)["variant"] == 35
    assert _plan(4096, 4096, 4096)["variant"] == 35
    p = _plan(4099, 3001, 777)
    assert p["variant"] == 35 and p["split"] > 1 and p["main_tiles"] > 0
    assert _plan(3000, 3000, 3000)["variant"] == 39


TMA_VARIANTS = (26, 30, 31, 32, 37, 38, 45)  # TMA-fed, A as stored (aligned copies if needed)
AT_VARIANTS = (35, 36, 39, 40)  # TMA-fed, reading a transposed copy of A (B copied if needed)


def test_plan_workspace_formula():
    """Workspace = the A^T copy of a k-major plan (K rows of ceil4(M) floats) and aligned
    copies of the operands a TMA-fed plan cannot address (rows of ceil4(cols) floats), each
    256-byte rounded, then one BM x BN float tile per K slice of every split tile.
    Launches = the copies + the GEMM + the split-K finish."""
    def r256(x):
        return -(-x // 256) * 256

    for shp in [(16, 4096, 4096), (4096, 16, 8192), (256, 256, 256), (1023, 1021, 4096),
                (8192, 8192, 8192), (4097, 4097, 4097), (4099, 3001, 777)]:
        M, N, K = shp
        p = _plan(M, N, K)
        info = sg.sgemm_f32_variant_info(p["variant"])
        tiles = -(-M // info["BM"]) * -(-N // info["BN"])
        split_tiles = tiles - p["main_tiles"]
        pre, copies = 0, 0
        if p["variant"] in AT_VARIANTS:
            pre, copies = pre + r256(4 * K * (-(-M // 4) * 4)), copies + 1
        if p["variant"] in TMA_VARIANTS and K % 4:
            pre, copies = pre + r256(4 * M * (-(-K // 4) * 4)), copies + 1
        if p["variant"] in TMA_VARIANTS + AT_VARIANTS and N % 4:
            pre, copies = pre + r256(4 * K * (-(-N // 4) * 4)), copies + 1
        if p["variant"] in THIN_CLUSTER:
            assert p["ws_bytes"] == 0 and p["launches"] == 1
        elif p["split"] > 1 and p["launches"] == 1 + copies:
            # every tile split into at most 8 slices that a thread-block cluster adds in
            # shared memory: no partial tiles, no reduce launch
            assert p["main_tiles"] == 0 and p["split"] <= 8 and p["ws_bytes"] == pre
        elif p["split"] > 1:
            assert split_tiles > 0 and p["launches"] == 2 + copies
            assert p["ws_bytes"] == pre + 4 * p["split"] * split_tiles * info["BM"] * info["BN"]
        else:
            assert p["main_tiles"] == tiles and p["ws_bytes"] == pre
            assert p["launches"] == 1 + copies


def test_plan_tail_split_keeps_whole_waves():
    """When the tiles overflow the last wave, whole waves stay unsplit."""
    p = _plan(8192, 8192, 8192)
    if p["split"] > 1 and p["main_tiles"] > 0:
        info = sg.sgemm_f32_variant_info(p["variant"])
        assert p["main_tiles"] % SMS == 0


def test_plan_split_never_exceeds_k_tiles():
    for K in (1, 7, 16, 17, 33, 100):
        p = _plan(64, 64, K)
        info = sg.sgemm_f32_variant_info(p["variant"])
        assert 1 <= p["split"] <= -(-K // info["BK"])


@pytest.mark.parametrize("args,code", [
    ((2, 0, 4, 4, 4, 1.0, 8, 4, 8, 4, 0.0, 8, 4), -1),     # transa not 0/1
    ((0, 5, 4, 4, 4, 1.0, 8, 4, 8, 4, 0.0, 8, 4), -2),     # transb not 0/1
    ((0, 0, -1, 4, 4, 1.0, 8, 4, 8, 4, 0.0, 8, 4), -3),    # M
    ((1, 0, 4, 6, 5, 1.0, 8, 3, 8, 6, 0.0, 8, 6), -8),     # lda < M when A is transposed
    ((0, 1, 4, 6, 5, 1.0, 8, 5, 8, 4, 0.0, 8, 6), -10),    # ldb < K when B is transposed
    ((0, 0, 4, 6, 5, 1.0, 8, 5, 8, 6, 0.0, None, 6), -12),  # C missing
    ((0, 0, 4, 6, 5, 1.0, 8, 5, 8, 6, 0.0, 8, 5), -13),    # ldc < N
])
def test_ex_argument_checks(args, code):
    assert sg.sgemm_f32_ex(*args, stream=0) == code


@pytest.mark.parametrize("args,code", [
    ((0, 0, -1, 4, 4, 1.0, 8, 4, 8, 4, 0.0, 8, 4), -3),    # m
    ((0, 0, 4, -1, 4, 1.0, 8, 4, 8, 4, 0.0, 8, 4), -4),    # n
    ((0, 0, 4, 6, 5, 1.0, 8, 3, 8, 5, 0.0, 8, 4), -8),     # lda < m (A is m x k, col-major)
    ((1, 0, 4, 6, 5, 1.0, 8, 4, 8, 5, 0.0, 8, 4), -8),     # lda < k when transposed
    ((0, 0, 4, 6, 5, 1.0, 8, 4, 8, 4, 0.0, 8, 4), -10),    # ldb < k
    ((0, 1, 4, 6, 5, 1.0, 8, 4, 8, 5, 0.0, 8, 4), -10),    # ldb < n when transposed
    ((0, 0, 4, 6, 5, 1.0, 8, 4, 8, 5, 0.0, 8, 3), -13),    # ldc < m
    ((0, 0, 4, 6, 5, 1.0, None, 4, 8, 5, 0.0, 8, 4), -7),  # A missing
])
def test_colmajor_argument_checks(args, code):
    assert sg.sgemm_f32_colmajor(*args, stream=0) == code


@pytest.mark.parametrize("args,code", [
    ((2, 4, 4, 1.0, 8, 4, 8, 1, 0.0, 8, 1), -1),
    ((0, -1, 4, 1.0, 8, 4, 8, 1, 0.0, 8, 1), -2),
    ((0, 4, -1, 1.0, 8, 4, 8, 1, 0.0, 8, 1), -3),
    ((0, 4, 4, 1.0, None, 4, 8, 1, 0.0, 8, 1), -5),
    ((0, 4, 4, 1.0, 8, 3, 8, 1, 0.0, 8, 1), -6),
    ((0, 4, 4, 1.0, 8, 4, None, 1, 0.0, 8, 1), -7),
    ((0, 4, 4, 1.0, 8, 4, 8, 0, 0.0, 8, 1), -8),
    ((0, 4, 4, 1.0, 8, 4, 8, 1, 0.0, None, 1), -10),
    ((0, 4, 4, 1.0, 8, 4, 8, 1, 0.0, 8, 0), -11),
])
def test_sgemv_argument_checks(args, code):
    assert sg.sgemv_f32(*args, stream=0) == code


@pytest.mark.parametrize("args,code", [
    ((-1, 8, 1, 8, 1, 8), -1), ((4, None, 1, 8, 1, 8), -2), ((4, 8, 0, 8, 1, 8), -3),
    ((4, 8, 1, None, 1, 8), -4), ((4, 8, 1, 8, 0, 8), -5), ((4, 8, 1, 8, 1, None), -6),
])
def test_sdot_argument_checks(args, code):
    assert sg.sdot_f32(*args, stream=0) == code
