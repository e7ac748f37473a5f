"""Pins for the CPU oracle: checks that do not trust the oracle's own formula.

Each check compares the oracle with something fixed from outside it: a worked example the
pages print (tests/golden), exact closed forms (identity, all-ones, rank-1, alpha = 0,
beta = 0, K = 0), brute force in exact Python integers on tiny shapes, the transposition
identity (A B)^T = B^T A^T, and a library matmul in float64 as a check. The last test
plants mistakes in copies of the oracle's C source and shows that the pins catch each one.
"""
import itertools
import json
import os
import random

import numpy as np
import pytest

import oracle
from workloads import make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _all_forms(orc, A, B, C, alpha, beta):
    """The three entry points of one oracle build, each returning full (R, S)."""
    M, N = A.shape[0], B.shape[1]
    R, S = orc.sgemm_f64(A, B, C, alpha, beta)
    yield "full", R, S
    rows = np.arange(M)[::-1].copy()
    Rr, Sr = orc.sgemm_f64_rows(A, B, C, alpha, beta, rows)
    yield "rows", Rr[::-1], Sr[::-1]
    ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    Re, Se = orc.sgemm_f64_entries(A, B, C, alpha, beta, ii.ravel(), jj.ravel())
    yield "entries", Re.reshape(M, N), Se.reshape(M, N)


# ---------------------------------------------------------------------------------------
# The individual pins. Each takes an Oracle instance and raises AssertionError on mismatch,
# so the same functions can be run against planted-mistake builds below.


def pin_golden_matvec(orc):
    g = _load("dense_matvec_example.json")
    A = _f32(g["A"])
    B = _f32(np.asarray(g["x"]).reshape(-1, 1))
    for form, R, _ in _all_forms(orc, A, B, None, 1.0, 0.0):
        assert R.ravel().tolist() == [float(v) for v in g["expected"]], form


def pin_golden_submatrix(orc):
    """Row-major reading of the column-major sub-block example: a 2 x 3 view at offset 6,
    ld 5, inside a 4 x 5 buffer; the oracle on that view equals the oracle on a packed
    copy, and padding outside the view (NaN) is never read."""
    g = _load("submatrix_view_example.json")
    rows_rm, cols_rm = g["parent_cols_colmajor"], g["parent_rows_colmajor"]  # 4 x 5
    r0, c0 = g["block_origin"][1], g["block_origin"][0]
    h, w = g["block_shape_colmajor"][1], g["block_shape_colmajor"][0]
    assert r0 * cols_rm + c0 == g["expected_offset"] and cols_rm == g["expected_ld"]
    buf = np.arange(1, 7, dtype=np.float32)
    assert buf.reshape(2, 3).tolist() == g["row_major_2x3"]
    assert buf.reshape(2, 3).T.tolist() == g["col_major_3x2"]
    parent = np.full((rows_rm, cols_rm), np.nan, np.float32)
    parent[r0:r0 + h, c0:c0 + w] = np.arange(1, h * w + 1, dtype=np.float32).reshape(h, w)
    view = parent[r0:r0 + h, c0:c0 + w]
    assert view.ctypes.data - parent.ctypes.data == 4 * g["expected_offset"]
    assert view.strides[0] == 4 * g["expected_ld"]
    B = _f32(np.arange(w * 2).reshape(w, 2) - 3)
    Cp = np.full((8, 9), np.nan, np.float32)
    Cv = Cp[2:2 + h, 3:5]
    Cv[...] = _f32([[1, -2], [3, 4]])
    R1, S1 = orc.sgemm_f64(view, B, Cv, 2.0, -1.0)
    R2, S2 = orc.sgemm_f64(np.ascontiguousarray(view), B, np.ascontiguousarray(Cv), 2.0, -1.0)
    assert np.array_equal(R1, R2) and np.array_equal(S1, S2)
    want = 2.0 * (np.arange(1, 7).reshape(2, 3) @ (np.arange(6).reshape(3, 2) - 3)) \
        - np.array([[1, -2], [3, 4]])
    assert R1.tolist() == want.astype(float).tolist()


def pin_bruteforce_integers(orc, seed=0):
    """(M, N, K) in {1..5}^3, small integer operands and scalars: every product and sum is
    an exact integer in double, so R and S must equal Python-int brute force exactly."""
    rng = random.Random(seed)
    for M, N, K in itertools.product(range(1, 6), repeat=3):
        a = [[rng.randint(-8, 8) for _ in range(K)] for _ in range(M)]
        b = [[rng.randint(-8, 8) for _ in range(N)] for _ in range(K)]
        c = [[rng.randint(-8, 8) for _ in range(N)] for _ in range(M)]
        alpha, beta = rng.choice([1, 2, -3]), rng.choice([0, 1, -2, 5])
        want = [[alpha * sum(a[i][k] * b[k][j] for k in range(K)) + beta * c[i][j]
                 for j in range(N)] for i in range(M)]
        want_s = [[sum(abs(a[i][k] * b[k][j]) for k in range(K)) for j in range(N)]
                  for i in range(M)]
        for form, R, S in _all_forms(orc, _f32(a), _f32(b), _f32(c), alpha, beta):
            assert R.tolist() == want, (form, M, N, K)
            assert S.tolist() == want_s, (form, M, N, K)


def pin_identity(orc):
    """A = I_K (M = K): R = alpha B + beta C exactly (one nonzero product per sum)."""
    A, B, C = make_inputs(7, 5, 7, seed=11)
    A = np.eye(7, dtype=np.float32)
    Bn, Cn = B.numpy().astype(np.float64), C.numpy().astype(np.float64)
    for form, R, S in _all_forms(orc, A, B, C, 0.75, -1.5):
        assert np.array_equal(R, 0.75 * Bn + (-1.5) * Cn), form
        assert np.array_equal(S, np.abs(Bn)), form


def pin_all_ones(orc):
    """A = 1, B = 1: every sum is K, so R = alpha K + beta C and S = K."""
    M, N, K = 6, 9, 13
    C = _f32(np.arange(M * N).reshape(M, N) * 0.25)
    for form, R, S in _all_forms(orc, np.ones((M, K), np.float32),
                                 np.ones((K, N), np.float32), C, 1.0, 2.0):
        assert np.array_equal(R, K + 2.0 * C.astype(np.float64)), form
        assert np.array_equal(S, np.full((M, N), float(K))), form
    R, _ = orc.sgemm_f64(np.ones((3, 4096), np.float32), np.ones((4096, 2), np.float32),
                         None, 1.0, 0.0)
    assert np.all(R == 4096.0)


def pin_alpha_zero(orc):
    """alpha = 0: R = beta C; A and B are not read (NaN-poisoned here)."""
    A = np.full((4, 3), np.nan, np.float32)
    B = np.full((3, 5), np.nan, np.float32)
    C = _f32(np.arange(20).reshape(4, 5) - 7)
    for form, R, S in _all_forms(orc, A, B, C, 0.0, -0.5):
        assert np.array_equal(R, -0.5 * C.astype(np.float64)), form
        assert np.all(S == 0.0), form


def pin_beta_zero(orc):
    """beta = 0: C is not read (NaN-poisoned here) and R = alpha A B."""
    A = _f32([[1, 2], [3, 4], [5, 6]])
    B = _f32([[1, -1, 2], [0, 3, -2]])
    C = np.full((3, 3), np.nan, np.float32)
    for form, R, _ in _all_forms(orc, A, B, C, 3.0, 0.0):
        assert np.array_equal(R, 3.0 * (A.astype(np.float64) @ B.astype(np.float64))), form


def pin_k_zero(orc):
    """K = 0: the sum is empty, R = beta C."""
    C = _f32([[1, 2], [3, 4]])
    A = np.zeros((2, 0), np.float32)
    B = np.zeros((0, 2), np.float32)
    for form, R, S in _all_forms(orc, A, B, C, 1.0, 3.0):
        assert np.array_equal(R, 3.0 * C.astype(np.float64)), form
        assert np.all(S == 0.0), form


def pin_rank_one(orc):
    """A_ik = u_i, B_kj = v_j with dyadic u, v: R = alpha K u_i v_j + beta c_ij exactly."""
    M, N, K = 5, 7, 11
    u = _f32([0.5, -1.25, 2.0, 0.125, -3.0])
    v = _f32([1.0, -0.75, 0.25, 4.0, -2.5, 0.0625, 1.5])
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[None, :], K, axis=0)
    C = _f32(np.arange(M * N).reshape(M, N) * 0.5 - 8)
    want = 0.5 * K * np.outer(u, v).astype(np.float64) + 1.5 * C.astype(np.float64)
    for form, R, S in _all_forms(orc, A, B, C, 0.5, 1.5):
        assert np.array_equal(R, want), form
        assert np.array_equal(S, K * np.abs(np.outer(u, v)).astype(np.float64)), form


def pin_transpose_identity(orc):
    """(A B)^T = B^T A^T: integer-valued operands make both sides exact, so they match
    bitwise. Catches a transposed operand or a swapped index."""
    rng = np.random.default_rng(5)
    M, N, K = 9, 4, 6
    A = _f32(rng.integers(-9, 10, (M, K)))
    B = _f32(rng.integers(-9, 10, (K, N)))
    C = _f32(rng.integers(-9, 10, (M, N)))
    R, S = orc.sgemm_f64(A, B, C, 2.0, -1.0)
    Rt, St = orc.sgemm_f64(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T),
                           np.ascontiguousarray(C.T), 2.0, -1.0)
    assert np.array_equal(R.T, Rt) and np.array_equal(S.T, St)


def pin_library_matmul(orc):
    """Random N(0,1) inputs: a float64 library matmul must agree with R to within the
    rounding of two different double summation orders, bounded by 2 K eps64 S."""
    A, B, C = make_inputs(33, 41, 57, seed=9)
    R, S = orc.sgemm_f64(A, B, C, 0.7, -1.3)
    An, Bn, Cn = (x.numpy().astype(np.float64) for x in (A, B, C))
    ref = np.float64(np.float32(0.7)) * (An @ Bn) + np.float64(np.float32(-1.3)) * Cn
    bound = 2 * 57 * np.finfo(np.float64).eps * (S + np.abs(Cn)) + 1e-300
    assert np.all(np.abs(R - ref) <= bound)
    assert np.all(S >= np.abs(An @ Bn) - bound)


PINS = [pin_golden_matvec, pin_golden_submatrix, pin_bruteforce_integers, pin_identity,
        pin_all_ones, pin_alpha_zero, pin_beta_zero, pin_k_zero, pin_rank_one,
        pin_transpose_identity, pin_library_matmul]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.default())


def test_phase_count_golden():
    """The phase (k-tile) count rounds up: the pages' worked boundary examples."""
    g = _load("phase_counts.json")
    for c in g["cases"]:
        assert -(-c["extent"] // c["tile"]) == c["phases"]
        assert c["extent"] // c["tile"] == c["truncating_division_phases"]


def test_oracle_rejects_bad_rows():
    with pytest.raises(ValueError):
        oracle.sgemm_f64_rows(np.ones((2, 2), np.float32), np.ones((2, 2), np.float32),
                              None, 1.0, 0.0, [2])


def test_oracle_threads_positive():
    assert oracle.threads() >= 1


# ---------------------------------------------------------------------------------------
# Planted mistakes: each mutation of the oracle source must be caught by at least one pin.

MUTATIONS = {
    "dropped_beta_term": ("beta * (double)C[i * ldc + j];\n        r[j] = ab + bc;",
                          "0.0 * (double)C[i * ldc + j];\n        r[j] = ab + bc;"),
    "wrong_sign": ("                r[j] += p;", "                r[j] -= p;"),
    "transposed_b": ("const double p = a * (double)brow[j];",
                     "const double p = a * (double)B[j * ldb + k]; (void)brow;"),
    "packed_lda": ("const double a = (double)A[i * lda + k];",
                   "const double a = (double)A[i * K + k];"),
    "dropped_last_k": ("        for (int64_t k = 0; k < K; ++k) {\n            const double a",
                       "        for (int64_t k = 0; k + 1 < K; ++k) {\n            const double a"),
    "alpha_on_beta_term": ("        r[j] = ab + bc;", "        r[j] = alpha * (r[j] + bc);"),
    "signed_magnitude_sum": ("                s[j] += fabs(p);", "                s[j] += p;"),
    "entries_dropped_beta": ("        R[t] = alpha * r + bc;", "        R[t] = alpha * r;"),
    "entries_transposed_b": ("(double)A[i * lda + k] * (double)B[k * ldb + j]",
                             "(double)A[i * lda + k] * (double)B[j * ldb + k]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mutated.c"
    mutated.write_text(src.replace(old, new))
    orc = oracle.Oracle(oracle.compile_oracle(str(mutated), str(tmp_path / "libmut.so")))
    caught = []
    for pin in PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
