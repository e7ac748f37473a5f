"""CPU FP64 oracle for row-major FP32 SGEMM (C = alpha * A * B + beta * C).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline leg
may import this package; the CUDA library never does. The arithmetic lives in
``sgemm_oracle.c`` (plain C, OpenMP over rows); this module compiles it with gcc on first
use and marshals numpy / torch CPU arrays into it.

Functions return ``(R, S)`` as float64 arrays: R is the FP64 result
alpha * sum_k a_ik b_kj + beta * c_ij and S is sum_k |a_ik b_kj|, the magnitude sum that the
error bound of the parity tests is built from.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "sgemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsgemm_oracle.so")


def compile_oracle(src: str, out: str) -> str:
    """gcc with OpenMP and strict IEEE (no fast-math, no FMA contraction), so the double
    sums are neither reassociated nor fused."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/libsgemm_oracle.so if missing or stale."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE))
    if force or stale:
        compile_oracle(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _as_f32(x, name):
    """Return (numpy float32 array sharing memory, row stride in elements)."""
    if x is None:
        return None, 1
    if hasattr(x, "detach"):  # torch CPU tensor, possibly a strided view
        x = x.detach().numpy()
    x = np.asarray(x)
    if x.dtype != np.float32:
        raise TypeError(f"{name} must be float32, got {x.dtype}")
    if x.ndim != 2:
        raise ValueError(f"{name} must be 2-D")
    if x.size == 0:
        return x, max(x.shape[1], 1)
    if x.shape[1] > 1 and x.strides[1] != 4:
        raise ValueError(f"{name} must have unit column stride")
    ld = x.strides[0] // 4 if x.shape[0] > 1 else max(x.shape[1], 1)
    return x, ld


def _ptr(x):
    return None if x is None or x.size == 0 else x.ctypes.data


def _dims(A, B, C, beta):
    if C is None and beta != 0.0:
        raise ValueError("C is required when beta != 0")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    if C is not None and tuple(C.shape) != (M, N):
        raise ValueError("C has the wrong shape")
    return M, N, K


class Oracle:
    """One loaded build of the oracle library (the default one, or a test's variant)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, dbl, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        common = [i64, i64, i64, dbl, vp, i64, vp, i64, dbl, vp, i64]
        lib.oracle_sgemm_f64.argtypes = common + [vp, vp]
        lib.oracle_sgemm_f64_rows.argtypes = common + [vp, i64, vp, vp]
        lib.oracle_sgemm_f64_entries.argtypes = common + [vp, vp, i64, vp, vp]
        lib.oracle_threads.argtypes = []
        for f in (lib.oracle_sgemm_f64, lib.oracle_sgemm_f64_rows,
                  lib.oracle_sgemm_f64_entries, lib.oracle_threads):
            f.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    def threads(self) -> int:
        """OpenMP threads the oracle runs on."""
        return int(self.lib.oracle_threads())

    def _prep(self, A, B, C, alpha, beta):
        A, lda = _as_f32(A, "A")
        B, ldb = _as_f32(B, "B")
        C, ldc = _as_f32(C, "C")
        M, N, K = _dims(A, B, C, beta)
        # alpha and beta are float32 scalars of the SGEMM call, widened exactly to double
        return (M, N, K, float(np.float32(alpha)), _ptr(A), lda, _ptr(B), ldb,
                float(np.float32(beta)), _ptr(C), ldc)

    def sgemm_f64(self, A, B, C, alpha: float, beta: float):
        """Full M x N result. A: M x K, B: K x N, C: M x N (may be None when beta == 0)."""
        args = self._prep(A, B, C, alpha, beta)
        M, N = args[0], args[1]
        R = np.empty((M, N), np.float64)
        S = np.empty((M, N), np.float64)
        rc = self.lib.oracle_sgemm_f64(*args, _ptr(R), _ptr(S))
        if rc != 0:
            raise ValueError(f"oracle rejected its arguments ({rc})")
        return R, S

    def sgemm_f64_rows(self, A, B, C, alpha: float, beta: float, rows):
        """Only the listed rows (all columns): R, S are len(rows) x N."""
        args = self._prep(A, B, C, alpha, beta)
        N = args[1]
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        R = np.empty((rows.size, N), np.float64)
        S = np.empty((rows.size, N), np.float64)
        rc = self.lib.oracle_sgemm_f64_rows(*args, _ptr(rows), rows.size, _ptr(R), _ptr(S))
        if rc != 0:
            raise ValueError(f"oracle rejected its arguments ({rc})")
        return R, S

    def sgemm_f64_entries(self, A, B, C, alpha: float, beta: float, ii, jj):
        """Single elements (ii[t], jj[t]): R, S are 1-D of length len(ii)."""
        args = self._prep(A, B, C, alpha, beta)
        ii = np.ascontiguousarray(np.asarray(ii, dtype=np.int64).reshape(-1))
        jj = np.ascontiguousarray(np.asarray(jj, dtype=np.int64).reshape(-1))
        if ii.shape != jj.shape:
            raise ValueError("ii and jj differ in length")
        R = np.empty(ii.size, np.float64)
        S = np.empty(ii.size, np.float64)
        rc = self.lib.oracle_sgemm_f64_entries(*args, _ptr(ii), _ptr(jj), ii.size, _ptr(R),
                                               _ptr(S))
        if rc != 0:
            raise ValueError(f"oracle rejected its arguments ({rc})")
        return R, S


_lock = threading.Lock()
_default: Oracle | None = None


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def threads() -> int:
    return default().threads()


def sgemm_f64(A, B, C, alpha, beta):
    return default().sgemm_f64(A, B, C, alpha, beta)


def sgemm_f64_rows(A, B, C, alpha, beta, rows):
    return default().sgemm_f64_rows(A, B, C, alpha, beta, rows)


def sgemm_f64_entries(A, B, C, alpha, beta, ii, jj):
    return default().sgemm_f64_entries(A, B, C, alpha, beta, ii, jj)
