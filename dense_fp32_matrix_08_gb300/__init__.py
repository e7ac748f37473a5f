"""Python binding of the sgemm_f32 C ABI (include/sgemm_f32.h).

Argument marshalling only: every step of C = alpha * A * B + beta * C runs in the CUDA
kernels of libsgemm_f32.so. Loading fails loudly if the library has not been built; there
is no fallback implementation.

Pointer arguments accept either integers (device addresses) or torch CUDA tensors (their
data_ptr() is passed; the tensor must be float32). `stream` accepts an integer handle, a
torch.cuda.Stream, or None for torch's current stream on the current device.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB as LIB_PATH

__all__ = [
    "LIB_PATH", "SgemmError", "lib", "sgemm_f32", "sgemm_f32_ws", "sgemm_f32_forced",
    "sgemm_f32_workspace_size", "sgemm_f32_plan", "sgemm_f32_num_variants",
    "sgemm_f32_variant_info", "sgemm_f32_version", "sgemm_f32_noalloc", "sgemm_f32_ex",
    "sgemm_f32_colmajor", "sgemv_f32", "sdot_f32", "sgemm_f32_status", "sgemm_f32_3xtf32",
    "sgemm_f32_3xtf32_workspace_size", "sgemm_f32_3xtf32_status", "sgemm_f32_ex_forced",
    "sgemm_f32_autotune", "sgemm_f32_tune_count", "sgemm_f32_tune_clear", "sgemm_f32_tune_save",
    "sgemm_f32_tune_load", "sgemm_f32_host", "sgemm_f32_wait_selftest",
    "sgemm_f32_release_workspace", "sgemm_f32_fma_probe", "sgemm_f32_cluster_capacity",
    "sgemm_f32_workspace_size_min",
    "sgemm", "EXPORTED",
]

# Every symbol include/sgemm_f32.h declares.
EXPORTED = ("sgemm_f32", "sgemm_f32_ws", "sgemm_f32_forced", "sgemm_f32_workspace_size",
            "sgemm_f32_plan", "sgemm_f32_num_variants", "sgemm_f32_variant_info",
            "sgemm_f32_version", "sgemm_f32_noalloc", "sgemm_f32_ex", "sgemm_f32_colmajor",
            "sgemv_f32", "sdot_f32", "sgemm_f32_status",
            "sgemm_f32_3xtf32",
            "sgemm_f32_3xtf32_workspace_size", "sgemm_f32_3xtf32_status",
            "sgemm_f32_ex_forced", "sgemm_f32_autotune", "sgemm_f32_tune_count",
            "sgemm_f32_tune_clear", "sgemm_f32_tune_save", "sgemm_f32_tune_load",
            "sgemm_f32_host", "sgemm_f32_wait_selftest", "sgemm_f32_release_workspace",
            "sgemm_f32_fma_probe", "sgemm_f32_cluster_capacity",
            "sgemm_f32_workspace_size_min")


class SgemmError(RuntimeError):
    """A nonzero status from the library: negative = illegal argument index, positive =
    cudaError_t."""

    def __init__(self, status: int, what: str = "sgemm_f32"):
        self.status = status
        super().__init__(f"{what} returned {status}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    i, f, vp, sz = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
    pi, psz = ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_size_t)
    gemm = [i, i, i, f, vp, i, vp, i, f, vp, i]
    L.sgemm_f32.argtypes = gemm + [vp]
    L.sgemm_f32_ws.argtypes = gemm + [vp, sz, vp]
    L.sgemm_f32_forced.argtypes = gemm + [i, i, vp]
    L.sgemm_f32_noalloc.argtypes = gemm + [vp]
    L.sgemm_f32_ex.argtypes = [i, i] + gemm + [vp]
    L.sgemm_f32_ex_forced.argtypes = [i, i] + gemm + [i, i, vp]
    L.sgemm_f32_autotune.argtypes = [i, i] + gemm + [i, vp, pi, pi, ctypes.POINTER(f)]
    L.sgemm_f32_tune_count.argtypes = []
    L.sgemm_f32_tune_clear.argtypes = []
    L.sgemm_f32_tune_save.argtypes = [ctypes.c_char_p]
    L.sgemm_f32_tune_load.argtypes = [ctypes.c_char_p]
    L.sgemm_f32_host.argtypes = gemm + [vp]
    L.sgemv_f32.argtypes = [i, i, i, f, vp, i, vp, i, f, vp, i, vp]
    L.sdot_f32.argtypes = [i, vp, i, vp, i, vp, vp]
    L.sgemm_f32_colmajor.argtypes = [i, i] + gemm + [vp]
    L.sgemm_f32_3xtf32.argtypes = gemm + [vp]
    L.sgemm_f32_3xtf32_workspace_size.argtypes = [i, i, i, psz]
    L.sgemm_f32_3xtf32_status.argtypes = [pi]
    L.sgemm_f32_status.argtypes = [pi]
    L.sgemm_f32_wait_selftest.argtypes = [pi, ctypes.POINTER(ctypes.c_float)]
    L.sgemm_f32_release_workspace.argtypes = [psz]
    L.sgemm_f32_cluster_capacity.argtypes = [i, i, pi]
    L.sgemm_f32_fma_probe.argtypes = [i, i, ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_float)]
    L.sgemm_f32_workspace_size.argtypes = [i, i, i, i, i, i, psz]
    L.sgemm_f32_workspace_size_min.argtypes = [i, i, i, i, i, i, psz]
    L.sgemm_f32_plan.argtypes = [i, i, i, i, i, i, f, f, i, pi, pi, pi, pi, psz]
    L.sgemm_f32_num_variants.argtypes = []
    L.sgemm_f32_variant_info.argtypes = [i] + [pi] * 7
    L.sgemm_f32_version.argtypes = []
    L.sgemm_f32_version.restype = ctypes.c_char_p
    for name in EXPORTED:
        if name != "sgemm_f32_version":
            getattr(L, name).restype = ctypes.c_int
    return L


lib = _load()


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    import torch
    if isinstance(x, torch.Tensor):
        if x.dtype != torch.float32:
            raise TypeError("tensor operands must be float32")
        if x.numel() and not x.is_cuda:
            raise TypeError("tensor operands must live on a CUDA device")
        return x.data_ptr() or None
    raise TypeError(f"cannot pass {type(x).__name__} as a device pointer")


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(s, int):
        return s or None
    return int(s.cuda_stream) or None


def sgemm_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """Mirror of the C entry point; returns its status (0 = success)."""
    return lib.sgemm_f32(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                         _stream(stream))


def sgemm_f32_ws(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, workspace, workspace_bytes,
                 stream=None) -> int:
    return lib.sgemm_f32_ws(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                            _ptr(workspace), workspace_bytes, _stream(stream))


def sgemm_f32_forced(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, variant, split,
                     stream=None) -> int:
    return lib.sgemm_f32_forced(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C),
                                ldc, variant, split, _stream(stream))


def sgemm_f32_ex_forced(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, variant,
                        split, stream=None) -> int:
    """sgemm_f32_ex with the tile configuration and split-K layout forced."""
    return lib.sgemm_f32_ex_forced(int(transa), int(transb), M, N, K, alpha, _ptr(A), lda,
                                   _ptr(B), ldb, beta, _ptr(C), ldc, variant, split,
                                   _stream(stream))


def sgemm_f32_autotune(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, reps=3,
                       stream=None) -> dict:
    """Time every configuration that can run this problem and record the fastest for its
    shape (see include/sgemm_f32.h). C is only read. Returns {"status", "variant", "split",
    "ms"}."""
    v, sp, ms = ctypes.c_int(-1), ctypes.c_int(0), ctypes.c_float(0.0)
    rc = lib.sgemm_f32_autotune(int(transa), int(transb), M, N, K, alpha, _ptr(A), lda,
                                _ptr(B), ldb, beta, _ptr(C), ldc, int(reps), _stream(stream),
                                ctypes.byref(v), ctypes.byref(sp), ctypes.byref(ms))
    return {"status": rc, "variant": v.value, "split": sp.value, "ms": ms.value}


def _host_ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    import torch
    if isinstance(x, torch.Tensor):
        if x.dtype != torch.float32:
            raise TypeError("tensor operands must be float32")
        if x.is_cuda:
            raise TypeError("sgemm_f32_host takes host (CPU) tensors")
        return x.data_ptr() or None
    raise TypeError(f"cannot pass {type(x).__name__} as a host pointer")


def sgemm_f32_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """C = alpha A B + beta C with A, B, C in host memory (pinned for overlap); the GPU
    computes it in row blocks while the copies of neighbouring blocks run. Asynchronous on
    `stream`: synchronise it before reading C."""
    return lib.sgemm_f32_host(M, N, K, alpha, _host_ptr(A), lda, _host_ptr(B), ldb, beta,
                              _host_ptr(C), ldc, _stream(stream))


def sgemm_f32_tune_count() -> int:
    return lib.sgemm_f32_tune_count()


def sgemm_f32_tune_clear() -> int:
    return lib.sgemm_f32_tune_clear()


def sgemm_f32_tune_save(path) -> int:
    return lib.sgemm_f32_tune_save(os.fsencode(path))


def sgemm_f32_tune_load(path) -> int:
    return lib.sgemm_f32_tune_load(os.fsencode(path))


def sgemm_f32_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """sgemm_f32 for callers that may not allocate device memory: any split-K workspace
    comes from the library's fixed per-device scratch array (see include/sgemm_f32.h).
    Returns the C status; -15 means the problem needs more scratch than that array."""
    return lib.sgemm_f32_noalloc(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C),
                                 ldc, _stream(stream))


def sgemm_f32_ex(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                 stream=None) -> int:
    """Row-major C = alpha op(A) op(B) + beta C with transpose flags (0 = N, 1 = T)."""
    return lib.sgemm_f32_ex(int(transa), int(transb), M, N, K, alpha, _ptr(A), lda, _ptr(B),
                            ldb, beta, _ptr(C), ldc, _stream(stream))


def sgemm_f32_colmajor(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc,
                       stream=None) -> int:
    """Column-major BLAS-style sgemm (transa/transb: 0 = N, 1 = T)."""
    return lib.sgemm_f32_colmajor(int(transa), int(transb), m, n, k, alpha, _ptr(A), lda,
                                  _ptr(B), ldb, beta, _ptr(C), ldc, _stream(stream))


def sgemv_f32(trans, M, N, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    """y = alpha op(A) x + beta y, A M x N row-major (trans: 0 = N, 1 = T)."""
    return lib.sgemv_f32(int(trans), M, N, alpha, _ptr(A), lda, _ptr(x), incx, beta, _ptr(y),
                         incy, _stream(stream))


def sdot_f32(n, x, incx, y, incy, result, stream=None) -> int:
    """*result (device) = sum x_i y_i."""
    return lib.sdot_f32(n, _ptr(x), incx, _ptr(y), incy, _ptr(result), _stream(stream))


def sgemm_f32_3xtf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """Tensor-core 3xTF32 variant (same contract and return codes as sgemm_f32)."""
    return lib.sgemm_f32_3xtf32(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C),
                                ldc, _stream(stream))


def sgemm_f32_3xtf32_workspace_size(M, N, K) -> tuple[int, int]:
    b = ctypes.c_size_t(0)
    rc = lib.sgemm_f32_3xtf32_workspace_size(M, N, K, ctypes.byref(b))
    return rc, b.value


def sgemm_f32_status() -> tuple[int, int]:
    """(call status, device status word of the TMA-fed FFMA kernel); reading clears it."""
    v = ctypes.c_int(0)
    rc = lib.sgemm_f32_status(ctypes.byref(v))
    return rc, v.value


def sgemm_f32_wait_selftest() -> dict:
    """Run the bounded-wait self-test: {"status", "timed_out", "seconds"} (see the header)."""
    t, sec = ctypes.c_int(0), ctypes.c_float(0.0)
    rc = lib.sgemm_f32_wait_selftest(ctypes.byref(t), ctypes.byref(sec))
    return {"status": rc, "timed_out": t.value, "seconds": sec.value}


def sgemm_f32_cluster_capacity(variant: int, cluster: int) -> tuple[int, int]:
    """(call status, CTAs the device holds at once in clusters of `cluster`) for a
    configuration, as the planner sees it (see the header)."""
    n = ctypes.c_int(0)
    rc = lib.sgemm_f32_cluster_capacity(variant, cluster, ctypes.byref(n))
    return rc, n.value


def sgemm_f32_fma_probe(iters: int = 1 << 17, reps: int = 5) -> dict:
    """Measure the FP32 FMA pipe: {"status", "tflops", "ms"} (see the header)."""
    t, ms = ctypes.c_double(0.0), ctypes.c_float(0.0)
    rc = lib.sgemm_f32_fma_probe(iters, reps, ctypes.byref(t), ctypes.byref(ms))
    return {"status": rc, "tflops": t.value, "ms": ms.value}


def sgemm_f32_release_workspace() -> tuple[int, int]:
    """(call status, bytes returned): hand the library pool's cached device memory on the
    current device back to the system (see the header)."""
    n = ctypes.c_size_t(0)
    rc = lib.sgemm_f32_release_workspace(ctypes.byref(n))
    return rc, n.value


def sgemm_f32_3xtf32_status() -> tuple[int, int]:
    """(call status, device status word); reading clears the word."""
    v = ctypes.c_int(0)
    rc = lib.sgemm_f32_3xtf32_status(ctypes.byref(v))
    return rc, v.value


def sgemm_f32_workspace_size(M, N, K, lda, ldb, ldc) -> tuple[int, int]:
    """(status, bytes)."""
    b = ctypes.c_size_t(0)
    rc = lib.sgemm_f32_workspace_size(M, N, K, lda, ldb, ldc, ctypes.byref(b))
    return rc, b.value


def sgemm_f32_workspace_size_min(M, N, K, lda, ldb, ldc) -> tuple[int, int]:
    """(status, bytes): the smallest workspace sgemm_f32_ws runs this problem with (the plan
    without its A^T copy; see the header)."""
    b = ctypes.c_size_t(0)
    rc = lib.sgemm_f32_workspace_size_min(M, N, K, lda, ldb, ldc, ctypes.byref(b))
    return rc, b.value


def sgemm_f32_plan(M, N, K, lda, ldb, ldc, alpha=1.0, beta=0.0, num_sms=0) -> dict:
    v, s, mt, n = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    ws = ctypes.c_size_t(0)
    rc = lib.sgemm_f32_plan(M, N, K, lda, ldb, ldc, alpha, beta, num_sms, ctypes.byref(v),
                            ctypes.byref(s), ctypes.byref(mt), ctypes.byref(n),
                            ctypes.byref(ws))
    return {"status": rc, "variant": v.value, "split": s.value, "main_tiles": mt.value,
            "launches": n.value, "ws_bytes": ws.value}


def sgemm_f32_num_variants() -> int:
    return lib.sgemm_f32_num_variants()


def sgemm_f32_variant_info(v: int) -> dict | None:
    """Shape of tile configuration v, with "built" False for a configuration kept in the
    table but not compiled (forcing it returns -14); None when v is out of range."""
    vals = [ctypes.c_int(0) for _ in range(7)]
    rc = lib.sgemm_f32_variant_info(v, *[ctypes.byref(x) for x in vals])
    if rc not in (0, 1):
        return None
    keys = ("BM", "BN", "BK", "threads", "TM", "TN", "stages")
    info = dict(zip(keys, (x.value for x in vals)))
    info["built"] = rc == 0
    return info


def sgemm_f32_version() -> str:
    return lib.sgemm_f32_version().decode()


def sgemm(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C = alpha * A @ B + beta * C in place on 2-D float32 CUDA tensors (row-major views
    with unit column stride; the row stride is passed as the leading dimension). Raises
    SgemmError on a nonzero status. Returns C."""
    for name, t in (("A", A), ("B", B), ("C", C)):
        if t.dim() != 2:
            raise ValueError(f"{name} must be 2-D")
        if t.size(1) > 1 and t.stride(1) != 1:
            raise ValueError(f"{name} must have unit column stride")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError("shape mismatch")

    def ld(t):
        return max(t.stride(0) if t.size(0) > 1 else t.size(1), 1)

    rc = sgemm_f32(M, N, K, alpha, A, ld(A), B, ld(B), beta, C, ld(C), stream)
    if rc != 0:
        raise SgemmError(rc)
    return C
