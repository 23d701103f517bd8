"""FP64 CPU oracle for C = A*B and y = A*x -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product (``gemv_tiled_gemm_gb300``)
never does, and the two share no code. The arithmetic lives in ``oracle.c``
(plain C, FP64, the textbook definitions; see that file for the sources it
follows). This module only builds that file with gcc and marshals numpy
arrays into it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile oracle.c into a shared library (no -ffast-math, no FMA fusion)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", *extra_flags,
           "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, cwd=os.path.dirname(src) or ".")
    return out


def _needs_build() -> bool:
    if not os.path.exists(_LIB):
        return True
    lib_t = os.path.getmtime(_LIB)
    return any(os.path.getmtime(os.path.join(_HERE, f)) > lib_t
               for f in ("oracle.c", "oracle.h"))


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; returns ctypes CDLL."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            if _needs_build():
                build()
            _lib = _bind(ctypes.CDLL(_LIB))
        return _lib


def _bind(lib):
    i64, dp, ci = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.c_int
    lib.oracle_gemm_f64.argtypes = [i64, i64, i64, dp, i64, dp, i64, dp, i64, dp, i64, ci]
    lib.oracle_gemm_f64.restype = ci
    lib.oracle_gemv_f64.argtypes = [i64, i64, dp, i64, dp, dp, dp]
    lib.oracle_gemv_f64.restype = ci
    lib.oracle_bias_act_f64.argtypes = [i64, i64, dp, i64, dp, ci, ci]
    lib.oracle_bias_act_f64.restype = ci
    lib.oracle_conv2d_f64.argtypes = [i64] * 13 + [dp, dp, dp, dp, ci]
    lib.oracle_conv2d_f64.restype = ci
    lib.oracle_threads_default.argtypes = []
    lib.oracle_threads_default.restype = ci
    return lib


def _as_f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype not in (np.float16, np.float32, np.float64):
        raise TypeError(f"oracle takes floating-point arrays, got {a.dtype}")
    return np.ascontiguousarray(a, dtype=np.float64)  # exact widening


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def threads_default() -> int:
    return int(load().oracle_threads_default())


def gemm(A, B, threads: int = 0, with_E: bool = True, lib=None):
    """C = A @ B in FP64 (and E = sum_k |a_ik b_kj|). Inputs are widened exactly."""
    lib = lib or load()
    A, B = _as_f64(A), _as_f64(B)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch {A.shape} x {B.shape}")
    M, K = A.shape
    N = B.shape[1]
    C = np.empty((M, N), dtype=np.float64)
    E = np.empty((M, N), dtype=np.float64) if with_E else None
    rc = lib.oracle_gemm_f64(M, N, K, _ptr(A), max(K, 1), _ptr(B), max(N, 1),
                             _ptr(C), max(N, 1),
                             _ptr(E) if with_E else None, max(N, 1), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_f64 returned {rc}")
    return (C, E) if with_E else C


def gemm_strided(M, N, K, A, lda, B, ldb, C, ldc, E=None, lde=0, threads=0, lib=None):
    """Leading-dimension form on flat FP64 buffers (used to pin padding)."""
    lib = lib or load()
    for arr in (A, B, C) + ((E,) if E is not None else ()):
        if arr.dtype != np.float64 or not arr.flags.c_contiguous:
            raise TypeError("flat contiguous float64 buffers required")
    rc = lib.oracle_gemm_f64(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc,
                             _ptr(E) if E is not None else None, lde, int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_f64 returned {rc}")


def gemv(A, x, with_E: bool = True, lib=None):
    """y = A @ x in FP64 (and E = sum_j |a_ij x_j|)."""
    lib = lib or load()
    A, x = _as_f64(A), _as_f64(x)
    if A.ndim != 2 or x.ndim != 1 or A.shape[1] != x.shape[0]:
        raise ValueError(f"shape mismatch {A.shape} x {x.shape}")
    M, N = A.shape
    y = np.empty(M, dtype=np.float64)
    E = np.empty(M, dtype=np.float64) if with_E else None
    rc = lib.oracle_gemv_f64(M, N, _ptr(A), max(N, 1), _ptr(x), _ptr(y),
                             _ptr(E) if with_E else None)
    if rc != 0:
        raise RuntimeError(f"oracle_gemv_f64 returned {rc}")
    return (y, E) if with_E else y


ACT = {"none": 0, "relu": 1}


def bias_act(C, bias=None, per_column=True, act="none", lib=None):
    """act(C + bias) in FP64 on a copy of C (bias per column, or per row)."""
    lib = lib or load()
    C = np.array(C, dtype=np.float64, order="C", copy=True)
    if C.ndim == 1:
        C = C[:, None]
        squeeze = True
    else:
        squeeze = False
    M, N = C.shape
    b = None if bias is None else _as_f64(bias)
    if b is not None and b.size != (N if per_column else M):
        raise ValueError("bias length must match the output columns (per_column) or rows")
    rc = lib.oracle_bias_act_f64(M, N, _ptr(C), max(N, 1), _ptr(b) if b is not None else None,
                                 1 if per_column else 0, ACT[act])
    if rc != 0:
        raise RuntimeError(f"oracle_bias_act_f64 returned {rc}")
    return C[:, 0] if squeeze else C


def dense_layer(A, B, bias=None, act="none", threads=0, lib=None):
    """act(A @ B + bias), bias per output column (a batch of inputs in A's rows)."""
    C, E = gemm(A, B, threads=threads, lib=lib)
    return bias_act(C, bias, True, act, lib=lib), E


def dense_vector(A, x, bias=None, act="none", lib=None):
    """act(A @ x + bias), bias per output row (one fully connected layer)."""
    y, E = gemv(A, x, lib=lib)
    return bias_act(y, bias, False, act, lib=lib), E


def _pair(v):
    return (int(v), int(v)) if np.isscalar(v) else (int(v[0]), int(v[1]))


def conv2d(X, Wt, stride=1, pad=0, dil=1, threads: int = 0, with_E: bool = True, lib=None):
    """Y = conv2d(X, Wt) in FP64 from the definition (zero padding), and E.

    X: N x H x W x C (channels last); Wt: KH x KW x C x CO; Y: N x OH x OW x CO.
    stride, pad, dil: an int or an (h, w) pair.
    """
    lib = lib or load()
    X, Wt = _as_f64(X), _as_f64(Wt)
    if X.ndim != 4 or Wt.ndim != 4 or X.shape[3] != Wt.shape[2]:
        raise ValueError(f"shape mismatch {X.shape} * {Wt.shape}")
    N, H, W, C = X.shape
    KH, KW, _, CO = Wt.shape
    (sh, sw), (ph, pw), (dh, dw) = _pair(stride), _pair(pad), _pair(dil)
    OH = (H + 2 * ph - dh * (KH - 1) - 1) // sh + 1
    OW = (W + 2 * pw - dw * (KW - 1) - 1) // sw + 1
    if OH < 1 or OW < 1:
        raise ValueError("kernel window larger than the padded image")
    Y = np.empty((N, OH, OW, CO), dtype=np.float64)
    E = np.empty((N, OH, OW, CO), dtype=np.float64) if with_E else None
    rc = lib.oracle_conv2d_f64(N, H, W, C, CO, KH, KW, sh, sw, ph, pw, dh, dw, _ptr(X), _ptr(Wt), _ptr(Y),
                               _ptr(E) if with_E else None, int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_conv2d_f64 returned {rc}")
    return (Y, E) if with_E else Y


def conv_layer(X, Wt, bias=None, act="none", stride=1, pad=0, dil=1, threads=0, lib=None):
    """act(conv2d(X, Wt) + bias), one bias per output channel."""
    Y, E = conv2d(X, Wt, stride, pad, dil, threads=threads, lib=lib)
    shape = Y.shape
    out = bias_act(Y.reshape(-1, shape[3]), bias, True, act, lib=lib).reshape(shape)
    return out, E
