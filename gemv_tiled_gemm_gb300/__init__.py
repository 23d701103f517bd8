"""gtg -- dense GEMM and GEMV on one NVIDIA GB300, through libgtg.so.

This module is argument marshalling only: every step of every product runs
in the CUDA kernels behind the C ABI declared in ``include/gtg.h``. PyTorch
supplies device memory and streams; nothing here computes a result. If the
library has not been built the first call raises ``GtgError`` -- there is no
fallback of any kind.

Two layers:
  * the raw C ABI under the same names (``gemm_f32``, ``gemm_tf32``,
    ``gemm_bf16``, ``gemv_f32``, ``gtg_sync_status`` ...) taking integers for
    pointers, sizes and the stream handle, returning the status code;
  * tensor helpers ``matmul`` and ``matvec`` that take torch tensors (CUDA
    tensors, or host tensors that are copied in and the result copied out).
"""

from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
# GTG_DEBUG=1 loads the checking build (kernels verify every address they
# compute; see _build.py), made by _build.build(debug=True)
DEBUG = os.environ.get("GTG_DEBUG") == "1"
LIB_PATH = os.path.join(_PKG, "libgtg_debug.so" if DEBUG else "libgtg.so")

GTG_OK, GTG_ERR_INVALID_VALUE, GTG_ERR_MISALIGNED, GTG_ERR_ALIAS = 0, 1, 2, 3
GTG_ERR_UNSUPPORTED, GTG_ERR_LAUNCH, GTG_ERR_TIMEOUT, GTG_ERR_DEVICE = 4, 5, 6, 7
GTG_ERR_SCRATCH_LIMIT = 8
GTG_ERR_BOUNDS = 9
PREC = {"f32": 0, "tf32": 1, "bf16": 2, "f16": 3}
KERNELS = {0: "none", 1: "simt", 2: "tcgen05", 3: "zero_fill", 4: "gemv"}

# names and C signatures of every exported function of include/gtg.h
_i64, _ptr, _int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int


class GtgPlan(ctypes.Structure):
    _fields_ = [("kernel", _int), ("bm", _int), ("bn", _int), ("bk", _int), ("stages", _int),
                ("grid", _int), ("threads", _int), ("smem", _int), ("cluster", _int), ("splits", _int)]

    def as_dict(self) -> dict:
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["kernel"] = KERNELS.get(self.kernel, str(self.kernel))
        return d


class GtgEpilogue(ctypes.Structure):
    _fields_ = [("bias", _ptr), ("activation", _int)]


ACT = {"none": 0, "relu": 1}
_ep = ctypes.POINTER(GtgEpilogue)

SIGNATURES = {
    "gemm_f32": (_int, [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr]),
    "gemm_tf32": (_int, [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr]),
    "gemm_bf16": (_int, [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr]),
    "gemv_f32": (_int, [_i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _int, _ptr]),
    "gemm_tf32_noalloc": (_int, [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr]),
    "gemm_f32_ex": (_int, [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ep, _ptr]),
    "gemm_tf32_ex": (_int, [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ep, _ptr]),
    "gemm_bf16_ex": (_int, [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ep, _ptr]),
    "gemm_f16": (_int, [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr]),
    "gemm_f16_ex": (_int, [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ep, _ptr]),
    "gemm_strided_batched": (_int, [_int, _i64, _i64, _i64, _ptr, _i64, _i64, _ptr, _i64, _i64, _ptr, _i64, _i64,
                                    _i64, _ep, _ptr]),
    "gemv_f32_ex": (_int, [_i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _int, _ep, _ptr]),
    "gemm_host": (_int, [_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ep]),
    "gtg_pool_trim": (_int, []),
    "conv2d_nhwc": (_int, [_int] + [_i64] * 13 + [_ptr, _ptr, _ptr, _ep, _ptr]),
    "gemv_bf16": (_int, [_i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _int, _ptr]),
    "gemv_bf16_ex": (_int, [_i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _int, _ep, _ptr]),
    "gtg_ablation_gemm_f32": (_int, [_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr]),
    "gtg_ablation_gemv_f32": (_int, [_int, _i64, _i64, _ptr, _i64, _ptr, _ptr, _ptr]),
    "gtg_status_string": (ctypes.c_char_p, [_int]),
    "gtg_sync_status": (_int, [_ptr]),
    "gtg_last_cuda_error": (ctypes.c_char_p, []),
    "gtg_plan_gemm": (_int, [_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64,
                             ctypes.POINTER(GtgPlan)]),
    "gtg_plan_gemv": (_int, [_i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _int,
                             ctypes.POINTER(GtgPlan)]),
    "gtg_plan_gemv_bf16": (_int, [_i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _int,
                             ctypes.POINTER(GtgPlan)]),
    "gtg_version": (_int, []),
}

# include/gtg_testing.h: path switches, failure-path hooks and probes for
# tests and tuning (the failure-path hooks act only with GTG_TESTING=1 in the
# environment)
TESTING_SIGNATURES = {
    "gtg_force_simt": (None, [_int]),
    "gtg_force_gemm_splits": (None, [_int]),
    "gtg_force_c_store": (None, [_int]),
    "gtg_conv_force_path": (None, [_int]),
    "gtg_gemv_force_path": (None, [_int]),
    "gtg_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "gtg_test_drop_load": (_int, [_int]),
    "gtg_test_skip_vector_copy": (_int, [_int]),
    "gtg_test_inject_launch_failure": (_int, [_int]),
    "gtg_test_workspace_allocations": (ctypes.c_uint64, []),
    "gtg_plan_gemm_tf32_noalloc": (_int, [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64,
                                          ctypes.POINTER(GtgPlan)]),
    "gtg_debug_build": (_int, []),
    "gtg_test_debug_shrink_extent": (_int, [_int]),
    "gtg_plan_conv2d": (_int, [_int] + [_i64] * 13 + [_ptr, _ptr, _ptr, ctypes.POINTER(GtgPlan)]),
}


class GtgError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        text = status_string(status) if status >= 0 and _lib is not None else ""
        super().__init__(f"{what}: gtg status {status} ({text})" if what else f"gtg status {status} ({text})")


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded libgtg.so (ctypes). Raises GtgError if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                how = ("python -m gemv_tiled_gemm_gb300._build --debug" if DEBUG
                       else "python -c 'import __graft_entry__ as g; g.build()'")
                raise GtgError(-1, f"{LIB_PATH} is missing: build it first ({how})")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in {**SIGNATURES, **TESTING_SIGNATURES}.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


# ---- raw C ABI, same names and argument order as include/gtg.h ---------------

def gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    return lib().gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_tf32(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    return lib().gemm_tf32(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    return lib().gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_f16(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    return lib().gemm_f16(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_f16_ex(M, N, K, A, lda, B, ldb, C, ldc, ep=None, stream=0) -> int:
    return lib().gemm_f16_ex(M, N, K, A, lda, B, ldb, C, ldc, ctypes.byref(ep) if ep else None, stream)


def gemm_strided_batched(precision, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, batch,
                         ep=None, stream=0) -> int:
    prec = PREC[precision] if isinstance(precision, str) else precision
    return lib().gemm_strided_batched(prec, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, batch,
                                      ctypes.byref(ep) if ep else None, stream)


def gemv_f32(M, N, A, lda, x, ldx, y, ldy, batch, stream=0) -> int:
    return lib().gemv_f32(M, N, A, lda, x, ldx, y, ldy, batch, stream)


def gemm_tf32_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """gemm_tf32 without any device allocation (fixed 16 MiB scratch; see gtg.h)."""
    return lib().gemm_tf32_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream)


def epilogue(bias=0, activation="none"):
    """A gtg_epilogue for the *_ex calls (bias: device address or 0)."""
    return GtgEpilogue(bias or None, ACT[activation] if isinstance(activation, str) else int(activation))


def gemm_f32_ex(M, N, K, A, lda, B, ldb, C, ldc, ep=None, stream=0) -> int:
    return lib().gemm_f32_ex(M, N, K, A, lda, B, ldb, C, ldc, ctypes.byref(ep) if ep else None, stream)


def gemm_tf32_ex(M, N, K, A, lda, B, ldb, C, ldc, ep=None, stream=0) -> int:
    return lib().gemm_tf32_ex(M, N, K, A, lda, B, ldb, C, ldc, ctypes.byref(ep) if ep else None, stream)


def gemm_bf16_ex(M, N, K, A, lda, B, ldb, C, ldc, ep=None, stream=0) -> int:
    return lib().gemm_bf16_ex(M, N, K, A, lda, B, ldb, C, ldc, ctypes.byref(ep) if ep else None, stream)


def gemv_f32_ex(M, N, A, lda, x, ldx, y, ldy, batch, ep=None, stream=0) -> int:
    return lib().gemv_f32_ex(M, N, A, lda, x, ldx, y, ldy, batch, ctypes.byref(ep) if ep else None, stream)


def gemv_bf16(M, N, A, lda, x, ldx, y, ldy, batch, stream=0) -> int:
    return lib().gemv_bf16(M, N, A, lda, x, ldx, y, ldy, batch, stream)


def gemv_bf16_ex(M, N, A, lda, x, ldx, y, ldy, batch, ep=None, stream=0) -> int:
    return lib().gemv_bf16_ex(M, N, A, lda, x, ldx, y, ldy, batch, ctypes.byref(ep) if ep else None, stream)


def gemm_host(precision, M, N, K, A, lda, B, ldb, C, ldc, ep=None) -> int:
    prec = PREC[precision] if isinstance(precision, str) else precision
    return lib().gemm_host(prec, M, N, K, A, lda, B, ldb, C, ldc, ctypes.byref(ep) if ep else None)


def gtg_pool_trim() -> int:
    return lib().gtg_pool_trim()


def conv2d_nhwc(precision, N, H, W, C, CO, KH, KW, stride_h, stride_w, pad_h, pad_w, dil_h, dil_w, X, Wt, Y,
                ep=None, stream=0) -> int:
    prec = PREC[precision] if isinstance(precision, str) else precision
    return lib().conv2d_nhwc(prec, N, H, W, C, CO, KH, KW, stride_h, stride_w, pad_h, pad_w, dil_h, dil_w, X, Wt, Y,
                             ctypes.byref(ep) if ep else None, stream)


def conv_out_size(H, W, KH, KW, stride=1, pad=0, dil=1):
    """(OH, OW) of conv2d_nhwc for these sizes."""
    (sh, sw), (ph, pw), (dh, dw) = _pair(stride), _pair(pad), _pair(dil)
    return (H + 2 * ph - dh * (KH - 1) - 1) // sh + 1, (W + 2 * pw - dw * (KW - 1) - 1) // sw + 1


def _pair(v):
    return (int(v), int(v)) if isinstance(v, int) else (int(v[0]), int(v[1]))


ABLATION_GEMM = {"naive16": 0, "naive32": 1, "tiled16": 2, "tiled32": 3}
ABLATION_GEMV = {"naive": 0, "shared": 1}


def gtg_ablation_gemm_f32(variant, M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    v = ABLATION_GEMM[variant] if isinstance(variant, str) else variant
    return lib().gtg_ablation_gemm_f32(v, M, N, K, A, lda, B, ldb, C, ldc, stream)


def gtg_ablation_gemv_f32(variant, M, N, A, lda, x, y, stream=0) -> int:
    v = ABLATION_GEMV[variant] if isinstance(variant, str) else variant
    return lib().gtg_ablation_gemv_f32(v, M, N, A, lda, x, y, stream)


def status_string(status: int) -> str:
    return lib().gtg_status_string(status).decode()


def gtg_sync_status(stream=0) -> int:
    return lib().gtg_sync_status(stream)


def last_cuda_error() -> str:
    return lib().gtg_last_cuda_error().decode()


# ---- testing and tuning hooks (include/gtg_testing.h) ---------------------------

def gtg_force_simt(force: bool) -> None:
    lib().gtg_force_simt(1 if force else 0)


GEMV_PATHS = {"auto": 0, "cuda_cores": 1, "tensor_cores": 2, "no_ring": 3, "no_xi": 4}


def gtg_gemv_force_path(path="auto") -> None:
    """Tuning/testing hook for the GEMV kernel choice: "auto" (the planner),
    "cuda_cores" or "tensor_cores" (BF16 matrices at batch 3-8, whenever the
    layout allows), "no_ring" (CUDA cores, and the streaming kernel
    instead of the ring kernel for one or two vectors) or "no_xi" (CUDA
    cores, and at batch 8 the vectors staged one after another instead of
    interleaved)."""
    lib().gtg_gemv_force_path(GEMV_PATHS[path] if isinstance(path, str) else int(path))


def gtg_conv_force_path(mode: str) -> None:
    """Testing hook: conv2d_nhwc path, "auto", "explicit" (im2col + GEMM),
    "implicit" (any tensor-core kernel), "implicit_single" (single-CTA tiles)
    or "implicit_pair" (CTA pairs)."""
    lib().gtg_conv_force_path({"auto": 0, "explicit": 1, "implicit": 2, "implicit_single": 3,
                               "implicit_pair": 4}[mode])


def plan_conv2d(precision, N, H, W, C, CO, KH, KW, stride_h, stride_w, pad_h, pad_w, dil_h, dil_w, X, Wt, Y) -> dict:
    """The kernel a conv2d_nhwc call with these arguments would run (testing probe)."""
    plan = GtgPlan()
    st = lib().gtg_plan_conv2d(PREC[precision], N, H, W, C, CO, KH, KW, stride_h, stride_w, pad_h, pad_w, dil_h,
                               dil_w, X, Wt, Y, ctypes.byref(plan))
    if st != GTG_OK:
        raise GtgError(st, "gtg_plan_conv2d")
    return plan.as_dict()


def gtg_force_gemm_splits(splits: int) -> None:
    """Testing / tuning hook: split K of tensor-core GEMMs `splits` ways (0: planner's choice)."""
    lib().gtg_force_gemm_splits(int(splits))


def gtg_force_c_store(mode: str) -> None:
    """Testing / tuning hook: C stores of the CTA-pair GEMM, "auto", "direct" or "tensor"."""
    lib().gtg_force_c_store({"auto": 0, "direct": 1, "tensor": 2}[mode])


def gtg_set_wait_limit_ns(ns: int) -> None:
    lib().gtg_set_wait_limit_ns(ns)


def gtg_test_drop_load(slice_index: int) -> int:
    """Failure-path hook (needs GTG_TESTING=1): the next tensor-core GEMM leaves out one K-slice load."""
    return lib().gtg_test_drop_load(slice_index)


def gtg_test_skip_vector_copy(on: bool) -> int:
    """Failure-path hook (needs GTG_TESTING=1): the next bulk-staged GEMV announces its
    vector copies but issues none."""
    return lib().gtg_test_skip_vector_copy(1 if on else 0)


def gtg_test_inject_launch_failure(n: int) -> int:
    """Failure-path hook (needs GTG_TESTING=1): the n-th dispatched call from now on
    returns GTG_ERR_LAUNCH before launching anything (0 cancels)."""
    return lib().gtg_test_inject_launch_failure(int(n))


def gtg_test_workspace_allocations() -> int:
    return int(lib().gtg_test_workspace_allocations())


def plan_gemm_tf32_noalloc(M, N, K, A, lda, B, ldb, C, ldc) -> dict:
    """The kernel gemm_tf32_noalloc would launch for these arguments."""
    plan = GtgPlan()
    st = lib().gtg_plan_gemm_tf32_noalloc(M, N, K, A, lda, B, ldb, C, ldc, ctypes.byref(plan))
    if st != GTG_OK:
        raise GtgError(st, "gtg_plan_gemm_tf32_noalloc")
    return plan.as_dict()


def gtg_debug_build() -> int:
    return lib().gtg_debug_build()


def gtg_test_debug_shrink_extent(elements: int) -> int:
    """GTG_DEBUG builds (needs GTG_TESTING=1): the GEMV kernels check their loads
    against an extent `elements` shorter than the matrix, so their checks fire."""
    return lib().gtg_test_debug_shrink_extent(int(elements))


def gtg_version() -> int:
    return lib().gtg_version()


def plan_gemm(precision, M, N, K, A, lda, B, ldb, C, ldc) -> dict:
    plan = GtgPlan()
    st = lib().gtg_plan_gemm(PREC[precision], M, N, K, A, lda, B, ldb, C, ldc, ctypes.byref(plan))
    if st != GTG_OK:
        raise GtgError(st, "gtg_plan_gemm")
    return plan.as_dict()


def plan_gemv(M, N, A, lda, x, ldx, y, ldy, batch, precision="f32") -> dict:
    """The kernel a gemv_f32 (precision "f32") or gemv_bf16 ("bf16") call
    with these arguments would launch."""
    plan = GtgPlan()
    name = {"f32": "gtg_plan_gemv", "bf16": "gtg_plan_gemv_bf16"}[precision]
    st = getattr(lib(), name)(M, N, A, lda, x, ldx, y, ldy, batch, ctypes.byref(plan))
    if st != GTG_OK:
        raise GtgError(st, name)
    return plan.as_dict()


# ---- torch tensor helpers ------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream_handle(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _rowmajor_ld(t, name) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D row-major tensor (unit column stride)")
    return max(int(t.stride(0)), int(t.shape[1]), 1)


def _check(status: int, what: str):
    if status != GTG_OK:
        extra = f" [{last_cuda_error()}]" if status in (GTG_ERR_LAUNCH, GTG_ERR_DEVICE) else ""
        raise GtgError(status, what + extra)


_IN_DTYPE = {"f32": "float32", "tf32": "float32", "bf16": "bfloat16", "f16": "float16"}
_GEMM_EX = {"f32": gemm_f32_ex, "tf32": gemm_tf32_ex, "bf16": gemm_bf16_ex, "f16": gemm_f16_ex}


def matmul(A, B, precision: str = "f32", out=None, stream=None, bias=None, activation="none"):
    """C = act(A @ B + bias) on the GPU through gemm_<precision>_ex; C is FP32.

    A (M x K) and B (K x N) are row-major torch tensors: float32 for "f32" and
    "tf32", bfloat16 for "bf16", float16 for "f16". `bias` (N float32 values, one per output
    column) and `activation` ("none" or "relu") form the fused epilogue.
    CUDA tensors are used in place (on `stream`). Host tensors go through
    gemm_host, which copies A in and C out in blocks of rows while the blocks
    before and after them are multiplied (pinned host memory lets the copies
    overlap); the call then returns a host tensor and has synchronised.
    """
    torch = _torch()
    want = getattr(torch, _IN_DTYPE[precision])
    if A.dtype != want or B.dtype != want:
        raise TypeError(f"{precision} GEMM takes {want} operands, got {A.dtype}, {B.dtype}")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch {tuple(A.shape)} x {tuple(B.shape)}")
    host = not A.is_cuda
    M, K = A.shape
    N = B.shape[1]
    if host:
        # host operands: gemm_host overlaps the copies with the product
        if B.is_cuda:
            raise ValueError("A and B must both be host tensors or both device tensors")
        C = out if out is not None else torch.empty((M, N), dtype=torch.float32, pin_memory=A.is_pinned())
        if C.is_cuda or C.dtype != torch.float32 or tuple(C.shape) != (M, N):
            raise ValueError("out must be a host float32 tensor of shape (M, N)")
        hbias = None
        if bias is not None:
            if bias.dtype != torch.float32 or bias.numel() != N:
                raise ValueError(f"bias must hold {N} float32 values")
            hbias = bias.reshape(-1).cpu().contiguous()
        ep = epilogue(hbias.data_ptr() if hbias is not None else 0, activation)
        st = gemm_host(PREC[precision], M, N, K, A.data_ptr(), _rowmajor_ld(A, "A"), B.data_ptr(),
                       _rowmajor_ld(B, "B"), C.data_ptr(), _rowmajor_ld(C, "C"), ep)
        _check(st, "gemm_host")
        return C
    dA, dB = A, B
    if out is not None:
        C = out
    else:
        C = torch.empty((M, N), dtype=torch.float32, device=dA.device)
    dbias = _device_bias(bias, N, dA.device)
    ep = epilogue(dbias.data_ptr() if dbias is not None else 0, activation)
    st = _GEMM_EX[precision](M, N, K, dA.data_ptr(), _rowmajor_ld(dA, "A"), dB.data_ptr(),
                             _rowmajor_ld(dB, "B"), C.data_ptr(), _rowmajor_ld(C, "C"), ep,
                             _stream_handle(stream))
    _check(st, f"gemm_{precision}")
    return C


def _device_bias(bias, n, device):
    if bias is None:
        return None
    torch = _torch()
    if bias.dtype != torch.float32 or bias.numel() != n:
        raise ValueError(f"bias must hold {n} float32 values")
    return bias.reshape(-1).to(device, non_blocking=True).contiguous()


def matvec(A, x, out=None, stream=None, bias=None, activation="none"):
    """y = act(A @ x + bias) (x of shape (N,)), or Y = act(X @ A^T + bias)
    per row of X (shape (batch, N)): a fully connected layer with weight A.

    A in float32 (gemv_f32_ex) or bfloat16 (gemv_bf16_ex); x, the bias and the
    result in float32; batch <= 8; `bias` holds M values (one per output).
    Host tensors are copied in and the result copied back, as in `matmul`.
    """
    torch = _torch()
    if A.dtype not in (torch.float32, torch.bfloat16) or x.dtype != torch.float32:
        raise TypeError("matvec takes a float32 or bfloat16 matrix and a float32 vector")
    fn, name = (gemv_bf16_ex, "gemv_bf16") if A.dtype == torch.bfloat16 else (gemv_f32_ex, "gemv_f32")
    single = x.dim() == 1
    X = x.unsqueeze(0) if single else x
    if A.dim() != 2 or X.dim() != 2 or X.shape[1] != A.shape[1]:
        raise ValueError(f"shape mismatch {tuple(A.shape)} x {tuple(x.shape)}")
    host = not A.is_cuda
    dA = A.to("cuda", non_blocking=True) if host else A
    dX = X.to("cuda", non_blocking=True) if host else X
    M, N = dA.shape
    batch = dX.shape[0]
    if out is not None and not host:
        Y = out.unsqueeze(0) if single else out
    else:
        Y = torch.empty((batch, M), dtype=torch.float32, device=dA.device)
    dbias = _device_bias(bias, M, dA.device)
    ep = epilogue(dbias.data_ptr() if dbias is not None else 0, activation)
    st = fn(M, N, dA.data_ptr(), _rowmajor_ld(dA, "A"), dX.data_ptr(), _rowmajor_ld(dX, "x"),
            Y.data_ptr(), _rowmajor_ld(Y, "y"), batch, ep, _stream_handle(stream))
    _check(st, name)
    if host:
        res = torch.empty((batch, M), dtype=torch.float32, pin_memory=A.is_pinned())
        res.copy_(Y, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        Y = res
        if out is not None:
            out.copy_(Y[0] if single else Y)
            return out
    return Y[0] if single else Y


def sync_status(stream=None) -> None:
    """Wait for the stream and raise GtgError if a kernel reported a device-side failure."""
    st = gtg_sync_status(_stream_handle(stream))
    _check(st, "device status")


def conv2d(X, Wt, stride=1, pad=0, dil=1, precision=None, out=None, stream=None, bias=None, activation="none"):
    """A convolutional layer: Y = act(conv(X, Wt) + bias) through conv2d_nhwc.

    X: (N, H, W, C) channels last; Wt: (KH, KW, C, CO); Y: (N, OH, OW, CO)
    float32. precision defaults to the tensors' type ("f32" for float32,
    "bf16" / "f16" for bfloat16 / float16); "tf32" runs float32 tensors on
    the TF32 tensor path. `bias` holds CO float32 values (one per output
    channel). Host tensors are copied in and the result copied back.
    """
    torch = _torch()
    kinds = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}
    if X.dtype not in kinds or Wt.dtype != X.dtype:
        raise TypeError("conv2d takes float32, bfloat16 or float16 X and Wt of the same type")
    prec = precision or kinds[X.dtype]
    if (prec in ("f32", "tf32")) != (X.dtype == torch.float32) or (prec in ("bf16", "f16") and kinds[X.dtype] != prec):
        raise TypeError(f"precision {prec} does not match tensors of type {X.dtype}")
    if X.dim() != 4 or Wt.dim() != 4 or X.shape[3] != Wt.shape[2]:
        raise ValueError(f"shape mismatch {tuple(X.shape)} * {tuple(Wt.shape)}")
    N, H, W, C = X.shape
    KH, KW, _, CO = Wt.shape
    (sh, sw), (ph, pw), (dh, dw) = _pair(stride), _pair(pad), _pair(dil)
    OH, OW = conv_out_size(H, W, KH, KW, (sh, sw), (ph, pw), (dh, dw))
    host = not X.is_cuda
    dX = (X.to("cuda", non_blocking=True) if host else X).contiguous()
    dW = (Wt.to("cuda", non_blocking=True) if host else Wt).contiguous()
    if out is not None and not host:
        Y = out
    else:
        Y = torch.empty((N, OH, OW, CO), dtype=torch.float32, device=dX.device)
    if not Y.is_contiguous() or tuple(Y.shape) != (N, OH, OW, CO):
        raise ValueError("out must be a contiguous (N, OH, OW, CO) float32 tensor")
    dbias = _device_bias(bias, CO, dX.device)
    ep = epilogue(dbias.data_ptr() if dbias is not None else 0, activation)
    st = conv2d_nhwc(prec, N, H, W, C, CO, KH, KW, sh, sw, ph, pw, dh, dw, dX.data_ptr(), dW.data_ptr(),
                     Y.data_ptr(), ep, _stream_handle(stream))
    _check(st, "conv2d_nhwc")
    if host:
        res = torch.empty_like(Y, device="cpu", pin_memory=X.is_pinned())
        res.copy_(Y, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        if out is not None:
            out.copy_(res)
            return out
        return res
    return Y
