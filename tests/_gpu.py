"""GPU-side test helpers: run the C-ABI calls with guard bands around the output."""

from __future__ import annotations

import numpy as np

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import bf16_bits_to_f32, f16_bits_to_f32
from tests._util import parity_ratio

CANARY = np.float32(-12345.5)
BF16_NAN = np.uint16(0x7FC0)
F16_NAN = np.uint16(0x7E00)


def torch():
    import torch as t
    return t


def _dev_buffer(values: np.ndarray, rows: int, cols: int, ld: int, offset: int, fill):
    """A flat device buffer holding `values` (rows x cols) at `offset` elements
    with leading dimension `ld`; every other element is `fill`."""
    t = torch()
    host = np.full(offset + rows * ld + 8, fill, dtype=values.dtype)
    if rows and cols:
        host[offset:offset + rows * ld].reshape(rows, ld)[:, :cols] = values
    if values.dtype == np.uint16:
        return t.from_numpy(host.view(np.int16)).cuda()
    return t.from_numpy(host).cuda()


def run_gemm(prec: str, A: np.ndarray, B: np.ndarray, lda=None, ldb=None, ldc=None,
             a_off=0, b_off=0, c_off=0, stream=None, expect_kernel=None):
    """C = A @ B through gemm_<prec>; checks guard bands; returns C (M x N float32)."""
    t = torch()
    M, K = A.shape
    N = B.shape[1]
    lda = lda or max(K, 1)
    ldb = ldb or max(N, 1)
    ldc = ldc or max(N, 1)
    fill = {"bf16": BF16_NAN, "f16": F16_NAN}.get(prec, np.float32(np.nan))
    dA = _dev_buffer(A, M, K, lda, a_off, fill)
    dB = _dev_buffer(B, K, N, ldb, b_off, fill)
    # C: one guard row above and below, padding columns, NaN in the interior
    guard = ldc
    host_c = np.full(c_off + (M + 2) * ldc + 8, CANARY, dtype=np.float32)
    body = np.zeros(host_c.shape, dtype=bool)
    body[c_off + guard:c_off + guard + M * ldc].reshape(M, ldc)[:, :N] = True
    host_c[body] = np.nan
    dC = t.from_numpy(host_c).cuda()
    esz = 2 if prec in ("bf16", "f16") else 4
    pA = dA.data_ptr() + a_off * esz
    pB = dB.data_ptr() + b_off * esz
    pC = dC.data_ptr() + (c_off + guard) * 4
    if expect_kernel is not None:
        plan = gtg.plan_gemm(prec, M, N, K, pA, lda, pB, ldb, pC, ldc)
        assert plan["kernel"] == expect_kernel, plan
    s = stream if stream is not None else t.cuda.current_stream()
    fn = {"f32": gtg.gemm_f32, "tf32": gtg.gemm_tf32, "bf16": gtg.gemm_bf16, "f16": gtg.gemm_f16}[prec]
    st = fn(M, N, K, pA, lda, pB, ldb, pC, ldc, int(s.cuda_stream))
    assert st == gtg.GTG_OK, gtg.status_string(st)
    assert gtg.gtg_sync_status(int(s.cuda_stream)) == gtg.GTG_OK
    out = dC.cpu().numpy()
    assert np.all(out[~body] == CANARY), "write outside C"
    return out[c_off + guard:c_off + guard + M * ldc].reshape(M, ldc)[:, :N].copy()


def run_gemv(A: np.ndarray, X: np.ndarray, lda=None, ldx=None, ldy=None, a_off=0, stream=None, prec="f32",
             x_off=0):
    """Y = X @ A^T through gemv_f32, or gemv_bf16 when prec == "bf16" (A then
    holds BF16 bit patterns); X: batch x N. Checks guard bands."""
    t = torch()
    M, N = A.shape
    batch = X.shape[0]
    lda = lda or max(N, 1)
    ldx = ldx or max(N, 1)
    ldy = ldy or max(M, 1)
    dA = _dev_buffer(A, M, N, lda, a_off, BF16_NAN if prec == "bf16" else np.float32(np.nan))
    dX = _dev_buffer(X, batch, N, ldx, x_off, np.float32(np.nan))
    host_y = np.full((batch + 2) * ldy + 8, CANARY, dtype=np.float32)
    body = np.zeros(host_y.shape, dtype=bool)
    body[ldy:ldy + batch * ldy].reshape(batch, ldy)[:, :M] = True
    host_y[body] = np.nan
    dY = t.from_numpy(host_y).cuda()
    s = stream if stream is not None else t.cuda.current_stream()
    fn, esz = (gtg.gemv_bf16, 2) if prec == "bf16" else (gtg.gemv_f32, 4)
    st = fn(M, N, dA.data_ptr() + esz * a_off, lda, dX.data_ptr() + 4 * x_off, ldx,
            dY.data_ptr() + 4 * ldy, ldy, batch, int(s.cuda_stream))
    assert st == gtg.GTG_OK, gtg.status_string(st)
    assert gtg.gtg_sync_status(int(s.cuda_stream)) == gtg.GTG_OK
    out = dY.cpu().numpy()
    assert np.all(out[~body] == CANARY), "write outside y"
    return out[ldy:ldy + batch * ldy].reshape(batch, ldy)[:, :M].copy()


def as_f32(prec, X):
    if prec == "bf16":
        return bf16_bits_to_f32(X)
    return f16_bits_to_f32(X) if prec == "f16" else X


def check_gemm(prec, A, B, C, rows=None):
    """Element-wise parity of C (or C[rows]) against the FP64 oracle."""
    Af, Bf = as_f32(prec, A), as_f32(prec, B)
    K = A.shape[1]
    if rows is not None:
        ref, E = oracle.gemm(Af[rows], Bf)
        got = C[rows]
    else:
        ref, E = oracle.gemm(Af, Bf)
        got = C
    ratio, bad = parity_ratio(got, ref, E, prec, K)
    assert bad == 0, f"{bad} elements out of bound (max ratio {ratio:.3g})"
    return ratio


def sample_rows(M, bm=128, seed=0):
    """First and last row plus one random row in every bm-row band."""
    rng = np.random.default_rng(seed)
    rows = {0, M - 1}
    for b0 in range(0, M, bm):
        rows.add(int(rng.integers(b0, min(b0 + bm, M))))
    return np.array(sorted(rows))
