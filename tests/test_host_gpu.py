"""gemm_host: products of operands in host memory (copies overlapped with the
product, row block by row block) against the FP64 oracle, element by element,
through the C ABI; and the host-tensor path of matmul, which calls it."""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from tests._gpu import CANARY, as_f32, check_gemm
from tests._util import parity_ratio
from seeded import PCG32

pytestmark = pytest.mark.gpu


def _t():
    import torch
    return torch


def _draw(prec, g, shape, sigma=1.0):
    if prec == "bf16":
        return g.normal_bf16(shape, sigma)
    if prec == "f16":
        return g.normal_f16(shape, sigma)
    return g.uniform_f32(shape)


def _host(values, rows, cols, ld, pinned):
    """A host buffer (torch tensor, pinned or pageable) holding `values` with
    leading dimension `ld`; padding columns hold NaN patterns."""
    torch = _t()
    fill = {np.dtype(np.uint16): np.uint16(0x7FC0)}.get(values.dtype, np.float32(np.nan))
    buf = np.full((max(rows, 1), ld), fill, dtype=values.dtype)
    buf[:rows, :cols] = values
    t = torch.from_numpy(buf.view(np.int16) if values.dtype == np.uint16 else buf)
    return t.pin_memory() if pinned else t


def run_host(prec, A, B, lda=None, ldb=None, ldc=None, pinned=True, bias=None, act="none"):
    """C through gemm_host with host buffers; a guard row after C is checked."""
    torch = _t()
    M, K = A.shape
    N = B.shape[1]
    lda, ldb, ldc = lda or max(K, 1), ldb or max(N, 1), ldc or max(N, 1)
    hA, hB = _host(A, M, K, lda, pinned), _host(B, K, N, ldb, pinned)
    hC = torch.full(((M + 1) * ldc,), float(CANARY))
    hC[:M * ldc].view(M, ldc)[:, :N] = float("nan")
    if pinned:
        hC = hC.pin_memory()
    hb = torch.from_numpy(bias) if bias is not None else None
    ep = gtg.epilogue(hb.data_ptr() if hb is not None else 0, act) if (bias is not None or act != "none") else None
    st = gtg.gemm_host(prec, M, N, K, hA.data_ptr(), lda, hB.data_ptr(), ldb, hC.data_ptr(), ldc, ep)
    assert st == gtg.GTG_OK, gtg.status_string(st)
    out = hC.numpy()
    full = out[:M * ldc].reshape(M, ldc)
    assert np.all(full[:, N:] == CANARY) and np.all(out[M * ldc:] == CANARY), "write outside C"
    return full[:, :N].copy()


CASES = [
    # (precision, M, N, K): several row blocks with a ragged last one, and one block
    ("bf16", 2300, 200, 136),
    ("f16", 1100, 72, 64),
    ("tf32", 777, 96, 100),
    ("f32", 1030, 33, 47),          # SIMT: odd sizes
    ("bf16", 100, 64, 32),          # a single block
    ("bf16", 5000, 300, 72),        # tall: every panel of B, then the rest of A
    ("f16", 300, 3000, 40),         # wide: every block of A, then the rest of B
    ("tf32", 1500, 1700, 36),       # both in pieces, ragged in both directions
    ("f32", 700, 530, 20),          # SIMT product regions
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(str(v) for v in c))
def test_gemm_host_matches_oracle(case):
    prec, M, N, K = case
    g = PCG32(3000 + M + N + K)
    A = _draw(prec, g, (M, K))
    B = _draw(prec, g, (K, N), K ** -0.5)
    C = run_host(prec, A, B)
    check_gemm(prec, A, B, C)


def test_gemm_host_padded_leading_dimensions_and_pageable_memory():
    g = PCG32(3100)
    M, N, K = 1500, 80, 96
    A = _draw("bf16", g, (M, K))
    B = _draw("bf16", g, (K, N), K ** -0.5)
    for pinned in (True, False):
        C = run_host("bf16", A, B, lda=K + 24, ldb=N + 8, ldc=N + 5, pinned=pinned)
        check_gemm("bf16", A, B, C)


@pytest.mark.parametrize("prec", ["bf16", "f32"])
def test_gemm_host_bias_and_relu(prec):
    g = PCG32(3200)
    M, N, K = 1300, 48, 64
    A = _draw(prec, g, (M, K))
    B = _draw(prec, g, (K, N), K ** -0.5)
    bias = g.uniform_f32((N,))
    C = run_host(prec, A, B, bias=bias, act="relu")
    ref, E = oracle.dense_layer(as_f32(prec, A), as_f32(prec, B), bias, "relu")
    ratio, bad = parity_ratio(C, ref, E, prec, K, rel=2.0 ** -23)
    assert bad == 0, f"{bad} elements out of bound (max ratio {ratio:.3g})"
    assert np.all(C >= 0)


def test_pool_trim_then_call_again():
    g = PCG32(3250)
    A = _draw("bf16", g, (700, 64))
    B = _draw("bf16", g, (64, 600), 0.125)
    C1 = run_host("bf16", A, B)
    assert gtg.gtg_pool_trim() == gtg.GTG_OK
    C2 = run_host("bf16", A, B)
    assert np.array_equal(C1, C2)
    check_gemm("bf16", A, B, C2)


def test_gemm_host_empty_reduction_gives_the_epilogue_of_zero():
    g = PCG32(3300)
    M, N = 600, 24
    bias = g.uniform_f32((N,))
    C = run_host("bf16", np.zeros((M, 0), np.uint16), np.zeros((0, N), np.uint16), bias=bias)
    assert np.array_equal(C, np.broadcast_to(bias, (M, N)))


def test_matmul_on_host_tensors_uses_gemm_host():
    torch = _t()
    g = PCG32(3400)
    M, N, K = 2049, 128, 256
    A = _draw("bf16", g, (M, K))
    B = _draw("bf16", g, (K, N), K ** -0.5)
    tA = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16)
    tB = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16)
    Ch = gtg.matmul(tA.pin_memory(), tB.pin_memory(), "bf16")
    assert not Ch.is_cuda
    check_gemm("bf16", A, B, Ch.numpy())
    # the same product as one launch on device operands, up to the rounding
    # order of the kernel each row block is planned with
    Cd = gtg.matmul(tA.cuda(), tB.cuda(), "bf16").cpu()
    ref, E = oracle.gemm(as_f32("bf16", A), as_f32("bf16", B))
    assert parity_ratio(Cd.numpy(), ref, E, "bf16", K)[1] == 0
