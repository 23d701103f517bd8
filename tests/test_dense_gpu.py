"""Fully connected layers: the fused epilogue act(product + bias) on every
kernel path, against the FP64 oracle (oracle.dense_layer / dense_vector).

Bound per output: the product's bound (E from the oracle) plus one FP32
rounding of the bias addition, 2^-23 |ref|; ReLU is 1-Lipschitz and so adds
nothing.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32, bf16_bits_to_f32
from tests._util import BOUNDS

pytestmark = pytest.mark.gpu


def _t():
    import torch
    return torch


def _check(got, ref, E, prec, K):
    bound = BOUNDS[prec](E, K) + 2.0 ** -23 * np.abs(ref)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(np.isfinite(got))
    bad = int((err > bound).sum())
    assert bad == 0, f"{bad} outputs out of bound (max ratio {float((err / np.maximum(bound, 1e-300)).max()):.3g})"


GEMM_CASES = [
    ("f32", (2048, 2048, 64), "simt"),     # 128 x 128 tiles, no split
    ("f32", (256, 256, 256), "simt"),      # split K: epilogue in the reduction
    ("tf32", (1024, 1024, 96), "tcgen05"),
    ("bf16", (1000, 712, 208), "tcgen05"),   # single-CTA kernel, ragged (16-byte rows)
    ("bf16", (4096, 4160, 128), "tcgen05"),  # CTA-pair kernel, partial last column tile
]


@pytest.mark.parametrize("act", ["relu", "none"])
@pytest.mark.parametrize("with_bias", [True, False])
@pytest.mark.parametrize("prec,shape,kernel", GEMM_CASES)
def test_dense_layer_gemm(prec, shape, kernel, with_bias, act):
    if not with_bias and act == "none":
        pytest.skip("plain product: covered by test_gemm_gpu")
    torch = _t()
    M, N, K = shape
    g = PCG32(500 + M % 97 + K)
    if prec == "bf16":
        Ab, Bb = g.normal_bf16((M, K)), g.normal_bf16((K, N))
        A, B = bf16_bits_to_f32(Ab), bf16_bits_to_f32(Bb)
        dA = torch.from_numpy(Ab.view(np.int16)).view(torch.bfloat16).cuda()
        dB = torch.from_numpy(Bb.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        A, B = g.uniform_f32((M, K)), g.uniform_f32((K, N))
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    bias = g.uniform_f32((N,)) if with_bias else None
    C = gtg.matmul(dA, dB, prec, bias=torch.from_numpy(bias).cuda() if with_bias else None,
                   activation=act)
    plan = gtg.plan_gemm(prec, M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, C.data_ptr(), N)
    assert plan["kernel"] == kernel
    got = C.cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 97)), [M - 1]]))
    ref, E = oracle.dense_layer(A[rows], B, bias, act)
    _check(got[rows], ref, E, prec, K)
    if act == "relu":
        assert np.all(got >= 0) and (got == 0).any()


GEMV_CASES = [
    (4096, 4096, 1, 0),      # streaming kernel
    (4096, 4096, 8, 0),      # column-split kernel
    (1523, 1030, 4, 2),      # column-split kernel, ragged width, padded rows
    (300, 7000, 8, 0),       # chunked x: round kernel
    (257, 1001, 3, 1),       # unaligned rows: scalar round kernel
    (257, 1001, 1, 1),       # unaligned rows at batch 1: peeled streaming kernel
]


@pytest.mark.parametrize("act", ["relu", "none"])
@pytest.mark.parametrize("M,N,batch,pad", GEMV_CASES)
def test_dense_layer_gemv(M, N, batch, pad, act):
    torch = _t()
    g = PCG32(600 + M + batch)
    A = g.uniform_f32((M, N))
    X = g.uniform_f32((batch, N))
    bias = g.uniform_f32((M,))
    lda = N + pad
    hostA = np.zeros((M, lda), dtype=np.float32)
    hostA[:, :N] = A
    dA = torch.from_numpy(hostA).cuda()
    dX = torch.from_numpy(X).cuda()
    dY = torch.full((batch, M), float("nan"), device="cuda")
    db = torch.from_numpy(bias).cuda()
    s = int(torch.cuda.current_stream().cuda_stream)
    st = gtg.gemv_f32_ex(M, N, dA.data_ptr(), lda, dX.data_ptr(), N, dY.data_ptr(), M, batch,
                         gtg.epilogue(db.data_ptr(), act), s)
    assert st == gtg.GTG_OK
    assert gtg.gtg_sync_status(s) == gtg.GTG_OK
    Y = dY.cpu().numpy()
    for b in range(batch):
        ref, E = oracle.dense_vector(A, X[b], bias, act)
        _check(Y[b], ref, E, "f32", N)


def test_tensor_helper_dense_vector():
    torch = _t()
    g = PCG32(700)
    W = g.uniform_f32((512, 768))
    x = g.uniform_f32((768,))
    b = g.uniform_f32((512,))
    y = gtg.matvec(torch.from_numpy(W).cuda(), torch.from_numpy(x).cuda(),
                   bias=torch.from_numpy(b).cuda(), activation="relu").cpu().numpy()
    ref, E = oracle.dense_vector(W, x, b, "relu")
    _check(y, ref, E, "f32", 768)


@pytest.mark.parametrize("prec", ["f32", "tf32", "bf16"])
def test_empty_product_gives_activated_bias(prec):
    torch = _t()
    M, N = 37, 45
    bias = PCG32(701).uniform_f32((N,))
    dt = torch.bfloat16 if prec == "bf16" else torch.float32
    A = torch.zeros((M, 0), dtype=dt, device="cuda")
    B = torch.zeros((0, N), dtype=dt, device="cuda")
    C = gtg.matmul(A, B, prec, bias=torch.from_numpy(bias).cuda(), activation="relu").cpu().numpy()
    assert np.array_equal(C, np.tile(np.maximum(bias, 0), (M, 1)))
    y = gtg.matvec(torch.zeros((N, 0), device="cuda"), torch.zeros((0,), device="cuda"),
                   bias=torch.from_numpy(bias).cuda()).cpu().numpy()
    assert np.array_equal(y, bias)
