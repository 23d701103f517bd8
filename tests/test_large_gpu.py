"""Maximum sizes: outputs and matrices with more than 2^31 elements, and very
long reductions. They check the 64-bit index arithmetic of every kernel (row
* leading dimension overflows 32 bits) and the accumulation over K far past
the tile depth. Inputs are closed forms built on the device (exact integers)
or seeded draws, compared with exact sums or with the FP64 oracle on sampled
rows.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32, bf16_bits_to_f32
from tests._util import parity_ratio

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _torch():
    import torch
    return torch


def _sync(stream):
    assert gtg.gtg_sync_status(int(stream.cuda_stream)) == gtg.GTG_OK


def test_gemv_matrix_beyond_2_31_elements():
    torch = _torch()
    M, N = 65536, 36868              # 2.42e9 elements (9.7 GB), N % 4 == 0
    A = torch.empty((M, N), dtype=torch.float32, device="cuda")
    j = torch.arange(N, device="cuda")
    for r0 in range(0, M, 4096):     # A[i][j] = ((i + j) mod 5) - 2, built in row blocks
        i = torch.arange(r0, r0 + 4096, device="cuda")[:, None]
        A[r0:r0 + 4096] = (((i + j[None, :]) % 5) - 2).float()
    x = torch.ones((2, N), dtype=torch.float32, device="cuda")
    x[1] = 2.0
    y = torch.full((2, M), float("nan"), device="cuda")
    s = torch.cuda.current_stream()
    st = gtg.gemv_f32(M, N, A.data_ptr(), N, x.data_ptr(), N, y.data_ptr(), M, 2, int(s.cuda_stream))
    assert st == gtg.GTG_OK
    _sync(s)
    # exact: for row i, sum_j ((i + j) mod 5) - 2 over j < N
    i = np.arange(M)
    q, r = divmod(N, 5)
    base = q * (0 + 1 + 2 + 3 + 4 - 10)          # full cycles contribute 0
    extra = np.zeros(M, dtype=np.int64)
    for t in range(r):                            # the r leftover columns j = 5q + t
        extra += ((i + 5 * q + t) % 5) - 2
    want = (base + extra).astype(np.float64)
    got = y.cpu().numpy()
    assert np.array_equal(got[0], want) and np.array_equal(got[1], 2 * want)
    del A


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
def test_gemm_output_beyond_2_31_elements(prec):
    torch = _torch()
    M = N = 49152                     # C has 2.42e9 elements (9.7 GB)
    K = 64 if prec == "bf16" else 32
    g = PCG32(77)
    if prec == "bf16":
        Ab, Bb = g.normal_bf16((M, K)), g.normal_bf16((K, N))
        Af, Bf = bf16_bits_to_f32(Ab), bf16_bits_to_f32(Bb)
        dA = torch.from_numpy(Ab.view(np.int16)).view(torch.bfloat16).cuda()
        dB = torch.from_numpy(Bb.view(np.int16)).view(torch.bfloat16).cuda()
        fn = gtg.gemm_bf16
    else:
        Af, Bf = g.uniform_f32((M, K)), g.uniform_f32((K, N))
        dA, dB = torch.from_numpy(Af).cuda(), torch.from_numpy(Bf).cuda()
        fn = gtg.gemm_tf32
    C = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream()
    st = fn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, C.data_ptr(), N, int(s.cuda_stream))
    assert st == gtg.GTG_OK
    _sync(s)
    rows = np.array([0, 1, 22000, 43690, 43691, M - 2, M - 1])   # 43691 * N > 2^31
    got = C[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref, E = oracle.gemm(Af[rows], Bf)
    ratio, bad = parity_ratio(got, ref, E, prec, K)
    assert bad == 0, ratio
    assert not torch.isnan(C).any().item()
    del C


def test_simt_output_beyond_2_31_elements():
    torch = _torch()
    M = N = 46400                     # 2.15e9 outputs
    K = 8
    g = PCG32(78)
    Af, Bf = g.uniform_f32((M, K)), g.uniform_f32((K, N))
    dA, dB = torch.from_numpy(Af).cuda(), torch.from_numpy(Bf).cuda()
    C = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream()
    assert gtg.gemm_f32(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, C.data_ptr(), N,
                        int(s.cuda_stream)) == gtg.GTG_OK
    _sync(s)
    rows = np.array([0, 46282, 46283, M - 1])                      # 46283 * N > 2^31
    got = C[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref, E = oracle.gemm(Af[rows], Bf)
    ratio, bad = parity_ratio(got, ref, E, "f32", K)
    assert bad == 0, ratio
    assert not torch.isnan(C).any().item()
    del C


@pytest.mark.parametrize("prec", ["bf16", "tf32", "f32"])
def test_very_long_reduction(prec):
    torch = _torch()
    M, N, K = 256, 256, 131072        # 2048 BF16 / 4096 TF32 K-slices per tile
    g = PCG32(79)
    if prec == "bf16":
        Ab, Bb = g.normal_bf16((M, K), K ** -0.5), g.normal_bf16((K, N), K ** -0.5)
        Af, Bf = bf16_bits_to_f32(Ab), bf16_bits_to_f32(Bb)
        dA = torch.from_numpy(Ab.view(np.int16)).view(torch.bfloat16).cuda()
        dB = torch.from_numpy(Bb.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        Af, Bf = g.uniform_f32((M, K)), g.uniform_f32((K, N))
        dA, dB = torch.from_numpy(Af).cuda(), torch.from_numpy(Bf).cuda()
    fn = {"bf16": gtg.gemm_bf16, "tf32": gtg.gemm_tf32, "f32": gtg.gemm_f32}[prec]
    C = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream()
    assert fn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, C.data_ptr(), N, int(s.cuda_stream)) == gtg.GTG_OK
    _sync(s)
    rows = np.array([0, 77, 128, 255])
    ref, E = oracle.gemm(Af[rows], Bf)
    ratio, bad = parity_ratio(C.cpu().numpy()[rows], ref, E, prec, K)
    assert bad == 0, ratio
