"""The pages' own kernel designs (naive and shared-memory tiled GEMM, naive and
shared-vector GEMV) compute the same products: parity with the FP64 oracle
within the FP32 bound 4 K 2^-24 E, on the workload shapes and ragged edges."""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32, gemm_uniform_f32, gemv_uniform_f32
from tests._util import parity_ratio

pytestmark = pytest.mark.gpu


def _t():
    import torch
    return torch


@pytest.mark.parametrize("variant", ["naive16", "naive32", "tiled16", "tiled32"])
@pytest.mark.parametrize("shape,seed", [((256, 256, 256), 1), ((1000, 700, 1500), 4),
                                        ((33, 65, 47), 9), ((1, 17, 5), 10)])
def test_ablation_gemm(variant, shape, seed):
    torch = _t()
    M, N, K = shape
    A, B = gemm_uniform_f32(seed, M, N, K)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.full((M, N), float("nan"), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    assert gtg.gtg_ablation_gemm_f32(variant, M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, C.data_ptr(), N, s) == 0
    ref, E = oracle.gemm(A, B)
    ratio, bad = parity_ratio(C.cpu().numpy(), ref, E, "f32", K)
    assert bad == 0, ratio


@pytest.mark.parametrize("variant", ["naive", "shared"])
@pytest.mark.parametrize("M,N", [(4096, 4096), (523, 1031), (300, 200), (257, 257)])
def test_ablation_gemv(variant, M, N):
    torch = _t()
    A, x, _ = gemv_uniform_f32(2 if M == 4096 else M + N, M, N, batch=1)
    dA, dx = torch.from_numpy(A).cuda(), torch.from_numpy(x).cuda()
    y = torch.full((M,), float("nan"), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    assert gtg.gtg_ablation_gemv_f32(variant, M, N, dA.data_ptr(), N, dx.data_ptr(), y.data_ptr(), s) == 0
    ref, E = oracle.gemv(A, x)
    ratio, bad = parity_ratio(y.cpu().numpy(), ref, E, "f32", N)
    assert bad == 0, ratio


def test_ablation_rejects_unknown_variant():
    assert gtg.gtg_ablation_gemm_f32(9, 4, 4, 4, 1 << 32, 4, 2 << 32, 4, 3 << 32, 4) == gtg.GTG_ERR_INVALID_VALUE
    assert gtg.gtg_ablation_gemv_f32(5, 4, 4, 1 << 32, 4, 2 << 32, 3 << 32) == gtg.GTG_ERR_INVALID_VALUE
