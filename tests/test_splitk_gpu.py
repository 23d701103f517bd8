"""Tensor-core GEMMs with K split into ranges (partial tiles added in order
by a second kernel), forced through the tuning hook, against the oracle."""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32, bf16_bits_to_f32
from tests._gpu import check_gemm, run_gemm
from tests._util import parity_ratio

pytestmark = pytest.mark.gpu


@pytest.fixture
def force_splits():
    yield gtg.gtg_force_gemm_splits
    gtg.gtg_force_gemm_splits(0)


def _inputs(prec, seed, M, N, K):
    g = PCG32(seed)
    if prec == "bf16":
        return g.normal_bf16((M, K)), g.normal_bf16((K, N))
    if prec == "f16":
        return g.normal_f16((M, K)), g.normal_f16((K, N))
    return g.uniform_f32((M, K)), g.uniform_f32((K, N))


@pytest.mark.parametrize("prec,M,N,K,splits", [
    ("bf16", 1024, 1024, 2048, 2),
    ("bf16", 300, 520, 1000, 3),        # ragged M, N and K (K not a multiple of 3 x 64)
    ("bf16", 100, 72, 960, 5),          # one tile
    ("f16", 640, 384, 4096, 4),
    ("tf32", 512, 512, 1500, 4),        # TF32: K slices of 32, transposed B
    ("bf16", 128, 64, 128, 8),          # 2 slices: a split cannot exceed them (taken as 1)
])
def test_split_k_matches_oracle(force_splits, prec, M, N, K, splits):
    A, B = _inputs(prec, 3000 + M + K, M, N, K)
    force_splits(splits)
    plan = gtg.plan_gemm(prec, M, N, K, 1 << 32, K, 2 << 32, N, 3 << 32, N)
    bk = 32 if prec == "tf32" else 64
    if (K + bk - 1) // bk >= 2 * splits:
        assert plan["splits"] == splits, plan
    else:
        assert plan["splits"] == 1, plan
    C = run_gemm(prec, A, B, ldc=N + 8, expect_kernel="tcgen05")
    check_gemm(prec, A, B, C)


def test_split_k_with_epilogue(force_splits):
    """The reduction applies bias and ReLU once, after all partial tiles are added."""
    torch = pytest.importorskip("torch")
    g = PCG32(3100)
    M, N, K = 700, 264, 1536
    A, B = g.normal_bf16((M, K)), g.normal_bf16((K, N))
    bias = g.uniform_f32((N,))
    force_splits(3)
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.empty((M, N), device="cuda")
    db = torch.from_numpy(bias).cuda()
    s = int(torch.cuda.current_stream().cuda_stream)
    st = gtg.gemm_bf16_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N,
                          gtg.epilogue(db.data_ptr(), "relu"), s)
    assert st == gtg.GTG_OK and gtg.gtg_sync_status(s) == gtg.GTG_OK
    ref, E = oracle.dense_layer(bf16_bits_to_f32(A), bf16_bits_to_f32(B), bias, "relu")
    ratio, bad = parity_ratio(dC.cpu().numpy(), ref, E, "bf16", K, rel=2.0 ** -23)
    assert bad == 0, ratio


def test_split_k_is_deterministic(force_splits):
    A, B = _inputs("bf16", 3200, 512, 512, 4096)
    force_splits(4)
    C1 = run_gemm("bf16", A, B)
    C2 = run_gemm("bf16", A, B)
    assert np.array_equal(C1, C2)


def test_split_k_leaves_batches_alone(force_splits):
    """Strided batches never split (each item keeps its whole K range)."""
    torch = pytest.importorskip("torch")
    g = PCG32(3300)
    batch, M, N, K = 3, 256, 192, 1024
    A, B = g.normal_bf16((batch, M, K)), g.normal_bf16((batch, K, N))
    force_splits(4)
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.empty((batch, M, N), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    assert gtg.gemm_strided_batched("bf16", M, N, K, dA.data_ptr(), K, M * K, dB.data_ptr(), N, K * N,
                                    dC.data_ptr(), N, M * N, batch, None, s) == gtg.GTG_OK
    assert gtg.gtg_sync_status(s) == gtg.GTG_OK
    C = dC.cpu().numpy()
    for b in range(batch):
        check_gemm("bf16", A[b], B[b], C[b])
