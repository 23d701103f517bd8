"""GEMM variants: FP16 inputs, and strided batches of independent products
(one call), against the FP64 oracle through the C ABI."""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32, bf16_bits_to_f32, f16_bits_to_f32
from tests._gpu import check_gemm, run_gemm, run_gemv, sample_rows
from tests._util import parity_ratio

pytestmark = pytest.mark.gpu


def _t():
    import torch
    return torch


# ---- FP16 ------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K,bm", [(4096, 4096, 256, 256), (1024, 1024, 320, 128), (130, 72, 24, 128),
                                      (1000, 712, 208, 128)])
def test_f16_tensor_core(M, N, K, bm):
    g = PCG32(800 + K)
    A, B = g.normal_f16((M, K)), g.normal_f16((K, N))
    C = run_gemm("f16", A, B, expect_kernel="tcgen05")
    Af, Bf = f16_bits_to_f32(A), f16_bits_to_f32(B)
    rows = sample_rows(M, seed=3) if M > 1024 else None
    ref, E = oracle.gemm(Af[rows] if rows is not None else Af, Bf)
    ratio, bad = parity_ratio(C[rows] if rows is not None else C, ref, E, "f16", K)
    assert bad == 0, ratio


def test_f16_unaligned_layouts_are_repacked():
    # bases off 16 bytes and odd leading dimensions: A and B are copied into
    # 16-byte rows and the tensor cores multiply them
    g = PCG32(810)
    M, N, K = 97, 61, 43
    A, B = g.normal_f16((M, K)), g.normal_f16((K, N))
    C = run_gemm("f16", A, B, a_off=1, b_off=3, expect_kernel="tcgen05")
    ref, E = oracle.gemm(f16_bits_to_f32(A), f16_bits_to_f32(B))
    ratio, bad = parity_ratio(C, ref, E, "f16", K)
    assert bad == 0, ratio


def test_f16_small_integers_exact():
    rng = np.random.default_rng(811)
    Ai = rng.integers(-8, 9, (256, 512))
    Bi = rng.integers(-8, 9, (512, 320))
    from seeded import f64_to_f16_bits
    C = run_gemm("f16", f64_to_f16_bits(Ai.astype(np.float64)), f64_to_f16_bits(Bi.astype(np.float64)))
    assert np.array_equal(C, (Ai @ Bi).astype(np.float32))


# ---- strided batches ---------------------------------------------------------

def _draw(prec, g, shape):
    if prec == "bf16":
        bits = g.normal_bf16(shape)
        return bits, bf16_bits_to_f32(bits)
    if prec == "f16":
        bits = g.normal_f16(shape)
        return bits, f16_bits_to_f32(bits)
    v = g.uniform_f32(shape)
    return v, v


def _dev(prec, host):
    torch = _t()
    if prec in ("bf16", "f16"):
        return torch.from_numpy(np.ascontiguousarray(host).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(host)).cuda()


@pytest.mark.parametrize("prec", ["bf16", "f16", "tf32", "f32"])
@pytest.mark.parametrize("case", ["packed", "shared_B", "padded", "unaligned"])
def test_strided_batched(prec, case):
    torch = _t()
    g = PCG32(900 + len(case))
    batch, M, N, K = 3, 300, 264, 136
    lda, ldb, ldc = K, N, N
    sA, sB, sC = M * lda, K * ldb, M * ldc
    if case == "shared_B":
        sB = 0
    if case == "padded":
        sA, sB, sC = sA + 64, sB + 128, sC + 40
    if case == "unaligned":            # strides that are not multiples of 16 bytes
        sA, sB = sA + 1, (sB + 3 if sB else 0)
    A_host, A_f = _draw(prec, g, (batch * sA + 8,))
    B_host, B_f = _draw(prec, g, (max(1, batch * sB) + K * ldb + 8,))
    dA, dB = _dev(prec, A_host), _dev(prec, B_host)
    dC = torch.full((batch * sC + 8,), float("nan"), device="cuda")
    bias = g.uniform_f32((N,))
    db = torch.from_numpy(bias).cuda()
    s = int(torch.cuda.current_stream().cuda_stream)
    st = gtg.gemm_strided_batched(prec, M, N, K, dA.data_ptr(), lda, sA, dB.data_ptr(), ldb, sB,
                                  dC.data_ptr(), ldc, sC, batch, gtg.epilogue(db.data_ptr(), "relu"), s)
    assert st == gtg.GTG_OK, gtg.status_string(st)
    assert gtg.gtg_sync_status(s) == gtg.GTG_OK
    C = dC.cpu().numpy()
    for b in range(batch):
        Ab = A_f[b * sA: b * sA + M * lda].reshape(M, lda)[:, :K]
        Bb = B_f[b * sB: b * sB + K * ldb].reshape(K, ldb)[:, :N]
        ref, E = oracle.dense_layer(Ab, Bb, bias, "relu")
        got = C[b * sC: b * sC + M * ldc].reshape(M, ldc)[:, :N]
        ratio, bad = parity_ratio(got, ref, E, prec, K, rel=2.0 ** -23)
        assert bad == 0, (b, ratio)
    # nothing written between the items (the padding keeps its NaN)
    if case == "padded":
        for b in range(batch - 1):
            assert np.all(np.isnan(C[b * sC + M * ldc: (b + 1) * sC]))


@pytest.mark.parametrize("mode", ["direct", "tensor"])
def test_strided_batched_c_stores(mode):
    # items large enough for the CTA-pair kernel (2000 x 1000: ragged last row
    # and column tiles), padded item strides, bias + ReLU: with tensor stores the
    # 3-D map (columns, rows, item) must clip each item at M and N and leave the
    # padding between items untouched
    torch = _t()
    g = PCG32(960)
    batch, M, N, K = 3, 2000, 1000, 200
    sA, sB, sC = M * K + 64, K * N + 128, M * N + 400
    A_host, A_f = _draw("bf16", g, (batch * sA + 8,))
    B_host, B_f = _draw("bf16", g, (batch * sB + 8,))
    dA, dB = _dev("bf16", A_host), _dev("bf16", B_host)
    dC = torch.full((batch * sC + 8,), float("nan"), device="cuda")
    bias = g.uniform_f32((N,))
    db = torch.from_numpy(bias).cuda()
    s = int(torch.cuda.current_stream().cuda_stream)
    gtg.gtg_force_c_store(mode)
    try:
        st = gtg.gemm_strided_batched("bf16", M, N, K, dA.data_ptr(), K, sA, dB.data_ptr(), N, sB,
                                      dC.data_ptr(), N, sC, batch, gtg.epilogue(db.data_ptr(), "relu"), s)
        assert st == gtg.GTG_OK, gtg.status_string(st)
        assert gtg.gtg_sync_status(s) == gtg.GTG_OK
    finally:
        gtg.gtg_force_c_store("auto")
    C = dC.cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(0, M, 37), np.arange(M - 100, M)]))
    for b in range(batch):
        Ab = A_f[b * sA: b * sA + M * K].reshape(M, K)
        Bb = B_f[b * sB: b * sB + K * N].reshape(K, N)
        ref, E = oracle.dense_layer(Ab[rows], Bb, bias, "relu")
        got = C[b * sC: b * sC + M * N].reshape(M, N)[rows]
        ratio, bad = parity_ratio(got, ref, E, "bf16", K, rel=2.0 ** -23)
        assert bad == 0, (b, ratio)
        assert np.all(np.isnan(C[b * sC + M * N: (b + 1) * sC]))


@pytest.mark.parametrize("prec", ["bf16", "f16", "tf32"])
@pytest.mark.parametrize("case", ["odd_strides", "odd_ld_shared_B", "odd_ld_shared_A"])
def test_strided_batched_repacked(prec, case):
    # item strides or leading dimensions off 16 bytes: the items are copied into
    # aligned rows (a shared operand once) and the batch runs as one
    # tensor-core launch; checked per item against the oracle
    torch = _t()
    g = PCG32(970 + len(case))
    batch, M, N, K = 3, 300, 264, 136
    lda, ldb, ldc = K, N, N
    sA, sB, sC = M * lda + 1, K * ldb + 3, M * ldc
    if case == "odd_ld_shared_B":
        lda, ldb = K + 1, N + 3
        sA, sB = M * lda, 0
    if case == "odd_ld_shared_A":
        lda, ldb = K + 3, N + 1
        sA, sB = 0, K * ldb
    A_host, A_f = _draw(prec, g, (max(1, batch * sA) + M * lda + 8,))
    B_host, B_f = _draw(prec, g, (max(1, batch * sB) + K * ldb + 8,))
    dA, dB = _dev(prec, A_host), _dev(prec, B_host)
    dC = torch.full((batch * sC + 8,), float("nan"), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    st = gtg.gemm_strided_batched(prec, M, N, K, dA.data_ptr(), lda, sA, dB.data_ptr(), ldb, sB,
                                  dC.data_ptr(), ldc, sC, batch, None, s)
    assert st == gtg.GTG_OK, gtg.status_string(st)
    assert gtg.gtg_sync_status(s) == gtg.GTG_OK
    C = dC.cpu().numpy()
    for b in range(batch):
        Ab = A_f[b * sA: b * sA + M * lda].reshape(M, lda)[:, :K]
        Bb = B_f[b * sB: b * sB + K * ldb].reshape(K, ldb)[:, :N]
        ref, E = oracle.gemm(Ab, Bb)
        got = C[b * sC: b * sC + M * ldc].reshape(M, ldc)[:, :N]
        ratio, bad = parity_ratio(got, ref, E, prec, K)
        assert bad == 0, (b, ratio)


def test_strided_batched_plans_one_launch_for_all_items():
    torch = _t()
    batch, M, N, K = 40, 512, 512, 64
    g = PCG32(950)
    A = g.normal_bf16((batch, M, K))
    B = g.normal_bf16((batch, K, N))
    dA, dB = _dev("bf16", A), _dev("bf16", B)
    dC = torch.empty((batch, M, N), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    assert gtg.gemm_strided_batched("bf16", M, N, K, dA.data_ptr(), K, M * K, dB.data_ptr(), N, K * N,
                                    dC.data_ptr(), N, M * N, batch, None, s) == gtg.GTG_OK
    C = dC.cpu().numpy()
    for b in (0, 17, batch - 1):
        ref, E = oracle.gemm(bf16_bits_to_f32(A[b]), bf16_bits_to_f32(B[b]))
        ratio, bad = parity_ratio(C[b], ref, E, "bf16", K)
        assert bad == 0, (b, ratio)


def test_f32_strided_batch_in_one_launch_past_the_grid_z_limit():
    """FP32 batches run on the SIMT kernel in one launch over blockIdx.z; more
    than 65535 items take a second launch. Tiny ragged items with one shared
    B: stacked, the items' A rows form one matrix whose product with B the
    oracle computes in a single call."""
    torch = _t()
    batch, M, N, K = 70001, 3, 5, 7
    g = PCG32(960)
    A = g.uniform_f32((batch, M, K))
    B = g.uniform_f32((K, N))
    dA, dB = _dev("f32", A), _dev("f32", B)
    dC = torch.full((batch, M, N), float("nan"), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    st = gtg.gemm_strided_batched("f32", M, N, K, dA.data_ptr(), K, M * K, dB.data_ptr(), N, 0,
                                  dC.data_ptr(), N, M * N, batch, None, s)
    assert st == gtg.GTG_OK and gtg.gtg_sync_status(s) == gtg.GTG_OK
    plan = gtg.plan_gemm("f32", M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N)
    assert plan["kernel"] == "simt"
    ref, E = oracle.gemm(A.reshape(batch * M, K), B)
    ratio, bad = parity_ratio(dC.cpu().numpy().reshape(batch * M, N), ref, E, "f32", K)
    assert bad == 0, ratio


def test_strided_batched_validation():
    A, B, C = 1 << 32, 2 << 32, 3 << 32
    f = gtg.gemm_strided_batched
    assert f("bf16", 4, 4, 4, A, 4, 16, B, 4, 16, C, 4, 10, 2) == gtg.GTG_ERR_INVALID_VALUE   # outputs overlap
    assert f("bf16", 4, 4, 4, A, 4, -16, B, 4, 16, C, 4, 16, 2) == gtg.GTG_ERR_INVALID_VALUE
    assert f("bf16", 4, 4, 4, A, 4, 16, B, 4, 16, C, 4, 16, -1) == gtg.GTG_ERR_INVALID_VALUE
    assert f(7, 4, 4, 4, A, 4, 16, B, 4, 16, C, 4, 16, 2) == gtg.GTG_ERR_INVALID_VALUE
    assert f("f32", 4, 4, 4, A, 4, 16, B, 4, 16, A + 64, 4, 16, 2) == gtg.GTG_ERR_ALIAS          # C reaches A's items
    assert f("f32", 4, 4, 4, A, 4, 16, B, 4, 16, C, 4, 16, 0) == gtg.GTG_OK


# ---- BF16 matrix GEMV ----------------------------------------------------------
# A in BF16 is widened exactly, so the reference is the FP64 product with the
# widened matrix and the FP32 bound of gemv_f32 applies unchanged.

def _check_gemv(Abits, X, Y):
    Af = bf16_bits_to_f32(Abits)
    for b in range(X.shape[0]):
        ref, E = oracle.gemv(Af, X[b])
        ratio, bad = parity_ratio(Y[b], ref, E, "f32", Af.shape[1])
        assert bad == 0, (b, ratio)


@pytest.mark.parametrize("M,N,batch", [(4096, 4096, 1), (4096, 4096, 8), (8192, 8192, 2), (523, 1031, 3),
                                       (151, 4097, 1), (2049, 130, 5), (1, 1, 1), (10, 100003, 2),
                                       (7, 9, 8), (300, 16, 4)])
def test_gemv_bf16(M, N, batch):
    g = PCG32(1000 + M + N + batch)
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((batch, N))
    _check_gemv(A, X, run_gemv(A, X, prec="bf16"))


@pytest.mark.parametrize("M,N,lda", [(1523, 1030, 1032), (4095, 4096, 4096), (153, 520, 520), (7, 4104, 4112)])
def test_gemv_bf16_batch2_two_rows_per_warp(M, N, lda):
    # BF16 rows at batch 2 stream two rows per warp: odd row counts per CTA
    # (a last task with one row), tails of N % 8 entries, padded rows
    g = PCG32(1080 + M + N)
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((2, N))
    gtg.gtg_gemv_force_path("no_ring")
    try:
        plan = gtg.plan_gemv(M, N, 1 << 32, lda, 2 << 32, N, 3 << 32, M, 2, precision="bf16")
        assert plan["kernel"] == "gemv" and plan["bm"] == 2 and plan["threads"] == 1024, plan
        _check_gemv(A, X, run_gemv(A, X, lda=lda, prec="bf16"))
        # batch 1 keeps one row per warp
        assert gtg.plan_gemv(M, N, 1 << 32, lda, 2 << 32, N, 3 << 32, M, 1, precision="bf16")["bm"] == 1
    finally:
        gtg.gtg_gemv_force_path("auto")


@pytest.mark.parametrize("M,N,batch", [(4096, 4096, 8), (300, 16, 4), (2000, 1000, 3)])
def test_gemv_bf16_cuda_cores(cuda_cores, M, N, batch):
    g = PCG32(1050 + M + N + batch)
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((batch, N))
    _check_gemv(A, X, run_gemv(A, X, prec="bf16"))


@pytest.mark.parametrize("lda,a_off", [(1040, 0), (1033, 0), (1032, 3), (1024, 1)])
def test_gemv_bf16_unaligned_and_padded_rows(lda, a_off):
    g = PCG32(1100 + lda + a_off)
    A = g.normal_bf16((333, 1024))
    X = g.uniform_f32((2, 1024))
    _check_gemv(A, X, run_gemv(A, X, lda=lda, a_off=a_off, prec="bf16"))


def test_gemv_bf16_matches_f32_on_the_widened_matrix_exactly_for_integers():
    rng = np.random.default_rng(1200)
    Ai = rng.integers(-64, 65, (777, 2056))
    xi = rng.integers(-64, 65, (3, 2056))
    from seeded import f64_to_bf16_bits
    Y = run_gemv(f64_to_bf16_bits(Ai.astype(np.float64)), xi.astype(np.float32), prec="bf16")
    assert np.array_equal(Y, (xi @ Ai.T).astype(np.float32))


def test_matvec_bf16_with_epilogue():
    torch = _t()
    g = PCG32(1300)
    A = g.normal_bf16((640, 520))
    x = g.uniform_f32((520,))
    bias = g.uniform_f32((640,))
    tA = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16)
    y = gtg.matvec(tA.cuda(), torch.from_numpy(x).cuda(), bias=torch.from_numpy(bias), activation="relu")
    ref, E = oracle.dense_vector(bf16_bits_to_f32(A), x, bias, "relu")
    ratio, bad = parity_ratio(y.cpu().numpy(), ref, E, "f32", 520, rel=2.0 ** -23)
    assert bad == 0, ratio
    # host tensors: copied in and out
    yh = gtg.matvec(tA, torch.from_numpy(x), bias=torch.from_numpy(bias), activation="relu")
    assert torch.equal(yh, y.cpu())


@pytest.fixture
def cuda_cores():
    """BF16 GEMVs of batch 3..8 on the CUDA-core kernels (the tensor-core
    path has its own tests)."""
    gtg.gtg_gemv_force_path("cuda_cores")
    yield
    gtg.gtg_gemv_force_path("auto")


@pytest.mark.parametrize("M,N,batch,lda,cluster", [(8192, 8192, 8, 8192, 2), (700, 20004, 3, 20008, 2),
                                                   (300, 16384, 8, 16384, 4)])
def test_gemv_bf16_column_blocks_over_a_cluster(cuda_cores, M, N, batch, lda, cluster):
    """Column blocks over a cluster; with 4-column units the second CTA's
    block of N = 20004 starts 8 bytes past a 16-byte boundary."""
    g = PCG32(1400 + M + batch)
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((batch, N))
    plan = gtg.plan_gemv(M, N, 1 << 32, lda, 2 << 32, N, 3 << 32, M, batch, precision="bf16")
    assert plan["cluster"] == cluster, plan
    Y = run_gemv(A, X, lda=lda, prec="bf16")
    rows = np.unique(np.concatenate([np.arange(0, M, 29), [M - 1]]))
    Af = bf16_bits_to_f32(A[rows])
    for b in range(batch):
        ref, E = oracle.gemv(Af, X[b])
        ratio, bad = parity_ratio(Y[b][rows], ref, E, "f32", N)
        assert bad == 0, (b, ratio)
