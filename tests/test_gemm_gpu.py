"""GPU parity of the three GEMM paths against the FP64 oracle, through the C ABI.

Bounds (per element, E = sum_k |a_ik b_kj| from the oracle):
  FP32 |c - ref| <= 4 K 2^-24 E,  TF32 <= 4 2^-11 E,  BF16 <= 4 2^-8 E.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
from seeded import PCG32, gemm_normal_bf16, gemm_uniform_f32
from tests._gpu import check_gemm, run_gemm, sample_rows

pytestmark = pytest.mark.gpu


def inputs(prec, M, N, K, seed):
    g = PCG32(seed)
    if prec == "bf16":
        return g.normal_bf16((M, K)), g.normal_bf16((K, N))
    if prec == "f16":
        return g.normal_f16((M, K)), g.normal_f16((K, N))
    return g.uniform_f32((M, K)), g.uniform_f32((K, N))


# ---- the workload configurations -------------------------------------------

def test_f32_256_cubed_seed1():
    A, B = gemm_uniform_f32(1, 256, 256, 256)
    C = run_gemm("f32", A, B, expect_kernel="simt")
    check_gemm("f32", A, B, C)


@pytest.mark.parametrize("prec,kernel", [("f32", "simt"), ("tf32", "tcgen05")])
def test_1024_cubed_seed3(prec, kernel):
    A, B = gemm_uniform_f32(3, 1024, 1024, 1024)
    C = run_gemm(prec, A, B, expect_kernel=kernel)
    check_gemm(prec, A, B, C)


@pytest.mark.parametrize("prec,kernel", [("f32", "simt"), ("tf32", "tcgen05")])
def test_ragged_1000x1500x700_seed4(prec, kernel):
    # M = 1000, K = 1500, N = 700: partial tiles in every dimension
    A, B = gemm_uniform_f32(4, 1000, 700, 1500)
    C = run_gemm(prec, A, B, expect_kernel=kernel)
    check_gemm(prec, A, B, C)


def test_bf16_4096_cubed_seed5():
    (A, B), = gemm_normal_bf16(5, [(4096, 4096, 4096)])
    C = run_gemm("bf16", A, B, expect_kernel="tcgen05")
    check_gemm("bf16", A, B, C, rows=sample_rows(4096))


@pytest.mark.slow
def test_bf16_large_and_skinny_seed6():
    # 8192^3 then 16384 x 4096 x 4096 from one continuing stream, sigma = 1/sqrt(K)
    shapes = [(8192, 8192, 8192), (16384, 4096, 4096)]
    for (M, N, K), (A, B) in zip(shapes, gemm_normal_bf16(6, shapes, lambda k: k ** -0.5)):
        C = run_gemm("bf16", A, B, expect_kernel="tcgen05")
        check_gemm("bf16", A, B, C, rows=sample_rows(M))


# ---- edges, tails and every tile width -----------------------------------------

EDGE = [(1, 1, 1), (7, 5, 3), (127, 129, 65), (129, 127, 1), (1, 300, 17), (300, 1, 17),
        (33, 65, 257), (128, 256, 64), (257, 513, 129)]


@pytest.mark.parametrize("M,N,K", EDGE)
def test_f32_edge_shapes(M, N, K):
    A, B = inputs("f32", M, N, K, 100 + M)
    check_gemm("f32", A, B, run_gemm("f32", A, B))


TC_EDGE = [(1, 8, 8), (128, 256, 64), (128, 256, 128), (130, 72, 24), (129, 264, 1000),
           (300, 64, 8), (512, 256, 4096), (1536, 1536, 64), (1, 520, 72)]


@pytest.mark.parametrize("prec", ["tf32", "bf16"])
@pytest.mark.parametrize("M,N,K", TC_EDGE)
def test_tcgen05_edge_shapes(prec, M, N, K):
    A, B = inputs(prec, M, N, K, 200 + N)
    check_gemm(prec, A, B, run_gemm(prec, A, B, expect_kernel="tcgen05"))


@pytest.mark.parametrize("prec", ["tf32", "bf16"])
def test_every_tile_width_is_exercised(prec):
    seen = set()
    # (1408 x 1664: 143 tiles of 128 x 128 fit one wave, while its 42 pair
    # tiles are too many to run as half tiles in one wave)
    for (M, N, K) in [(4096, 4096, 64), (1408, 1664, 64), (1024, 1024, 64)]:
        A, B = inputs(prec, M, N, K, 7)
        C = run_gemm(prec, A, B, expect_kernel="tcgen05")
        check_gemm(prec, A, B, C, rows=sample_rows(M))
        t = gtg_plan(prec, M, N, K)
        seen.add(t["bn"])
    assert seen == {64, 128, 256}


def gtg_plan(prec, M, N, K):
    import torch
    esz = 2 if prec == "bf16" else 4
    a = torch.empty(M * K * esz // 4 + 4, dtype=torch.float32, device="cuda")
    b = torch.empty(K * N * esz // 4 + 4, dtype=torch.float32, device="cuda")
    c = torch.empty(M * N + 4, dtype=torch.float32, device="cuda")
    return gtg.plan_gemm(prec, M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N)


@pytest.mark.parametrize("prec", ["tf32", "bf16"])
def test_many_tiles_per_cta(prec):
    # ~7 output tiles per persistent CTA: exercises both TMEM accumulators and
    # several phases of every pipeline barrier
    M, N, K = 8192, 4096, 96
    A, B = inputs(prec, M, N, K, 9)
    C = run_gemm(prec, A, B, expect_kernel="tcgen05")
    check_gemm(prec, A, B, C, rows=sample_rows(M, seed=1))
    # and every row of one band of tiles, every column
    check_gemm(prec, A, B, C, rows=np.arange(1024, 1152))


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("M,N,K", [(4252, 4160, 520), (4224, 4160, 72), (4096, 4096, 8)])
def test_cta_pair_kernel_ragged(prec, M, N, K):
    # shapes the planner gives to the CTA-pair kernel (256 x 256 tiles): the
    # odd CTA's rows of the last pair tile lie partly or wholly past M, the
    # last column tile is partial, and K ends inside a 128-byte slice (TF32:
    # B^T staged K-major in each CTA)
    A, B = inputs(prec, M, N, K, 300 + K)
    C = run_gemm(prec, A, B, expect_kernel="tcgen05")
    assert gtg_plan(prec, M, N, K)["bm"] == 256
    check_gemm(prec, A, B, C, rows=np.concatenate([sample_rows(M, seed=2), np.arange(M - 200, M)]))


@pytest.mark.parametrize("prec", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(4000, 4000, 200), (4096, 4096, 72), (2048, 1024, 512), (1536, 1528, 512), (3000, 2008, 1024)])
def test_cta_pair_kernel_half_tiles(prec, M, N, K):
    # a last wave of 256 x 256 tiles that would leave clusters idle runs as
    # 128-wide halves (4000: 256 tiles on 76 clusters, 28 left, their second
    # halves only 32 columns wide at the right edge; 2048 x 1024 and 1536 x 1528:
    # every tile in halves)
    A, B = inputs(prec, M, N, K, 400 + K)
    C = run_gemm(prec, A, B, expect_kernel="tcgen05")
    assert gtg_plan(prec, M, N, K)["bm"] == 256
    rows = np.concatenate([sample_rows(M, seed=3), np.arange(max(0, M - 300), M)])
    check_gemm(prec, A, B, C, rows=np.unique(rows))


@pytest.mark.parametrize("mode", ["direct", "tensor"])
@pytest.mark.parametrize("prec,M,N,K,cpad", [("bf16", 4252, 4160, 520, 0), ("bf16", 4000, 4000, 200, 4),
                                             ("f16", 3000, 2008, 1024, 12), ("tf32", 4224, 4160, 72, 4),
                                             ("bf16", 4096, 4104, 64, 2), ("bf16", 2048, 1544, 256, 8)])
def test_cta_pair_kernel_c_stores(mode, prec, M, N, K, cpad):
    # the pair kernel's two ways of writing C (direct row stores, or 32 x 32
    # blocks through shared memory and tensor stores that clip at M and N):
    # ragged last row and column tiles, half tiles, padded ldc (ldc = N + 2
    # has 8-byte rows, so tensor stores are not allowed and direct ones run);
    # the guard bands around C check that nothing is written past N or M
    A, B = inputs(prec, M, N, K, 500 + K + cpad)
    gtg.gtg_force_c_store(mode)
    try:
        C = run_gemm(prec, A, B, ldc=N + cpad, expect_kernel="tcgen05")
        assert gtg_plan(prec, M, N, K)["bm"] == 256
    finally:
        gtg.gtg_force_c_store("auto")
    rows = np.concatenate([sample_rows(M, seed=4), np.arange(M - 130, M)])
    check_gemm(prec, A, B, C, rows=np.unique(rows))


@pytest.mark.parametrize("M,N,K,bm,threads,splits", [
    (1024, 1024, 1024, 128, 256, 2),    # 64 big tiles in 2 K ranges: one 8-warp CTA on 128 of 152 SMs
    (1000, 1100, 2000, 128, 256, 2),    # ragged edges, K ranges of 63 slices
    (256, 256, 256, 64, 128, None),     # small: 4-warp 64 x 64 tiles (K split by the wave model)
    (4096, 4096, 512, 128, 256, 1),     # enough big tiles for every SM
    (3000, 3000, 3000, 256, 256, 1),    # 256 x 128 tiles (16 x 8 outputs per thread), ragged edges
    (2999, 3012, 1001, 256, 256, 1),    # the same with scalar loads (K rows not 16-byte aligned)
])
def test_simt_tile_choice_and_parity(M, N, K, bm, threads, splits):
    p = gtg_plan("f32", M, N, K)
    assert p["kernel"] == "simt" and p["bm"] == bm and p["threads"] == threads, p
    if splits is not None:
        assert p["splits"] == splits, p
    if M * N * K <= 3e10:
        A, B = inputs("f32", M, N, K, 700 + M)
        C = run_gemm("f32", A, B, expect_kernel="simt")
        check_gemm("f32", A, B, C, rows=np.unique(np.concatenate([sample_rows(M, seed=5), np.arange(M - 70, M)])))


# ---- layouts the tensor-memory path cannot take: the SIMT fallback --------------

@pytest.mark.parametrize("cpad", [5, 4, 8])
@pytest.mark.parametrize("prec", ["f32", "tf32", "bf16"])
def test_padded_leading_dimensions(prec, cpad):
    # ldc padding 5 / 4 / 8 selects the epilogue's 4-, 16- and 32-byte stores
    M, N, K = 200, 136, 96
    A, B = inputs(prec, M, N, K, 11)
    C = run_gemm(prec, A, B, lda=K + 8, ldb=N + 24, ldc=N + cpad,
                 expect_kernel="simt" if prec == "f32" else "tcgen05")
    check_gemm(prec, A, B, C)


@pytest.mark.parametrize("prec", ["f32", "tf32", "bf16"])
def test_unaligned_layouts(prec):
    # odd leading dimensions and bases off 16 bytes: the tensor-core paths copy
    # A (and 16-bit B) into 16-byte rows first; FP32 stays on the SIMT kernel
    M, N, K = 97, 61, 43
    A, B = inputs(prec, M, N, K, 12)
    C = run_gemm(prec, A, B, a_off=1, b_off=3, c_off=1, expect_kernel="simt" if prec == "f32" else "tcgen05")
    check_gemm(prec, A, B, C)


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (5, 3, 1), (130, 9, 17), (2, 257, 3), (129, 1, 1001)])
def test_repacked_tiny_operands(prec, M, N, K):
    # degenerate sizes whose rows are shorter than 16 bytes: the copies pad
    # them to whole 16-byte rows and TMA fills the rest of each box with zeros
    A, B = inputs(prec, M, N, K, 1400 + M + N + K)
    check_gemm(prec, A, B, run_gemm(prec, A, B, expect_kernel="tcgen05"))


@pytest.mark.parametrize("prec,M,N,K,a_off,b_off", [
    ("bf16", 1000, 701, 1501, 0, 0),     # odd K and N: neither A's nor B's rows are 16-byte multiples
    ("f16", 513, 264, 1500, 3, 0),       # A's base 6 bytes off, K * 2 = 3000-byte rows
    ("bf16", 300, 1100, 256, 0, 5),      # only B repacked (N * 2 = 2200-byte rows, base off)
    ("tf32", 700, 500, 1501, 1, 1),      # TF32: A repacked, B through its transpose as always
    ("bf16", 4000, 3000, 2001, 0, 0),    # large enough for the CTA-pair kernel after the copy
])
def test_repacked_operands_on_the_tensor_cores(prec, M, N, K, a_off, b_off):
    A, B = inputs(prec, M, N, K, 1300 + K)
    C = run_gemm(prec, A, B, a_off=a_off, b_off=b_off, expect_kernel="tcgen05")
    rows = np.unique(np.concatenate([sample_rows(M, seed=7), np.arange(max(0, M - 70), M)]))
    check_gemm(prec, A, B, C, rows=rows)


@pytest.mark.parametrize("prec", ["tf32", "bf16"])
def test_forced_simt_matches_bound(prec):
    M, N, K = 256, 192, 320
    A, B = inputs(prec, M, N, K, 13)
    gtg.gtg_force_simt(True)
    try:
        C = run_gemm(prec, A, B, expect_kernel="simt")
    finally:
        gtg.gtg_force_simt(False)
    check_gemm(prec, A, B, C)


# ---- closed forms, exactness, degenerate sizes, determinism --------------------

@pytest.mark.parametrize("prec", ["f32", "tf32", "bf16"])
def test_identity_gives_B_exactly(prec):
    M = K = 256
    N = 320
    g = PCG32(14)
    if prec == "bf16":
        A = np.full((M, K), 0, dtype=np.uint16)
        A[np.arange(M), np.arange(K)] = 0x3F80          # 1.0
        B = g.normal_bf16((K, N))
        from seeded import bf16_bits_to_f32
        ref = bf16_bits_to_f32(B)
    else:
        A = np.eye(M, K, dtype=np.float32)
        B = g.uniform_f32((K, N))
        if prec == "tf32":   # values with at most 11 significant bits pass through
            B = (np.round(B * 1024) / 1024).astype(np.float32)
        ref = B
    C = run_gemm(prec, A, B)
    assert np.array_equal(C, ref)


@pytest.mark.parametrize("prec", ["f32", "tf32", "bf16"])
def test_all_ones_gives_K(prec):
    M, N, K = 130, 260, 1000
    if prec == "bf16":
        A = np.full((M, K), 0x3F80, dtype=np.uint16)
        B = np.full((K, N), 0x3F80, dtype=np.uint16)
    else:
        A = np.ones((M, K), dtype=np.float32)
        B = np.ones((K, N), dtype=np.float32)
    assert np.all(run_gemm(prec, A, B) == K)


@pytest.mark.parametrize("prec", ["f32", "tf32", "bf16"])
def test_small_integers_are_exact(prec):
    # |entries| <= 8, K <= 1024: every partial sum is an integer below 2^24
    M, N, K = 192, 272, 1024
    rng = np.random.default_rng(15)
    Ai = rng.integers(-8, 9, (M, K))
    Bi = rng.integers(-8, 9, (K, N))
    ref = (Ai @ Bi).astype(np.float32)
    if prec == "bf16":
        from seeded import f64_to_bf16_bits
        A, B = f64_to_bf16_bits(Ai.astype(np.float64)), f64_to_bf16_bits(Bi.astype(np.float64))
    else:
        A, B = Ai.astype(np.float32), Bi.astype(np.float32)
    assert np.array_equal(run_gemm(prec, A, B), ref)


@pytest.mark.parametrize("prec", ["f32", "tf32", "bf16"])
def test_K_zero_writes_zeros(prec):
    M, N = 37, 45
    dt = np.uint16 if prec == "bf16" else np.float32
    C = run_gemm(prec, np.zeros((M, 0), dtype=dt), np.zeros((0, N), dtype=dt))
    assert np.all(C == 0)


@pytest.mark.parametrize("prec", ["f32", "tf32", "bf16"])
def test_deterministic(prec):
    M, N, K = 640, 512, 768
    A, B = inputs(prec, M, N, K, 16)
    C1 = run_gemm(prec, A, B)
    C2 = run_gemm(prec, A, B)
    assert np.array_equal(C1, C2)


def test_side_stream_and_tensor_helper():
    import torch
    A, B = gemm_uniform_f32(17, 300, 200, 100)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C = gtg.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), "tf32")
    s.synchronize()
    check_gemm("tf32", A, B, C.cpu().numpy())
    # host tensors in, host tensor out (the end-to-end form)
    Ch = gtg.matmul(torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(), "f32")
    assert not Ch.is_cuda
    check_gemm("f32", A, B, Ch.numpy())
