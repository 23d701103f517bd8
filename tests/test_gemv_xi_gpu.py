"""GPU parity of the row-block GEMV kernel at batch 8 with the vectors staged
interleaved (the eight values of a column side by side, two vectors per
packed FMA) against the FP64 oracle, through the C ABI: in one CTA per block
of rows, and over clusters (each CTA its own block of columns) when the
vectors are too long for one CTA.

The threads stage x themselves: 16-byte reads of each vector where x is
16-byte aligned with ldx a multiple of 4, single reads otherwise and for the
last partial group of four columns. The cases cover both, trailing entries
(N not a multiple of 4), padded rows, rows shorter than one load and fewer
rows than SMs, for FP32 and BF16 matrices. The packed FMAs take each sum's
products in the same order as the plain staging, so the two must agree bit
for bit ("no_xi" forces the plain staging). Bound per output:
|y - ref| <= 4 N 2^-24 E, E = sum_j |a_ij x_j|.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32, bf16_bits_to_f32
from tests._gpu import run_gemv
from tests._util import parity_ratio

pytestmark = pytest.mark.gpu


def check(Af, X, Y):
    for b in range(X.shape[0]):
        ref, E = oracle.gemv(Af, X[b])
        ratio, bad = parity_ratio(Y[b], ref, E, "f32", Af.shape[1])
        assert bad == 0, f"vector {b}: {bad} outputs out of bound (max ratio {ratio:.3g})"


def plan_of(M, N, batch, prec="f32", lda=None):
    return gtg.plan_gemv(M, N, 1 << 32, lda or N, 2 << 32, N, 3 << 32, M, batch, precision=prec)


def is_xi(plan, N, batch=8):
    # the row-block kernel (512 threads, 4 rows per task, one CTA per block
    # of rows) whose staged vectors take (4 * batch + 4) floats per group of
    # four columns instead of batch floats per column
    return (plan["kernel"] == "gemv" and plan["threads"] == 512 and plan["bm"] == 4 and plan["cluster"] == 1
            and plan["bn"] * batch >= (N + 3) // 4 * (4 * batch + 4))


F32_CASES = [(4096, 4096, None), (1000, 3000, None), (997, 1001, 1004), (152, 8, None), (333, 1027, 1028),
             (20000, 100, None), (5, 4099, 4100), (303, 2049, 2052), (4096, 6000, None), (1, 13, 16)]


@pytest.mark.parametrize("M,N,lda", F32_CASES)
def test_f32_batch8(M, N, lda):
    g = PCG32(3600 + M + N)
    A = g.uniform_f32((M, N))
    X = g.uniform_f32((8, N))
    if N >= 8:
        assert is_xi(plan_of(M, N, 8, lda=lda), N)
    check(A, X, run_gemv(A, X, lda=lda))


@pytest.mark.parametrize("M,N,ldx,x_off", [(997, 1001, 1002, 0), (1000, 3000, 3000, 1), (64, 4097, 4099, 3)])
def test_f32_batch8_vectors_off_16_bytes(M, N, ldx, x_off):
    """x not 16-byte aligned, or ldx not a multiple of 4: single reads."""
    g = PCG32(3700 + M + N + x_off)
    A = g.uniform_f32((M, N))
    X = g.uniform_f32((8, N))
    lda = (N + 3) // 4 * 4
    check(A, X, run_gemv(A, X, lda=lda, ldx=ldx, x_off=x_off))


@pytest.mark.parametrize("M,N,lda", [(4096, 4096, None), (1000, 3000, None), (997, 1001, 1008), (152, 16, None),
                                     (16384, 1024, None), (301, 5003, 5008)])
def test_bf16_batch8(M, N, lda):
    g = PCG32(3800 + M + N)
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((8, N))
    gtg.gtg_gemv_force_path("cuda_cores")
    try:
        assert is_xi(plan_of(M, N, 8, "bf16", lda), N)
        Y = run_gemv(A, X, lda=lda, prec="bf16")
    finally:
        gtg.gtg_gemv_force_path("auto")
    check(bf16_bits_to_f32(A), X, Y)


@pytest.mark.parametrize("prec,M,N,lda,ldx,x_off", [("f32", 997, 1001, 1004, None, 0), ("f32", 4096, 4096, None, None, 0),
                                                    ("f32", 333, 1027, 1028, 1029, 1),
                                                    ("bf16", 1000, 3000, None, None, 0),
                                                    ("bf16", 997, 1001, 1008, 1003, 2)])
def test_same_bits_as_the_plain_staging(prec, M, N, lda, ldx, x_off):
    g = PCG32(3900 + M + N)
    A = g.normal_bf16((M, N)) if prec == "bf16" else g.uniform_f32((M, N))
    X = g.uniform_f32((8, N))
    gtg.gtg_gemv_force_path("cuda_cores")
    try:
        assert is_xi(plan_of(M, N, 8, prec, lda), N)
        y_xi = run_gemv(A, X, lda=lda, ldx=ldx, x_off=x_off, prec=prec)
        gtg.gtg_gemv_force_path("no_xi")
        assert not is_xi(plan_of(M, N, 8, prec, lda), N)
        y_plain = run_gemv(A, X, lda=lda, ldx=ldx, x_off=x_off, prec=prec)
    finally:
        gtg.gtg_gemv_force_path("auto")
    assert np.array_equal(y_xi.view(np.uint32), y_plain.view(np.uint32))


def test_small_integer_products_are_exact():
    # |a|, |x| <= 8 and N = 2001: every partial sum is an integer below 2^24
    g = PCG32(4000)
    M, N = 777, 2001
    A = np.floor(g.uniform_f32((M, N)) * 8).astype(np.float32)
    X = np.floor(g.uniform_f32((8, N)) * 8).astype(np.float32)
    assert is_xi(plan_of(M, N, 8, lda=2004), N)
    Y = run_gemv(A, X, lda=2004)
    assert np.array_equal(Y, (X.astype(np.int64) @ A.astype(np.int64).T).astype(np.float32))


def test_deterministic():
    g = PCG32(4100)
    A = g.uniform_f32((4096, 4096))
    X = g.uniform_f32((8, 4096))
    assert np.array_equal(run_gemv(A, X), run_gemv(A, X))


@pytest.mark.parametrize("batch", [3, 4, 6, 7])
def test_other_batches_keep_the_plain_staging(batch):
    assert not is_xi(plan_of(4096, 4096, batch), 4096, batch)


def _plans(M, N, prec="f32", lda=None):
    """The plan at batch 8 with the interleaved staging and with the vectors
    staged one after another (mode "no_xi")."""
    gtg.gtg_gemv_force_path("cuda_cores")
    try:
        xi = plan_of(M, N, 8, prec, lda)
        gtg.gtg_gemv_force_path("no_xi")
        plain = plan_of(M, N, 8, prec, lda)
    finally:
        gtg.gtg_gemv_force_path("auto")
    return xi, plain


CLUSTER_CASES = [("f32", 1000, 8192, None), ("f32", 333, 9001, 9004), ("f32", 2048, 16384, None),
                 ("f32", 77, 12345, 12348), ("bf16", 1000, 8192, None), ("bf16", 301, 10001, 10008)]


@pytest.mark.parametrize("prec,M,N,lda", CLUSTER_CASES)
def test_batch8_over_clusters(prec, M, N, lda):
    xi, plain = _plans(M, N, prec, lda)
    assert xi["cluster"] > 1 and plain["cluster"] > 1, (xi, plain)
    assert xi["bn"] > plain["bn"], (xi, plain)   # 36 floats per four columns instead of 32
    g = PCG32(4200 + M + N)
    A = g.normal_bf16((M, N)) if prec == "bf16" else g.uniform_f32((M, N))
    X = g.uniform_f32((8, N))
    gtg.gtg_gemv_force_path("cuda_cores")
    try:
        Y = run_gemv(A, X, lda=lda, prec=prec)
    finally:
        gtg.gtg_gemv_force_path("auto")
    check(bf16_bits_to_f32(A) if prec == "bf16" else A, X, Y)


@pytest.mark.parametrize("prec,M,N,lda,ldx,x_off", [("f32", 77, 12345, 12348, None, 0),
                                                    ("f32", 500, 8192, None, 8195, 1),
                                                    ("bf16", 301, 10001, 10008, None, 0)])
def test_clusters_same_bits_as_the_plain_staging(prec, M, N, lda, ldx, x_off):
    g = PCG32(4300 + M + N)
    A = g.normal_bf16((M, N)) if prec == "bf16" else g.uniform_f32((M, N))
    X = g.uniform_f32((8, N))
    gtg.gtg_gemv_force_path("cuda_cores")
    try:
        y_xi = run_gemv(A, X, lda=lda, ldx=ldx, x_off=x_off, prec=prec)
        gtg.gtg_gemv_force_path("no_xi")
        y_plain = run_gemv(A, X, lda=lda, ldx=ldx, x_off=x_off, prec=prec)
    finally:
        gtg.gtg_gemv_force_path("auto")
    assert np.array_equal(y_xi.view(np.uint32), y_plain.view(np.uint32))
