"""GPU parity of the ring GEMV kernel (one or two vectors, 16-byte aligned
rows, x in one CTA) against the FP64 oracle, through the C ABI.

The kernel cuts each CTA's rows x steps into one equal range per warp, so a
range may start and end inside a row and span several short rows; these
cases pick shapes where that happens, with trailing entries (N not a multiple
of the 16-byte load), rows shorter than one load, fewer rows than SMs and
padded rows. Bound per output: |y - ref| <= 4 N 2^-24 E, E = sum_j |a_ij x_j|.
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


def is_ring(plan, batch):
    # the ring kernel: 1024 threads, one row per step, 4 loads per ring set
    # ahead of the arithmetic, and shared memory for its per-warp partial
    # sums beside the staged vectors
    return (plan["kernel"] == "gemv" and plan["threads"] == 1024 and plan["bm"] == 1 and plan["bk"] == 4
            and plan["smem"] > 4 * batch * plan["bn"] and plan["cluster"] == 1)


@pytest.mark.parametrize("M,N,batch,lda", [(1000, 3000, 1, None), (1000, 3000, 2, None), (997, 1001, 2, 1004),
                                           (152, 8, 1, None), (151, 3, 1, 4), (4096, 511, 2, 512),
                                           (4096, 513, 1, 516), (20000, 100, 2, None), (2000, 25600, 1, None),
                                           (5, 4099, 2, 4100), (1523, 1030, 2, 1032), (1, 1, 1, 4),
                                           (303, 2049, 1, 2052)])
def test_f32_ranges_across_rows(M, N, batch, lda):
    g = PCG32(3100 + M + N + batch)
    A = g.uniform_f32((M, N))
    X = g.uniform_f32((batch, N))
    assert is_ring(plan_of(M, N, batch, lda=lda), batch)
    check(A, X, run_gemv(A, X, lda=lda))


@pytest.mark.parametrize("M,N,lda", [(8192, 4096, None), (4099, 8195, 8200), (16384, 2048, None)])
def test_bf16_batch1_from_2_to_the_25(M, N, lda):
    g = PCG32(3200 + M + N)
    A = g.normal_bf16((M, N))
    x = g.uniform_f32((1, N))
    assert is_ring(plan_of(M, N, 1, "bf16", lda), 1)
    Y = run_gemv(A, x, lda=lda, prec="bf16")
    rows = np.unique(np.concatenate([np.arange(0, M, 7), [M - 1]]))
    Af = bf16_bits_to_f32(A[rows])
    ref, E = oracle.gemv(Af, x[0])
    ratio, bad = parity_ratio(Y[0][rows], ref, E, "f32", N)
    assert bad == 0, ratio


def test_bf16_stays_on_the_streaming_kernel_below_2_to_the_25_and_at_batch_2():
    assert not is_ring(plan_of(4096, 4096, 1, "bf16"), 1)
    assert not is_ring(plan_of(8192, 8192, 2, "bf16"), 2)


def test_small_integer_products_are_exact():
    # |a|, |x| <= 8 and N = 2000: every partial sum is an integer below 2^24,
    # so any order of addition gives the exact result
    g = PCG32(3300)
    M, N = 3001, 2000
    A = np.floor(g.uniform_f32((M, N)) * 8).astype(np.float32)
    X = np.floor(g.uniform_f32((2, N)) * 8).astype(np.float32)
    assert is_ring(plan_of(M, N, 2), 2)
    Y = run_gemv(A, X)
    assert np.array_equal(Y, (X.astype(np.int64) @ A.astype(np.int64).T).astype(np.float32))


def test_deterministic():
    g = PCG32(3400)
    A = g.uniform_f32((4096, 4096))
    X = g.uniform_f32((2, 4096))
    assert np.array_equal(run_gemv(A, X), run_gemv(A, X))


@pytest.mark.parametrize("batch", [1, 2])
def test_streaming_kernel_still_right_when_forced(batch):
    """gtg_gemv_force_path("no_ring") keeps the streaming kernel reachable for
    comparison; it must give results within the same bound."""
    g = PCG32(3500 + batch)
    A = g.uniform_f32((1523, 1030))
    X = g.uniform_f32((batch, 1030))
    gtg.gtg_gemv_force_path("no_ring")
    try:
        assert not is_ring(plan_of(1523, 1030, batch, lda=1032), batch)
        check(A, X, run_gemv(A, X, lda=1032))
    finally:
        gtg.gtg_gemv_force_path("auto")
