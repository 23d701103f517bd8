"""Pins for the FP64 oracle: it is checked against things other than itself.

Each `pin_*` function takes the loaded oracle library so that the mutation
test (test_oracle_mutants.py) can run the same pins against copies of the
oracle with a planted mistake and show that every mistake is caught.
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests._util import read_golden


# ---- pins ------------------------------------------------------------------

def pin_golden_gemm(lib):
    """Hand-worked 2x3 * 3x4 product (non-square: catches transposes)."""
    g = read_golden("gemm_hand_2x3x4.txt")
    C, E = oracle.gemm(g["A"], g["B"], lib=lib)
    assert np.array_equal(C, g["C"])
    assert np.array_equal(E, g["E"])


def pin_golden_gemv(lib):
    """Hand-worked 3x4 matrix-vector product."""
    g = read_golden("gemv_hand_3x4.txt")
    y, E = oracle.gemv(g["A"], g["x"][:, 0], lib=lib)
    assert np.array_equal(y, g["y"][:, 0])
    assert np.array_equal(E, g["E"][:, 0])


def pin_identity(lib):
    """A = I gives C = B exactly; B = I gives C = A exactly."""
    rng = np.random.default_rng(11)
    for (m, n) in [(1, 1), (5, 3), (17, 9)]:
        B = rng.uniform(-1, 1, (m, n))
        C, _ = oracle.gemm(np.eye(m), B, lib=lib)
        assert np.array_equal(C, B)
        A = rng.uniform(-1, 1, (n, m))
        C, _ = oracle.gemm(A, np.eye(m), lib=lib)
        assert np.array_equal(C, A)


def pin_all_ones(lib):
    """All-ones operands: every output (and its magnitude) equals K."""
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (8, 2, 129)]:
        C, E = oracle.gemm(np.ones((M, K)), np.ones((K, N)), lib=lib)
        assert np.all(C == K) and np.all(E == K)
        y, Ey = oracle.gemv(np.ones((M, K)), np.ones(K), lib=lib)
        assert np.all(y == K) and np.all(Ey == K)


def pin_small_integers_exact(lib):
    """Small-integer operands are exact in FP64: must equal integer matmul."""
    rng = np.random.default_rng(12)
    for (M, N, K) in [(1, 1, 1), (2, 3, 4), (7, 5, 9), (9, 8, 1), (33, 17, 65)]:
        A = rng.integers(-9, 10, (M, K))
        B = rng.integers(-9, 10, (K, N))
        ref = A.astype(np.int64) @ B.astype(np.int64)          # exact integer product
        C, E = oracle.gemm(A.astype(np.float64), B.astype(np.float64), lib=lib)
        assert np.array_equal(C, ref.astype(np.float64))
        refE = np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64)
        assert np.array_equal(E, refE.astype(np.float64))
        x = rng.integers(-9, 10, K)
        y, Ey = oracle.gemv(A.astype(np.float64), x.astype(np.float64), lib=lib)
        assert np.array_equal(y, (A.astype(np.int64) @ x).astype(np.float64))
        assert np.array_equal(Ey, (np.abs(A).astype(np.int64) @ np.abs(x)).astype(np.float64))


def pin_exact_rational(lib):
    """Random real operands on tiny shapes: within the FP64 summation bound
    of the exact (rational) product, |C - C_exact| <= (K + 1) 2^-53 E."""
    rng = np.random.default_rng(13)
    for (M, N, K) in [(1, 1, 1), (2, 2, 3), (3, 4, 5), (4, 3, 9)]:
        A = rng.uniform(-1, 1, (M, K))
        B = rng.uniform(-1, 1, (K, N))
        C, E = oracle.gemm(A, B, lib=lib)
        for i in range(M):
            for j in range(N):
                exact = sum(Fraction(A[i, k]) * Fraction(B[k, j]) for k in range(K))
                mag = sum(abs(Fraction(A[i, k]) * Fraction(B[k, j])) for k in range(K))
                assert abs(Fraction(C[i, j]) - exact) <= Fraction(K + 1, 2 ** 53) * mag
                assert abs(Fraction(E[i, j]) - mag) <= Fraction(K + 1, 2 ** 53) * mag


def pin_rank_one(lib):
    """A = u 1^T, B = 1 v^T gives C = K u v^T (powers of two: exact)."""
    u = np.array([1.0, -2.0, 0.5, 4.0])
    v = np.array([0.25, -1.0, 8.0])
    K = 6
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[None, :], K, axis=0)
    C, E = oracle.gemm(A, B, lib=lib)
    assert np.array_equal(C, K * np.outer(u, v))
    assert np.array_equal(E, K * np.abs(np.outer(u, v)))


def pin_gemv_is_gemm_with_one_column(lib):
    """The matrix-vector product is the GEMM with N = 1 (two separate loops)."""
    rng = np.random.default_rng(14)
    A = rng.uniform(-1, 1, (37, 53))
    x = rng.uniform(-1, 1, 53)
    y, Ey = oracle.gemv(A, x, lib=lib)
    C, E = oracle.gemm(A, x[:, None], lib=lib)
    assert np.array_equal(y, C[:, 0]) and np.array_equal(Ey, E[:, 0])


def pin_magnitude(lib):
    """E >= |C|, E == C for non-negative operands, E == |A| @ |B| (numpy)."""
    rng = np.random.default_rng(15)
    A = rng.uniform(-1, 1, (19, 23))
    B = rng.uniform(-1, 1, (23, 29))
    C, E = oracle.gemm(A, B, lib=lib)
    assert np.all(E >= np.abs(C))
    ref = np.abs(A) @ np.abs(B)
    assert np.allclose(E, ref, rtol=64 * 2.0 ** -53, atol=0)
    Cp, Ep = oracle.gemm(np.abs(A), np.abs(B), lib=lib)
    assert np.array_equal(Cp, Ep)


def pin_vs_library_matmul(lib):
    """Against numpy's own FP64 matmul, within the summation bound."""
    rng = np.random.default_rng(16)
    for (M, N, K) in [(64, 48, 200), (7, 130, 31)]:
        A = rng.uniform(-1, 1, (M, K))
        B = rng.uniform(-1, 1, (K, N))
        C, E = oracle.gemm(A, B, lib=lib)
        assert np.all(np.abs(C - A @ B) <= 2 * (K + 1) * 2.0 ** -53 * E)
        x = rng.uniform(-1, 1, K)
        y, Ey = oracle.gemv(A, x, lib=lib)
        assert np.all(np.abs(y - A @ x) <= 2 * (K + 1) * 2.0 ** -53 * Ey)


def pin_leading_dimensions(lib):
    """Padded rows (lda > K, ldb > N, ldc > N) give the same product, read no
    padding and write none."""
    rng = np.random.default_rng(17)
    M, N, K = 5, 6, 7
    lda, ldb, ldc = K + 3, N + 2, N + 5
    A = rng.uniform(-1, 1, (M, K))
    B = rng.uniform(-1, 1, (K, N))
    Ap = np.full((M, lda), np.nan)
    Ap[:, :K] = A
    Bp = np.full((K, ldb), np.nan)
    Bp[:, :N] = B
    Cp = np.full((M, ldc), -7.0)
    Ep = np.full((M, ldc), -7.0)
    oracle.gemm_strided(M, N, K, Ap.reshape(-1), lda, Bp.reshape(-1), ldb,
                        Cp.reshape(-1), ldc, Ep.reshape(-1), ldc, lib=lib)
    C, E = oracle.gemm(A, B, lib=lib)
    assert np.array_equal(Cp[:, :N], C) and np.array_equal(Ep[:, :N], E)
    assert np.all(Cp[:, N:] == -7.0) and np.all(Ep[:, N:] == -7.0)


def pin_empty_sum(lib):
    """K = 0: every output is the empty sum, 0."""
    C, E = oracle.gemm(np.zeros((3, 0)), np.zeros((0, 4)), lib=lib)
    assert C.shape == (3, 4) and np.all(C == 0) and np.all(E == 0)
    y, Ey = oracle.gemv(np.zeros((3, 0)), np.zeros(0), lib=lib)
    assert np.all(y == 0) and np.all(Ey == 0)


def pin_thread_invariance(lib):
    """Rows have one owner each: any thread count gives identical bits."""
    rng = np.random.default_rng(18)
    A = rng.uniform(-1, 1, (41, 77))
    B = rng.uniform(-1, 1, (77, 13))
    ref = oracle.gemm(A, B, threads=1, lib=lib)
    for t in (2, 3, 0, 64):
        got = oracle.gemm(A, B, threads=t, lib=lib)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def pin_golden_dense_layer(lib):
    """Hand-worked batch of a fully connected layer: bias per column, ReLU."""
    g = read_golden("dense_layer_hand.txt")
    lin, _ = oracle.dense_layer(g["X"], g["WT"], g["bias"][0], "none", lib=lib)
    out, _ = oracle.dense_layer(g["X"], g["WT"], g["bias"][0], "relu", lib=lib)
    assert np.array_equal(lin, g["linear"]) and np.array_equal(out, g["relu"])


def pin_bias_act_closed_forms(lib):
    """A = 0 gives act(bias); ReLU keeps non-negative values and zeroes the
    rest; a GEMV bias is per row, a GEMM bias per column."""
    rng = np.random.default_rng(19)
    b = rng.uniform(-1, 1, 6)
    out, _ = oracle.dense_layer(np.zeros((4, 5)), np.zeros((5, 6)), b, "relu", lib=lib)
    assert np.array_equal(out, np.tile(np.maximum(b, 0), (4, 1)))
    y, _ = oracle.dense_vector(np.zeros((6, 3)), np.ones(3), b, "none", lib=lib)
    assert np.array_equal(y, b)
    v = rng.uniform(-1, 1, (7, 9))
    r = oracle.bias_act(v, None, True, "relu", lib=lib)
    assert np.array_equal(r, np.where(v > 0, v, 0.0))
    rows = oracle.bias_act(np.zeros((3, 2)), np.array([1.0, -2.0, 3.0]), False, "none", lib=lib)
    assert np.array_equal(rows, np.array([[1.0, 1.0], [-2.0, -2.0], [3.0, 3.0]]))


def pin_conv_golden(lib):
    """Hand-worked convolutions: padding, stride, dilation, a non-square
    kernel and two input and output channels (catches swapped indices)."""
    g = read_golden("conv2d_hand.txt")
    X1 = g["X1"].reshape(1, 3, 3, 1)
    W1 = g["W1"].reshape(2, 2, 1, 1)
    Y, _ = oracle.conv2d(X1, W1, lib=lib)
    assert np.array_equal(Y[0, :, :, 0], g["Y1_valid"])
    Y, _ = oracle.conv2d(X1, W1, stride=2, pad=1, lib=lib)
    assert np.array_equal(Y[0, :, :, 0], g["Y1_s2p1"])
    X2 = np.stack([g["X2c0"], g["X2c1"]], axis=-1)[None]
    W2 = np.stack([g["W2k0"], g["W2k1"]])[:, None]          # KH=2, KW=1, C=2, CO=2
    Y, E = oracle.conv2d(X2, W2, lib=lib)
    assert Y.shape == (1, 1, 3, 2)
    assert np.array_equal(Y[0, 0], g["Y2"]) and np.array_equal(E[0, 0], g["E2"])
    X3 = np.arange(1, 17, dtype=np.float64).reshape(1, 4, 4, 1)
    Y, _ = oracle.conv2d(X3, W1, dil=2, lib=lib)
    assert np.array_equal(Y[0, :, :, 0], g["Y3"])


def pin_conv_1x1_is_gemm(lib):
    """A 1x1 kernel at stride 1 is the matrix product of pixels x channels
    with the C x CO weight matrix (the GEMM, a separate loop nest); same
    ascending channel order, so bit-identical."""
    rng = np.random.default_rng(30)
    X = rng.uniform(-1, 1, (2, 5, 7, 6))
    Wt = rng.uniform(-1, 1, (1, 1, 6, 4))
    Y, E = oracle.conv2d(X, Wt, lib=lib)
    C, Eg = oracle.gemm(X.reshape(-1, 6), Wt.reshape(6, 4), lib=lib)
    assert np.array_equal(Y.reshape(-1, 4), C) and np.array_equal(E.reshape(-1, 4), Eg)


def pin_conv_vs_library_correlate(lib):
    """Against scipy's 2-D cross-correlation, one (input, output) channel pair
    at a time: stride by subsampling the stride-1 result, padding by padding
    the image, dilation by spreading the kernel with zeros."""
    signal = pytest.importorskip("scipy.signal")
    rng = np.random.default_rng(31)
    for (H, W_, C, CO, KH, KW, s, p, d) in [(7, 9, 3, 2, 3, 2, 1, 0, 1), (8, 6, 2, 3, 3, 3, 2, 1, 1),
                                             (9, 9, 2, 2, 2, 3, 1, 2, 2), (6, 11, 1, 2, 1, 4, 3, 1, 1)]:
        X = rng.uniform(-1, 1, (2, H, W_, C))
        Wt = rng.uniform(-1, 1, (KH, KW, C, CO))
        Y, E = oracle.conv2d(X, Wt, stride=s, pad=p, dil=d, lib=lib)
        Kd = np.zeros((d * (KH - 1) + 1, d * (KW - 1) + 1, C, CO))
        Kd[::d, ::d] = Wt
        for n in range(2):
            for co in range(CO):
                ref = sum(signal.correlate2d(np.pad(X[n, :, :, ci], p), Kd[:, :, ci, co], mode="valid")
                          for ci in range(C))[::s, ::s]
                assert ref.shape == Y.shape[1:3]
                assert np.all(np.abs(Y[n, :, :, co] - ref) <= 4 * KH * KW * C * 2.0 ** -53 * E[n, :, :, co])


def pin_conv_delta_kernel_shifts(lib):
    """A kernel that is one at (kh0, kw0, ci0 -> co0) and zero elsewhere copies
    channel ci0, shifted by the tap, into output channel co0 (zeros where the
    tap falls in the padding); every other output channel is zero."""
    rng = np.random.default_rng(32)
    X = rng.uniform(-1, 1, (1, 5, 6, 3))
    Wt = np.zeros((3, 3, 3, 2))
    Wt[2, 0, 1, 1] = 1.0
    Y, _ = oracle.conv2d(X, Wt, pad=1, lib=lib)
    assert np.all(Y[..., 0] == 0)
    want = np.zeros((5, 6))
    want[:4, 1:] = X[0, 1:, :5, 1]        # output (oh, ow) reads input (oh + 1, ow - 1)
    assert np.array_equal(Y[0, :, :, 1], want)


def pin_conv_magnitude(lib):
    """E >= |Y|; E == Y for non-negative operands; all-ones counts the taps
    inside the image times C."""
    rng = np.random.default_rng(33)
    X = rng.uniform(-1, 1, (1, 6, 5, 2))
    Wt = rng.uniform(-1, 1, (3, 2, 2, 3))
    Y, E = oracle.conv2d(X, Wt, stride=(2, 1), pad=(1, 2), lib=lib)
    assert np.all(E >= np.abs(Y))
    Yp, Ep = oracle.conv2d(np.abs(X), np.abs(Wt), stride=(2, 1), pad=(1, 2), lib=lib)
    assert np.array_equal(Yp, Ep)
    Y1, _ = oracle.conv2d(np.ones((1, 4, 4, 3)), np.ones((3, 3, 3, 1)), pad=1, lib=lib)
    # interior outputs see 9 taps, edges 6, corners 4
    assert np.array_equal(Y1[0, :, :, 0], 3 * np.array([[4, 6, 6, 4], [6, 9, 9, 6], [6, 9, 9, 6], [4, 6, 6, 4]]))


PINS = [pin_conv_golden, pin_conv_1x1_is_gemm, pin_conv_vs_library_correlate, pin_conv_delta_kernel_shifts,
        pin_conv_magnitude, pin_golden_dense_layer, pin_bias_act_closed_forms, pin_golden_gemm, pin_golden_gemv, pin_identity, pin_all_ones,
        pin_small_integers_exact, pin_exact_rational, pin_rank_one,
        pin_gemv_is_gemm_with_one_column, pin_magnitude, pin_vs_library_matmul,
        pin_leading_dimensions, pin_empty_sum, pin_thread_invariance]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.load())


def test_oracle_rejects_bad_arguments():
    lib = oracle.load()
    a = np.zeros(4)
    with pytest.raises(RuntimeError):
        oracle.gemm_strided(2, 2, 2, a, 1, a, 2, a, 2, lib=lib)   # lda < K
    with pytest.raises(ValueError):
        oracle.gemm(np.zeros((2, 3)), np.zeros((2, 3)), lib=lib)
