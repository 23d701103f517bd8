"""TF32 convolutional layers as an implicit GEMM against the FP64 oracle's
direct convolution, element by element, through the C ABI.

A TF32 layer with C a multiple of 32 reads its patches with TMA im2col loads
(32 FP32 channels = one 128-byte block) from a copy of the image rounded to
the nearest TF32 value, and the weights from a rounded W^T; the single-CTA
and CTA-pair kernels are each forced in turn, so a silent fall-back to the
patch matrix fails the tests. Bound per output: 4 * 2^-11 * E with
K = KH*KW*C and E the oracle's sum of |x*w| over the window.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32
from tests.test_conv_gpu import _draw, check, run_conv

pytestmark = pytest.mark.gpu


@pytest.fixture
def conv_path():
    yield gtg.gtg_conv_force_path
    gtg.gtg_conv_force_path("auto")
    gtg.gtg_force_gemm_splits(0)


def _plan(N, H, W, C, CO, KH, KW, s, p, d):
    (sh, sw), (ph, pw), (dh, dw) = [(v, v) if isinstance(v, int) else v for v in (s, p, d)]
    return gtg.plan_conv2d("tf32", N, H, W, C, CO, KH, KW, sh, sw, ph, pw, dh, dw, 1 << 32, 2 << 32, 3 << 32)


TF32_CASES = [
    (2, 14, 14, 64, 64, 3, 3, 1, 1, 1),
    (1, 17, 13, 32, 48, 3, 3, 2, 1, 1),              # one 32-channel block, stride 2, ragged output
    (1, 12, 10, 96, 40, 3, 3, 1, 2, 2),              # three channel blocks, dilation 2
    (2, 8, 20, 32, 16, 1, 5, 1, (0, 2), 1),          # 1 x 5, padding along W only
    (1, 9, 7, 64, 24, 3, 2, (2, 1), (1, 0), (1, 2)),  # per-axis strides, paddings, dilations
    (2, 32, 32, 32, 128, 7, 7, 2, 3, 1),             # 7 x 7 / 2
    (3, 5, 6, 32, 8, 1, 1, 2, 0, 1),                 # 1 x 1 / 2
    (5, 11, 13, 64, 264, 3, 3, 1, 1, 1),             # CO beyond one 256-wide tile
    (3, 23, 19, 32, 300, 3, 3, 1, 1, 1),             # ragged pair row-tiles and column tile
]


@pytest.mark.parametrize("path", ["implicit_single", "implicit_pair"])
@pytest.mark.parametrize("case", TF32_CASES, ids=lambda c: "x".join(str(v) for v in c))
def test_tf32_implicit_conv(conv_path, path, case):
    N, H, W, C, CO, KH, KW, s, p, d = case
    conv_path(path)
    plan = _plan(N, H, W, C, CO, KH, KW, s, p, d)
    assert plan["kernel"] == "tcgen05" and plan["bk"] == 32, plan
    assert (plan["cluster"] == 2) == (path == "implicit_pair"), plan
    g = PCG32(5100 + N * H * W + C * CO + KH)
    X, Xf = _draw("tf32", g, (N, H, W, C))
    Wt, Wf = _draw("tf32", g, (KH, KW, C, CO), (KH * KW * C) ** -0.5)
    Y = run_conv("tf32", X, Wt, s, p, d)
    check("tf32", Xf, Wf, Y, s, p, d)


def test_tf32_conv_takes_the_implicit_route_by_default():
    plan = _plan(2, 14, 14, 64, 64, 3, 3, 1, 1, 1)
    assert plan["kernel"] == "tcgen05" and plan["bk"] == 32, plan
    # C not a multiple of 32: the patch matrix, then gemm_tf32
    g = PCG32(5200)
    X, Xf = _draw("tf32", g, (1, 9, 9, 24))
    Wt, Wf = _draw("tf32", g, (3, 3, 24, 16), 216 ** -0.5)
    Y = run_conv("tf32", X, Wt, 1, 1, 1)
    check("tf32", Xf, Wf, Y, 1, 1, 1)


@pytest.mark.parametrize("path", ["implicit_single", "implicit_pair"])
def test_tf32_implicit_conv_bias_relu_and_split_k(conv_path, path):
    g = PCG32(5300)
    X, Xf = _draw("tf32", g, (2, 15, 13, 96))
    Wt, Wf = _draw("tf32", g, (3, 3, 96, 72), (9 * 96) ** -0.5)
    bias = g.uniform_f32((72,))
    conv_path(path)
    for splits in (0, 3):
        gtg.gtg_force_gemm_splits(splits)
        Y = run_conv("tf32", X, Wt, 2, 1, 1, bias, "relu")
        check("tf32", Xf, Wf, Y, 2, 1, 1, bias, "relu")
        assert np.all(Y >= 0)


def test_tf32_implicit_conv_rounds_to_nearest(conv_path):
    """Every input 1 + 2^-10 - 2^-23 times a power of two, all positive: the 13
    bits TF32 drops are all ones, so truncation would lose almost 2^-10 of
    each operand and reach the whole bound; rounding to nearest loses 2^-23."""
    c = np.float32(1 + 2.0 ** -10 - 2.0 ** -23)
    g = PCG32(5400)
    N, H, W, C, CO = 2, 12, 12, 64, 48
    ex = (g.next_u32(N * H * W * C) % 3).astype(np.int64).reshape(N, H, W, C) - 1
    ew = (g.next_u32(9 * C * CO) % 3).astype(np.int64).reshape(3, 3, C, CO) - 1
    X = (c * np.ldexp(np.float32(1), ex)).astype(np.float32)
    Wt = (c * np.ldexp(np.float32(1), ew) / 64).astype(np.float32)
    for path in ("implicit_single", "implicit_pair"):
        conv_path(path)
        Y = run_conv("tf32", X, Wt, 1, 1, 1)
        ratio = check("tf32", X, Wt, Y, 1, 1, 1)
        ref, E = oracle.conv_layer(X, Wt, None, "none", stride=1, pad=1, dil=1)
        rel = np.abs(Y.astype(np.float64) - ref) / E
        assert rel.max() < 2.0 ** -12, (path, rel.max(), ratio)   # far below the truncation level (~2^-9)
