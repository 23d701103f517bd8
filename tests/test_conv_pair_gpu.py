"""Implicit-GEMM convolution on the CTA-pair tensor-core kernel (256 x 256
tiles of Y, each CTA's 128 output pixels of a K slice one TMA im2col load)
against the FP64 oracle's direct convolution, element by element, through the
C ABI. The tests force that kernel (gtg_conv_force_path "implicit_pair"), so
a silent fall-back to another kernel fails them."""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
from seeded import PCG32
from tests.test_conv_gpu import IMPLICIT_CASES, _draw, check, run_conv

pytestmark = pytest.mark.gpu


@pytest.fixture
def pair_path():
    gtg.gtg_conv_force_path("implicit_pair")
    yield
    gtg.gtg_conv_force_path("auto")
    gtg.gtg_force_gemm_splits(0)


def _plan(prec, N, H, W, C, CO, KH, KW, s, p, d):
    (sh, sw), (ph, pw), (dh, dw) = [(v, v) if isinstance(v, int) else v for v in (s, p, d)]
    return gtg.plan_conv2d(prec, N, H, W, C, CO, KH, KW, sh, sw, ph, pw, dh, dw, 1 << 32, 2 << 32, 3 << 32)


PAIR_CASES = IMPLICIT_CASES + [
    (3, 23, 19, 64, 320, 3, 3, 1, 1, 1),     # M = 1311 (ragged pair row-tiles), CO = 320 (ragged column tile)
    (5, 64, 64, 64, 64, 3, 3, 1, 1, 1),      # 80 pair tiles on 76 clusters: a second wave, whose K runs backwards
]


@pytest.mark.parametrize("prec", ["bf16", "f16"])
@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: "x".join(str(v) for v in c))
def test_pair_implicit_gemm_conv(pair_path, prec, case):
    N, H, W, C, CO, KH, KW, s, p, d = case
    plan = _plan(prec, N, H, W, C, CO, KH, KW, s, p, d)
    assert plan["kernel"] == "tcgen05" and plan["cluster"] == 2 and plan["bm"] == 256, plan
    g = PCG32(4500 + N * H * W + C * CO + KH)
    X, Xf = _draw(prec, g, (N, H, W, C))
    Wt, Wf = _draw(prec, g, (KH, KW, C, CO), (KH * KW * C) ** -0.5)
    Y = run_conv(prec, X, Wt, s, p, d)
    check(prec, Xf, Wf, Y, s, p, d)


def test_pair_conv_with_bias_relu_and_tensor_stores(pair_path):
    # stride 2, bias and ReLU in the epilogue; 2 K slices per unit, so Y goes
    # out by tensor stores (32 x 32 blocks clipped at the edges)
    g = PCG32(4600)
    X, Xf = _draw("bf16", g, (2, 20, 18, 128))
    Wt, Wf = _draw("bf16", g, (1, 1, 128, 200), 128 ** -0.5)
    bias = g.uniform_f32((200,))
    Y = run_conv("bf16", X, Wt, 2, 0, 1, bias, "relu")
    check("bf16", Xf, Wf, Y, 2, 0, 1, bias, "relu")
    assert np.all(Y >= 0)


@pytest.mark.parametrize("splits", [2, 3])
def test_pair_conv_split_k(pair_path, splits):
    g = PCG32(4700 + splits)
    X, Xf = _draw("bf16", g, (2, 15, 13, 192))
    Wt, Wf = _draw("bf16", g, (3, 3, 192, 272), (9 * 192) ** -0.5)
    bias = g.uniform_f32((272,))
    gtg.gtg_force_gemm_splits(splits)
    plan = _plan("bf16", 2, 15, 13, 192, 272, 3, 3, 2, 1, 1)
    assert plan["cluster"] == 2 and plan["splits"] == splits, plan
    Y = run_conv("bf16", X, Wt, 2, 1, 1, bias, "relu")
    check("bf16", Xf, Wf, Y, 2, 1, 1, bias, "relu")


def test_pair_conv_small_integers_exact_and_repeatable(pair_path):
    rng = np.random.default_rng(4800)
    Xi = rng.integers(-4, 5, (3, 17, 19, 64))
    Wi = rng.integers(-4, 5, (3, 3, 64, 136))
    from seeded import f64_to_bf16_bits
    import oracle
    Xb, Wb = f64_to_bf16_bits(Xi.astype(np.float64)), f64_to_bf16_bits(Wi.astype(np.float64))
    Y1 = run_conv("bf16", Xb, Wb, 1, 1, 1)
    Y2 = run_conv("bf16", Xb, Wb, 1, 1, 1)
    ref, _ = oracle.conv2d(Xi.astype(np.float64), Wi.astype(np.float64), pad=1)
    assert np.array_equal(Y1, ref.astype(np.float32))
    assert np.array_equal(Y1, Y2)


def test_single_cta_choice_still_reachable():
    gtg.gtg_conv_force_path("implicit_single")
    try:
        plan = _plan("bf16", 4, 14, 14, 256, 256, 3, 3, 1, 1, 1)
        assert plan["cluster"] == 1 and plan["bm"] == 128, plan
    finally:
        gtg.gtg_conv_force_path("auto")
