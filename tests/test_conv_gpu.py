"""Convolutional layers through conv2d_nhwc (im2col + GEMM) against the FP64
oracle's direct convolution, element by element, through the C ABI.

Bound per output: the GEMM bound of the precision with K = KH*KW*C and E the
oracle's sum of |x*w| over the window (plus one FP32 rounding of the bias add
when an epilogue is applied)."""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32, bf16_bits_to_f32, f16_bits_to_f32
from tests._util import parity_ratio

pytestmark = pytest.mark.gpu

CANARY = np.float32(-12345.5)


def _t():
    import torch
    return torch


def _draw(prec, g, shape, sigma=1.0):
    if prec == "bf16":
        bits = g.normal_bf16(shape, sigma)
        return bits, bf16_bits_to_f32(bits)
    if prec == "f16":
        bits = g.normal_f16(shape, sigma)
        return bits, f16_bits_to_f32(bits)
    v = g.uniform_f32(shape)
    return v, v


def _dev(host):
    torch = _t()
    if host.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(host).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(host)).cuda()


def run_conv(prec, X, Wt, stride=1, pad=0, dil=1, bias=None, act="none"):
    """Y through conv2d_nhwc, with canaries after Y; returns Y (float32)."""
    torch = _t()
    N, H, W, C = X.shape
    KH, KW, _, CO = Wt.shape
    OH, OW = gtg.conv_out_size(H, W, KH, KW, stride, pad, dil)
    dX, dW = _dev(X), _dev(Wt)
    ny = N * OH * OW * CO
    dY = torch.full((ny + 64,), float("nan"), device="cuda")
    dY[ny:] = float(CANARY)
    db = torch.from_numpy(bias).cuda() if bias is not None else None
    ep = gtg.epilogue(db.data_ptr() if db is not None else 0, act) if (bias is not None or act != "none") else None
    (sh, sw), (ph, pw), (dh, dw) = [(v, v) if isinstance(v, int) else v for v in (stride, pad, dil)]
    s = int(torch.cuda.current_stream().cuda_stream)
    st = gtg.conv2d_nhwc(prec, N, H, W, C, CO, KH, KW, sh, sw, ph, pw, dh, dw, dX.data_ptr(), dW.data_ptr(),
                         dY.data_ptr(), ep, s)
    assert st == gtg.GTG_OK, gtg.status_string(st)
    assert gtg.gtg_sync_status(s) == gtg.GTG_OK
    out = dY.cpu().numpy()
    assert np.all(out[ny:] == CANARY), "write past Y"
    return out[:ny].reshape(N, OH, OW, CO)


def check(prec, Xf, Wf, Y, stride=1, pad=0, dil=1, bias=None, act="none"):
    ref, E = oracle.conv_layer(Xf, Wf, bias, act, stride=stride, pad=pad, dil=dil)
    K = Wf.shape[0] * Wf.shape[1] * Wf.shape[2]
    ratio, bad = parity_ratio(Y, ref, E, prec, K, rel=2.0 ** -23 if (bias is not None or act != "none") else 0.0)
    assert bad == 0, f"{bad} outputs out of bound (max ratio {ratio:.3g})"
    return ratio


CASES = [
    # (N, H, W, C, CO, KH, KW, stride, pad, dil)
    (2, 14, 14, 64, 64, 3, 3, 1, 1, 1),        # a 3x3 layer, 16-byte im2col chunks
    (1, 17, 13, 32, 48, 3, 3, 2, 1, 1),        # stride 2, ragged output
    (2, 32, 32, 3, 16, 7, 7, 2, 3, 1),         # first-layer shape: C = 3, element-wise im2col
    (3, 9, 11, 64, 32, 1, 1, 1, 0, 1),         # 1x1 stride 1: X is the patch matrix, no gather
    (1, 15, 15, 40, 24, 1, 1, 2, 0, 1),        # 1x1 stride 2: gathered
    (1, 12, 10, 16, 40, 3, 3, 1, 2, 2),        # dilation 2
    (2, 8, 20, 24, 16, 1, 5, 1, (0, 2), 1),    # non-square window
    (1, 6, 7, 12, 8, 3, 2, (2, 1), (1, 0), (1, 2)),   # mixed strides, paddings, dilations
]


@pytest.mark.parametrize("prec", ["bf16", "f16", "tf32", "f32"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(str(v) for v in c))
def test_conv_matches_direct_definition(prec, case):
    N, H, W, C, CO, KH, KW, s, p, d = case
    g = PCG32(2000 + N * H * W + C * CO + KH)
    X, Xf = _draw(prec, g, (N, H, W, C))
    Wt, Wf = _draw(prec, g, (KH, KW, C, CO), (KH * KW * C) ** -0.5)
    Y = run_conv(prec, X, Wt, s, p, d)
    check(prec, Xf, Wf, Y, s, p, d)


@pytest.mark.parametrize("prec", ["bf16", "f32"])
def test_conv_layer_with_bias_and_relu(prec):
    g = PCG32(2100)
    X, Xf = _draw(prec, g, (2, 10, 10, 32))
    Wt, Wf = _draw(prec, g, (3, 3, 32, 24), (9 * 32) ** -0.5)
    bias = g.uniform_f32((24,))
    Y = run_conv(prec, X, Wt, 1, 1, 1, bias, "relu")
    check(prec, Xf, Wf, Y, 1, 1, 1, bias, "relu")
    assert np.all(Y >= 0)


def test_resnet_stage_layer_bf16():
    """A 3x3, 64 -> 64 channel layer on 56 x 56 images, batch 4 (the widths of
    a residual network's first stage)."""
    g = PCG32(2200)
    X, Xf = _draw("bf16", g, (4, 56, 56, 64))
    Wt, Wf = _draw("bf16", g, (3, 3, 64, 64), 576 ** -0.5)
    Y = run_conv("bf16", X, Wt, 1, 1, 1)
    check("bf16", Xf, Wf, Y, 1, 1, 1)


def test_small_integer_convolution_is_exact():
    rng = np.random.default_rng(2300)
    Xi = rng.integers(-4, 5, (2, 9, 9, 16))
    Wi = rng.integers(-4, 5, (3, 3, 16, 8))
    from seeded import f64_to_bf16_bits
    Y = run_conv("bf16", f64_to_bf16_bits(Xi.astype(np.float64)), f64_to_bf16_bits(Wi.astype(np.float64)), 1, 1, 1)
    ref, _ = oracle.conv2d(Xi.astype(np.float64), Wi.astype(np.float64), pad=1)
    assert np.array_equal(Y, ref.astype(np.float32))


def test_conv2d_helper_on_torch_tensors():
    torch = _t()
    g = PCG32(2400)
    X, Xf = _draw("bf16", g, (1, 12, 12, 16))
    Wt, Wf = _draw("bf16", g, (3, 3, 16, 8), 144 ** -0.5)
    tX = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16)
    tW = torch.from_numpy(Wt.view(np.int16)).view(torch.bfloat16)
    Yd = gtg.conv2d(tX.cuda(), tW.cuda(), stride=1, pad=1)
    Yh = gtg.conv2d(tX, tW, stride=1, pad=1)                # host tensors: copied in and out
    assert torch.equal(Yd.cpu(), Yh)
    check("bf16", Xf, Wf, Yh.numpy(), 1, 1, 1)


# ---- implicit GEMM: the tensor-core kernel loads the patches from X with TMA
# in im2col mode (16-bit inputs, C a multiple of 64); the tests require that
# path, so a silent fall-back to the patch matrix fails them

@pytest.fixture
def conv_path():
    yield gtg.gtg_conv_force_path
    gtg.gtg_conv_force_path("auto")


IMPLICIT_CASES = [
    (2, 14, 14, 64, 64, 3, 3, 1, 1, 1),
    (1, 17, 13, 128, 96, 3, 3, 2, 1, 1),             # stride 2, ragged output, CO = 96
    (1, 12, 10, 64, 40, 3, 3, 1, 2, 2),              # dilation 2
    (2, 8, 20, 64, 16, 1, 5, 1, (0, 2), 1),          # 1 x 5, padding along W only
    (1, 9, 7, 64, 24, 3, 2, (2, 1), (1, 0), (1, 2)),  # per-axis strides, paddings, dilations
    (2, 32, 32, 64, 128, 7, 7, 2, 3, 1),             # 7 x 7 / 2
    (3, 5, 6, 64, 8, 1, 1, 2, 0, 1),                 # 1 x 1 / 2
    (1, 7, 7, 192, 64, 3, 3, 1, 1, 1),               # three 64-channel blocks
    (3, 9, 11, 64, 32, 1, 1, 1, 0, 1),               # 1 x 1 / 1
    (5, 11, 13, 64, 264, 3, 3, 1, 1, 1),             # CO beyond one 256-wide tile
]


@pytest.mark.parametrize("prec", ["bf16", "f16"])
@pytest.mark.parametrize("case", IMPLICIT_CASES, ids=lambda c: "x".join(str(v) for v in c))
def test_implicit_gemm_conv(conv_path, prec, case):
    N, H, W, C, CO, KH, KW, s, p, d = case
    g = PCG32(2500 + N * H * W + C * CO + KH)
    X, Xf = _draw(prec, g, (N, H, W, C))
    Wt, Wf = _draw(prec, g, (KH, KW, C, CO), (KH * KW * C) ** -0.5)
    conv_path("implicit")
    Y = run_conv(prec, X, Wt, s, p, d)
    check(prec, Xf, Wf, Y, s, p, d)


def test_implicit_gemm_conv_with_epilogue_and_both_paths(conv_path):
    g = PCG32(2600)
    X, Xf = _draw("bf16", g, (2, 20, 18, 128))
    Wt, Wf = _draw("bf16", g, (3, 3, 128, 72), (9 * 128) ** -0.5)
    bias = g.uniform_f32((72,))
    for path in ("implicit", "explicit"):
        conv_path(path)
        Y = run_conv("bf16", X, Wt, 2, 1, 1, bias, "relu")
        check("bf16", Xf, Wf, Y, 2, 1, 1, bias, "relu")


def test_implicit_gemm_refuses_what_it_cannot_take(conv_path):
    torch = _t()
    conv_path("implicit")
    X = torch.zeros((1, 8, 8, 32), dtype=torch.int16, device="cuda")          # C = 32: not a 64-channel block
    Wt = torch.zeros((3, 3, 32, 16), dtype=torch.int16, device="cuda")
    Y = torch.empty((1, 6, 6, 16), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    st = gtg.conv2d_nhwc("bf16", 1, 8, 8, 32, 16, 3, 3, 1, 1, 0, 0, 1, 1, X.data_ptr(), Wt.data_ptr(), Y.data_ptr(),
                         None, s)
    assert st == gtg.GTG_ERR_UNSUPPORTED


@pytest.mark.parametrize("splits", [2, 3, 5])
def test_implicit_gemm_conv_split_k(conv_path, splits):
    # K split into ranges (forced): each range's partial tiles go to a workspace
    # slab and the ordered reduction adds them and applies bias + ReLU; ragged
    # output (stride 2), three 64-channel blocks x 9 taps = 27 K slices, CO = 72
    g = PCG32(2700 + splits)
    X, Xf = _draw("bf16", g, (2, 15, 13, 192))
    Wt, Wf = _draw("bf16", g, (3, 3, 192, 72), (9 * 192) ** -0.5)
    bias = g.uniform_f32((72,))
    conv_path("implicit")
    gtg.gtg_force_gemm_splits(splits)
    try:
        Y = run_conv("bf16", X, Wt, 2, 1, 1, bias, "relu")
    finally:
        gtg.gtg_force_gemm_splits(0)
    check("bf16", Xf, Wf, Y, 2, 1, 1, bias, "relu")


def test_deep_layer_takes_k_ranges_and_matches():
    # 3 x 3, 512 -> 512 channels on 7 x 7 images: few tiles, 72 K slices; the
    # planner splits K here (parity only: the split is the planner's choice)
    g = PCG32(2800)
    X, Xf = _draw("bf16", g, (4, 7, 7, 512))
    Wt, Wf = _draw("bf16", g, (3, 3, 512, 512), (9 * 512) ** -0.5)
    Y = run_conv("bf16", X, Wt, 1, 1, 1)
    check("bf16", Xf, Wf, Y, 1, 1, 1)
