"""The seeded input generator follows its published definition."""

import numpy as np

from seeded import (PCG32, bf16_bits_to_f32, f16_bits_to_f32, f64_to_bf16_bits, f64_to_f16_bits,
                    gemm_normal_bf16, gemm_uniform_f32, gemv_uniform_f32)


def test_pcg32_published_stream():
    # First outputs of PCG32 seeded with initstate=42, initseq=54, as printed
    # by the PCG reference distribution's demo program (pcg32-demo).
    g = PCG32(42, 54)
    want = [0xA15C02B7, 0x7B47F409, 0xBA1D3330, 0x83D2F293, 0xBFA4784B, 0xCBED606E]
    assert [int(v) for v in g.next_u32(6)] == want


def test_vectorised_draw_equals_scalar_recurrence():
    a, b = PCG32(5), PCG32(5)
    n = 3 * (1 << 16) + 77
    got = np.concatenate([a.next_u32(5), a.next_u32(n), a.next_u32(1)])
    ref = np.array([b.next_u32_scalar() for _ in range(n + 6)], dtype=np.uint32)
    assert np.array_equal(got, ref)
    assert a.state == b.state


def test_uniform_values_exact_and_in_range():
    x = PCG32(1).uniform_f32((300, 301))
    assert x.dtype == np.float32 and x.min() >= -1.0 and x.max() < 1.0
    k = (x.astype(np.float64) + 1.0) * 2.0 ** 23        # must be an integer < 2^24
    assert np.array_equal(k, np.round(k)) and k.max() < 2 ** 24
    assert abs(float(x.mean())) < 0.01


def test_normal_moments():
    z = PCG32(9).normal_f64((400000,), sigma=0.5)
    assert abs(z.mean()) < 0.005 and abs(z.std() - 0.5) < 0.005


def _bf16_nearest_reference(x):
    """Nearest BF16 by explicit search over neighbouring candidates."""
    f = x.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    cands = np.stack([f - np.uint32(0x10000), f, f + np.uint32(0x10000)])
    vals = cands.view(np.float32).astype(np.float64)
    d = np.abs(vals - x[None, :])
    best = d.min(axis=0)
    pick = np.empty(x.size, dtype=np.uint32)
    for i in range(x.size):
        ties = [int(c) for c, dd in zip(cands[:, i], d[:, i]) if dd == best[i]]
        even = [c for c in ties if ((c >> 16) & 1) == 0]
        pick[i] = (even or ties)[0]
    return (pick >> np.uint32(16)).astype(np.uint16)


def test_bf16_rounding_is_nearest_even():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(20000) * 3.0
    # exact midpoints between neighbouring BF16 values (ties must go to even)
    base = bf16_bits_to_f32(f64_to_bf16_bits(rng.standard_normal(200))).astype(np.float64)
    ulp = np.abs(base) * 2.0 ** -7
    x = np.concatenate([x, base + ulp / 2, base - ulp / 2])
    got = f64_to_bf16_bits(x)
    ref = _bf16_nearest_reference(x)
    assert np.array_equal(got, ref)


def test_recipes_shapes_and_stream_continuation():
    A, B = gemm_uniform_f32(4, 10, 7, 15)
    assert A.shape == (10, 15) and B.shape == (15, 7)
    g = PCG32(4)
    assert np.array_equal(A, g.uniform_f32((10, 15)))
    assert np.array_equal(B, g.uniform_f32((15, 7)))
    (A1, B1), (A2, B2) = gemm_normal_bf16(6, [(4, 3, 5), (2, 6, 3)], lambda k: k ** -0.5)
    g = PCG32(6)
    assert np.array_equal(A1, g.normal_bf16((4, 5), 5 ** -0.5))
    assert np.array_equal(B1, g.normal_bf16((5, 3), 5 ** -0.5))
    assert np.array_equal(A2, g.normal_bf16((2, 3), 3 ** -0.5))
    A, x, X = gemv_uniform_f32(2, 6, 9, batch=8)
    assert A.shape == (6, 9) and x.shape == (9,) and X.shape == (8, 9)


def test_f16_rounding_is_nearest_even():
    rng = np.random.default_rng(4)
    x = rng.standard_normal(20000) * 3.0
    base = f16_bits_to_f32(f64_to_f16_bits(rng.standard_normal(300))).astype(np.float64)
    up = np.nextafter(base.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    x = np.concatenate([x, (base + up) / 2])            # exact midpoints: ties to even
    got = f64_to_f16_bits(x)
    h = x.astype(np.float32).astype(np.float16)          # a nearby candidate
    cands = np.stack([np.nextafter(h, np.float16(-np.inf)), h, np.nextafter(h, np.float16(np.inf))])
    d = np.abs(cands.astype(np.float64) - x[None, :])
    best = d.min(axis=0)
    for i in range(x.size):
        ties = [c for c, dd in zip(cands[:, i], d[:, i]) if dd == best[i]]
        even = [c for c in ties if (int(np.array(c).view(np.uint16)) & 1) == 0]
        want = (even or ties)[0]
        assert got[i] == np.array(want).view(np.uint16), (x[i], got[i])
