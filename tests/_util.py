"""Shared test helpers: golden-file parsing and the per-element acceptance bounds."""

from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

U32 = 2.0 ** -24   # unit roundoff of FP32 (round to nearest)

# Per-element bounds |c - ref| <= bound, with E = sum_k |a_ik b_kj| from the
# oracle. FP32 scales with the reduction length; the tensor-core paths round
# their operands, so their bound is a fixed relative multiple of E.
def bound_f32(E, K):
    return 4.0 * max(int(K), 1) * U32 * np.asarray(E)


def bound_tf32(E, K=None):
    return 4.0 * 2.0 ** -11 * np.asarray(E)


def bound_bf16(E, K=None):
    return 4.0 * 2.0 ** -8 * np.asarray(E)


def bound_f16(E, K=None):
    # FP16 inputs are exact in the products (11 x 11 significant bits fit in
    # FP32); what rounds is the FP32 accumulation, far inside 4 * 2^-11 E for
    # every K used here (K * 2^-24 <= 2^-11 up to K = 8192)
    return 4.0 * 2.0 ** -11 * np.asarray(E)


BOUNDS = {"f32": bound_f32, "tf32": bound_tf32, "bf16": bound_bf16, "f16": bound_f16}


def read_golden(name: str) -> dict[str, np.ndarray]:
    """Parse a fixture: `NAME rows cols` headers followed by rows of numbers."""
    out, cur, rows, want = {}, None, [], 0
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if cur is None or len(rows) == want:
                if cur is not None:
                    out[cur] = np.array(rows, dtype=np.float64)
                cur, want, ncols, rows = parts[0], int(parts[1]), int(parts[2]), []
                continue
            vals = [float(v) for v in parts]
            assert len(vals) == ncols, line
            rows.append(vals)
    if cur is not None:
        out[cur] = np.array(rows, dtype=np.float64)
    return out


def parity_ratio(c, ref, E, path, K, rel=0.0):
    """max |c - ref| / bound, and how many elements exceed their bound.
    `rel` adds rel * |ref| to the bound (2^-23 for an epilogue: one FP32
    rounding of the bias add; ReLU cannot increase an error)."""
    c = np.asarray(c, dtype=np.float64)
    bnd = BOUNDS[path](E, K) + rel * np.abs(ref)
    # an exactly-zero E means the reference is exactly zero: demand exactness
    err = np.where(np.isfinite(c), np.abs(c - ref), np.inf)
    ok = err <= bnd
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bnd > 0, err / np.where(bnd > 0, bnd, 1.0), np.where(err > 0, np.inf, 0.0))
    return float(ratio.max()) if ratio.size else 0.0, int((~ok).sum())
