"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module only draws numbers. It holds none of the arithmetic of the
matrix products: it produces the matrices and vectors that both the CUDA path
and the FP64 oracle consume, so that the two sides see bit-identical inputs.

Generator: PCG32, i.e. PCG-XSH-RR with 64-bit state and 32-bit output
(M. E. O'Neill, "PCG: A Family of Simple Fast Space-Efficient Statistically
Good Algorithms for Random Number Generation", 2014). The state advances by
the 64-bit LCG  s <- s * 6364136223846793005 + inc  (mod 2^64) and each output
is an xorshift-high + random-rotation permutation of the *old* state. Seeding
follows the reference "srandom" procedure with initstate = initseq = seed.

Because the LCG is affine, the state k steps ahead is  A_k * s + C_k  with
(A_k, C_k) the k-fold composition of the step. This module uses that to draw
large blocks with numpy (vectorised jump-ahead), producing exactly the same
sequence as the scalar recurrence.

Distributions:
  * uniform [-1, 1):  x = (r >> 8) * 2^-23 - 1, exactly representable in FP32.
  * normal(0, sigma): Box-Muller in FP64 from a pair of 24-bit uniforms
    u1 = ((r0 >> 8) + 1) * 2^-24 in (0, 1], u2 = (r1 >> 8) * 2^-24 in [0, 1);
    z0 = sqrt(-2 ln u1) cos(2 pi u2), z1 = sqrt(-2 ln u1) sin(2 pi u2), both
    used, in that order; then scaled by sigma.
  * BF16 and FP16: round-to-nearest-even directly from the FP64 value.
"""

from __future__ import annotations

import numpy as np

_MULT = 6364136223846793005
_MASK = (1 << 64) - 1
_BLOCK = 1 << 16          # states produced per vectorised jump
_CHUNK = 1 << 22          # outputs converted per pass (bounds temporary memory)


def _compose(a1: int, c1: int, a2: int, c2: int) -> tuple[int, int]:
    """Affine map (a2, c2) applied after (a1, c1): s -> a2 (a1 s + c1) + c2."""
    return (a2 * a1) & _MASK, (a2 * c1 + c2) & _MASK


class PCG32:
    """PCG-XSH-RR 64/32 generator with a vectorised block draw."""

    def __init__(self, initstate: int, initseq: int | None = None):
        if initseq is None:
            initseq = initstate
        self.inc = ((int(initseq) << 1) | 1) & _MASK
        s = 0
        s = (s * _MULT + self.inc) & _MASK
        s = (s + (int(initstate) & _MASK)) & _MASK
        s = (s * _MULT + self.inc) & _MASK
        self.state = s
        # offsets of one block: state_i = A_i * s0 + C_i for i in [0, _BLOCK)
        a_i = np.empty(_BLOCK, dtype=np.uint64)
        c_i = np.empty(_BLOCK, dtype=np.uint64)
        a, c = 1, 0
        for i in range(_BLOCK):
            a_i[i] = a
            c_i[i] = c
            a, c = _compose(a, c, _MULT, self.inc)
        self._a_i, self._c_i = a_i, c_i
        self._a_block, self._c_block = a, c          # jump of _BLOCK steps

    # scalar path, used by tests to cross-check the vectorised draw
    def next_u32_scalar(self) -> int:
        old = self.state
        self.state = (old * _MULT + self.inc) & _MASK
        xs = (((old >> 18) ^ old) >> 27) & 0xFFFFFFFF
        rot = old >> 59
        return ((xs >> rot) | (xs << ((-rot) & 31))) & 0xFFFFFFFF

    @staticmethod
    def _output(old: np.ndarray) -> np.ndarray:
        xs = (((old >> np.uint64(18)) ^ old) >> np.uint64(27)) & np.uint64(0xFFFFFFFF)
        rot = old >> np.uint64(59)
        left = (np.uint64(32) - rot) & np.uint64(31)
        out = (xs >> rot) | (xs << left)
        return (out & np.uint64(0xFFFFFFFF)).astype(np.uint32)

    def next_u32(self, n: int) -> np.ndarray:
        """The next n outputs as uint32, identical to n scalar draws."""
        out = np.empty(n, dtype=np.uint32)
        pos = 0
        with np.errstate(over="ignore"):
            while pos < n:
                take = min(_BLOCK, n - pos)
                s0 = np.uint64(self.state)
                states = self._a_i[:take] * s0 + self._c_i[:take]
                out[pos:pos + take] = self._output(states)
                pos += take
                if take == _BLOCK:
                    self.state = (self._a_block * self.state + self._c_block) & _MASK
                else:
                    a, c = int(self._a_i[take - 1]), int(self._c_i[take - 1])
                    a, c = _compose(a, c, _MULT, self.inc)
                    self.state = (a * self.state + c) & _MASK
        return out

    # ---- distributions -------------------------------------------------
    def uniform_f32(self, shape) -> np.ndarray:
        """i.i.d. uniform [-1, 1) in FP32 (every value exactly representable)."""
        n = int(np.prod(shape))
        out = np.empty(n, dtype=np.float32)
        for p in range(0, n, _CHUNK):
            r = self.next_u32(min(_CHUNK, n - p))
            out[p:p + r.size] = ((r >> np.uint32(8)).astype(np.float64) * 2.0 ** -23 - 1.0)
        return out.reshape(shape)

    def _normal_chunks(self, n: int, sigma: float):
        """Yield (offset, FP64 block) covering n normal(0, sigma) draws."""
        pairs = (n + 1) // 2
        step = _CHUNK // 2
        for p in range(0, pairs, step):
            m = min(step, pairs - p)
            r = self.next_u32(2 * m).reshape(m, 2)
            u1 = ((r[:, 0] >> np.uint32(8)).astype(np.float64) + 1.0) * 2.0 ** -24
            u2 = (r[:, 1] >> np.uint32(8)).astype(np.float64) * 2.0 ** -24
            rad = np.sqrt(-2.0 * np.log(u1))
            ang = 2.0 * np.pi * u2
            z = np.empty((m, 2), dtype=np.float64)
            z[:, 0] = rad * np.cos(ang)
            z[:, 1] = rad * np.sin(ang)
            z = z.reshape(-1)[: min(2 * m, n - 2 * p)]
            yield 2 * p, z * sigma

    def normal_f64(self, shape, sigma: float = 1.0) -> np.ndarray:
        """i.i.d. normal(0, sigma) in FP64 by Box-Muller (pairs, z0 then z1)."""
        n = int(np.prod(shape))
        out = np.empty(n, dtype=np.float64)
        for off, z in self._normal_chunks(n, sigma):
            out[off:off + z.size] = z
        return out.reshape(shape)

    def normal_f16(self, shape, sigma: float = 1.0) -> np.ndarray:
        """normal(0, sigma) rounded to FP16; returned as uint16 bit patterns."""
        n = int(np.prod(shape))
        out = np.empty(n, dtype=np.uint16)
        for off, z in self._normal_chunks(n, sigma):
            out[off:off + z.size] = f64_to_f16_bits(z)
        return out.reshape(shape)

    def normal_bf16(self, shape, sigma: float = 1.0) -> np.ndarray:
        """normal(0, sigma) rounded to BF16; returned as uint16 bit patterns."""
        n = int(np.prod(shape))
        out = np.empty(n, dtype=np.uint16)
        for off, z in self._normal_chunks(n, sigma):
            out[off:off + z.size] = f64_to_bf16_bits(z)
        return out.reshape(shape)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round FP64 values to the nearest BF16 (ties to even); uint16 bits.

    Values are assumed finite and inside the BF16 normal range (the inputs
    drawn here are); the FP64 significand is rounded to 7 explicit bits and
    the exactly-representable result is narrowed to FP32, whose top half is
    the BF16 pattern.
    """
    b = np.ascontiguousarray(x, dtype=np.float64).view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    r = (b + (np.uint64((1 << 44) - 1) + lsb)) & ~np.uint64((1 << 45) - 1)
    f = r.view(np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def f64_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round FP64 values to the nearest IEEE binary16 (ties to even); uint16 bits."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of binary16 bit patterns to FP32."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns to FP32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---- the workloads' input recipes -------------------------------------------
# Each returns host numpy arrays; the draw order is fixed and documented.

def gemm_uniform_f32(seed: int, M: int, N: int, K: int):
    """A (MxK) then B (KxN), uniform [-1, 1) FP32, one stream seeded `seed`."""
    g = PCG32(seed)
    A = g.uniform_f32((M, K))
    B = g.uniform_f32((K, N))
    return A, B


def gemm_normal_bf16(seed: int, shapes, sigma_of_k=None):
    """For each (M, N, K) in `shapes`, in order: A then B from one stream.

    Entries are normal(0, sigma) rounded to BF16 with sigma = sigma_of_k(K)
    (sigma = 1 when `sigma_of_k` is None). Returns a list of (A_bits, B_bits)
    uint16 arrays. Later shapes continue the same stream.
    """
    g = PCG32(seed)
    out = []
    for (M, N, K) in shapes:
        s = 1.0 if sigma_of_k is None else float(sigma_of_k(K))
        A = g.normal_bf16((M, K), s)
        B = g.normal_bf16((K, N), s)
        out.append((A, B))
    return out


def gemv_uniform_f32(seed: int, M: int, N: int, batch: int = 8):
    """A (MxN), then x (N), then `batch` further vectors (batch x N)."""
    g = PCG32(seed)
    A = g.uniform_f32((M, N))
    x = g.uniform_f32((N,))
    X = g.uniform_f32((batch, N))
    return A, x, X
