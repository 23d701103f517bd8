"""gemv_bf16 at batch 3..8 on the tensor cores (each vector entry as three
BF16 pieces, stream-K over the SMs) against the FP64 oracle, element by
element, with the FP32 GEMV bound (K -> N), through the C ABI."""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32, bf16_bits_to_f32, f64_to_bf16_bits
from tests._gpu import run_gemv
from tests._util import parity_ratio

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tensor_cores():
    """The tensor-core path at every size (by default only from 2^25 elements)."""
    gtg.gtg_gemv_force_path("tensor_cores")
    yield
    gtg.gtg_gemv_force_path("auto")


def _plan(M, N, batch, lda=None):
    return gtg.plan_gemv(M, N, 1 << 32, lda or N, 2 << 32, N, 3 << 32, M, batch, precision="bf16")


def _check(A, X, Y, rows=None):
    Af = bf16_bits_to_f32(A if rows is None else A[rows])
    for b in range(X.shape[0]):
        ref, E = oracle.gemv(Af, X[b])
        got = Y[b] if rows is None else Y[b][rows]
        ratio, bad = parity_ratio(got, ref, E, "f32", A.shape[1])
        assert bad == 0, (b, ratio)
    return ratio


CASES = [
    # (M, N, batch): tiles of 128 rows x slices of 64 columns cut into 152 ranges
    (4096, 4096, 8),      # 32 tiles x 64 slices: every tile shared by ~5 CTAs
    (4096, 4096, 3),
    (1000, 1000, 5),      # ragged rows and columns
    (130, 72, 8),         # fewer units than SMs: ranges of one slice, ragged everywhere
    (300, 64, 4),         # one slice per tile: no tile shared
    (300, 16, 6),         # K shorter than a slice
    (5, 20000, 7),        # one tile over 152 CTAs (152 parts)
    (19456, 64, 8),       # 152 tiles of one slice: one whole tile per CTA
    (3000, 336, 3),       # 144 units
]


@pytest.mark.parametrize("M,N,batch", CASES, ids=lambda v: str(v))
def test_tc_gemv_matches_oracle(M, N, batch):
    g = PCG32(3500 + M + N + batch)
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((batch, N))
    plan = _plan(M, N, batch)
    assert plan["kernel"] == "tcgen05", plan
    Y = run_gemv(A, X, prec="bf16")
    rows = None if M * N <= 4_000_000 else np.unique(np.concatenate([np.arange(0, M, 7), [M - 1]]))
    _check(A, X, Y, rows)


def test_tc_gemv_padded_rows_and_vectors():
    g = PCG32(3600)
    M, N, batch = 777, 1000, 8
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((batch, N))
    assert _plan(M, N, batch, lda=1016)["kernel"] == "tcgen05"
    Y = run_gemv(A, X, lda=1016, ldx=1003, ldy=800, prec="bf16")
    _check(A, X, Y)


def test_planner_sizes():
    gtg.gtg_gemv_force_path("auto")
    assert _plan(8192, 4096, 8)["kernel"] == "tcgen05"    # 2^25 elements
    assert _plan(4096, 4096, 8)["kernel"] == "gemv"       # below: the CUDA cores
    assert _plan(8192, 8192, 2)["kernel"] == "gemv"       # batch 1-2: the streaming kernel
    assert _plan(8192, 8192, 5)["kernel"] == "gemv"       # batch 3-5: the CUDA cores
    assert _plan(8192, 8192, 6)["kernel"] == "tcgen05"


def test_tc_gemv_unaligned_rows_take_the_cuda_cores():
    assert _plan(500, 1000, 8, lda=1001)["kernel"] == "gemv"   # lda * 2 not a multiple of 16
    g = PCG32(3650)
    A = g.normal_bf16((500, 1000))
    X = g.uniform_f32((8, 1000))
    _check(A, X, run_gemv(A, X, lda=1001, prec="bf16"))


def test_tc_gemv_exact_for_small_integers():
    # integer vectors are their own first piece; every partial sum is an
    # integer below 2^24, so the tensor-core result is exact
    rng = np.random.default_rng(3700)
    Ai = rng.integers(-64, 65, (1500, 2048))
    xi = rng.integers(-64, 65, (8, 2048))
    Y = run_gemv(f64_to_bf16_bits(Ai.astype(np.float64)), xi.astype(np.float32), prec="bf16")
    assert np.array_equal(Y, (xi @ Ai.T).astype(np.float32))


def test_tc_gemv_needs_all_three_pieces():
    # N = 8: the bound is 4 * 8 * 2^-24 * E = 2^-19 E. Vector entries with
    # 24 significant bits leave a residual of up to 2^-9 of |x| after one BF16
    # piece and 2^-18 after two, so over 4096 x 8 outputs a kernel that
    # dropped the third piece (or the second) would exceed the bound
    g = PCG32(3750)
    M, N, batch = 4096, 8, 8
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((batch, N))
    assert _plan(M, N, batch)["kernel"] == "tcgen05"
    _check(A, X, run_gemv(A, X, prec="bf16"))


def test_tc_gemv_deterministic_and_close_to_the_cuda_cores():
    g = PCG32(3800)
    M, N, batch = 2048, 3000, 8
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((batch, N))
    Y1 = run_gemv(A, X, prec="bf16")
    Y2 = run_gemv(A, X, prec="bf16")
    assert np.array_equal(Y1, Y2)
    gtg.gtg_gemv_force_path("cuda_cores")
    try:
        assert _plan(M, N, batch)["kernel"] == "gemv"
        Yc = run_gemv(A, X, prec="bf16")
    finally:
        gtg.gtg_gemv_force_path("tensor_cores")
    _check(A, X, Yc)
    _check(A, X, Y1)


@pytest.mark.parametrize("act", ["none", "relu"])
def test_tc_gemv_epilogue(act):
    torch = pytest.importorskip("torch")
    g = PCG32(3900)
    M, N, batch = 1100, 900, 6     # tiles shared between CTAs: the epilogue runs in the gather
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((batch, N))
    bias = g.uniform_f32((M,))
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dX = torch.from_numpy(X).cuda()
    dY = torch.empty((batch, M), device="cuda")
    db = torch.from_numpy(bias).cuda()
    ep = gtg.epilogue(db.data_ptr(), act)
    s = int(torch.cuda.current_stream().cuda_stream)
    st = gtg.gemv_bf16_ex(M, N, dA.data_ptr(), N, dX.data_ptr(), N, dY.data_ptr(), M, batch, ep, s)
    assert st == gtg.GTG_OK and gtg.gtg_sync_status(s) == gtg.GTG_OK
    Y = dY.cpu().numpy()
    Af = bf16_bits_to_f32(A)
    for b in range(batch):
        ref, E = oracle.dense_vector(Af, X[b], bias, act)
        ratio, bad = parity_ratio(Y[b], ref, E, "f32", N, rel=2.0 ** -23)
        assert bad == 0, (b, ratio)
    if act == "relu":
        assert np.all(Y >= 0)
