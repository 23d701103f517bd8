"""GPU parity of gemv_f32 against the FP64 oracle, through the C ABI.

Bound per output: |y - ref| <= 4 N 2^-24 E with E = sum_j |a_ij x_j|.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32, gemv_uniform_f32
from tests._gpu import run_gemv
from tests._util import parity_ratio

pytestmark = pytest.mark.gpu


def check(A, X, Y):
    worst = 0.0
    for b in range(X.shape[0]):
        ref, E = oracle.gemv(A, X[b])
        ratio, bad = parity_ratio(Y[b], ref, E, "f32", A.shape[1])
        assert bad == 0, f"vector {b}: {bad} outputs out of bound (max ratio {ratio:.3g})"
        worst = max(worst, ratio)
    return worst


def test_fc_layer_4096_seed2_batch1_and_batch8():
    A, x, X = gemv_uniform_f32(2, 4096, 4096, batch=8)
    check(A, x[None, :], run_gemv(A, x[None, :]))
    check(A, X, run_gemv(A, X))


@pytest.mark.parametrize("n", [8192, 16384])
def test_larger_square(n):
    A, x, X = gemv_uniform_f32(2, n, n, batch=8)
    check(A, x[None, :], run_gemv(A, x[None, :]))
    check(A, X[:2], run_gemv(A, X[:2]))


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 6, 7, 8])
def test_every_batch_size(batch):
    g = PCG32(20 + batch)
    A = g.uniform_f32((523, 1031))
    X = g.uniform_f32((batch, 1031))
    check(A, X, run_gemv(A, X))


@pytest.mark.parametrize("M,N", [(1, 1), (1, 5), (5, 1), (3, 7), (31, 33), (152, 4), (151, 4097),
                                 (2049, 130), (10, 100003)])
def test_edge_shapes(M, N):
    g = PCG32(M * 7 + N)
    A = g.uniform_f32((M, N))
    X = g.uniform_f32((2, N))
    check(A, X[:1], run_gemv(A, X[:1]))
    check(A, X, run_gemv(A, X))


@pytest.mark.parametrize("batch", [3, 4, 5, 6, 7, 8])
def test_column_split_kernel_with_ragged_rows_and_width(batch):
    # aligned rows (lda % 4 == 0) but N % 4 != 0, and a row count that leaves
    # partial 4-row groups in the CTAs: the kernel for batch >= 3
    g = PCG32(40 + batch)
    M, N, lda = 1523, 1030, 1032
    A = g.uniform_f32((M, N))
    X = g.uniform_f32((batch, N))
    check(A, X, run_gemv(A, X, lda=lda))
    import torch
    dA = torch.empty(M * lda, device="cuda")
    dX = torch.empty((batch, N), device="cuda")
    dY = torch.empty((batch, M), device="cuda")
    plan = gtg.plan_gemv(M, N, dA.data_ptr(), lda, dX.data_ptr(), N, dY.data_ptr(), M, batch)
    assert plan["bm"] == 4 and plan["threads"] == 512


def test_vectors_that_do_not_fit_shared_memory():
    # batch 8 x 7000 entries and batch 1 x 60000 entries exceed one staging
    # chunk: the chunked loop with barriers on both sides is used
    g = PCG32(31)
    A = g.uniform_f32((300, 7000))
    X = g.uniform_f32((8, 7000))
    check(A, X, run_gemv(A, X))
    A = g.uniform_f32((97, 60000))
    x = g.uniform_f32((1, 60000))
    check(A, x, run_gemv(A, x))


@pytest.mark.parametrize("M,N,lda,batch", [(37, 3, 4, 1), (37, 3, 4, 2), (300, 1, 4, 1), (5, 2, 8, 2), (200, 7, 8, 1)])
def test_rows_shorter_than_one_16_byte_unit(M, N, lda, batch):
    # aligned, padded rows with fewer than four FP32 entries: the streaming
    # kernel's only work per row is its trailing-entry step
    g = PCG32(35 + N + lda)
    A = g.uniform_f32((M, N))
    X = g.uniform_f32((batch, N))
    check(A, X, run_gemv(A, X, lda=lda))


@pytest.mark.parametrize("M,N,lda,batch", [(37, 7, 8, 1), (100, 5, 16, 2), (64, 1, 8, 1)])
def test_bf16_rows_shorter_than_one_16_byte_unit(M, N, lda, batch):
    from seeded import bf16_bits_to_f32
    g = PCG32(36 + N + lda)
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((batch, N))
    Y = run_gemv(A, X, lda=lda, prec="bf16")
    check(bf16_bits_to_f32(A), X, Y)


@pytest.mark.parametrize("batch", [1, 2])
@pytest.mark.parametrize("M,N,lda,a_off", [(1000, 4095, 4095, 0), (333, 1001, 1003, 1), (301, 517, 517, 2),
                                           (64, 3, 3, 1), (77, 5, 7, 3), (40, 2, 2, 0), (2000, 8190, 8190, 0)])
def test_unaligned_rows_at_batch_1_and_2(batch, M, N, lda, a_off):
    # FP32 rows off 16 bytes: each row's first entries up to its 16-byte
    # boundary are single loads, the rest aligned 16-byte loads (rows shorter
    # than a unit are all head and tail)
    g = PCG32(37 + N + lda + a_off)
    A = g.uniform_f32((M, N))
    X = g.uniform_f32((batch, N))
    check(A, X, run_gemv(A, X, lda=lda, a_off=a_off))


@pytest.mark.parametrize("batch", [3, 5, 8])
@pytest.mark.parametrize("M,N,lda,a_off", [(1000, 4095, 4095, 0), (333, 1001, 1003, 1), (301, 517, 518, 2),
                                           (700, 2048, 2048, 1), (64, 3, 3, 1), (77, 5, 7, 3), (40, 2, 2, 0),
                                           (609, 9, 9, 2), (2000, 4094, 4094, 0), (151, 6000, 6001, 3)])
def test_unaligned_rows_at_batch_3_to_8(batch, M, N, lda, a_off):
    # FP32 rows off 16 bytes at batch >= 3: tasks of four rows four apart
    # (the same offset from a 16-byte boundary), each row's head by single
    # loads and the rest by aligned 16-byte loads; lda % 4 of 3, 1, 2 and 0
    # (with A off 16 bytes), fewer than 16 rows per CTA (row groups left
    # empty), rows shorter than one unit
    g = PCG32(38 + N + lda + a_off + batch)
    A = g.uniform_f32((M, N))
    X = g.uniform_f32((batch, N))
    if a_off == 0:
        plan = _plan(A, X, lda=lda)
        assert plan["bm"] == 4 and plan["bk"] == 2 and plan["threads"] == 512 and plan["cluster"] == 1, plan
    check(A, X, run_gemv(A, X, lda=lda, a_off=a_off))


@pytest.mark.parametrize("batch", [1, 2, 3, 8])
@pytest.mark.parametrize("M,N,lda,a_off", [(1000, 4095, 4095, 0), (333, 1001, 1003, 1), (301, 517, 518, 2),
                                           (700, 2048, 2052, 0), (64, 3, 3, 1), (77, 5, 7, 3), (609, 9, 9, 2),
                                           (151, 6000, 6001, 3), (500, 4100, 4100, 5)])
def test_bf16_unaligned_rows_take_peeled_row_blocks(batch, M, N, lda, a_off):
    # BF16 rows off 16 bytes: tasks of four rows four apart share the offset
    # from an 8-byte boundary (the lane load), their heads are single loads;
    # lda % 8 of 7, 3, 6, 4 (8-byte aligned rows, h = 0) and 5 with offsets
    from seeded import bf16_bits_to_f32
    g = PCG32(41 + N + lda + a_off + batch)
    A = g.normal_bf16((M, N))
    X = g.uniform_f32((batch, N))
    if a_off == 0:
        plan = _plan(A, X, prec="bf16", lda=lda)
        assert plan["kernel"] == "gemv" and plan["bm"] == 4 and plan["bk"] == 4 and plan["threads"] == 512, plan
    check(bf16_bits_to_f32(A), X, run_gemv(A, X, lda=lda, a_off=a_off, prec="bf16"))


def test_unaligned_rows_at_batch_8_are_deterministic():
    g = PCG32(39)
    A = g.uniform_f32((3001, 3001))
    X = g.uniform_f32((8, 3001))
    Y1, Y2 = run_gemv(A, X), run_gemv(A, X)
    assert np.array_equal(Y1, Y2)
    check(A, X, Y1)


def test_scalar_path_for_unaligned_rows():
    # batch 3 here takes the peeled row-block kernel; x too long for one
    # staging chunk at batch 8 takes the chunked scalar kernel
    g = PCG32(32)
    A = g.uniform_f32((257, 1001))
    X = g.uniform_f32((3, 1001))
    check(A, X, run_gemv(A, X, a_off=1))               # A not 16-byte aligned
    check(A, X, run_gemv(A, X, lda=1003))              # lda not a multiple of 4
    A = g.uniform_f32((150, 9001))
    X = g.uniform_f32((8, 9001))
    assert _plan(A, X)["bm"] == 2 and _plan(A, X)["stages"] > 1
    check(A, X, run_gemv(A, X))


def test_padded_batch_strides():
    g = PCG32(33)
    A = g.uniform_f32((400, 512))
    X = g.uniform_f32((4, 512))
    check(A, X, run_gemv(A, X, lda=520, ldx=515, ldy=405))


def test_closed_forms():
    M, N = 300, 4096
    ones = run_gemv(np.ones((M, N), dtype=np.float32), np.ones((2, N), dtype=np.float32))
    assert np.all(ones == N)
    # A with one non-zero per row picks out entries of x exactly
    rng = np.random.default_rng(34)
    cols = rng.integers(0, N, M)
    A = np.zeros((M, N), dtype=np.float32)
    A[np.arange(M), cols] = 1.0
    x = PCG32(34).uniform_f32((1, N))
    assert np.array_equal(run_gemv(A, x)[0], x[0, cols])


def test_N_zero_writes_zeros():
    y = run_gemv(np.zeros((17, 0), dtype=np.float32), np.zeros((3, 0), dtype=np.float32))
    assert np.all(y == 0)


def test_deterministic_and_plan():
    A, x, X = gemv_uniform_f32(2, 4096, 4096, batch=8)
    assert np.array_equal(run_gemv(A, X), run_gemv(A, X))
    import torch
    dA = torch.from_numpy(A).cuda()
    dX = torch.from_numpy(X).cuda()
    dY = torch.empty((8, 4096), device="cuda")
    plan = gtg.plan_gemv(4096, 4096, dA.data_ptr(), 4096, dX.data_ptr(), 4096, dY.data_ptr(), 4096, 8)
    assert plan["kernel"] == "gemv"
    assert plan["grid"] % torch.cuda.get_device_properties(0).multi_processor_count == 0


def test_tensor_helper_host_and_device():
    import torch
    A, x, X = gemv_uniform_f32(2, 512, 768, batch=3)
    y = gtg.matvec(torch.from_numpy(A).cuda(), torch.from_numpy(x).cuda()).cpu().numpy()
    check(A, x[None, :], y[None, :])
    Y = gtg.matvec(torch.from_numpy(A).pin_memory(), torch.from_numpy(X).pin_memory())
    assert not Y.is_cuda
    check(A, X, Y.numpy())


@pytest.mark.parametrize("batch,ldx,x_off", [(1, 1024, 1), (2, 1025, 0), (2, 1024, 3), (5, 1026, 0), (8, 1024, 2)])
def test_vectors_staged_by_threads_when_not_16_byte_aligned(batch, ldx, x_off):
    """x rows that are not 16-byte aligned cannot be staged by bulk copies;
    the kernels then stage them with plain loads (same results)."""
    g = PCG32(70 + batch + ldx + x_off)
    A = g.uniform_f32((700, 1024))
    X = g.uniform_f32((batch, 1024))
    check(A, X, run_gemv(A, X, ldx=ldx, x_off=x_off))


def _plan(A, X, prec="f32", lda=None):
    """The plan of the call run_gemv makes (fake, aligned, non-overlapping addresses)."""
    M, N = A.shape
    return gtg.plan_gemv(M, N, 1 << 32, lda or N, 2 << 32, N, 3 << 32, M, X.shape[0], precision=prec)


@pytest.mark.parametrize("M,N,batch,lda,cluster", [(8192, 8192, 8, None, 2), (3000, 20000, 3, None, 2),
                                                   (200, 60000, 1, None, 2), (300, 16384, 8, None, 4),
                                                   (10, 30000, 8, None, 8), (999, 20003, 3, 20004, 2),
                                                   (517, 13000, 6, None, 2)])
def test_column_blocks_over_a_cluster(M, N, batch, lda, cluster):
    """Vectors too large for one CTA's shared memory: the CTAs of a cluster
    each stage one block of columns and add their partial sums through
    distributed shared memory (fewer rows than clusters included; N = 20003
    has trailing entries and x rows that bulk copies cannot take)."""
    g = PCG32(90 + M + N + batch)
    A = g.uniform_f32((M, N))
    X = g.uniform_f32((batch, N))
    plan = _plan(A, X, lda=lda)
    assert plan["cluster"] == cluster, plan
    Y = run_gemv(A, X, lda=lda)
    if M > 2048:
        rows = np.unique(np.concatenate([np.arange(0, M, 37), [M - 1]]))
        for b in range(batch):
            ref, E = oracle.gemv(A[rows], X[b])
            ratio, bad = parity_ratio(Y[b][rows], ref, E, "f32", N)
            assert bad == 0, (b, ratio)
    else:
        check(A, X, Y)


def test_cluster_results_do_not_depend_on_the_run():
    g = PCG32(95)
    A = g.uniform_f32((1500, 24000))
    X = g.uniform_f32((4, 24000))
    assert _plan(A, X)["cluster"] == 2
    Y1, Y2 = run_gemv(A, X), run_gemv(A, X)
    assert np.array_equal(Y1, Y2)
