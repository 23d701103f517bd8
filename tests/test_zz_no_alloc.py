"""gemm_tf32_noalloc: the TF32 GEMM for callers that cannot allocate device memory.

Some callers cannot allocate GPU memory while they run: a serving process
whose allocator already holds nearly all of the device's memory, a set-up
without stream-ordered memory pools, or a latency-critical loop that allows
no allocation calls. For them gemm_tf32_noalloc stages B^T in a fixed 16 MiB
array inside the library instead of a pool buffer. These tests call it
through the C ABI and compare it with the FP64 oracle and with gemm_tf32 on
the same inputs, twice in a row (the array keeps the previous call's
contents, which must not leak into the next result); they check that a call
takes no workspace and leaves the device's free memory unchanged, and they
cover its SIMT side (layouts the tensor-memory accelerator cannot read, and
the forced SIMT path). This file is collected last on purpose.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import gemm_uniform_f32
from tests._util import bound_f32, bound_tf32

LIMIT = 16 << 20   # bytes of the fixed array


def _run(fn, A, B, lda=None, a_off=0):
    """C = A @ B through fn (a gemm_tf32-like entry point) with A stored at
    leading dimension lda, a_off elements into its buffer; returns C and the
    plan of that call."""
    import torch
    M, K = A.shape
    N = B.shape[1]
    lda = lda or K
    hA = np.full(a_off + M * lda, np.nan, dtype=np.float32)
    hA[a_off:].reshape(M, lda)[:, :K] = A
    dA = torch.from_numpy(hA).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.full((M, N), float("nan"), device="cuda")
    pA = dA.data_ptr() + 4 * a_off
    s = int(torch.cuda.current_stream().cuda_stream)
    if fn is gtg.gemm_tf32_noalloc:
        plan = gtg.plan_gemm_tf32_noalloc(M, N, K, pA, lda, dB.data_ptr(), N, dC.data_ptr(), N)
    else:
        plan = gtg.plan_gemm("tf32", M, N, K, pA, lda, dB.data_ptr(), N, dC.data_ptr(), N)
    st = fn(M, N, K, pA, lda, dB.data_ptr(), N, dC.data_ptr(), N, s)
    assert st == gtg.GTG_OK, gtg.status_string(st)
    assert gtg.gtg_sync_status(s) == gtg.GTG_OK
    return dC.cpu().numpy(), plan


def _check(got, A, B, bound):
    ref, E = oracle.gemm(A, B)
    assert np.all(np.isfinite(got))
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= bound(E, A.shape[1])), float((err / bound(E, A.shape[1])).max())


@pytest.mark.gpu
def test_noalloc_matches_the_oracle_and_gemm_tf32_on_two_calls_in_a_row():
    gtg.gtg_force_simt(False)
    # first call fills the whole array (N * K * 4 = 16 MiB), the second uses
    # less of it with different values and a ragged shape
    cases = [gemm_uniform_f32(41, 2048, 2048, 2048), gemm_uniform_f32(4, 1000, 700, 1500)]
    for A, B in cases:
        M, K = A.shape
        N = B.shape[1]
        assert N * ((K + 3) // 4 * 4) * 4 <= LIMIT
        got, plan = _run(gtg.gemm_tf32_noalloc, A, B)
        # the tensor-core path that stages B^T in the fixed array: one CTA per
        # tile (no CTA pair), K never split
        assert plan["kernel"] == "tcgen05" and plan["cluster"] == 1 and plan["splits"] == 1, plan
        assert plan["grid"] <= ((M + 127) // 128) * ((N + plan["bn"] - 1) // plan["bn"])
        _check(got, A, B, bound_tf32)
        want, _ = _run(gtg.gemm_tf32, A, B)
        assert np.all(np.abs(got.astype(np.float64) - want) <= bound_tf32(oracle.gemm(A, B)[1]))


@pytest.mark.gpu
def test_noalloc_takes_no_workspace_and_no_device_memory():
    import torch
    A, B = gemm_uniform_f32(43, 1024, 2048, 2048)
    M, K = A.shape
    N = B.shape[1]
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.empty((M, N), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    args = (M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N, s)
    # warm the library's per-device state (device facts, the array's address)
    assert gtg.gemm_tf32_noalloc(*args) == gtg.GTG_OK
    torch.cuda.synchronize()
    ws0 = gtg.gtg_test_workspace_allocations()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        assert gtg.gemm_tf32_noalloc(*args) == gtg.GTG_OK
    torch.cuda.synchronize()
    assert gtg.gtg_test_workspace_allocations() == ws0
    assert torch.cuda.mem_get_info()[0] == free0
    # the counter does see the pool: gemm_tf32 takes its B^T from it
    assert gtg.gemm_tf32(*args) == gtg.GTG_OK
    torch.cuda.synchronize()
    assert gtg.gtg_test_workspace_allocations() > ws0
    assert gtg.gtg_sync_status(s) == gtg.GTG_OK


@pytest.mark.gpu
@pytest.mark.parametrize("shape,lda,a_off,force_simt", [
    ((300, 257, 515), 517, 0, False),     # lda % 4 != 0: A's rows are off 16 bytes
    ((129, 200, 64), 64, 1, False),       # A's base off 16 bytes
    ((1000, 700, 1500), None, 0, True),   # the SIMT kernel forced
])
def test_noalloc_simt_side_against_the_oracle(shape, lda, a_off, force_simt):
    """Layouts the tensor-memory accelerator cannot read would need a copied
    operand (pool memory) on the tensor-core path, so gemm_tf32_noalloc runs
    them on the SIMT kernel in one K range: exact FP32 arithmetic, within the
    FP32 bound (tighter than the TF32 one)."""
    M, N, K = shape
    A, B = gemm_uniform_f32(44 + M, M, N, K)
    gtg.gtg_force_simt(force_simt)
    try:
        got, plan = _run(gtg.gemm_tf32_noalloc, A, B, lda=lda, a_off=a_off)
        got2, _ = _run(gtg.gemm_tf32_noalloc, A, B, lda=lda, a_off=a_off)
    finally:
        gtg.gtg_force_simt(False)
    assert plan["kernel"] == "simt" and plan["splits"] == 1, plan
    _check(got, A, B, bound_f32)
    assert np.array_equal(got, got2)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # fake, aligned, disjoint addresses: the size check happens before any
    # device work, so this runs without a GPU
    A, B, C = 1 << 32, 3 << 32, 5 << 32
    K = 2048
    assert gtg.gemm_tf32_noalloc(8, 2049, K, A, K, B, 2049, C, 2049) == gtg.GTG_ERR_SCRATCH_LIMIT
    assert gtg.gemm_tf32_noalloc(8, 2048, 2049, A, 2049, B, 2048, C, 2048) == gtg.GTG_ERR_SCRATCH_LIMIT
    with pytest.raises(gtg.GtgError) as e:
        gtg.plan_gemm_tf32_noalloc(8, 2049, K, A, K, B, 2049, C, 2049)
    assert e.value.status == gtg.GTG_ERR_SCRATCH_LIMIT
    assert "16 MiB" in gtg.status_string(gtg.GTG_ERR_SCRATCH_LIMIT)
    # ordinary argument errors are reported as for gemm_tf32
    assert gtg.gemm_tf32_noalloc(-1, 4, 4, A, 4, B, 4, C, 4) == gtg.GTG_ERR_INVALID_VALUE
