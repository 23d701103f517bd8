"""gemm_tf32_noalloc: the TF32 GEMM for callers that cannot allocate device memory.

Some callers cannot allocate GPU memory while they run: a serving process
whose allocator already holds nearly all of the device's memory, a set-up
without stream-ordered memory pools, or a latency-critical loop that allows
no allocation calls. For them gemm_tf32_noalloc stages B^T in a fixed 16 MiB
array inside the library instead of a pool buffer. These tests call it
through the C ABI and compare it with gemm_tf32 on the same inputs, twice in
a row (the array keeps the previous call's contents, which must not leak
into the next result). This file is collected last on purpose.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import gemm_uniform_f32
from tests._util import bound_tf32

LIMIT = 16 << 20   # bytes of the fixed array


def _run(fn, A, B):
    import torch
    M, K = A.shape
    N = B.shape[1]
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.full((M, N), float("nan"), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    st = fn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N, s)
    assert st == gtg.GTG_OK, gtg.status_string(st)
    assert gtg.gtg_sync_status(s) == gtg.GTG_OK
    plan = gtg.plan_gemm("tf32", M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N)
    return dC.cpu().numpy(), plan


@pytest.mark.gpu
def test_noalloc_matches_gemm_tf32_on_two_calls_in_a_row():
    gtg.gtg_force_simt(False)
    # first call fills the whole array (N * K * 4 = 16 MiB), the second uses
    # less of it with different values and a ragged shape
    cases = [gemm_uniform_f32(41, 2048, 2048, 2048), gemm_uniform_f32(4, 1000, 700, 1500)]
    for A, B in cases:
        M, K = A.shape
        N = B.shape[1]
        assert N * ((K + 3) // 4 * 4) * 4 <= LIMIT
        got, plan = _run(gtg.gemm_tf32_noalloc, A, B)
        assert plan["kernel"] == "tcgen05"       # the path that uses the scratch
        want, _ = _run(gtg.gemm_tf32, A, B)
        _, E = oracle.gemm(A, B)
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got.astype(np.float64) - want) <= bound_tf32(E))
        # same kernels, same summation order: identical bits in practice
        assert np.array_equal(got, want)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # fake, aligned, disjoint addresses: the size check happens before any
    # device work, so this runs without a GPU
    A, B, C = 1 << 32, 3 << 32, 5 << 32
    K = 2048
    assert gtg.gemm_tf32_noalloc(8, 2049, K, A, K, B, 2049, C, 2049) == gtg.GTG_ERR_SCRATCH_LIMIT
    assert gtg.gemm_tf32_noalloc(8, 2048, 2049, A, 2049, B, 2048, C, 2048) == gtg.GTG_ERR_SCRATCH_LIMIT
    assert "16 MiB" in gtg.status_string(gtg.GTG_ERR_SCRATCH_LIMIT)
    # ordinary argument errors are reported as for gemm_tf32
    assert gtg.gemm_tf32_noalloc(-1, 4, 4, A, 4, B, 4, C, 4) == gtg.GTG_ERR_INVALID_VALUE
