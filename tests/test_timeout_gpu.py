"""Failure detection without a GPU fault.

Every mbarrier wait in the tensor-core kernels is bounded in time. Here a
testing hook leaves out one K-slice load, so one wait can only run out (a
barrier that nothing completes). The kernel must then stop, drain the copies
and multiplies it has in flight, free its tensor memory and exit; the host
reads GTG_ERR_TIMEOUT from gtg_sync_status, and the same context keeps
working for the calls that follow.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
from seeded import PCG32, bf16_bits_to_f32
from tests._gpu import check_gemm, run_gemm

pytestmark = pytest.mark.gpu

SHORT_LIMIT_NS = 20_000_000   # 20 ms instead of the 2 s default


def _operands(prec, M, N, K, seed):
    g = PCG32(seed)
    if prec == "bf16":
        return g.normal_bf16((M, K)), g.normal_bf16((K, N))
    return g.uniform_f32((M, K)), g.uniform_f32((K, N))


def _launch(prec, A, B):
    import torch
    M, K = A.shape
    N = B.shape[1]
    if prec == "bf16":
        dA = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()
        dB = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.zeros((M, N), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    fn = {"bf16": gtg.gemm_bf16, "tf32": gtg.gemm_tf32}[prec]
    st = fn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, C.data_ptr(), N, s)
    return st, gtg.gtg_sync_status(s), gtg.plan_gemm(prec, M, N, K, dA.data_ptr(), K, dB.data_ptr(), N,
                                                      C.data_ptr(), N)


@pytest.mark.parametrize("prec,shape,kernel_bm", [
    ("bf16", (1024, 1024, 512), 128),    # single-CTA tensor-core kernel
    ("tf32", (1024, 1024, 512), 128),    # same kernel behind the B^T transpose
    ("bf16", (4096, 4096, 256), 256),    # CTA-pair kernel
    ("tf32", (4096, 4096, 256), 256),    # CTA-pair kernel, B^T staged K-major
])
def test_wait_that_runs_out_is_reported_and_context_survives(prec, shape, kernel_bm):
    M, N, K = shape
    A, B = _operands(prec, M, N, K, 90)
    gtg.gtg_set_wait_limit_ns(SHORT_LIMIT_NS)
    try:
        assert gtg.gtg_test_drop_load(2) == gtg.GTG_OK
        st, status, plan = _launch(prec, A, B)
    finally:
        gtg.gtg_test_drop_load(-1)
        gtg.gtg_set_wait_limit_ns(0)
    assert plan["kernel"] == "tcgen05" and plan["bm"] == kernel_bm
    assert st == gtg.GTG_OK                  # the launch itself succeeded
    assert status == gtg.GTG_ERR_TIMEOUT     # the kernel reported the wait it gave up
    # the status word is cleared by reading it, and the context still works
    assert gtg.gtg_sync_status(0) == gtg.GTG_OK
    C = run_gemm(prec, A[:256], B[:, :320])  # run_gemm also checks the status is OK
    check_gemm(prec, A[:256], B[:, :320], C)
    st, status, _ = _launch(prec, A, B)
    assert st == gtg.GTG_OK and status == gtg.GTG_OK


def test_wait_limit_default_restored():
    # a normal call after the hooks were used takes the normal path
    A, B = _operands("bf16", 512, 512, 512, 91)
    st, status, _ = _launch("bf16", A, B)
    assert st == gtg.GTG_OK and status == gtg.GTG_OK


@pytest.mark.parametrize("M,N,batch,kernel", [
    (4096, 4096, 1, "stream"),       # one row per warp, vectors in one bulk copy each
    (4096, 4096, 4, "split"),        # 4 rows x half the columns per task (batch 8 stages x by threads)
    (2048, 16384, 4, "cluster"),     # column blocks over a 2-CTA cluster (batch 8 stages x by threads)
])
def test_gemv_vector_wait_that_runs_out_is_reported(M, N, batch, kernel):
    """The GEMV kernels wait (bounded) for their bulk-copied vectors; a hook
    announces the copies but issues none, so that wait can only run out."""
    import torch
    from tests._gpu import run_gemv
    from tests.test_gemv_gpu import check
    g = PCG32(95 + batch)
    A = torch.from_numpy(g.uniform_f32((M, N))).cuda()
    X = torch.from_numpy(g.uniform_f32((batch, N))).cuda()
    Y = torch.zeros((batch, M), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    plan = gtg.plan_gemv(M, N, A.data_ptr(), N, X.data_ptr(), N, Y.data_ptr(), M, batch)
    assert (plan["bm"] == 1) == (kernel == "stream") and (plan["cluster"] > 1) == (kernel == "cluster"), plan
    gtg.gtg_set_wait_limit_ns(SHORT_LIMIT_NS)
    try:
        assert gtg.gtg_test_skip_vector_copy(True) == gtg.GTG_OK
        st = gtg.gemv_f32(M, N, A.data_ptr(), N, X.data_ptr(), N, Y.data_ptr(), M, batch, s)
        status = gtg.gtg_sync_status(s)
    finally:
        gtg.gtg_test_skip_vector_copy(False)
        gtg.gtg_set_wait_limit_ns(0)
    assert st == gtg.GTG_OK
    assert status == gtg.GTG_ERR_TIMEOUT
    # the context still works and the hook was used up
    Ah, Xh = g.uniform_f32((333, 1024)), g.uniform_f32((batch, 1024))
    check(Ah, Xh, run_gemv(Ah, Xh))


@pytest.mark.parametrize("M,N", [(8192, 4096), (4096, 4096)])
def test_tensor_core_gemv_wait_that_runs_out_is_reported(M, N):
    """The BF16 batch-8 GEMV on the tensor cores: one slice load of A left out,
    so the MMA thread's wait runs out; the kernel drains, frees its tensor
    memory and returns, and the following calls work."""
    import torch
    from tests._gpu import run_gemv
    from tests._util import parity_ratio
    import oracle
    g = PCG32(96)
    A = torch.from_numpy(g.normal_bf16((M, N)).view(np.int16)).cuda()
    X = torch.from_numpy(g.uniform_f32((8, N))).cuda()
    Y = torch.zeros((8, M), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    gtg.gtg_gemv_force_path("tensor_cores")
    gtg.gtg_set_wait_limit_ns(SHORT_LIMIT_NS)
    try:
        plan = gtg.plan_gemv(M, N, A.data_ptr(), N, X.data_ptr(), N, Y.data_ptr(), M, 8, precision="bf16")
        assert plan["kernel"] == "tcgen05", plan
        assert gtg.gtg_test_drop_load(1) == gtg.GTG_OK
        st = gtg.gemv_bf16(M, N, A.data_ptr(), N, X.data_ptr(), N, Y.data_ptr(), M, 8, s)
        status = gtg.gtg_sync_status(s)
    finally:
        gtg.gtg_test_drop_load(-1)
        gtg.gtg_set_wait_limit_ns(0)
    try:
        assert st == gtg.GTG_OK
        assert status == gtg.GTG_ERR_TIMEOUT
        # the context still works
        Ah, Xh = g.normal_bf16((300, 1024)), g.uniform_f32((8, 1024))
        Yh = run_gemv(Ah, Xh, prec="bf16")
        ref, E = oracle.gemv(bf16_bits_to_f32(Ah), Xh[3])
        assert parity_ratio(Yh[3], ref, E, "f32", 1024)[1] == 0
    finally:
        gtg.gtg_gemv_force_path("auto")
