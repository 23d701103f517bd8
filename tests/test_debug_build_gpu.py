"""The GTG_DEBUG build: kernels check every address they compute.

libgtg_debug.so (built by gemv_tiled_gemm_gb300._build.build(debug=True)) is
loaded instead of libgtg.so when GTG_DEBUG=1 is in the environment. Its
index-heavy kernels (the GEMV kernels, the peeled unaligned-row paths, the
im2col gathers, the operand copies and the TF32 transpose) check each global
address against its operand's extent and each shared-memory write against
the dynamic allocation; a failed check latches GTG_ERR_BOUNDS and skips the
access. The whole GPU suite is run once under this build (every parity test
asserts gtg_sync_status() == GTG_OK after its calls, so a check that fired
fails it). These tests show that the checks are live: with the checked
extent of the matrix shortened by one element, the last load of a call fails
its check, without any access outside the real matrix.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32
from tests._util import parity_ratio

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gtg.DEBUG, reason="needs the GTG_DEBUG build (GTG_DEBUG=1)")]


def test_the_debug_build_is_loaded():
    assert gtg.gtg_debug_build() == 1


def _gemv(A, X, lda):
    import torch
    M, N = A.shape
    batch = X.shape[0]
    host = np.zeros(M * lda + 8, dtype=np.float32)
    host[:M * lda].reshape(M, lda)[:, :N] = A
    dA = torch.from_numpy(host).cuda()
    dX = torch.from_numpy(np.ascontiguousarray(X)).cuda()
    dY = torch.zeros((batch, M), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    st = gtg.gemv_f32(M, N, dA.data_ptr(), lda, dX.data_ptr(), N, dY.data_ptr(), M, batch, s)
    assert st == gtg.GTG_OK
    return gtg.gtg_sync_status(s), dY.cpu().numpy()


@pytest.mark.parametrize("M,N,lda,batch", [
    (700, 1024, 1024, 1),    # ring kernel (one or two vectors)
    (700, 1024, 1024, 8),    # row blocks, vectors staged interleaved by the threads
    (700, 1024, 1024, 4),    # row blocks, vectors by bulk copies
    (700, 1023, 1025, 1),    # peeled rows, one per warp
    (700, 1023, 1025, 5),    # peeled row blocks
])
def test_bounds_checks_fire_and_skip_the_access(M, N, lda, batch):
    g = PCG32(500 + batch)
    A = g.uniform_f32((M, N))
    X = g.uniform_f32((batch, N))
    assert gtg.gtg_test_debug_shrink_extent(1) == gtg.GTG_OK
    try:
        status, _ = _gemv(A, X, lda)
    finally:
        assert gtg.gtg_test_debug_shrink_extent(0) == gtg.GTG_OK
    assert status == gtg.GTG_ERR_BOUNDS
    # the real extent again: no check fires and the result is right
    status, Y = _gemv(A, X, lda)
    assert status == gtg.GTG_OK
    for b in range(batch):
        ref, E = oracle.gemv(A, X[b])
        assert parity_ratio(Y[b], ref, E, "f32", N)[1] == 0
