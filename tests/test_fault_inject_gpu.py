"""Host-side fault injection in the dispatcher (no GPU fault is involved).

gtg_test_inject_launch_failure(n) makes the n-th dispatched call fail with
GTG_ERR_LAUNCH before it launches anything. A failed call must leave its
output untouched and the library usable; inside gemm_host (which dispatches
one product per region of C while its copies are in flight) a failure must
end the call cleanly, with every stream drained and every buffer returned.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import gemm_uniform_f32
from tests._util import parity_ratio

pytestmark = pytest.mark.gpu


def test_injected_failure_launches_nothing_and_the_next_call_works():
    import torch
    A, B = gemm_uniform_f32(81, 300, 200, 100)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.full((300, 200), float("nan"), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    args = (300, 200, 100, dA.data_ptr(), 100, dB.data_ptr(), 200, dC.data_ptr(), 200, s)
    assert gtg.gtg_test_inject_launch_failure(1) == gtg.GTG_OK
    assert gtg.gemm_tf32(*args) == gtg.GTG_ERR_LAUNCH
    assert gtg.last_cuda_error() == "injected launch failure"
    assert gtg.gtg_sync_status(s) == gtg.GTG_OK
    assert torch.isnan(dC).all()            # nothing ran
    assert gtg.gemm_tf32(*args) == gtg.GTG_OK
    assert gtg.gtg_sync_status(s) == gtg.GTG_OK
    ref, E = oracle.gemm(A, B)
    assert parity_ratio(dC.cpu().numpy(), ref, E, "tf32", 100)[1] == 0


def test_injected_failure_inside_gemm_host():
    import torch
    M, N, K = 2048, 2048, 512
    A, B = gemm_uniform_f32(82, M, N, K)
    hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
    hC = torch.full((M, N), float("nan")).pin_memory()
    call = lambda: gtg.gemm_host("f32", M, N, K, hA.data_ptr(), K, hB.data_ptr(), N, hC.data_ptr(), N)
    # the call itself is dispatch 1; its first region's product is dispatch 2
    for n in (1, 2, 3):
        assert gtg.gtg_test_inject_launch_failure(n) == gtg.GTG_OK
        assert call() == gtg.GTG_ERR_LAUNCH
    assert gtg.gtg_test_inject_launch_failure(0) == gtg.GTG_OK
    # the library and its streams still work: a full product afterwards
    assert call() == gtg.GTG_OK
    rows = np.arange(0, M, 97)
    ref, E = oracle.gemm(A[rows], B)
    assert parity_ratio(hC.numpy()[rows], ref, E, "f32", K)[1] == 0
