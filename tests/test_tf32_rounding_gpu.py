"""TF32 products at their worst case for the 4 * 2^-11 * E bound.

"Matrix Operations" ("Performance Considerations") notes that tensor cores
and reduced-precision formats buy speed with a little accuracy; the bound
for the TF32 path is 4 * 2^-11 * sum_k |a_ik * b_kj|. An FP32 value reduced
to TF32 keeps 10 explicit mantissa bits. Truncation loses up to 2^-10 of the
value, so with both operands truncated a product can be off by 2^-9 relative,
which is the whole bound; rounding to nearest loses at most 2^-11 per operand,
half the bound per product.

The operands below are all positive (so E is the exact result and the error
over E is the relative error) with mantissa patterns that make the reduction
as large as it can be:

  * 1 + 2^-10 - 2^-23 (the 13 dropped bits all ones): truncation loses
    almost 2^-10, rounding to nearest loses 2^-23;
  * 1 + 2^-11 (exactly half a TF32 unit): either way the loss is 2^-11.

On this GPU the TF32 MMA truncates (measured: the first pattern gave 0.998 of
the bound), so the library rounds both operands to nearest before the MMA.
The test checks every element against the FP64 oracle at the bound, and that
the first pattern's error is far below the truncation level.
"""

import numpy as np
import pytest

import gemv_tiled_gemm_gb300 as gtg
import oracle
from seeded import PCG32
from tests._gpu import sample_rows
from tests._util import bound_tf32

pytestmark = pytest.mark.gpu

PATTERNS = {
    "dropped_bits_all_ones": np.float32(1 + 2.0 ** -10 - 2.0 ** -23),
    "half_unit_tie": np.float32(1 + 2.0 ** -11),
}


def _operands(M, N, K, c, seed):
    g = PCG32(seed)
    ea = (g.next_u32(M * K) % 3).astype(np.int64).reshape(M, K) - 1
    eb = (g.next_u32(K * N) % 3).astype(np.int64).reshape(K, N) - 1
    A = (c * np.ldexp(np.float32(1), ea)).astype(np.float32)
    B = (c * np.ldexp(np.float32(1), eb)).astype(np.float32)
    return A, B


def _run(fn, A, B, plan_fn):
    import torch
    M, K = A.shape
    N = B.shape[1]
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.full((M, N), float("nan"), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    plan = plan_fn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N)
    st = fn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N, s)
    assert st == gtg.GTG_OK, gtg.status_string(st)
    assert gtg.gtg_sync_status(s) == gtg.GTG_OK
    return dC.cpu().numpy(), plan


def _worst_ratio(A, B, C):
    rows = sample_rows(A.shape[0], 128, seed=A.shape[1])
    ref, E = oracle.gemm(A[rows], B)
    err = np.abs(C[rows].astype(np.float64) - ref)
    assert np.all(np.isfinite(C[rows]))
    return float((err / bound_tf32(E)).max())


@pytest.mark.parametrize("pattern", sorted(PATTERNS))
@pytest.mark.parametrize("M,N,K,kernel", [
    (256, 256, 64, "single"),      # single-CTA kernel, one K range
    (256, 256, 1024, "single"),    # single-CTA kernel, K split across CTAs
    (256, 256, 8192, "single"),
    (2048, 2048, 64, "pair"),      # CTA-pair kernel (256 x 256 tiles)
    (2048, 2048, 1024, "pair"),
    (2048, 2048, 8192, "pair"),
])
def test_tf32_worst_case_operands(pattern, M, N, K, kernel):
    A, B = _operands(M, N, K, PATTERNS[pattern], 60 + K)
    C, plan = _run(gtg.gemm_tf32, A, B, lambda *a: gtg.plan_gemm("tf32", *a))
    assert plan["kernel"] == "tcgen05" and plan["cluster"] == (2 if kernel == "pair" else 1), plan
    ratio = _worst_ratio(A, B, C)
    assert ratio <= 1.0
    if pattern == "dropped_bits_all_ones":
        # rounded to nearest: 2^-23 per operand; truncated it would be 0.998
        assert ratio < 0.05, ratio
    else:
        # half a TF32 unit per operand: 0.5 of the bound, plus accumulation
        assert ratio < 0.6, ratio


@pytest.mark.parametrize("pattern", sorted(PATTERNS))
def test_tf32_worst_case_operands_without_allocation(pattern):
    # gemm_tf32_noalloc: B^T staged in the fixed array, the single-CTA kernel
    A, B = _operands(512, 1024, 2048, PATTERNS[pattern], 77)
    C, plan = _run(gtg.gemm_tf32_noalloc, A, B, gtg.plan_gemm_tf32_noalloc)
    assert plan["kernel"] == "tcgen05", plan
    ratio = _worst_ratio(A, B, C)
    assert ratio < (0.05 if pattern == "dropped_bits_all_ones" else 0.6), ratio


def test_tf32_strided_batch_worst_case():
    # the batched launch (pair kernel over batch items, B^T of every item
    # transposed and rounded in one launch)
    import torch
    batch, M, N, K = 3, 512, 512, 1024
    c = PATTERNS["dropped_bits_all_ones"]
    items = [_operands(M, N, K, c, 90 + b) for b in range(batch)]
    A = np.stack([a for a, _ in items])
    B = np.stack([b for _, b in items])
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.full((batch, M, N), float("nan"), device="cuda")
    s = int(torch.cuda.current_stream().cuda_stream)
    st = gtg.gemm_strided_batched("tf32", M, N, K, dA.data_ptr(), K, M * K, dB.data_ptr(), N, K * N,
                                  dC.data_ptr(), N, M * N, batch, None, s)
    assert st == gtg.GTG_OK and gtg.gtg_sync_status(s) == gtg.GTG_OK
    C = dC.cpu().numpy()
    for b in range(batch):
        assert _worst_ratio(A[b], B[b], C[b]) < 0.05
