"""pq2_gemm_small_noalloc: the small-batch matmul for callers that cannot
allocate device memory (no allocator of their own, or allocation not allowed
where they run), with its scratch in a fixed array inside the library.

It runs the same kernel, grid and fixed-order reduction as pq2_gemm_small
with a caller-owned workspace, so its y must be the same bits.  Each case
calls it twice through the C ABI: the second call reuses the array exactly
as the first one left it.  The cases cover the tensor-core kernel with row
tiles shared by several CTAs (partial sums and counters in the array), a
ragged last tile, and a token count that takes the DP4A kernel (which needs
no scratch).  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gemm_pq2_ternary_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = [
    inputs.small_batch(16, 6144, 5120),
    inputs.small_batch(8, 5120, 17408),
    # 300 rows: two full 128-row tiles and a ragged one; 12 groups in quads
    # of 4 give 9 items, so each tile is shared by three CTAs
    inputs.Problem("noalloc_ragged_m5", 5, 1536, 300, "p343", "outliers", 72),
    inputs.Problem("noalloc_dp4a_m3", 3, 384, 77, "p343", "outliers", 71),
]


def _noalloc(pq2, qp, S, T, codes, ws_d, y, M, N, K):
    return pq2._lib.pq2_gemm_small_noalloc(
        ctypes.c_void_p(qp.data_ptr()), ctypes.c_void_p(S.data_ptr()),
        ctypes.c_void_p(T.data_ptr()), ctypes.c_void_p(codes.data_ptr()),
        ctypes.c_void_p(ws_d.data_ptr()), ctypes.c_void_p(y.data_ptr()), M, N, K,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("prob", CASES, ids=lambda p: p.name)
def test_noalloc_matches_workspace_path(prob):
    from gemm_pq2_ternary_gb300 import binding as pq2
    tern, ws, x = inputs.generate(prob)
    codes, ws_d = pq2.pack(torch.from_numpy(tern).cuda(), torch.from_numpy(ws).cuda())
    qp, S, T = pq2.quantize(torch.from_numpy(x).cuda())
    M, N, K = prob.M, prob.N, prob.K

    ref = torch.full((M, N), float("nan"), device="cuda")
    pq2.pq2_gemm_small(qp, S, T, codes, ws_d, ref,
                       pq2.alloc_workspace(pq2.PQ2_OP_SMALL, M, N, K))
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    if M * N * K <= 16 * 1024 * 1024:
        # the workspace path itself against the oracle, on the small cases
        oqp, oS, _ = oracle.quantize_act(x)
        want, A = oracle.matmul(oqp, oS, oracle.pack(tern), ws)
        err = np.abs(ref.cpu().numpy().astype(np.float64) - want)
        assert np.all(err <= oracle.fp32_tolerance(want, A, K // 128))

    for call in range(2):
        y = torch.full((M, N), float("nan"), device="cuda")
        st = _noalloc(pq2, qp, S, T, codes, ws_d, y, M, N, K)
        assert st == pq2.PQ2_OK, pq2.pq2_status_string(st)
        torch.cuda.synchronize()
        assert pq2.pq2_last_device_error() == pq2.PQ2_OK
        assert torch.equal(y, ref), f"call {call}: differs from the workspace path"
