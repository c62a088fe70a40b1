"""pq2_gemm_small_noalloc: the small-batch matmul for callers that cannot
allocate device memory, with its split-K scratch in a fixed array inside the
library.  Called through the C ABI, its output must match pq2_gemm_small (the
same kernel with a caller-owned workspace) within the tolerance the other
parity tests use, on two calls in a row (the second call reuses the array the
first one left behind).  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gemm_pq2_ternary_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("prob", [inputs.small_batch(16, 6144, 5120),
                                  inputs.small_batch(8, 5120, 17408),
                                  inputs.Problem("noalloc_ragged", 3, 384, 77, "p343",
                                                 "outliers", 71)],
                         ids=lambda p: p.name)
def test_noalloc_matches_workspace_path(prob):
    from gemm_pq2_ternary_gb300 import binding as pq2
    tern, ws, x = inputs.generate(prob)
    codes, ws_d = pq2.pack(torch.from_numpy(tern).cuda(), torch.from_numpy(ws).cuda())
    qp, S, T = pq2.quantize(torch.from_numpy(x).cuda())
    M, N, K = prob.M, prob.N, prob.K

    ref = torch.empty((M, N), device="cuda")
    pq2.pq2_gemm_small(qp, S, T, codes, ws_d, ref,
                       pq2.alloc_workspace(pq2.PQ2_OP_SMALL, M, N, K))
    torch.cuda.synchronize()
    ref_h = ref.cpu().numpy().astype(np.float64)
    # magnitude term of the parity tolerance, from the oracle
    oqp, oS, _ = oracle.quantize_act(x)
    _, A = oracle.matmul(oqp, oS, oracle.pack(tern), ws)
    tol = oracle.fp32_tolerance(ref_h, A, K // 128)

    for call in range(2):
        y = torch.full((M, N), float("nan"), device="cuda")
        st = pq2._lib.pq2_gemm_small_noalloc(
            ctypes.c_void_p(qp.data_ptr()), ctypes.c_void_p(S.data_ptr()),
            ctypes.c_void_p(T.data_ptr()), ctypes.c_void_p(codes.data_ptr()),
            ctypes.c_void_p(ws_d.data_ptr()), ctypes.c_void_p(y.data_ptr()), M, N, K,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == pq2.PQ2_OK, pq2.pq2_status_string(st)
        torch.cuda.synchronize()
        assert pq2.pq2_last_device_error() == pq2.PQ2_OK
        got = y.cpu().numpy().astype(np.float64)
        err = np.abs(got - ref_h)
        assert np.all(err <= tol), f"call {call}: max err {np.nanmax(err)}"
