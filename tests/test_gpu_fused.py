"""GPU parity of the fused M = 1 path (pq2_matmul with M = 1: the GEMV
kernel quantises the fp16 activations itself) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from gemm_pq2_ternary_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("prob", [inputs.PR1, inputs.DECODE, inputs.mlp_gate_up(1),
                                  inputs.mlp_down(1),
                                  inputs.Problem("fused_g13", 1, 128 * 13, 301, "p343",
                                                 "outliers", 61)],
                         ids=lambda p: p.name)
def test_fused_gemv_parity(prob):
    from gemm_pq2_ternary_gb300 import binding as pq2
    tern, ws, x = inputs.generate(prob)
    if prob.K >= 256:
        x[0, 128:256] = 0  # an all-zero group
    codes, ws_d = pq2.pack(torch.from_numpy(tern).cuda(), torch.from_numpy(ws).cuda())
    y = torch.full((1, prob.N), float("nan"), device="cuda")
    assert pq2.pq2_workspace_bytes(pq2.PQ2_OP_MATMUL, 1, prob.N, prob.K) == 0
    pq2.pq2_matmul(torch.from_numpy(x).cuda(), codes, ws_d, y, None)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    oqp, oS, oT = oracle.quantize_act(x)
    ocodes = oracle.pack(tern)
    if prob.N * prob.K <= 64 * 1024 * 1024:
        ref, A = oracle.matmul(oqp, oS, ocodes, ws)
        got = y.cpu().numpy().astype(np.float64)
    else:
        ns = np.unique(np.concatenate([np.random.default_rng(0).integers(0, prob.N, 600),
                                       [0, prob.N - 1]]))
        ms = np.zeros_like(ns)
        ref, A = oracle.matmul_entries(oqp, oS, ocodes, ws, ms, ns)
        ref, A = ref[None], A[None]
        got = y.cpu().numpy()[:, ns].astype(np.float64)
    tol = oracle.fp32_tolerance(ref, A, prob.K // 128)
    err = np.abs(got - ref)
    assert np.all(err <= tol), f"max err {err.max()}"
