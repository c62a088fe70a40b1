"""GPU parity of the SwiGLU + quantise step (pq2_quantize_swiglu: bit-exact
qp, S, T against the oracle) and of the down projection from a gate/up
output (pq2_mlp_down_swiglu: y within the fp32 tolerance).  The gate/up
values are drawn on the host; nothing the oracle reads comes from the
library."""
import numpy as np
import pytest
import torch

import oracle
from gemm_pq2_ternary_gb300 import inputs

pytestmark = pytest.mark.gpu


def _gu(M, I, seed):
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal((M, I)) * 3.0).astype(np.float32)
    u = (rng.standard_normal((M, I)) * 2.0).astype(np.float32)
    # edge values: zeros, large gates of both signs (exp clamped), a product
    # beyond the fp16 range (saturates), exp's reduction boundaries
    g[0, :8] = [0.0, 95.0, -95.0, 87.5, -88.5, 20.0, 0.3465736, -0.3465736]
    u[0, :8] = [1.0, 1.0, 1.0, 1.0, 1.0, 5000.0, 1.0, 1.0]
    if I >= 256:
        g[0, 128:256] = 0.0                     # a group of zeros: h = 0, s = t = 0
    return np.concatenate([g, u], axis=1)


@pytest.mark.parametrize("M,I", [(1, 128), (1, 17408), (3, 1280), (16, 512)])
def test_quantize_swiglu_is_bit_exact(M, I):
    from gemm_pq2_ternary_gb300 import binding as pq2
    gu = _gu(M, I, 100 + M)
    qp, S, T = pq2.alloc_act(M, I)
    pq2.pq2_quantize_swiglu(torch.from_numpy(gu).cuda(), qp, S, T)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    oqp, oS, oT = oracle.quantize_act(oracle.swiglu(gu))
    assert np.array_equal(qp.cpu().numpy(), oqp)
    assert np.array_equal(S.cpu().numpy(), oS)
    assert np.array_equal(T.cpu().numpy(), oT)


@pytest.mark.parametrize("M,I,N", [(1, 1280, 777), (4, 1280, 300), (16, 512, 1000),
                                   (40, 384, 257)])
def test_mlp_down_swiglu_parity(M, I, N):
    from gemm_pq2_ternary_gb300 import binding as pq2
    gu = _gu(M, I, 200 + M)
    tern, ws, _ = inputs.generate(inputs.Problem("down", M, I, N, "uniform", "normal", 300 + M))
    codes, ws_d = pq2.pack(torch.from_numpy(tern).cuda(), torch.from_numpy(ws).cuda())
    y = torch.full((M, N), float("nan"), device="cuda")
    wsp = pq2.alloc_workspace(pq2.PQ2_OP_SWIGLU_DOWN, M, N, I)
    assert wsp is not None
    pq2.pq2_mlp_down_swiglu(torch.from_numpy(gu).cuda(), codes, ws_d, y, wsp)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    oqp, oS, _ = oracle.quantize_act(oracle.swiglu(gu))
    ref, A = oracle.matmul(oqp, oS, oracle.pack(tern), ws)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= oracle.fp32_tolerance(ref, A, I // 128)), f"max err {err.max()}"
