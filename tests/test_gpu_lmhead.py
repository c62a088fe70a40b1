"""GPU parity of an lm_head-scale decode GEMV (M = 1, K = 5120, N = 248,320):
an extreme N, so every CTA owns ~1600 rows and the last one a ragged tail.

The weights are drawn on the device (torch's seeded generator; 1.3 GB of
ternary values) and only the sampled rows travel to the host, where the
oracle packs them itself: no oracle input comes from the library."""
import numpy as np
import pytest
import torch

import oracle
from gemm_pq2_ternary_gb300 import inputs

pytestmark = pytest.mark.gpu

K, N = 5120, 248320


def _sampled_rows(n_rows, count, seed):
    rng = np.random.default_rng(seed)
    tail = np.arange(n_rows - 40, n_rows)          # the last CTA's ragged tail
    head = np.arange(0, 8)
    return np.unique(np.concatenate([rng.integers(0, n_rows, count), head, tail]))


@pytest.mark.parametrize("flags", [0, 1], ids=["default", "static_weights"])
def test_lmhead_gemv_parity(flags):
    from gemm_pq2_ternary_gb300 import binding as pq2
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(2024)
    tern = inputs.draw_ternary_torch(N, K, "uniform", gen, dev)
    ws = inputs.draw_ws_torch(N, K, gen, dev)
    codes, ws_d = pq2.pack(tern, ws)
    x = inputs.generate_x(1, K, "outliers", seed=77)
    torch.cuda.synchronize()
    y = torch.full((1, N), float("nan"), device=dev)
    pq2.pq2_matmul_ex(torch.from_numpy(x).to(dev), codes, ws_d, y, flags, None)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    assert not torch.isnan(y).any()

    ns = _sampled_rows(N, 600, 5)
    idx = torch.from_numpy(ns).to(dev)
    tern_s = tern.index_select(0, idx).cpu().numpy()
    ws_s = ws.index_select(0, idx).cpu().numpy()
    oqp, oS, _ = oracle.quantize_act(x)
    ref, A = oracle.matmul_entries(oqp, oS, oracle.pack(tern_s), ws_s,
                                   np.zeros(len(ns), dtype=np.int64),
                                   np.arange(len(ns), dtype=np.int64))
    got = y.cpu().numpy()[0, ns].astype(np.float64)
    tol = oracle.fp32_tolerance(ref, A, K // 128)
    err = np.abs(got - ref)
    assert np.all(err <= tol), f"max err {err.max()}"
