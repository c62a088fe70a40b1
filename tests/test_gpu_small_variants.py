"""GPU checks of the two small-batch kernels: the tensor-core kernel forced
at token counts the DP4A kernel would otherwise take (child process: the
library reads PQ2_SMALL_DP4A_MAX_M once per process), and the DP4A kernel's
per-token rows against the M = 1 GEMV on the same token, bit for bit (both
sum the same group terms in the same order), at 2, 3 and 4 tokens."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from gemm_pq2_ternary_gb300 import inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_tensor_core_kernel_at_few_tokens():
    names = ["m2", "m5", "m8"]  # (m5, m8: the default routing already takes this kernel)
    env = dict(os.environ, PQ2_SMALL_DP4A_MAX_M="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "small_variant_child.py"),
                        *names], env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    for n in names:
        assert f"ok {n}" in r.stdout, r.stdout


@pytest.mark.parametrize("M,K,N", [(2, 6144, 5120), (3, 5120, 17408), (4, 1280, 999)])
def test_dp4a_rows_equal_the_single_token_gemv(M, K, N):
    from gemm_pq2_ternary_gb300 import binding as pq2
    tern, ws, x = inputs.generate(inputs.Problem("bitid", M, K, N, "p343", "outliers", 80 + M))
    dev = torch.device("cuda")
    codes, ws_d = pq2.pack(torch.from_numpy(tern).to(dev), torch.from_numpy(ws).to(dev))
    qp, S, T = pq2.quantize(torch.from_numpy(x).to(dev))
    y = torch.empty((M, N), device=dev)
    pq2.pq2_gemm_small(qp, S, T, codes, ws_d, y,
                       pq2.alloc_workspace(pq2.PQ2_OP_SMALL, M, N, K))
    for m in range(M):
        y1 = torch.empty((1, N), device=dev)
        pq2.pq2_gemv(qp[m:m + 1].clone(), S[m:m + 1].clone(), T[m:m + 1].clone(),
                     codes, ws_d, y1)
        torch.cuda.synchronize()
        assert torch.equal(y[m], y1[0]), f"token {m}"
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
