"""Child process of test_gpu_small_variants: runs pq2_gemm_small and the
small-batch integer-dot view on the problems named on the command line, with
PQ2_SMALL_DP4A_MAX_M taken from the environment (read once per process by
the library), and checks them against the oracle.  Prints "ok <name>" per
problem; exits non-zero on a mismatch."""
import sys

import numpy as np
import torch

import oracle
from gemm_pq2_ternary_gb300 import binding as pq2
from gemm_pq2_ternary_gb300 import inputs

PROBLEMS = {
    "m2": inputs.Problem("tc_m2", 2, 384, 77, "p343", "outliers", 70),
    "m5": inputs.Problem("tc_m5", 5, 1280, 300, "uniform", "outliers", 71),
    "m8": inputs.Problem("tc_m8", 8, 6144, 640, "p343", "outliers", 72),
}


def check(name):
    prob = PROBLEMS[name]
    tern, ws, x = inputs.generate(prob)
    dev = torch.device("cuda")
    codes, ws_d = pq2.pack(torch.from_numpy(tern).to(dev), torch.from_numpy(ws).to(dev))
    qp, S, T = pq2.quantize(torch.from_numpy(x).to(dev))
    wsp = pq2.alloc_workspace(pq2.PQ2_OP_SMALL, prob.M, prob.N, prob.K)
    y = torch.full((prob.M, prob.N), float("nan"), device=dev)
    pq2.pq2_gemm_small(qp, S, T, codes, ws_d, y, wsp)
    dots = torch.empty((prob.M, prob.N, prob.K // 128), dtype=torch.int32, device=dev)
    pq2.pq2_group_dots(pq2.PQ2_OP_SMALL, qp, T, codes, dots, wsp)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK, name
    oqp, oS, _ = oracle.quantize_act(x)
    ocodes = oracle.pack(tern)
    if not np.array_equal(dots.cpu().numpy(), oracle.group_dots(oqp, ocodes)):
        print(f"FAIL {name}: group dots differ", flush=True)
        sys.exit(1)
    ref, A = oracle.matmul(oqp, oS, ocodes, ws)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    if not np.all(err <= oracle.fp32_tolerance(ref, A, prob.K // 128)):
        print(f"FAIL {name}: max err {err.max():.3e}", flush=True)
        sys.exit(1)
    print(f"ok {name}", flush=True)


if __name__ == "__main__":
    for n in sys.argv[1:]:
        check(n)
