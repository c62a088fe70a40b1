"""Child process of test_gpu_prefill_variants: runs pq2_gemm_prefill on the
problems named on the command line with PQ2_PREFILL_WIDE taken from the
environment (read once per process by the library) and checks y against the
oracle.  Prints "ok <name>" per problem; exits non-zero on a mismatch."""
import sys

import numpy as np
import torch

import oracle
from gemm_pq2_ternary_gb300 import binding as pq2
from gemm_pq2_ternary_gb300 import inputs

PROBLEMS = {
    "ragged": inputs.Problem("wide_ragged", 37, 384, 200, "uniform", "outliers", 60),
    "m17": inputs.Problem("wide_m17", 17, 640, 129, "p343", "outliers", 61),
    "m300": inputs.Problem("wide_m300", 300, 1024, 520, "uniform", "normal", 62),
    "m129": inputs.Problem("wide_m129", 129, 1280, 777, "p343", "outliers", 63),
    "n512": inputs.Problem("wide_n512", 256, 2048, 512, "uniform", "outliers", 64),
    "m4096": inputs.prefill(4096),
}


def check(name):
    prob = PROBLEMS[name]
    tern, ws, x = inputs.generate(prob)
    dev = torch.device("cuda")
    codes, ws_d = pq2.pack(torch.from_numpy(tern).to(dev), torch.from_numpy(ws).to(dev))
    qp, S, T = pq2.quantize(torch.from_numpy(x).to(dev))
    y = torch.full((prob.M, prob.N), float("nan"), device=dev)
    pq2.pq2_gemm_prefill(qp, S, T, codes, ws_d, y,
                         pq2.alloc_workspace(pq2.PQ2_OP_PREFILL, prob.M, prob.N, prob.K))
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK, name
    oqp, oS, _ = oracle.quantize_act(x)
    ocodes = oracle.pack(tern)
    yh = y.cpu().numpy().astype(np.float64)
    if prob.M * prob.N * prob.K <= 64 * 1024 * 1024:
        ref, A = oracle.matmul(oqp, oS, ocodes, ws)
        got = yh
    else:
        rng = np.random.default_rng(7)
        ms = np.concatenate([rng.integers(0, prob.M, 2048), [0, prob.M - 1, 0, prob.M - 1]])
        ns = np.concatenate([rng.integers(0, prob.N, 2048), [0, prob.N - 1, prob.N - 1, 0]])
        ref, A = oracle.matmul_entries(oqp, oS, ocodes, ws, ms, ns)
        got = yh[ms, ns]
    err = np.abs(got - ref)
    tol = oracle.fp32_tolerance(ref, A, prob.K // 128)
    if not np.all(err <= tol):
        print(f"FAIL {name}: max err {err.max():.3e}", flush=True)
        sys.exit(1)
    print(f"ok {name}", flush=True)


if __name__ == "__main__":
    for n in sys.argv[1:]:
        check(n)
