"""GPU parity of the small bf16 split-K projection (pq2_gemm_bf16_splitk):
the in_proj_ba shape (N = 96, K = 5120) at every token count up to 17,
ragged N and K, a K long enough that threads loop, K = 0, exact integer
cases compared bit for bit, and the fixed-order reduction's determinism.
Inputs are drawn on the host; nothing the oracle reads comes from the
library."""
import numpy as np
import pytest
import torch

import oracle
from gemm_pq2_ternary_gb300 import inputs

pytestmark = pytest.mark.gpu


def _dev(bits):
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def _run(xb, wb, flags=0):
    from gemm_pq2_ternary_gb300 import binding as pq2
    M, N = xb.shape[0], wb.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    pq2.pq2_gemm_bf16_splitk(_dev(xb), _dev(wb), y, flags)
    torch.cuda.synchronize()
    return y.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K", [(1, 96, 5120), (2, 96, 5120), (3, 96, 5120),
                                   (4, 96, 5120), (5, 96, 5120), (8, 96, 5120),
                                   (13, 96, 5120), (16, 96, 5120), (17, 96, 5120),
                                   (40, 100, 1032), (3, 7, 8), (6, 33, 16384),
                                   (2, 5, 24)])
def test_bf16_splitk_parity(M, N, K):
    xb, wb = inputs.generate_bf16(M, N, K, seed=1000 + M + N + K)
    got = oracle.bf16_to_f64(_run(xb, wb))
    ref, A = oracle.gemm_bf16(xb, wb)
    err = np.abs(got - ref)
    tol = oracle.bf16_gemm_tolerance(ref, A, K)
    assert np.all(err <= tol), f"max err {err.max()} (tol there {tol.flat[err.argmax()]})"


@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_bf16_splitk_integer_inputs_are_bit_exact(M):
    # every partial sum is an integer below 2^24, exact in fp32 in any
    # order; the one rounding to bf16 is then the oracle's own
    xb, wb = inputs.generate_bf16(M, 96, 5120, seed=77 + M, x="integer", w="integer")
    ref, _ = oracle.gemm_bf16(xb, wb)
    assert np.array_equal(_run(xb, wb), oracle.f64_to_bf16(ref))


def test_bf16_splitk_zero_k_writes_zeros():
    from gemm_pq2_ternary_gb300 import binding as pq2
    x = torch.empty((3, 0), dtype=torch.bfloat16, device="cuda")
    w = torch.empty((10, 0), dtype=torch.bfloat16, device="cuda")
    y = torch.full((3, 10), float("nan"), dtype=torch.bfloat16, device="cuda")
    pq2.pq2_gemm_bf16_splitk(x, w, y)
    torch.cuda.synchronize()
    assert torch.equal(y.float(), torch.zeros((3, 10), device="cuda"))


def test_bf16_splitk_is_deterministic_and_static_flag_agrees():
    from gemm_pq2_ternary_gb300 import binding as pq2
    xb, wb = inputs.generate_bf16(4, 96, 5120, seed=5)
    first = _run(xb, wb)
    for _ in range(20):
        assert np.array_equal(_run(xb, wb), first)
    assert np.array_equal(_run(xb, wb, pq2.PQ2_WEIGHTS_STATIC), first)
