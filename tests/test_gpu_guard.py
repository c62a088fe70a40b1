"""Guard bands around y for every kernel: the output is placed inside a larger
buffer filled with a sentinel, and after the call every element before and
after y still holds it.  Shapes are ragged (N not a multiple of 4 or of the
tile width, G not a multiple of 4, tokens that leave part of a token tile
empty), so the scalar tail stores and the last tiles' guards are exercised;
each kernel is forced through pq2_debug_force_kernel.  y itself is checked
against the oracle within the fp32 tolerance (bf16: the bf16 bound)."""
import numpy as np
import pytest
import torch

import oracle
from gemm_pq2_ternary_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
PAD = 64  # sentinel elements on each side (256 bytes: y stays 16-byte aligned)
SENTINEL = 123.0


@pytest.fixture(scope="module")
def pq2():
    from gemm_pq2_ternary_gb300 import binding
    yield binding
    for op in (binding.PQ2_OP_GEMV, binding.PQ2_OP_SMALL, binding.PQ2_OP_PREFILL):
        binding.pq2_debug_force_kernel(op, binding.PQ2_VARIANT_DEFAULT)


def _guarded(M, N, dtype=torch.float32):
    buf = torch.full((2 * PAD + M * N,), SENTINEL, dtype=dtype, device=DEV)
    return buf, buf[PAD:PAD + M * N].view(M, N)


def _check_guard(buf, M, N, what):
    torch.cuda.synchronize()
    head = buf[:PAD].float().cpu().numpy()
    tail = buf[PAD + M * N:].float().cpu().numpy()
    assert np.all(head == SENTINEL) and np.all(tail == SENTINEL), f"{what}: wrote outside y"


def _check_y(y, tern, ws, x, what):
    oqp, oS, _ = oracle.quantize_act(x)
    ref, A = oracle.matmul(oqp, oS, oracle.pack(tern), ws)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= oracle.fp32_tolerance(ref, A, x.shape[1] // 128)), f"{what}: max err {err.max()}"


# (op, variant name, problem): every kernel of the three matmul entry points
CASES = [
    ("gemv", "GEMV_DIRECT", inputs.Problem("gd_direct", 1, 640, 97, "uniform", "normal", 140)),
    ("gemv", "GEMV_RING", inputs.Problem("gd_ring", 1, 640, 97, "uniform", "normal", 141)),
    # the staged kernel takes slices of at least 16 KB a CTA: G = 13, ragged N
    ("gemv_x", "GEMV_STAGED", inputs.Problem("gd_staged", 1, 1664, 6083, "p343", "outliers", 142)),
    ("small", "SMALL_DP4A", inputs.Problem("gd_dp4a", 3, 384, 77, "p343", "outliers", 143)),
    ("small", "SMALL_TC", inputs.Problem("gd_small", 5, 640, 300, "p343", "outliers", 144)),
    ("small", "SMALL_TILE", inputs.Problem("gd_tile16", 7, 1664, 301, "uniform", "outliers", 145)),
    ("small", "SMALL_WTILE", inputs.Problem("gd_wtile16", 9, 1664, 301, "uniform", "outliers", 146)),
    ("prefill", "PREFILL_TILE", inputs.Problem("gd_tile32", 23, 640, 261, "p343", "outliers", 147)),
    ("prefill", "PREFILL_WTILE", inputs.Problem("gd_wtile64", 41, 640, 261, "p343", "outliers", 148)),
    ("prefill", "PREFILL_128", inputs.Problem("gd_pf128", 37, 384, 200, "uniform", "normal", 149)),
    ("prefill", "PREFILL_WIDE", inputs.Problem("gd_pfwide", 37, 384, 200, "uniform", "normal", 150)),
    ("matmul", "DEFAULT", inputs.Problem("gd_mm_small", 6, 640, 299, "p343", "outliers", 151)),
    ("matmul", "DEFAULT", inputs.Problem("gd_mm_tile", 19, 640, 299, "p343", "outliers", 152)),
    ("matmul", "DEFAULT", inputs.Problem("gd_mm_wtile", 45, 640, 299, "p343", "outliers", 153)),
]


@pytest.mark.parametrize("op,variant,prob", CASES, ids=lambda v: getattr(v, "name", str(v)))
def test_guard_bands(pq2, op, variant, prob):
    from gemm_pq2_ternary_gb300.binding import alloc_workspace
    tern, ws, x = inputs.generate(prob)
    codes, ws_d = pq2.pack(torch.from_numpy(tern).to(DEV), torch.from_numpy(ws).to(DEV))
    xd = torch.from_numpy(x).to(DEV)
    M, N, K = prob.M, prob.N, prob.K
    buf, y = _guarded(M, N)
    var = getattr(pq2, "PQ2_VARIANT_" + variant)
    if op in ("gemv", "gemv_x"):
        with pq2.forced_kernel(pq2.PQ2_OP_GEMV, var):
            if op == "gemv":
                qp, S, T = pq2.quantize(xd)
                pq2.pq2_gemv(qp, S, T, codes, ws_d, y)
            else:
                pq2.pq2_matmul_ex(xd, codes, ws_d, y, pq2.PQ2_WEIGHTS_STATIC, None)
    elif op in ("small", "prefill"):
        opc = pq2.PQ2_OP_SMALL if op == "small" else pq2.PQ2_OP_PREFILL
        fn = pq2.pq2_gemm_small if op == "small" else pq2.pq2_gemm_prefill
        qp, S, T = pq2.quantize(xd)
        with pq2.forced_kernel(opc, var):
            fn(qp, S, T, codes, ws_d, y, alloc_workspace(opc, M, N, K))
    else:
        pq2.pq2_matmul(xd, codes, ws_d, y, alloc_workspace(pq2.PQ2_OP_MATMUL, M, N, K))
    _check_guard(buf, M, N, prob.name)
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    _check_y(y, tern, ws, x, prob.name)


def test_guard_bands_bf16(pq2):
    xb, wb = inputs.generate_bf16(5, 97, 640, seed=12)
    xd = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
    wd = torch.from_numpy(wb.view(np.int16)).to(DEV).view(torch.bfloat16)
    buf, y = _guarded(5, 97, torch.bfloat16)
    pq2.pq2_gemm_bf16_splitk(xd, wd, y)
    _check_guard(buf, 5, 97, "bf16 projection")
    got = oracle.bf16_to_f64(y.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
    ref, A = oracle.gemm_bf16(xb, wb)
    assert np.all(np.abs(got - ref) <= oracle.bf16_gemm_tolerance(ref, A, 640))
