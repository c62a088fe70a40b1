"""The bounds-checked build (libpq2_debug.so, PQ2_DEBUG=1): every kernel store
to y, to the integer-dot output and to the split-K scratch checks its index
against its buffer first; a store outside is skipped and reported as
PQ2_ERR_BOUNDS.  It stands in for a memory checker, which cannot be run on
these GPUs.

1. Every kernel, forced on the ragged shapes of the guard-band tests, reports
   no bounds error in the checked build and gives the same bits as the normal
   build (y, and the integer dots of the three matmul entry points).
2. With pq2_debug_shrink_bounds(1) the checks treat the last element of every
   buffer as outside: every kernel must then report PQ2_ERR_BOUNDS (each
   writes y's last element), skip the store, and still write nothing around
   y.  No memory outside the buffers is touched in either test.
"""
import numpy as np
import pytest
import torch

from gemm_pq2_ternary_gb300 import inputs
from test_gpu_guard import CASES, PAD, SENTINEL, _guarded

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def libs():
    from gemm_pq2_ternary_gb300 import _build, binding
    release = binding._lib
    debug = binding.load_library(_build.build(debug=True))
    yield binding, release, debug
    binding._lib = release
    for lib in (release, debug):
        for op in (binding.PQ2_OP_GEMV, binding.PQ2_OP_SMALL, binding.PQ2_OP_PREFILL):
            lib.pq2_debug_force_kernel(op, binding.PQ2_VARIANT_DEFAULT)
    debug.pq2_debug_shrink_bounds(0)


def _run(pq2, op, variant, prob, data):
    """y of one call (inside a guarded buffer) with the library pq2._lib."""
    from gemm_pq2_ternary_gb300.binding import alloc_workspace
    codes, ws_d, xd = data
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
    torch.cuda.synchronize()
    return buf, y


def _data(pq2, prob):
    tern, ws, x = inputs.generate(prob)
    codes, ws_d = pq2.pack(torch.from_numpy(tern).to(DEV), torch.from_numpy(ws).to(DEV))
    return codes, ws_d, torch.from_numpy(x).to(DEV)


def test_build_flags(libs):
    pq2, release, debug = libs
    assert release.pq2_bounds_checked() == 0
    assert debug.pq2_bounds_checked() == 1


@pytest.mark.parametrize("op,variant,prob", CASES, ids=lambda v: getattr(v, "name", str(v)))
def test_checked_build_matches_and_reports_nothing(libs, op, variant, prob):
    pq2, release, debug = libs
    pq2._lib = release
    data = _data(pq2, prob)
    _, y_rel = _run(pq2, op, variant, prob, data)
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    pq2._lib = debug
    buf, y_dbg = _run(pq2, op, variant, prob, data)
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    pq2._lib = release
    assert torch.equal(y_rel, y_dbg)
    assert torch.all(buf[:PAD] == SENTINEL) and torch.all(buf[PAD + prob.M * prob.N:] == SENTINEL)


@pytest.mark.parametrize("op,prob", [
    ("gemv", inputs.Problem("bd_dots_gemv", 1, 640, 97, "uniform", "normal", 160)),
    ("small", inputs.Problem("bd_dots_small", 5, 640, 300, "p343", "outliers", 161)),
    ("small", inputs.Problem("bd_dots_dp4a", 3, 384, 77, "p343", "outliers", 162)),
    ("prefill", inputs.Problem("bd_dots_tile", 23, 640, 261, "p343", "outliers", 163)),
    ("prefill", inputs.Problem("bd_dots_pf", 37, 384, 200, "uniform", "normal", 164)),
], ids=lambda v: getattr(v, "name", str(v)))
def test_checked_build_dots(libs, op, prob):
    pq2, release, debug = libs
    from gemm_pq2_ternary_gb300.binding import alloc_workspace
    opc = {"gemv": pq2.PQ2_OP_GEMV, "small": pq2.PQ2_OP_SMALL, "prefill": pq2.PQ2_OP_PREFILL}[op]
    pq2._lib = release
    codes, _, xd = _data(pq2, prob)
    qp, S, T = pq2.quantize(xd)
    out = []
    for lib in (release, debug):
        pq2._lib = lib
        dots = torch.empty((prob.M, prob.N, prob.K // 128), dtype=torch.int32, device=DEV)
        pq2.pq2_group_dots(opc, qp, T, codes, dots, alloc_workspace(opc, prob.M, prob.N, prob.K))
        torch.cuda.synchronize()
        assert pq2.pq2_last_device_error() == pq2.PQ2_OK
        out.append(dots)
    pq2._lib = release
    assert torch.equal(out[0], out[1])


@pytest.mark.parametrize("op,variant,prob", CASES, ids=lambda v: getattr(v, "name", str(v)))
def test_checked_build_reports_a_store_outside(libs, op, variant, prob):
    pq2, release, debug = libs
    pq2._lib = debug
    data = _data(pq2, prob)
    try:
        pq2.pq2_debug_shrink_bounds(1)
        buf, y = _run(pq2, op, variant, prob, data)
        assert pq2.pq2_last_device_error() == pq2.PQ2_ERR_BOUNDS
    finally:
        pq2.pq2_debug_shrink_bounds(0)
        pq2._lib = release
    assert torch.all(buf[:PAD] == SENTINEL) and torch.all(buf[PAD + prob.M * prob.N:] == SENTINEL)
    # the skipped store is y's last element (a 4-wide store: its last four)
    assert buf[PAD + prob.M * prob.N - 1].item() == SENTINEL
