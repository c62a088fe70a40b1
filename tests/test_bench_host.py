"""CPU checks of bench.py's host side: workload sizing, launch counts and the
oracle baseline sample (the CPU arm the GPU bench line and --impl reference
both report), for one workload of each kind."""
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _args(workload, m=1, shape="5120,17408"):
    return types.SimpleNamespace(workload=workload, m=m, shape=shape)


@pytest.mark.parametrize("workload,m,units,launches", [
    ("decode", 1, 6144 * 5120 // 4 + 2 * 5120 * 48 + 2 * 6144 + 4 * 5120, 1),
    ("small", 16, None, 3),
    ("small", 4, None, 2),
    ("mlp_swiglu", 1, None, 1 + 2),
    ("in_proj_ba", 4, 2 * (96 * 5120 + 4 * 5120 + 4 * 96), 1),
    ("prefill", 128, 2.0 * 128 * 17408 * 5120, 3),
])
def test_workload_sizing(workload, m, units, launches):
    name, layer, kind = bench.workload_spec(_args(workload, m))
    assert kind == ("TOPS" if workload == "prefill" else "GB/s")
    got = bench.per_layer_units(layer, kind, name)
    if units is not None:
        assert got == units
    assert bench.layer_launches(layer, name) == launches


@pytest.mark.parametrize("workload,m", [("decode", 1), ("small", 4), ("mlp_swiglu", 1),
                                        ("in_proj_ba", 4)])
def test_oracle_sample_runs(workload, m):
    name, layer, kind = bench.workload_spec(_args(workload, m))
    value, desc, threads, dt = bench.oracle_sample(layer, kind, 0.05)
    assert value > 0 and threads >= 1 and dt > 0 and "output rows" in desc


def test_oracle_single_core_sample_and_thread_independence():
    import numpy as np

    import oracle
    from gemm_pq2_ternary_gb300 import inputs
    name, layer, kind = bench.workload_spec(_args("decode", 1))
    single = bench.oracle_single_core(layer, kind, 0.05)
    assert single["cores"] == 1 and single["value"] > 0
    assert bench.oracle_single_core(*bench.workload_spec(_args("in_proj_ba", 4))[1:], 0.05) is None
    # the oracle's parallel loops split output rows only: the same bits on one thread
    tern, ws, x = inputs.generate(inputs.Problem("thr", 3, 512, 40, "p343", "outliers", 9))
    qp, S, _ = oracle.quantize_act(x)
    codes = oracle.pack(tern)
    before = oracle.threads()
    try:
        oracle.set_threads(1)
        y1, _ = oracle.matmul(qp, S, codes, ws)
    finally:
        oracle.set_threads(before)
    yn, _ = oracle.matmul(qp, S, codes, ws)
    assert np.array_equal(y1, yn)
