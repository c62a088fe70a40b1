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
    ("small", 16, None, 2),  # quantise into the token tiles, then small_kernel
    ("small", 4, None, 2),   # quantise, then the DP4A kernel
    ("mid", 32, None, 2),    # quantise into the token tiles, then tile_kernel
    ("mid", 64, None, 3),    # quantise, token preparation, prefill_kernel (9 items a CTA)
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


def test_every_suite_configuration_has_a_workload():
    names = set()
    for (w, m, shape) in bench.SUITE:
        name, layer, kind = bench.workload_spec(_args(w, m, shape or "5120,17408"))
        assert bench.per_layer_units(layer, kind, name) > 0
        assert bench.layer_launches(layer, name) >= 1
        names.add(name)
    assert len(names) == len(bench.SUITE)
    # the five configurations the benchmark is quoted on are all there
    for want in ["pr1_gemv_m1_k1024_n256", "small_m16_k5120_n17408", "small_m2_k6144_n5120",
                 "mlp_pair_m1", "mlp_pair_m16", "prefill_m128_k5120_n17408",
                 "prefill_m4096_k5120_n17408"]:
        assert want in names


def test_accuracy_measures():
    import numpy as np

    import oracle
    from gemm_pq2_ternary_gb300 import inputs
    tern, ws, x = inputs.generate(inputs.Problem("acc", 4, 512, 64, "p343", "outliers", 3))
    qp, S, _ = oracle.quantize_act(x)
    ref, A = oracle.matmul(qp, S, oracle.pack(tern), ws)
    sample = dict(bf16=False, K=512, tern=tern, ws=ws, x=x, y=ref.astype(np.float32))
    got = bench.accuracy(sample)
    assert got["within_tolerance"] and got["rel_rms"] < 1e-7 and got["outputs"] == 4 * 64
    # a 1% error on one output shows in both measures and fails the bound
    bad = ref.astype(np.float32).copy()
    i = np.unravel_index(np.argmax(np.abs(ref)), ref.shape)
    bad[i] *= 1.01
    got = bench.accuracy(dict(sample, y=bad))
    assert not got["within_tolerance"] and got["max_rel_err"] > 0.009 and got["rel_rms"] > 1e-4
