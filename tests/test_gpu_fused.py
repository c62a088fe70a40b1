"""GPU parity of the fused M = 1 path (pq2_matmul with M = 1: the GEMV
kernel quantises the fp16 activations itself) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from gemm_pq2_ternary_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("prob", [inputs.PR1, inputs.DECODE, inputs.mlp_gate_up(1),
                                  inputs.mlp_down(1),
                                  inputs.Problem("fused_g13", 1, 128 * 13, 301, "p343",
                                                 "outliers", 61)],
                         ids=lambda p: p.name)
def test_fused_gemv_parity(prob):
    from gemm_pq2_ternary_gb300 import binding as pq2
    tern, ws, x = inputs.generate(prob)
    if prob.K >= 256:
        x[0, 128:256] = 0  # an all-zero group
    codes, ws_d = pq2.pack(torch.from_numpy(tern).cuda(), torch.from_numpy(ws).cuda())
    y = torch.full((1, prob.N), float("nan"), device="cuda")
    assert pq2.pq2_workspace_bytes(pq2.PQ2_OP_MATMUL, 1, prob.N, prob.K) == 0
    pq2.pq2_matmul(torch.from_numpy(x).cuda(), codes, ws_d, y, None)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    oqp, oS, oT = oracle.quantize_act(x)
    ocodes = oracle.pack(tern)
    if prob.N * prob.K <= 64 * 1024 * 1024:
        ref, A = oracle.matmul(oqp, oS, ocodes, ws)
        got = y.cpu().numpy().astype(np.float64)
    else:
        ns = np.unique(np.concatenate([np.random.default_rng(0).integers(0, prob.N, 600),
                                       [0, prob.N - 1]]))
        ms = np.zeros_like(ns)
        ref, A = oracle.matmul_entries(oqp, oS, ocodes, ws, ms, ns)
        ref, A = ref[None], A[None]
        got = y.cpu().numpy()[:, ns].astype(np.float64)
    tol = oracle.fp32_tolerance(ref, A, prob.K // 128)
    err = np.abs(got - ref)
    assert np.all(err <= tol), f"max err {err.max()}"


# Shapes for the static-weights path (staged where a CTA's weight slice is at
# least 16 KB; PR1 and static_n1 stay on the direct variant): G < 48 groups
# (several teams per group),
# G not a multiple of 8 (scales staged by plain loads), G > 48 (two passes,
# the second with only some teams busy), ragged N (short last CTA).
STATIC_PROBS = [inputs.PR1, inputs.DECODE,
                inputs.Problem("static_g8", 1, 1024, 10000, "p343", "outliers", 60),
                inputs.Problem("static_g13", 1, 128 * 13, 6000, "p343", "outliers", 61),
                inputs.Problem("static_g50", 1, 128 * 50, 2000, "uniform", "outliers", 62),
                inputs.Problem("static_g96", 1, 128 * 96, 1000, "p343", "normal", 63),
                inputs.Problem("static_n1", 1, 2048, 1, "uniform", "normal", 64)]


def _oracle_check(prob, tern, ws, x, y):
    oqp, oS, oT = oracle.quantize_act(x)
    ref, A = oracle.matmul(oqp, oS, oracle.pack(tern), ws)
    tol = oracle.fp32_tolerance(ref, A, prob.K // 128)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= tol), f"max err {err.max()}"


@pytest.mark.parametrize("prob", STATIC_PROBS, ids=lambda p: p.name)
def test_static_weights_match_default_path(prob):
    """PQ2_WEIGHTS_STATIC (weights staged before the dependency wait) gives
    bit-identical y to pq2_matmul, and y matches the oracle."""
    from gemm_pq2_ternary_gb300 import binding as pq2
    tern, ws, x = inputs.generate(prob)
    codes, ws_d = pq2.pack(torch.from_numpy(tern).cuda(), torch.from_numpy(ws).cuda())
    xd = torch.from_numpy(x).cuda()
    torch.cuda.synchronize()  # the weights are complete before the static calls
    y0 = torch.full((1, prob.N), float("nan"), device="cuda")
    y1 = torch.full((1, prob.N), float("nan"), device="cuda")
    pq2.pq2_matmul(xd, codes, ws_d, y0, None)
    pq2.pq2_matmul_ex(xd, codes, ws_d, y1, pq2.PQ2_WEIGHTS_STATIC, None)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    assert torch.equal(y0, y1)
    if prob.N * prob.K <= 16 * 1024 * 1024:
        _oracle_check(prob, tern, ws, x, y1)


def test_static_weights_back_to_back():
    """Several static-weight calls queued without synchronisation, eagerly and
    replayed from a CUDA graph: each call's weights are read while the
    previous call may still run, and its x only after that call is done (each
    x is written by the kernel just before it)."""
    from gemm_pq2_ternary_gb300 import binding as pq2
    n_calls = 6
    probs = [inputs.Problem(f"chain{i}", 1, 6144 if i % 2 == 0 else 4096,
                            5120 if i % 2 == 0 else 4096, "p343", "outliers", 70 + i)
             for i in range(n_calls)]
    data = [inputs.generate(p) for p in probs]
    dev = [pq2.pack(torch.from_numpy(t).cuda(), torch.from_numpy(w).cuda()) for t, w, _ in data]
    xs = [torch.from_numpy(x).cuda() for _, _, x in data]
    xs_live = [torch.empty_like(x) for x in xs]
    torch.cuda.synchronize()
    want = []
    for (codes, ws_d), x, p in zip(dev, xs, probs):
        y = torch.empty((1, p.N), device="cuda")
        pq2.pq2_matmul(x, codes, ws_d, y, None)
        want.append(y)
    torch.cuda.synchronize()

    def chain(outs):
        for i, ((codes, ws_d), p) in enumerate(zip(dev, probs)):
            xs_live[i].copy_(xs[i])  # x written by the kernel right before the call
            pq2.pq2_matmul_ex(xs_live[i], codes, ws_d, outs[i], pq2.PQ2_WEIGHTS_STATIC, None)

    outs = [torch.full((1, p.N), float("nan"), device="cuda") for p in probs]
    chain(outs)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    for a, b in zip(outs, want):
        assert torch.equal(a, b)

    gouts = [torch.full((1, p.N), float("nan"), device="cuda") for p in probs]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            chain(gouts)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        for o in gouts:
            o.fill_(float("nan"))
        g.replay()
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    for a, b in zip(gouts, want):
        assert torch.equal(a, b)


@pytest.mark.parametrize("prob", [inputs.mlp_gate_up(1), inputs.mlp_down(1)], ids=lambda p: p.name)
def test_static_weights_fall_back_where_slices_are_too_large(prob):
    """Where a CTA's weight slice does not fit the staged kernel, the flag
    changes nothing: y is bit-identical to pq2_matmul."""
    from gemm_pq2_ternary_gb300 import binding as pq2
    tern, ws, x = inputs.generate(prob)
    codes, ws_d = pq2.pack(torch.from_numpy(tern).cuda(), torch.from_numpy(ws).cuda())
    xd = torch.from_numpy(x).cuda()
    torch.cuda.synchronize()
    y0 = torch.full((1, prob.N), float("nan"), device="cuda")
    y1 = torch.full((1, prob.N), float("nan"), device="cuda")
    pq2.pq2_matmul(xd, codes, ws_d, y0, None)
    pq2.pq2_matmul_ex(xd, codes, ws_d, y1, pq2.PQ2_WEIGHTS_STATIC, None)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    assert torch.equal(y0, y1)


FEW_TOKEN_STATIC = ([inputs.Problem(f"static_m{M}_k{K}_n{N}", M, K, N, "p343", "outliers", 90 + M)
                     for M in (2, 3, 4, 5, 8, 16) for (K, N) in inputs.SMALL_SHAPES] +
                    # fewer items per CTA than the producer's stages, ragged N and G
                    [inputs.Problem("static_m8_k384_n300", 8, 384, 300, "p343", "outliers", 89),
                     inputs.Problem("static_m16_k1664_n200", 16, 1664, 200, "uniform", "outliers", 88)])


@pytest.mark.parametrize("prob", FEW_TOKEN_STATIC, ids=lambda p: p.name)
def test_static_weights_few_tokens_match_default_path(prob):
    """2 to 16 tokens: with PQ2_WEIGHTS_STATIC the DP4A kernel (2-4 tokens)
    requests its weights before the dependency wait, and the tensor-core
    kernel (5-16) ignores the flag; y is bit-identical to pq2_matmul."""
    from gemm_pq2_ternary_gb300 import binding as pq2
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_MATMUL
    tern, ws, x = inputs.generate(prob)
    codes, ws_d = pq2.pack(torch.from_numpy(tern).cuda(), torch.from_numpy(ws).cuda())
    xd = torch.from_numpy(x).cuda()
    wsb = alloc_workspace(PQ2_OP_MATMUL, prob.M, prob.N, prob.K)
    torch.cuda.synchronize()
    y0 = torch.full((prob.M, prob.N), float("nan"), device="cuda")
    y1 = torch.full((prob.M, prob.N), float("nan"), device="cuda")
    pq2.pq2_matmul(xd, codes, ws_d, y0, wsb)
    pq2.pq2_matmul_ex(xd, codes, ws_d, y1, pq2.PQ2_WEIGHTS_STATIC, wsb)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    assert torch.equal(y0, y1)


def test_static_weights_few_tokens_back_to_back():
    """Static-weight calls of 2 and 4 tokens queued back to back, each x
    written by the kernel right before its call: y equals pq2_matmul's."""
    from gemm_pq2_ternary_gb300 import binding as pq2
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_MATMUL
    probs = [inputs.Problem(f"fchain{i}", 2 if i % 2 == 0 else 4, 6144, 5120, "p343", "outliers", 95 + i)
             for i in range(4)]
    data = [inputs.generate(p) for p in probs]
    dev = [pq2.pack(torch.from_numpy(t).cuda(), torch.from_numpy(w).cuda()) for t, w, _ in data]
    xs = [torch.from_numpy(x).cuda() for _, _, x in data]
    xs_live = [torch.empty_like(x) for x in xs]
    wsbs = [alloc_workspace(PQ2_OP_MATMUL, p.M, p.N, p.K) for p in probs]
    torch.cuda.synchronize()
    want = []
    for (codes, ws_d), x, p, wsb in zip(dev, xs, probs, wsbs):
        y = torch.empty((p.M, p.N), device="cuda")
        pq2.pq2_matmul(x, codes, ws_d, y, wsb)
        want.append(y)
    torch.cuda.synchronize()
    outs = [torch.full((p.M, p.N), float("nan"), device="cuda") for p in probs]
    for i, ((codes, ws_d), p) in enumerate(zip(dev, probs)):
        xs_live[i].copy_(xs[i])
        pq2.pq2_matmul_ex(xs_live[i], codes, ws_d, outs[i], pq2.PQ2_WEIGHTS_STATIC, wsbs[i])
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    for a, b in zip(outs, want):
        assert torch.equal(a, b)


# pq2_matmul for 2-16 tokens on the tensor-core small-batch kernel: one kernel
# quantises x straight into the kernel's token tiles and (s, t) table.  y must
# be bit-identical to pq2_quantize_act + pq2_gemm_small (the same per-group
# quantiser), and within the fp32 tolerance of the oracle; tokens past M, G
# not a multiple of 4, ragged N, an all-zero group and 2-4 tokens at a shape
# the DP4A kernel cannot take are covered.
SMALL_FROM_X = ([inputs.Problem(f"smx_m{M}_k{K}_n{N}", M, K, N, "p343", "outliers", 110 + M)
                 for M in (5, 8, 16) for (K, N) in inputs.SMALL_SHAPES] +
                [inputs.Problem("smx_m7_k640_n300", 7, 640, 300, "uniform", "outliers", 120),
                 inputs.Problem("smx_m13_k1664_n1000", 13, 1664, 1000, "p343", "normal", 121),
                 inputs.Problem("smx_m3_k24576_n640", 3, 24576, 640, "p343", "outliers", 122)])


@pytest.mark.parametrize("prob", SMALL_FROM_X, ids=lambda p: p.name)
def test_matmul_small_from_x_matches_two_step_path(prob):
    from gemm_pq2_ternary_gb300 import binding as pq2
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_MATMUL, PQ2_OP_SMALL
    tern, ws, x = inputs.generate(prob)
    x[prob.M - 1, 128:256] = 0  # an all-zero group
    codes, ws_d = pq2.pack(torch.from_numpy(tern).cuda(), torch.from_numpy(ws).cuda())
    xd = torch.from_numpy(x).cuda()
    y1 = torch.full((prob.M, prob.N), float("nan"), device="cuda")
    pq2.pq2_matmul(xd, codes, ws_d, y1, alloc_workspace(PQ2_OP_MATMUL, prob.M, prob.N, prob.K))
    qp, S, T = pq2.quantize(xd)
    y2 = torch.full((prob.M, prob.N), float("nan"), device="cuda")
    pq2.pq2_gemm_small(qp, S, T, codes, ws_d, y2, alloc_workspace(PQ2_OP_SMALL, prob.M, prob.N, prob.K))
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    assert torch.equal(y1, y2)
    oqp, oS, _ = oracle.quantize_act(x)
    ocodes = oracle.pack(tern)
    rng = np.random.default_rng(3)
    ms = np.concatenate([rng.integers(0, prob.M, 512), [0, prob.M - 1]])
    ns = np.concatenate([rng.integers(0, prob.N, 512), [prob.N - 1, 0]])
    ref, A = oracle.matmul_entries(oqp, oS, ocodes, ws, ms, ns)
    err = np.abs(y1.cpu().numpy()[ms, ns].astype(np.float64) - ref)
    assert np.all(err <= oracle.fp32_tolerance(ref, A, prob.K // 128)), f"max err {err.max()}"


# The same for 17-64 tokens where pq2_gemm_prefill takes a token-tile kernel
# (tile_kernel up to 32 tokens, wtile_kernel from 33 where a CTA gets few
# items): y bit-identical to pq2_quantize_act + pq2_gemm_prefill.
PREFILL_FROM_X = [inputs.Problem("pfx_m17_k5120_n17408", 17, 5120, 17408, "p343", "outliers", 130),
                  inputs.Problem("pfx_m32_k6144_n5120", 32, 6144, 5120, "p343", "outliers", 131),
                  inputs.Problem("pfx_m24_k640_n300", 24, 640, 300, "uniform", "outliers", 132),
                  inputs.Problem("pfx_m33_k6144_n5120", 33, 6144, 5120, "p343", "outliers", 133),
                  inputs.Problem("pfx_m64_k6144_n5120", 64, 6144, 5120, "p343", "outliers", 134),
                  inputs.Problem("pfx_m50_k1664_n700", 50, 1664, 700, "uniform", "normal", 135),
                  inputs.Problem("pfx_m48_k5120_n17408", 48, 5120, 17408, "p343", "outliers", 136)]


@pytest.mark.parametrize("prob", PREFILL_FROM_X, ids=lambda p: p.name)
def test_matmul_token_tiles_from_x_match_two_step_path(prob):
    from gemm_pq2_ternary_gb300 import binding as pq2
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_MATMUL, PQ2_OP_PREFILL
    tern, ws, x = inputs.generate(prob)
    x[prob.M - 1, 128:256] = 0  # an all-zero group
    codes, ws_d = pq2.pack(torch.from_numpy(tern).cuda(), torch.from_numpy(ws).cuda())
    xd = torch.from_numpy(x).cuda()
    y1 = torch.full((prob.M, prob.N), float("nan"), device="cuda")
    pq2.pq2_matmul(xd, codes, ws_d, y1, alloc_workspace(PQ2_OP_MATMUL, prob.M, prob.N, prob.K))
    qp, S, T = pq2.quantize(xd)
    y2 = torch.full((prob.M, prob.N), float("nan"), device="cuda")
    pq2.pq2_gemm_prefill(qp, S, T, codes, ws_d, y2,
                         alloc_workspace(PQ2_OP_PREFILL, prob.M, prob.N, prob.K))
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    assert torch.equal(y1, y2)
    oqp, oS, _ = oracle.quantize_act(x)
    rng = np.random.default_rng(4)
    ms = np.concatenate([rng.integers(0, prob.M, 512), [0, prob.M - 1]])
    ns = np.concatenate([rng.integers(0, prob.N, 512), [prob.N - 1, 0]])
    ref, A = oracle.matmul_entries(oqp, oS, oracle.pack(tern), ws, ms, ns)
    err = np.abs(y1.cpu().numpy()[ms, ns].astype(np.float64) - ref)
    assert np.all(err <= oracle.fp32_tolerance(ref, A, prob.K // 128)), f"max err {err.max()}"


# Forced kernels on pq2_matmul's path: a forced token-tile kernel also takes
# its tiles straight from x (a forced 128-token or DP4A kernel keeps the
# two-step path); y is bit-identical to quantise + the forced entry point.
FORCED_FROM_X = [
    ("small", "SMALL_TC", inputs.Problem("fx_tc_m3", 3, 384, 77, "p343", "outliers", 170)),
    ("small", "SMALL_DP4A", inputs.Problem("fx_dp4a_m3", 3, 384, 77, "p343", "outliers", 171)),
    ("prefill", "PREFILL_TILE", inputs.Problem("fx_tile_m40", 40, 640, 261, "p343", "outliers", 172)),
    ("prefill", "PREFILL_WTILE", inputs.Problem("fx_wtile_m20", 20, 640, 261, "uniform", "outliers", 173)),
    ("prefill", "PREFILL_128", inputs.Problem("fx_pf128_m20", 20, 640, 261, "uniform", "normal", 174)),
]


@pytest.mark.parametrize("op,variant,prob", FORCED_FROM_X, ids=lambda v: getattr(v, "name", str(v)))
def test_forced_kernels_from_x_match_two_step_path(op, variant, prob):
    from gemm_pq2_ternary_gb300 import binding as pq2
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_MATMUL
    tern, ws, x = inputs.generate(prob)
    codes, ws_d = pq2.pack(torch.from_numpy(tern).cuda(), torch.from_numpy(ws).cuda())
    xd = torch.from_numpy(x).cuda()
    opc = pq2.PQ2_OP_SMALL if op == "small" else pq2.PQ2_OP_PREFILL
    fn = pq2.pq2_gemm_small if op == "small" else pq2.pq2_gemm_prefill
    var = getattr(pq2, "PQ2_VARIANT_" + variant)
    y1 = torch.full((prob.M, prob.N), float("nan"), device="cuda")
    y2 = torch.full((prob.M, prob.N), float("nan"), device="cuda")
    with pq2.forced_kernel(opc, var):
        pq2.pq2_matmul(xd, codes, ws_d, y1, alloc_workspace(PQ2_OP_MATMUL, prob.M, prob.N, prob.K))
        qp, S, T = pq2.quantize(xd)
        fn(qp, S, T, codes, ws_d, y2, alloc_workspace(opc, prob.M, prob.N, prob.K))
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    assert torch.equal(y1, y2)
    oqp, oS, _ = oracle.quantize_act(x)
    ref, A = oracle.matmul(oqp, oS, oracle.pack(tern), ws)
    err = np.abs(y1.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= oracle.fp32_tolerance(ref, A, prob.K // 128)), f"max err {err.max()}"
