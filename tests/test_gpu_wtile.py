"""GPU checks of the weights-wide token-tile kernel (wtile_kernel: 128 weight
rows per MMA, the tokens' hi and lo parts as the 128-row operand), forced
through pq2_debug_force_kernel for the small-batch and prefill entry points,
and of pq2_gemm_prefill's default routing of 33-64 tokens to it.

Its integer group dots must equal the oracle's bit for bit and y must meet
the fp32 tolerance (on every output at small sizes, on sampled outputs at the
sweep shapes); repeated calls give the same bits ([P1] "Choose the
configuration with the proxy": split partial sums added in a fixed order);
a withheld stage ends in PQ2_ERR_TIMEOUT with the next call correct.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_pq2_ternary_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pq2():
    from gemm_pq2_ternary_gb300 import binding
    yield binding
    for op in (binding.PQ2_OP_SMALL, binding.PQ2_OP_PREFILL):
        binding.pq2_debug_force_kernel(op, binding.PQ2_VARIANT_DEFAULT)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


class Case:
    def __init__(self, pq2, prob):
        self.p = prob
        tern, ws, x = inputs.generate(prob)
        self.ws = ws
        self.codes, self.ws_d = pq2.pack(_dev(tern), _dev(ws))
        self.qp, self.S, self.T = pq2.quantize(_dev(x))
        self.oqp, self.oS, _ = oracle.quantize_act(x)
        self.ocodes = oracle.pack(tern)


def _op_variant(pq2, M):
    if M <= 16:
        return pq2.PQ2_OP_SMALL, pq2.PQ2_VARIANT_SMALL_WTILE, pq2.pq2_gemm_small
    return pq2.PQ2_OP_PREFILL, pq2.PQ2_VARIANT_PREFILL_WTILE, pq2.pq2_gemm_prefill


def _run(pq2, c):
    M, N, K = c.p.M, c.p.N, c.p.K
    op, var, fn = _op_variant(pq2, M)
    y = torch.full((M, N), float("nan"), device=DEV)
    with pq2.forced_kernel(op, var):
        fn(c.qp, c.S, c.T, c.codes, c.ws_d, y, pq2.alloc_workspace(op, M, N, K))
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    return y


def _dots(pq2, c):
    M, N, K = c.p.M, c.p.N, c.p.K
    op, var, _ = _op_variant(pq2, M)
    dots = torch.empty((M, N, K // 128), dtype=torch.int32, device=DEV)
    with pq2.forced_kernel(op, var):
        pq2.pq2_group_dots(op, c.qp, c.T, c.codes, dots, pq2.alloc_workspace(op, M, N, K))
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    return dots.cpu().numpy()


def _tol_check(c, y, ref, A, what):
    err = np.abs(y.astype(np.float64) - ref)
    tol = oracle.fp32_tolerance(ref, A, c.p.K // 128)
    assert np.all(err <= tol), f"{c.p.name} {what}: max err {err.max():.3e}"


# ragged shapes: N not a multiple of 128, G not a multiple of 4, tokens that
# leave part of each 16/32/64-token tile empty
RAGGED = [
    inputs.Problem("wt_m2", 2, 384, 77, "p343", "outliers", 170),
    inputs.Problem("wt_m5", 5, 1280, 300, "uniform", "outliers", 171),
    inputs.Problem("wt_m8", 8, 6144, 640, "p343", "outliers", 172),
    inputs.Problem("wt_m16", 16, 640, 600, "p343", "outliers", 173),
    inputs.Problem("wt_m17", 17, 640, 300, "p343", "outliers", 174),
    inputs.Problem("wt_m31", 31, 1152, 513, "uniform", "outliers", 175),
    inputs.Problem("wt_m33", 33, 640, 260, "p343", "outliers", 176),
    inputs.Problem("wt_m64", 64, 1280, 700, "p343", "outliers", 177),
]


@pytest.mark.parametrize("prob", RAGGED, ids=lambda p: p.name)
def test_wtile_forced_parity_and_dots(pq2, prob):
    c = Case(pq2, prob)
    y = _run(pq2, c)
    ref, A = oracle.matmul(c.oqp, c.oS, c.ocodes, c.ws)
    _tol_check(c, y.cpu().numpy(), ref, A, "y")
    assert np.array_equal(_dots(pq2, c), oracle.group_dots(c.oqp, c.ocodes))


SWEEP = [inputs.Problem(f"wt_m{M}_k{K}_n{N}", M, K, N, "p343", "outliers", 180 + M)
         for M in (8, 16, 32, 64) for (K, N) in inputs.SMALL_SHAPES]


@pytest.mark.parametrize("prob", SWEEP, ids=lambda p: p.name)
def test_wtile_forced_sweep_shapes_sampled(pq2, prob):
    c = Case(pq2, prob)
    y = _run(pq2, c).cpu().numpy()
    rng = np.random.default_rng(1)
    ms = np.concatenate([rng.integers(0, prob.M, 1024), [0, prob.M - 1, 0, prob.M - 1]])
    ns = np.concatenate([rng.integers(0, prob.N, 1024), [0, prob.N - 1, prob.N - 1, 0]])
    ref, A = oracle.matmul_entries(c.oqp, c.oS, c.ocodes, c.ws, ms, ns)
    _tol_check(c, y[ms, ns], ref, A, "sampled y")


@pytest.mark.parametrize("prob", [SWEEP[3], SWEEP[7]], ids=lambda p: p.name)
def test_wtile_forced_sweep_dots_rows(pq2, prob):
    # the dots of the first and last 256 rows (two 128-row tiles each; the last ragged)
    c = Case(pq2, prob)
    got = _dots(pq2, c)
    rows = np.r_[0:256, prob.N - 256:prob.N]
    assert np.array_equal(got[:, rows], oracle.group_dots(c.oqp, c.ocodes[rows]))


@pytest.mark.parametrize("prob", [SWEEP[2], SWEEP[4], SWEEP[7]], ids=lambda p: p.name)
def test_wtile_deterministic(pq2, prob):
    # tiles shared by several CTAs: the last contributor adds the partials in
    # CTA order, so every call gives the same bits
    c = Case(pq2, prob)
    first = _run(pq2, c)
    for _ in range(4):
        assert torch.equal(_run(pq2, c), first)


@pytest.mark.parametrize("prob", [inputs.Problem("wt_timeout16", 8, 1280, 640, "p343", "outliers", 190),
                                  inputs.Problem("wt_timeout64", 40, 1280, 640, "p343", "outliers", 191)],
                         ids=lambda p: p.name)
def test_wtile_reports_timeout(pq2, prob):
    # the producer withholds its first code box; the other roles give up after
    # the limit, the producer waits for the copies it did issue, every role
    # reaches the teardown, and the host reads PQ2_ERR_TIMEOUT; the next call
    # is correct
    c = Case(pq2, prob)
    op, var, fn = _op_variant(pq2, prob.M)
    y = torch.empty((prob.M, prob.N), device=DEV)
    with pq2.forced_kernel(op, var):
        wsp = pq2.alloc_workspace(op, prob.M, prob.N, prob.K)
        try:
            pq2.pq2_debug_set_wait_limit_ns(20_000_000)
            pq2.pq2_debug_skip_stage(0)
            fn(c.qp, c.S, c.T, c.codes, c.ws_d, y, wsp)
            assert pq2.pq2_last_device_error() == pq2.PQ2_ERR_TIMEOUT
        finally:
            pq2.pq2_debug_skip_stage(-1)
            pq2.pq2_debug_set_wait_limit_ns(2_000_000_000)
    y = _run(pq2, c)
    ref, A = oracle.matmul(c.oqp, c.oS, c.ocodes, c.ws)
    _tol_check(c, y.cpu().numpy(), ref, A, "y after the timeout")


@pytest.mark.parametrize("M,K,N,want", [(48, 6144, 5120, "wtile"), (64, 6144, 5120, "wtile"),
                                        (48, 5120, 17408, "128")], ids=lambda v: str(v))
def test_prefill_routes_mid_token_counts(pq2, M, K, N, want):
    # 33-64 tokens take the weights-wide kernel where a CTA gets at most 4
    # items (128 rows x 4 groups), else the 128 x 128 tile kernel: the
    # default call is bit-identical to the forced one, and bench.py's mirror
    # of the rule agrees
    import bench
    assert bench.prefill_takes_wtile(M, N, K) == (want == "wtile")
    c = Case(pq2, inputs.Problem(f"route_m{M}", M, K, N, "p343", "outliers", 200 + M))
    ws = pq2.alloc_workspace(pq2.PQ2_OP_PREFILL, M, N, K)
    y_def = torch.empty((M, N), device=DEV)
    pq2.pq2_gemm_prefill(c.qp, c.S, c.T, c.codes, c.ws_d, y_def, ws)
    var = pq2.PQ2_VARIANT_PREFILL_WTILE if want == "wtile" else pq2.PQ2_VARIANT_PREFILL_128
    y_f = torch.empty((M, N), device=DEV)
    with pq2.forced_kernel(pq2.PQ2_OP_PREFILL, var):
        pq2.pq2_gemm_prefill(c.qp, c.S, c.T, c.codes, c.ws_d, y_f, ws)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    assert torch.equal(y_def, y_f)
