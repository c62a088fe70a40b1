"""GPU parity: every entry point of the C ABI against the CPU oracle on the
same seeded inputs.

Bar: bit-exact for the integer and byte outputs (quantised activations, S,
T, packed codes, per-group integer dots); for fp32 y, every element within
oracle.fp32_tolerance (1e-3 relative to the float64 reference plus the fp32
rounding bound of the group sum).  Full-size problems that the oracle cannot
finish in seconds are checked on sampled outputs, in the same launch
configuration the benchmark uses (the library picks it from the shape).
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_pq2_ternary_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pq2():
    from gemm_pq2_ternary_gb300 import binding
    return binding


DEV = "cuda"


def _to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


class Case:
    """A generated problem, its device copies and the oracle's quantities."""

    def __init__(self, pq2, prob, need_full=True):
        self.p = prob
        tern, ws, x = inputs.generate(prob)
        self.tern, self.ws, self.x = tern, ws, x
        self.codes_d, self.ws_d = pq2.pack(_to_dev(tern), _to_dev(ws))
        self.qp_d, self.S_d, self.T_d = pq2.quantize(_to_dev(x))
        self.oqp, self.oS, self.oT = oracle.quantize_act(x)
        self.ocodes = oracle.pack(tern)


def _check_close(y, ref, A, G, what):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - ref)
    tol = oracle.fp32_tolerance(ref, A, G)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; "
                           f"max err {err.max():.3e}, worst ratio {(err / tol).max():.2f}")


def _check_full(pq2, case, y_d):
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    ref, A = oracle.matmul(case.oqp, case.oS, case.ocodes, case.ws)
    _check_close(y_d.cpu().numpy(), ref, A, case.p.K // 128, case.p.name)


def _check_sampled(pq2, case, y_d, count=512, seed=0):
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    M, N = case.p.M, case.p.N
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, M, size=count)
    ns = rng.integers(0, N, size=count)
    # always include the corners and the ragged tail
    ms = np.concatenate([ms, [0, M - 1, 0, M - 1]])
    ns = np.concatenate([ns, [0, N - 1, N - 1, 0]])
    ref, A = oracle.matmul_entries(case.oqp, case.oS, case.ocodes, case.ws, ms, ns)
    y = y_d.cpu().numpy()[ms, ns]
    _check_close(y, ref, A, case.p.K // 128, case.p.name + " (sampled)")


# ----------------------------------------------------------------------------
# quantise and pack: bit-exact
# ----------------------------------------------------------------------------
QUANT_SHAPES = [(1, 128), (1, 1024), (1, 6144), (3, 384), (16, 5120), (16, 17408), (128, 5120),
                (37, 640)]


@pytest.mark.parametrize("M,K", QUANT_SHAPES)
def test_quantize_bit_exact(pq2, M, K):
    x = inputs.generate_x(M, K, "outliers", seed=M * 7 + K)
    if M >= 3:
        x[1, 128:256] = 0          # an all-zero group
        x[2, 5] = np.float16(60000.0)  # a large outlier
    qp, S, T = pq2.quantize(_to_dev(x))
    torch.cuda.synchronize()
    oqp, oS, oT = oracle.quantize_act(x)
    assert np.array_equal(qp.cpu().numpy(), oqp)
    assert np.array_equal(S.cpu().numpy().view(np.uint32), oS.view(np.uint32))
    assert np.array_equal(T.cpu().numpy(), oT)


def test_quantize_exact_ties(pq2):
    d = 0.125
    vals = [127 * d, 0.5 * d, 1.5 * d, 2.5 * d, -0.5 * d, -1.5 * d, -2.5 * d, 3 * d, -127 * d]
    x = np.zeros((1, 128), dtype=np.float16)
    x[0, :len(vals)] = vals
    qp, S, T = pq2.quantize(_to_dev(x))
    torch.cuda.synchronize()
    oqp, oS, oT = oracle.quantize_act(x)
    assert np.array_equal(qp.cpu().numpy(), oqp) and np.array_equal(T.cpu().numpy(), oT)


@pytest.mark.parametrize("N,K", [(1, 128), (77, 384), (5120, 6144)])
def test_pack_bit_exact(pq2, N, K):
    tern = inputs.draw_ternary(np.random.default_rng(N), N, K, "p343")
    ws = inputs.draw_ws(np.random.default_rng(K), N, K)
    codes, ws_out = pq2.pack(_to_dev(tern), _to_dev(ws))
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    assert np.array_equal(codes.cpu().numpy(), oracle.pack(tern))
    assert np.array_equal(ws_out.cpu().numpy(), ws)


def test_pack_flags_non_ternary(pq2):
    tern = np.zeros((4, 128), dtype=np.int8)
    tern[2, 9] = 3
    codes = torch.empty((4, 32), dtype=torch.uint8, device=DEV)
    pq2.pq2_pack_weights(_to_dev(tern), None, codes, None)
    assert pq2.pq2_last_device_error() == pq2.PQ2_ERR_INVALID_ARG
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK   # the word was cleared


# ----------------------------------------------------------------------------
# M = 1
# ----------------------------------------------------------------------------
GEMV_PROBLEMS = [
    inputs.PR1,
    inputs.Problem("gemv_ragged", 1, 384, 77, "p343", "outliers", 11),
    inputs.Problem("gemv_k128", 1, 128, 1000, "uniform", "normal", 12),
    inputs.Problem("gemv_n1", 1, 2048, 1, "uniform", "outliers", 13),
    inputs.Problem("gemv_g_odd", 1, 128 * 13, 301, "p343", "outliers", 14),
    inputs.DECODE,
    inputs.mlp_gate_up(1),
    inputs.mlp_down(1),
]


@pytest.mark.parametrize("prob", GEMV_PROBLEMS, ids=lambda p: p.name)
def test_gemv_parity(pq2, prob):
    c = Case(pq2, prob)
    y = torch.full((1, prob.N), float("nan"), device=DEV)
    pq2.pq2_gemv(c.qp_d, c.S_d, c.T_d, c.codes_d, c.ws_d, y)
    if prob.N * prob.K <= 64 * 1024 * 1024:
        _check_full(pq2, c, y)
    else:
        _check_sampled(pq2, c, y)


@pytest.mark.parametrize("prob", [inputs.PR1, GEMV_PROBLEMS[1], GEMV_PROBLEMS[4], inputs.DECODE],
                         ids=lambda p: p.name)
def test_gemv_group_dots_bit_exact(pq2, prob):
    c = Case(pq2, prob)
    G = prob.K // 128
    dots = torch.empty((1, prob.N, G), dtype=torch.int32, device=DEV)
    pq2.pq2_group_dots(pq2.PQ2_OP_GEMV, c.qp_d, c.T_d, c.codes_d, dots)
    torch.cuda.synchronize()
    assert np.array_equal(dots.cpu().numpy(), oracle.group_dots(c.oqp, c.ocodes))


def test_gemv_deterministic(pq2):
    c = Case(pq2, inputs.DECODE)
    ys = []
    for _ in range(3):
        y = torch.empty((1, c.p.N), device=DEV)
        pq2.pq2_gemv(c.qp_d, c.S_d, c.T_d, c.codes_d, c.ws_d, y)
        ys.append(y.cpu().numpy())
    assert all(np.array_equal(ys[0].view(np.uint32), v.view(np.uint32)) for v in ys[1:])


def test_gemv_constant_codes(pq2):
    # all codes 0 (all weights -1): y = -sum_g T * S * WS
    K, N = 768, 33
    x = inputs.generate_x(1, K, "outliers", seed=3)
    qp, S, T = pq2.quantize(_to_dev(x))
    codes = torch.zeros((N, K // 4), dtype=torch.uint8, device=DEV)
    ws = _to_dev(inputs.draw_ws(np.random.default_rng(1), N, K))
    y = torch.empty((1, N), device=DEV)
    pq2.pq2_gemv(qp, S, T, codes, ws, y)
    torch.cuda.synchronize()
    oqp, oS, oT = oracle.quantize_act(x)
    ref, A = oracle.matmul(oqp, oS, codes.cpu().numpy(), ws.cpu().numpy())
    want = -np.einsum("g,g,ng->n", oT[0].astype(np.float64), oS[0].astype(np.float64),
                      ws.cpu().numpy().astype(np.float64))
    np.testing.assert_allclose(ref[0], want, rtol=1e-12)
    _check_close(y.cpu().numpy(), ref, A, K // 128, "all-minus-one")


def test_gemv_guard_band(pq2):
    # y is written exactly for n < N: a larger buffer keeps its tail
    c = Case(pq2, inputs.Problem("guard", 1, 640, 97, "uniform", "normal", 5))
    buf = torch.full((1, 97 + 64), 123.0, device=DEV)
    y = buf[:, :97]
    assert y.is_contiguous()
    pq2.pq2_gemv(c.qp_d, c.S_d, c.T_d, c.codes_d, c.ws_d, y)
    torch.cuda.synchronize()
    assert torch.all(buf[0, 97:] == 123.0)


# ----------------------------------------------------------------------------
# 2 <= M <= 16
# ----------------------------------------------------------------------------
SMALL_PROBLEMS = ([inputs.Problem("small_ragged", M, 384, 77, "p343", "outliers", 20 + M)
                   for M in (2, 3, 5, 16)] +
                  [inputs.small_batch(M, K, N) for (K, N) in inputs.SMALL_SHAPES
                   for M in inputs.SMALL_MS] +
                  [inputs.mlp_gate_up(16), inputs.mlp_down(16)])


@pytest.mark.parametrize("prob", SMALL_PROBLEMS, ids=lambda p: p.name)
def test_small_parity(pq2, prob):
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_SMALL
    c = Case(pq2, prob)
    y = torch.full((prob.M, prob.N), float("nan"), device=DEV)
    pq2.pq2_gemm_small(c.qp_d, c.S_d, c.T_d, c.codes_d, c.ws_d, y,
                       alloc_workspace(PQ2_OP_SMALL, prob.M, prob.N, prob.K))
    if prob.M * prob.N * prob.K <= 64 * 1024 * 1024:
        _check_full(pq2, c, y)
    else:
        _check_sampled(pq2, c, y)


@pytest.mark.parametrize("prob", SMALL_PROBLEMS[:4] + [inputs.small_batch(16, 5120, 17408)],
                         ids=lambda p: p.name)
def test_small_group_dots_bit_exact(pq2, prob):
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_SMALL
    c = Case(pq2, prob)
    G = prob.K // 128
    dots = torch.empty((prob.M, prob.N, G), dtype=torch.int32, device=DEV)
    pq2.pq2_group_dots(pq2.PQ2_OP_SMALL, c.qp_d, c.T_d, c.codes_d, dots,
                       alloc_workspace(PQ2_OP_SMALL, prob.M, prob.N, prob.K))
    torch.cuda.synchronize()
    got = dots.cpu().numpy()
    if prob.M * prob.N * prob.K <= 64 * 1024 * 1024:
        assert np.array_equal(got, oracle.group_dots(c.oqp, c.ocodes))
    else:
        rows = slice(0, 512)
        want = oracle.group_dots(c.oqp, c.ocodes[rows])
        assert np.array_equal(got[:, rows], want)


# ----------------------------------------------------------------------------
# prefill
# ----------------------------------------------------------------------------
PREFILL_PROBLEMS = [
    inputs.Problem("prefill_ragged", 37, 384, 200, "uniform", "outliers", 30),
    inputs.Problem("prefill_m17", 17, 640, 129, "p343", "outliers", 31),
    inputs.Problem("prefill_m300", 300, 1024, 520, "uniform", "normal", 32),
    inputs.prefill(128),
    inputs.prefill(4096),
]


@pytest.mark.parametrize("prob", PREFILL_PROBLEMS, ids=lambda p: p.name)
def test_prefill_parity(pq2, prob):
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_PREFILL
    c = Case(pq2, prob)
    y = torch.full((prob.M, prob.N), float("nan"), device=DEV)
    pq2.pq2_gemm_prefill(c.qp_d, c.S_d, c.T_d, c.codes_d, c.ws_d, y,
                         alloc_workspace(PQ2_OP_PREFILL, prob.M, prob.N, prob.K))
    if prob.M * prob.N * prob.K <= 64 * 1024 * 1024:
        _check_full(pq2, c, y)
    else:
        _check_sampled(pq2, c, y, count=2048)


@pytest.mark.parametrize("prob", PREFILL_PROBLEMS[:3], ids=lambda p: p.name)
def test_prefill_group_dots_bit_exact(pq2, prob):
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_PREFILL
    c = Case(pq2, prob)
    dots = torch.empty((prob.M, prob.N, prob.K // 128), dtype=torch.int32, device=DEV)
    pq2.pq2_group_dots(pq2.PQ2_OP_PREFILL, c.qp_d, c.T_d, c.codes_d, dots,
                       alloc_workspace(PQ2_OP_PREFILL, prob.M, prob.N, prob.K))
    torch.cuda.synchronize()
    assert np.array_equal(dots.cpu().numpy(), oracle.group_dots(c.oqp, c.ocodes))


# ----------------------------------------------------------------------------
# 17 to 64 tokens (pq2_gemm_prefill, token-tile kernel)
# ----------------------------------------------------------------------------
MID_PROBLEMS = ([inputs.Problem(f"mid_ragged_m{M}", M, 640, 300, "p343", "outliers", 110 + M)
                 for M in (17, 31, 33, 50)] +
                [inputs.Problem(f"mid_m{M}_k{K}_n{N}", M, K, N, "p343", "outliers", 120 + M)
                 for M in (17, 32, 48, 64) for (K, N) in inputs.SMALL_SHAPES])


@pytest.mark.parametrize("prob", MID_PROBLEMS, ids=lambda p: p.name)
def test_mid_parity(pq2, prob):
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_PREFILL
    c = Case(pq2, prob)
    y = torch.full((prob.M, prob.N), float("nan"), device=DEV)
    pq2.pq2_gemm_prefill(c.qp_d, c.S_d, c.T_d, c.codes_d, c.ws_d, y,
                         alloc_workspace(PQ2_OP_PREFILL, prob.M, prob.N, prob.K))
    if prob.M * prob.N * prob.K <= 64 * 1024 * 1024:
        _check_full(pq2, c, y)
    else:
        _check_sampled(pq2, c, y, count=2048)


@pytest.mark.parametrize("prob", MID_PROBLEMS[:4] + [MID_PROBLEMS[-1]], ids=lambda p: p.name)
def test_mid_group_dots_bit_exact(pq2, prob):
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_PREFILL
    c = Case(pq2, prob)
    G = prob.K // 128
    dots = torch.empty((prob.M, prob.N, G), dtype=torch.int32, device=DEV)
    pq2.pq2_group_dots(pq2.PQ2_OP_PREFILL, c.qp_d, c.T_d, c.codes_d, dots,
                       alloc_workspace(PQ2_OP_PREFILL, prob.M, prob.N, prob.K))
    torch.cuda.synchronize()
    got = dots.cpu().numpy()
    if prob.M * prob.N * prob.K <= 64 * 1024 * 1024:
        assert np.array_equal(got, oracle.group_dots(c.oqp, c.ocodes))
    else:
        rows = np.r_[0:256, prob.N - 256:prob.N]
        assert np.array_equal(got[:, rows], oracle.group_dots(c.oqp, c.ocodes[rows]))


# ----------------------------------------------------------------------------
# whole path from fp16 and error reporting
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("M", [1, 6, 40])
def test_matmul_entry_point(pq2, M):
    from gemm_pq2_ternary_gb300.binding import alloc_workspace, PQ2_OP_MATMUL
    prob = inputs.Problem(f"mm{M}", M, 512, 150, "p343", "outliers", 40 + M)
    c = Case(pq2, prob)
    y = torch.empty((M, prob.N), device=DEV)
    pq2.pq2_matmul(_to_dev(c.x), c.codes_d, c.ws_d, y,
                   alloc_workspace(PQ2_OP_MATMUL, M, prob.N, prob.K))
    _check_full(pq2, c, y)


def test_bounded_wait_reports_timeout(pq2):
    # The producer withholds stage 0; the consumers' waits run out after the
    # (shortened) limit, the kernel exits cleanly and the host reads
    # PQ2_ERR_TIMEOUT.  A normal call afterwards is correct again.
    c = Case(pq2, inputs.Problem("timeout", 1, 1024, 4096, "uniform", "normal", 50))
    y = torch.empty((1, 4096), device=DEV)
    try:
        pq2.pq2_debug_set_wait_limit_ns(20_000_000)
        pq2.pq2_debug_skip_stage(0)
        pq2.pq2_gemv(c.qp_d, c.S_d, c.T_d, c.codes_d, c.ws_d, y)
        assert pq2.pq2_last_device_error() == pq2.PQ2_ERR_TIMEOUT
    finally:
        pq2.pq2_debug_skip_stage(-1)
        pq2.pq2_debug_set_wait_limit_ns(2_000_000_000)
    pq2.pq2_gemv(c.qp_d, c.S_d, c.T_d, c.codes_d, c.ws_d, y)
    _check_full(pq2, c, y)


@pytest.mark.parametrize("op,variant,prob", [
    ("small", "tc", inputs.Problem("timeout_small", 8, 1280, 640, "p343", "outliers", 51)),
    ("small", "tile", inputs.Problem("timeout_tile16", 8, 1280, 640, "p343", "outliers", 54)),
    ("prefill", "tile", inputs.Problem("timeout_tile64", 40, 1280, 640, "p343", "outliers", 55)),
    ("prefill", "128", inputs.Problem("timeout_pf128", 37, 384, 200, "uniform", "normal", 52)),
    ("prefill", "wide", inputs.Problem("timeout_pfwide", 37, 384, 200, "uniform", "normal", 53)),
], ids=["small_kernel", "tile_kernel_16", "tile_kernel_64", "prefill_kernel",
        "prefill_wide_kernel"])
def test_tensor_core_pipelines_report_timeout(pq2, op, variant, prob):
    # As above for the tcgen05 pipelines: the producer of each CTA withholds
    # its first stage; the MMA issuers and the other roles give up after the
    # limit, the producer waits for the copies it did issue, every role
    # reaches the teardown (tensor memory freed), and the host reads
    # PQ2_ERR_TIMEOUT.  The next normal call is correct.
    from gemm_pq2_ternary_gb300.binding import alloc_workspace
    opc = pq2.PQ2_OP_SMALL if op == "small" else pq2.PQ2_OP_PREFILL
    var = {("small", "tc"): pq2.PQ2_VARIANT_SMALL_TC, ("small", "tile"): pq2.PQ2_VARIANT_SMALL_TILE,
           ("prefill", "tile"): pq2.PQ2_VARIANT_PREFILL_TILE,
           ("prefill", "128"): pq2.PQ2_VARIANT_PREFILL_128,
           ("prefill", "wide"): pq2.PQ2_VARIANT_PREFILL_WIDE}[(op, variant)]
    fn = pq2.pq2_gemm_small if op == "small" else pq2.pq2_gemm_prefill
    c = Case(pq2, prob)
    y = torch.empty((prob.M, prob.N), device=DEV)
    with pq2.forced_kernel(opc, var):
        wsp = alloc_workspace(opc, prob.M, prob.N, prob.K)
        try:
            pq2.pq2_debug_set_wait_limit_ns(20_000_000)
            pq2.pq2_debug_skip_stage(0)
            fn(c.qp_d, c.S_d, c.T_d, c.codes_d, c.ws_d, y, wsp)
            assert pq2.pq2_last_device_error() == pq2.PQ2_ERR_TIMEOUT
        finally:
            pq2.pq2_debug_skip_stage(-1)
            pq2.pq2_debug_set_wait_limit_ns(2_000_000_000)
        y = torch.full((prob.M, prob.N), float("nan"), device=DEV)
        fn(c.qp_d, c.S_d, c.T_d, c.codes_d, c.ws_d, y, wsp)
    _check_full(pq2, c, y)
