"""GPU checks that every kernel variant of an entry point computes the same
bits, and that repeated calls do too.

The library routes each call to one kernel by shape; pq2_debug_force_kernel
makes a chosen kernel take shapes the routing would give to another, so
each kernel's integer group dots are compared bit for bit with the oracle's
(the fp32 tolerance cannot see an integer dot that is off by a few units:
that changes y by about 1e-5 relative) and its y bit for bit with the other
kernels of the same entry point, which sum the same terms in the same order.

Determinism: the same inputs give the same bits on every call ([P1] "Choose
the configuration with the proxy" and "Speed up a small unquantised
projection": split partial sums added in the fixed order 0, 1, 2, ...), also
where several CTAs share an output tile.
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
    for op in (binding.PQ2_OP_GEMV, binding.PQ2_OP_SMALL, binding.PQ2_OP_PREFILL):
        binding.pq2_debug_force_kernel(op, binding.PQ2_VARIANT_DEFAULT)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


class Case:
    def __init__(self, pq2, prob):
        self.p = prob
        tern, ws, x = inputs.generate(prob)
        self.tern, self.ws, self.x = tern, ws, x
        self.codes, self.ws_d = pq2.pack(_dev(tern), _dev(ws))
        self.qp, self.S, self.T = pq2.quantize(_dev(x))
        self.oqp, self.oS, _ = oracle.quantize_act(x)
        self.ocodes = oracle.pack(tern)


def _run(pq2, c, op, variant=None):
    """y of `op` (PQ2_OP_SMALL or PQ2_OP_PREFILL) on case c, with `variant`
    forced (None: the library's routing)."""
    M, N, K = c.p.M, c.p.N, c.p.K
    y = torch.full((M, N), float("nan"), device=DEV)
    fn = pq2.pq2_gemm_small if op == pq2.PQ2_OP_SMALL else pq2.pq2_gemm_prefill
    if variant is None:
        fn(c.qp, c.S, c.T, c.codes, c.ws_d, y, pq2.alloc_workspace(op, M, N, K))
    else:
        with pq2.forced_kernel(op, variant):
            fn(c.qp, c.S, c.T, c.codes, c.ws_d, y, pq2.alloc_workspace(op, M, N, K))
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    return y


def _dots(pq2, c, op, variant):
    M, N, K = c.p.M, c.p.N, c.p.K
    dots = torch.empty((M, N, K // 128), dtype=torch.int32, device=DEV)
    with pq2.forced_kernel(op, variant):
        pq2.pq2_group_dots(op, c.qp, c.T, c.codes, dots, pq2.alloc_workspace(op, M, N, K))
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    return dots.cpu().numpy()


def _check_oracle(c, y):
    ref, A = oracle.matmul(c.oqp, c.oS, c.ocodes, c.ws)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    tol = oracle.fp32_tolerance(ref, A, c.p.K // 128)
    assert np.all(err <= tol), f"{c.p.name}: max err {err.max():.3e}"


# ----------------------------------------------------------------------------
# small batches: the DP4A kernel and the tensor-core kernel on each other's shapes
# ----------------------------------------------------------------------------
SMALL_FORCED = [
    inputs.Problem("tc_m2", 2, 384, 77, "p343", "outliers", 70),
    inputs.Problem("tc_m5", 5, 1280, 300, "uniform", "outliers", 71),
    inputs.Problem("tc_m8", 8, 6144, 640, "p343", "outliers", 72),
    inputs.Problem("tc_m16", 16, 640, 129, "p343", "outliers", 73),
]


@pytest.mark.parametrize("prob", SMALL_FORCED, ids=lambda p: p.name)
def test_small_tensor_core_kernel_forced(pq2, prob):
    c = Case(pq2, prob)
    y = _run(pq2, c, pq2.PQ2_OP_SMALL, pq2.PQ2_VARIANT_SMALL_TC)
    _check_oracle(c, y)
    got = _dots(pq2, c, pq2.PQ2_OP_SMALL, pq2.PQ2_VARIANT_SMALL_TC)
    assert np.array_equal(got, oracle.group_dots(c.oqp, c.ocodes))


@pytest.mark.parametrize("prob", SMALL_FORCED, ids=lambda p: p.name)
def test_small_token_tile_kernel_forced(pq2, prob):
    # forced (the default for 5 to 16 tokens is small_kernel), also at 2 tokens
    c = Case(pq2, prob)
    y = _run(pq2, c, pq2.PQ2_OP_SMALL, pq2.PQ2_VARIANT_SMALL_TILE)
    _check_oracle(c, y)
    got = _dots(pq2, c, pq2.PQ2_OP_SMALL, pq2.PQ2_VARIANT_SMALL_TILE)
    assert np.array_equal(got, oracle.group_dots(c.oqp, c.ocodes))


@pytest.mark.parametrize("prob", [SMALL_FORCED[1], SMALL_FORCED[2]], ids=lambda p: p.name)
def test_small_dp4a_kernel_forced(pq2, prob):
    # 5 and 8 tokens: the routing gives them to the tensor cores
    c = Case(pq2, prob)
    y = _run(pq2, c, pq2.PQ2_OP_SMALL, pq2.PQ2_VARIANT_SMALL_DP4A)
    _check_oracle(c, y)
    got = _dots(pq2, c, pq2.PQ2_OP_SMALL, pq2.PQ2_VARIANT_SMALL_DP4A)
    assert np.array_equal(got, oracle.group_dots(c.oqp, c.ocodes))
    # each token's row equals the M = 1 GEMV on that token, bit for bit
    for m in range(prob.M):
        y1 = torch.empty((1, prob.N), device=DEV)
        pq2.pq2_gemv(c.qp[m:m + 1].clone(), c.S[m:m + 1].clone(), c.T[m:m + 1].clone(),
                     c.codes, c.ws_d, y1)
        torch.cuda.synchronize()
        assert torch.equal(y[m], y1[0]), f"token {m}"


def test_forced_dp4a_rejects_what_it_cannot_take(pq2):
    c = Case(pq2, SMALL_FORCED[3])  # 16 tokens: beyond the DP4A kernel's 8
    with pytest.raises(pq2.PQ2Error) as e:
        _run(pq2, c, pq2.PQ2_OP_SMALL, pq2.PQ2_VARIANT_SMALL_DP4A)
    assert e.value.status == pq2.PQ2_ERR_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("M,K,N", [(2, 6144, 5120), (3, 5120, 17408), (4, 1280, 999)])
def test_dp4a_rows_equal_the_single_token_gemv(pq2, M, K, N):
    c = Case(pq2, inputs.Problem("bitid", M, K, N, "p343", "outliers", 80 + M))
    y = _run(pq2, c, pq2.PQ2_OP_SMALL)
    for m in range(M):
        y1 = torch.empty((1, N), device=DEV)
        pq2.pq2_gemv(c.qp[m:m + 1].clone(), c.S[m:m + 1].clone(), c.T[m:m + 1].clone(),
                     c.codes, c.ws_d, y1)
        torch.cuda.synchronize()
        assert torch.equal(y[m], y1[0]), f"token {m}"


# ----------------------------------------------------------------------------
# prefill: the 128 x 128 and the 128 x 256 tile kernels
# ----------------------------------------------------------------------------
PREFILL_FORCED = [
    inputs.Problem("wide_ragged", 37, 384, 200, "uniform", "outliers", 60),
    inputs.Problem("wide_m17", 17, 640, 129, "p343", "outliers", 61),
    inputs.Problem("wide_m300", 300, 1024, 520, "uniform", "normal", 62),
    inputs.Problem("wide_m129", 129, 1280, 777, "p343", "outliers", 63),
    inputs.Problem("wide_n512", 256, 2048, 512, "uniform", "outliers", 64),
]


@pytest.mark.parametrize("prob", PREFILL_FORCED, ids=lambda p: p.name)
def test_prefill_kernels_forced_agree_bit_for_bit(pq2, prob):
    c = Case(pq2, prob)
    y_wide = _run(pq2, c, pq2.PQ2_OP_PREFILL, pq2.PQ2_VARIANT_PREFILL_WIDE)
    y_128 = _run(pq2, c, pq2.PQ2_OP_PREFILL, pq2.PQ2_VARIANT_PREFILL_128)
    _check_oracle(c, y_wide)
    assert torch.equal(y_wide, y_128)
    want = oracle.group_dots(c.oqp, c.ocodes)
    assert np.array_equal(_dots(pq2, c, pq2.PQ2_OP_PREFILL, pq2.PQ2_VARIANT_PREFILL_WIDE), want)
    assert np.array_equal(_dots(pq2, c, pq2.PQ2_OP_PREFILL, pq2.PQ2_VARIANT_PREFILL_128), want)


@pytest.mark.parametrize("prob", PREFILL_FORCED[:2] + [
    inputs.Problem("tile_m64", 64, 1024, 520, "uniform", "normal", 65),
    inputs.Problem("tile_m5", 5, 384, 300, "p343", "outliers", 66)], ids=lambda p: p.name)
def test_prefill_token_tile_kernel_forced(pq2, prob):
    # the token-tile kernel through pq2_gemm_prefill (its default up to 32
    # tokens), and the 128 x 128 tile kernel forced on the same shapes
    c = Case(pq2, prob)
    y_tile = _run(pq2, c, pq2.PQ2_OP_PREFILL, pq2.PQ2_VARIANT_PREFILL_TILE)
    _check_oracle(c, y_tile)
    want = oracle.group_dots(c.oqp, c.ocodes)
    assert np.array_equal(_dots(pq2, c, pq2.PQ2_OP_PREFILL, pq2.PQ2_VARIANT_PREFILL_TILE), want)
    y_128 = _run(pq2, c, pq2.PQ2_OP_PREFILL, pq2.PQ2_VARIANT_PREFILL_128)
    _check_oracle(c, y_128)


def test_prefill_full_size_kernels_agree_bit_for_bit(pq2):
    # M = 4096, 5120 -> 17408: the routing takes the 128 x 256 kernel; the
    # 128 x 128 kernel forced on the same call must give the same bits, and
    # repeated calls of the default must too
    c = Case(pq2, inputs.prefill(4096))
    y0 = _run(pq2, c, pq2.PQ2_OP_PREFILL)
    y_128 = _run(pq2, c, pq2.PQ2_OP_PREFILL, pq2.PQ2_VARIANT_PREFILL_128)
    assert torch.equal(y0, y_128)
    for _ in range(2):
        assert torch.equal(_run(pq2, c, pq2.PQ2_OP_PREFILL), y0)
    # and a sample of it against the oracle
    rng = np.random.default_rng(5)
    ms = np.concatenate([rng.integers(0, c.p.M, 1024), [0, c.p.M - 1]])
    ns = np.concatenate([rng.integers(0, c.p.N, 1024), [c.p.N - 1, 0]])
    ref, A = oracle.matmul_entries(c.oqp, c.oS, c.ocodes, c.ws, ms, ns)
    err = np.abs(y0.cpu().numpy()[ms, ns].astype(np.float64) - ref)
    assert np.all(err <= oracle.fp32_tolerance(ref, A, c.p.K // 128))


# ----------------------------------------------------------------------------
# M = 1: the direct, ring and staged kernels
# ----------------------------------------------------------------------------
def test_gemv_kernels_agree_bit_for_bit(pq2):
    c = Case(pq2, inputs.DECODE)
    N = c.p.N
    x = _dev(c.x)
    ys = {}
    for v in (pq2.PQ2_VARIANT_GEMV_DIRECT, pq2.PQ2_VARIANT_GEMV_RING):
        y = torch.full((1, N), float("nan"), device=DEV)
        with pq2.forced_kernel(pq2.PQ2_OP_GEMV, v):
            pq2.pq2_gemv(c.qp, c.S, c.T, c.codes, c.ws_d, y)
            ys[v] = y
        yf = torch.full((1, N), float("nan"), device=DEV)
        with pq2.forced_kernel(pq2.PQ2_OP_GEMV, v):
            pq2.pq2_matmul(x, c.codes, c.ws_d, yf, None)  # the fused kernels
        ys[(v, "fused")] = yf
    ys["staged"] = torch.full((1, N), float("nan"), device=DEV)
    with pq2.forced_kernel(pq2.PQ2_OP_GEMV, pq2.PQ2_VARIANT_GEMV_STAGED):
        pq2.pq2_matmul_ex(x, c.codes, c.ws_d, ys["staged"], pq2.PQ2_WEIGHTS_STATIC, None)
    torch.cuda.synchronize()
    assert pq2.pq2_last_device_error() == pq2.PQ2_OK
    first = ys[pq2.PQ2_VARIANT_GEMV_DIRECT]
    for k, y in ys.items():
        assert torch.equal(y, first), k
    ref, A = oracle.matmul(c.oqp, c.oS, c.ocodes, c.ws)
    err = np.abs(first.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= oracle.fp32_tolerance(ref, A, c.p.K // 128))


# ----------------------------------------------------------------------------
# determinism: repeated calls give the same bits
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("K,N", inputs.SMALL_SHAPES)
def test_small_deterministic(pq2, K, N):
    # 16 tokens: row tiles shared by several CTAs, partial sums added by the
    # last contributor in CTA order
    c = Case(pq2, inputs.small_batch(16, K, N))
    y0 = _run(pq2, c, pq2.PQ2_OP_SMALL)
    for _ in range(4):
        assert torch.equal(_run(pq2, c, pq2.PQ2_OP_SMALL), y0)


@pytest.mark.parametrize("M", [32, 64])
def test_mid_deterministic(pq2, M):
    # 32 tokens: the token-tile kernel; 64: the 128 x 128 tile kernel
    c = Case(pq2, inputs.Problem(f"det_mid_m{M}", M, 5120, 17408, "p343", "outliers", 95 + M))
    y0 = _run(pq2, c, pq2.PQ2_OP_PREFILL)
    for _ in range(4):
        assert torch.equal(_run(pq2, c, pq2.PQ2_OP_PREFILL), y0)


@pytest.mark.parametrize("M", [128, 300])
def test_prefill_deterministic(pq2, M):
    c = Case(pq2, inputs.Problem(f"det_m{M}", M, 5120, 17408 if M == 128 else 1040,
                                 "uniform", "normal", 90 + M))
    y0 = _run(pq2, c, pq2.PQ2_OP_PREFILL)
    for _ in range(4):
        assert torch.equal(_run(pq2, c, pq2.PQ2_OP_PREFILL), y0)


def test_mma_rate_probe(pq2):
    # the measurement hook behind the prefill roofline's tensor probe: N = 256
    # runs the pipe near its e4m3 peak (about 8190 multiply-adds per cycle per
    # SM measured), N = 32 is bound by the issue cost (about 46 cycles each)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cycles = torch.zeros(sms, dtype=torch.int64, device=DEV)
    for n, lo, hi in ((256, 4000.0, 9000.0), (32, 500.0, 9000.0)):
        pq2.pq2_debug_mma_rate(n, 2048, cycles)
        torch.cuda.synchronize()
        assert pq2.pq2_last_device_error() == pq2.PQ2_OK
        c = cycles.cpu().numpy().astype(np.float64)
        assert (c > 0).all()
        rate = 128.0 * n * 32 * 2048 / c.mean()
        assert lo < rate < hi, (n, rate)
    with pytest.raises(pq2.PQ2Error):
        pq2.pq2_debug_mma_rate(48, 16, cycles)
