"""Pins of the oracle's bf16 split-K GEMM (the unquantised in_proj_ba
projection of the pages): exact integer-valued products, the identity,
pure-Python brute force on a tiny case, bf16 conversions, and the tolerance's
bound against a deliberately perturbed summation order."""
import itertools

import numpy as np

import oracle


def _bits(v):
    return oracle.f64_to_bf16(np.asarray(v, dtype=np.float64))


def test_bf16_conversions_round_trip_and_round_half_even():
    vals = np.array([0.0, 1.0, -2.5, 3.140625, 1e-3, 65504.0, -1.0e30])
    back = oracle.bf16_to_f64(_bits(vals))
    assert np.all(np.abs(back - vals) <= np.abs(vals) * 2.0 ** -8)
    # 1 + 2^-8 is halfway between bf16 1 and 1 + 2^-7: ties go to even (1)
    assert oracle.bf16_to_f64(_bits([1.0 + 2.0 ** -8]))[0] == 1.0
    assert oracle.bf16_to_f64(_bits([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6
    assert oracle.bf16_to_f64(_bits([-0.0])).tolist() == [0.0]
    # just above the halfway point rounds up (a route through float32 would
    # drop the 2^-40 and then tie to 1.0: double rounding)
    assert oracle.bf16_to_f64(_bits([1.0 + 2.0 ** -8 + 2.0 ** -40]))[0] == 1.0 + 2.0 ** -7


def test_integer_valued_products_are_exact():
    rng = np.random.default_rng(3)
    x = rng.integers(-8, 9, size=(5, 384)).astype(np.float64)
    w = rng.integers(-8, 9, size=(7, 384)).astype(np.float64)
    ref, A = oracle.gemm_bf16(_bits(x), _bits(w))
    assert np.array_equal(ref, x @ w.T)
    assert np.array_equal(A, np.abs(x) @ np.abs(w).T)


def test_identity_weights_return_x():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 96))
    ref, _ = oracle.gemm_bf16(_bits(x), _bits(np.eye(96)))
    assert np.array_equal(ref, oracle.bf16_to_f64(_bits(x)))


def test_brute_force_tiny():
    rng = np.random.default_rng(5)
    xb = _bits(rng.standard_normal((2, 6)))
    wb = _bits(rng.standard_normal((3, 6)))
    x, w = oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb)
    ref, _ = oracle.gemm_bf16(xb, wb)
    for m, n in itertools.product(range(2), range(3)):
        s = 0.0
        for k in range(6):
            s += x[m, k] * w[n, k]
        assert abs(ref[m, n] - s) <= 1e-15 * (abs(s) + 1)


def test_tolerance_covers_fp32_split_sums_and_bf16_rounding():
    rng = np.random.default_rng(6)
    K = 5120
    xb = _bits(rng.standard_normal((4, K)))
    wb = _bits(rng.standard_normal((96, K)) * 0.02)
    ref, A = oracle.gemm_bf16(xb, wb)
    x32 = oracle.bf16_to_f64(xb).astype(np.float32)
    w32 = oracle.bf16_to_f64(wb).astype(np.float32)
    # 20 splits of 256, each summed in fp32, then the splits in order, in fp32
    parts = [x32[:, s:s + 256] @ w32[:, s:s + 256].T for s in range(0, K, 256)]
    acc = np.zeros_like(parts[0])
    for p in parts:
        acc = (acc + p).astype(np.float32)
    y = oracle.bf16_to_f64(oracle.f64_to_bf16(acc.astype(np.float64)))
    assert np.all(np.abs(y - ref) <= oracle.bf16_gemm_tolerance(ref, A, K))
