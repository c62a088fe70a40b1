"""Pins of the oracle's SwiGLU activation (an assumed activation between the
MLP projections; the pages do not define it) and of its stated fp32 exp.

Each check ties the oracle to mathematics rather than to itself: the fp64
exponential, the exact value exp(0) = 1, the identity
silu(g) - silu(-g) = g, the limits silu(g) -> g and silu(g) -> 0, and fp16
saturation."""
import math

import numpy as np

import oracle


def test_exp_is_within_one_ulp_of_the_fp64_exponential():
    x = np.concatenate([np.linspace(-87, 88, 40001, dtype=np.float32),
                        np.float32([-1e-7, 1e-7, -0.5, 0.5, -math.log(2), math.log(2)])])
    y = oracle.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(y - ref) / ulp) <= 1.0


def test_exp_special_values_and_clamp():
    y = oracle.exp_f32(np.float32([0.0, -100.0, -87.0, 100.0, 88.0]))
    assert y[0] == 1.0
    assert y[1] == y[2] and y[3] == y[4]          # clamped to [-87, 88]
    assert np.isfinite(y).all() and y[2] > 0


def _swiglu_fp64(g, u):
    g = g.astype(np.float64)
    return g / (1.0 + np.exp(-g)) * u.astype(np.float64)


def test_swiglu_matches_the_fp64_formula_to_fp16_rounding():
    rng = np.random.default_rng(11)
    g = (rng.standard_normal((3, 512)) * 4).astype(np.float32)
    u = (rng.standard_normal((3, 512)) * 3).astype(np.float32)
    h = oracle.swiglu(np.concatenate([g, u], axis=1)).astype(np.float64)
    ref = _swiglu_fp64(g, u)
    # one fp16 rounding (half an fp16 ulp) plus a few fp32 ulps of the steps
    bound = 0.5 * np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64) + 4e-7 * np.abs(ref) + 1e-30
    assert np.all(np.abs(h - ref) <= bound)


def test_swiglu_identity_and_limits():
    g = np.float32([0.0, 0.5, 1.0, 2.0, 3.0, 7.0])
    one = np.ones_like(g)
    h_pos = oracle.swiglu(np.concatenate([g, one])[None]).astype(np.float64)[0]
    h_neg = oracle.swiglu(np.concatenate([-g, one])[None]).astype(np.float64)[0]
    # silu(g) - silu(-g) = g, to fp16 rounding of each side
    assert np.all(np.abs((h_pos - h_neg) - g) <= 2 * np.spacing(np.float16(8.0)).astype(np.float64))
    assert h_pos[0] == 0.0
    # large gates: silu(g) -> g (exact in fp16 at g = 20), silu(-g) -> 0
    big = oracle.swiglu(np.float32([[20.0, -30.0, 1.0, 1.0]]))[0]
    assert big[0] == np.float16(20.0)
    assert abs(float(big[1])) < 1e-9


def test_swiglu_saturates_at_the_largest_fp16():
    g = np.float32([20.0, -20.0])
    u = np.float32([5000.0, 5000.0])
    h = oracle.swiglu(np.concatenate([g, u])[None])[0]
    assert h[0] == np.float16(65504.0)              # 1e5 saturates instead of overflowing
    ref = float(_swiglu_fp64(g[1:], u[1:])[0])      # about -2.06e-4, well inside fp16
    assert abs(float(h[1]) - ref) <= 0.5 * float(np.spacing(np.float16(ref)))
