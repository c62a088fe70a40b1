"""CPU oracle for the PQ2_0 ternary matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library and its Python binding never
import it, and it imports nothing from them.

The arithmetic lives in ``pq2_oracle.c`` (plain C loops, each function citing
the passage of the pages it follows); this module converts numpy arrays and
calls it.  The fp16 inputs (activations x, group scales WS) are widened here
with numpy's exact fp16 -> fp32/fp64 conversion, a library primitive.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        sigs = {
            "pq2o_threads": [],
            "pq2o_set_threads": [ctypes.c_int],
            "pq2o_quantize": [p, i64, i64, p, p, p],
            "pq2o_plane_order": [p, i64, i64, p],
            "pq2o_natural_order": [p, i64, i64, p],
            "pq2o_pack": [p, i64, i64, p],
            "pq2o_unpack": [p, i64, i64, p],
            "pq2o_group_dots": [p, p, i64, i64, i64, p],
            "pq2o_codes_dots": [p, p, i64, i64, i64, p],
            "pq2o_matmul_rows": [p, p, p, p, i64, i64, i64, i64, i64, p, p],
            "pq2o_matmul_entries": [p, p, p, p, i64, i64, i64, i64, p, p, p, p],
            "pq2o_exp": [p, i64, p],
            "pq2o_swiglu": [p, i64, i64, p],
        }
        for name, args in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: error code {rc}")


def threads() -> int:
    """Host threads the oracle's parallel loops use."""
    return int(_lib().pq2o_threads())


def set_threads(n: int) -> int:
    """Sets the oracle's thread count (n >= 1); returns the count in effect."""
    return int(_lib().pq2o_set_threads(int(n)))


def quantize(x_f16: np.ndarray):
    """x fp16 [M,K] -> (q natural int8 [M,K], S fp32 [M,G], T int32 [M,G])."""
    x = np.ascontiguousarray(np.asarray(x_f16, dtype=np.float16).astype(np.float32))
    M, K = x.shape
    q = np.empty((M, K), dtype=np.int8)
    S = np.empty((M, K // 128), dtype=np.float32)
    T = np.empty((M, K // 128), dtype=np.int32)
    _check(_lib().pq2o_quantize(_ptr(x), M, K, _ptr(q), _ptr(S), _ptr(T)), "quantize")
    return q, S, T


def plane_order(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8)
    M, K = q.shape
    qp = np.empty_like(q)
    _check(_lib().pq2o_plane_order(_ptr(q), M, K, _ptr(qp)), "plane_order")
    return qp


def natural_order(qp: np.ndarray) -> np.ndarray:
    qp = np.ascontiguousarray(qp, dtype=np.int8)
    M, K = qp.shape
    q = np.empty_like(qp)
    _check(_lib().pq2o_natural_order(_ptr(qp), M, K, _ptr(q)), "natural_order")
    return q


def quantize_act(x_f16: np.ndarray):
    """The full activation step: (qp plane-ordered int8, S, T)."""
    q, S, T = quantize(x_f16)
    return plane_order(q), S, T


def pack(tern: np.ndarray) -> np.ndarray:
    """ternary int8 [N,K] in {-1,0,1} -> codes uint8 [N,K/4]."""
    t = np.ascontiguousarray(tern, dtype=np.int8)
    N, K = t.shape
    codes = np.empty((N, K // 4), dtype=np.uint8)
    _check(_lib().pq2o_pack(_ptr(t), N, K, _ptr(codes)), "pack")
    return codes


def unpack(codes: np.ndarray, K: int) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    N = c.shape[0]
    t = np.empty((N, K), dtype=np.int8)
    _check(_lib().pq2o_unpack(_ptr(c), N, K, _ptr(t)), "unpack")
    return t


def group_dots(qp: np.ndarray, codes: np.ndarray) -> np.ndarray:
    """int32 [M,N,G]: per-group ternary dots sum((code-1)*q)."""
    qp = np.ascontiguousarray(qp, dtype=np.int8)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    M, K = qp.shape
    N = codes.shape[0]
    out = np.empty((M, N, K // 128), dtype=np.int32)
    _check(_lib().pq2o_group_dots(_ptr(qp), _ptr(codes), M, N, K, _ptr(out)), "group_dots")
    return out


def codes_dots(qp: np.ndarray, codes: np.ndarray) -> np.ndarray:
    """int32 [M,N,G]: per-group sum(code*q) with no offset."""
    qp = np.ascontiguousarray(qp, dtype=np.int8)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    M, K = qp.shape
    N = codes.shape[0]
    out = np.empty((M, N, K // 128), dtype=np.int32)
    _check(_lib().pq2o_codes_dots(_ptr(qp), _ptr(codes), M, N, K, _ptr(out)), "codes_dots")
    return out


def _ws64(ws):
    return np.ascontiguousarray(np.asarray(ws).astype(np.float64))


def matmul(qp, S, codes, ws_f16, rows=None):
    """(y float64 [M,N], A float64 [M,N]); rows=(n0,n1) limits to a slice,
    returning [M, n1-n0] arrays."""
    qp = np.ascontiguousarray(qp, dtype=np.int8)
    S = np.ascontiguousarray(S, dtype=np.float32)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    WS = _ws64(ws_f16)
    M, K = qp.shape
    N = codes.shape[0]
    n0, n1 = (0, N) if rows is None else rows
    y = np.zeros((M, N), dtype=np.float64)
    A = np.zeros((M, N), dtype=np.float64)
    _check(_lib().pq2o_matmul_rows(_ptr(qp), _ptr(S), _ptr(codes), _ptr(WS), M, N, K,
                                   n0, n1, _ptr(y), _ptr(A)), "matmul")
    return y[:, n0:n1].copy(), A[:, n0:n1].copy()


def matmul_entries(qp, S, codes, ws_f16, ms, ns):
    """y, A at the listed (m, n) pairs only (float64 [len])."""
    qp = np.ascontiguousarray(qp, dtype=np.int8)
    S = np.ascontiguousarray(S, dtype=np.float32)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    WS = _ws64(ws_f16)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    M, K = qp.shape
    N = codes.shape[0]
    y = np.empty(len(ms), dtype=np.float64)
    A = np.empty(len(ms), dtype=np.float64)
    _check(_lib().pq2o_matmul_entries(_ptr(qp), _ptr(S), _ptr(codes), _ptr(WS), M, N, K,
                                      len(ms), _ptr(ms), _ptr(ns), _ptr(y), _ptr(A)),
           "matmul_entries")
    return y, A


def fp32_tolerance(ref, A, G):
    """Allowed |y - ref| for an fp32 kernel result: 1e-3 relative to the
    float64 reference, plus the fp32 rounding bound gamma_{G+2} * A, where
    A = sum_g |dot_g * s * ws| and gamma_n = n*u/(1-n*u), u = 2^-24 (the
    classical bound for n roundings in any summation order).  The second term
    only matters where cancellation makes |ref| small against A."""
    u = 2.0 ** -24
    n = G + 2
    gamma = n * u / (1.0 - n * u)
    return 1e-3 * np.abs(ref) + gamma * A


def exp_f32(x: np.ndarray) -> np.ndarray:
    """The oracle's fp32 exp (Cody-Waite reduction + Taylor polynomial)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    _check(_lib().pq2o_exp(_ptr(x), x.size, _ptr(y)), "exp")
    return y


FP16_MAX = 65504.0


def swiglu(gu: np.ndarray) -> np.ndarray:
    """h = fp16(silu(gate) * up) of a gate/up output gu float32 [M, 2I]
    (gate = first half, up = second half).  The fp32 product is clamped to
    +-65504 and rounded to fp16 (IEEE round-half-even, numpy's conversion),
    i.e. fp16 conversion that saturates instead of overflowing."""
    gu = np.ascontiguousarray(gu, dtype=np.float32)
    M, I2 = gu.shape
    if I2 % 2:
        raise ValueError("gu must have an even number of columns")
    I = I2 // 2
    h = np.empty((M, I), dtype=np.float32)
    _check(_lib().pq2o_swiglu(_ptr(gu), M, I, _ptr(h)), "swiglu")
    return np.clip(h, -FP16_MAX, FP16_MAX).astype(np.float16)


# ---------------------------------------------------------------------------
# The pages' second, unquantised workload: a small bf16 projection
# (in_proj_ba, N = 96, K = 5120) computed as a split-K GEMM whose fp32 partial
# sums are reduced in the fixed order 0, 1, 2, ... and rounded once to bf16
# ("Making a ternary reasoning model fast in vLLM", page "From CUDA to Triton
# and Gluon", section "Speed up a small unquantised projection").  The result
# has a plain definition: y = bf16(x @ w^T); the oracle is that definition in
# float64 (numpy's matmul as the primitive) and the kernels' fp32 summation
# order is covered by bf16_gemm_tolerance.
# ---------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 values stored as uint16 bit patterns -> float64 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(v: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, rounded once to nearest, ties to even
    (bf16 keeps 8 significant bits).  Domain: zero and finite values whose
    magnitude lies in the normal bf16 range [2^-126, 2^128); the rounded
    value is exact in float32, whose upper 16 bits are the bf16 pattern."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                       # v = m * 2^e, 0.5 <= |m| < 1
    r = np.ldexp(np.round(m * 256.0) / 256.0, e)   # np.round: half to even
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def gemm_bf16(x_bits: np.ndarray, w_bits: np.ndarray):
    """x [M, K], w [N, K] as bf16 bit patterns -> (ref float64 [M, N],
    A = sum |x w| float64 [M, N]).  ref is the exact product sum (float64 is
    exact here: every bf16 x bf16 product has at most 16 significant bits and
    K <= 2^20 terms keep the sum well inside the 53-bit mantissa for the
    magnitudes the tests use)."""
    x = bf16_to_f64(x_bits)
    w = bf16_to_f64(w_bits)
    return x @ w.T, np.abs(x) @ np.abs(w).T


def bf16_gemm_tolerance(ref, A, K):
    """|y - ref| bound for y = bf16(fp32 sum of the K products in any order):
    the fp32 summation error gamma_K * A plus one bf16 rounding of the result
    (half a bf16 ulp, 2^-9 relative, of a value within gamma_K * A of ref)."""
    gam = K * 2.0 ** -24 / (1 - K * 2.0 ** -24)
    return 2.0 ** -8 * (np.abs(ref) + gam * A) + gam * A + 1e-30
