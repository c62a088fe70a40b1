"""Pins for the CPU oracle, against facts fixed by the pages and by
mathematics rather than by the oracle itself.

Each test names what pins it:
  * the worked lookup example of "Chasing llama.cpp at batch one",
    section "Recover four weights with one lookup" (tests/golden/);
  * the plane-order statement of "From CUDA to Triton and Gluon",
    section "One token at a time" (tests/golden/) and one-hot cases;
  * the identity dot(codes,q) - sum(q) = sum((code-1)*q) of the same section;
  * special cases (all codes 0 / 1 / 2), brute force in pure Python on tiny
    inputs, the integer matmul (numpy int64 @) with unit scales;
  * the word/plane formulation the same section prints for the M=1 kernel,
    re-expressed with numpy bit operations (an independent route to y);
  * exact quantisation cases (scales that are powers of two times 127,
    half-way ties, zero groups) and the rounding invariant.
"""
import os

import numpy as np
import pytest

import oracle
from gemm_pq2_ternary_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------------
# code map
# --------------------------------------------------------------------------
def test_lookup_worked_example():
    g = {r[0]: r[1:] for r in _read_golden("prmt_worked_example.txt")}
    lut = int(g["lut"][0], 16)
    codes = [int(c) for c in g["codes"]]
    selector = int(g["selector"][0], 16)
    want_bytes = [int(b, 16) for b in g["bytes"]]
    weights = [int(w) for w in g["weights"]]
    # the selector the page builds: one code per nibble
    assert sum(c << (4 * i) for i, c in enumerate(codes)) == selector
    # byte-select semantics on the lookup constant
    lut_bytes = [(lut >> (8 * i)) & 0xFF for i in range(4)]
    got = [lut_bytes[(selector >> (4 * i)) & 0xF] for i in range(4)]
    assert got == want_bytes
    assert [b - 256 if b >= 128 else b for b in got] == weights
    # the oracle's packing puts these codes in one byte and decodes them back
    t = np.array([weights], dtype=np.int8)
    packed = oracle.pack(t)
    assert packed.shape == (1, 1)
    assert [(int(packed[0, 0]) >> (2 * s)) & 3 for s in range(4)] == codes
    assert oracle.unpack(packed, 4).tolist() == [weights]


def test_pack_roundtrip_and_layout():
    rng = np.random.default_rng(5)
    t = rng.integers(-1, 2, size=(7, 256), dtype=np.int8)
    c = oracle.pack(t)
    assert c.shape == (7, 64)
    # weight k of row n in byte k>>2 at bits 2*(k&3)
    for n in range(7):
        for k in range(256):
            assert ((int(c[n, k >> 2]) >> (2 * (k & 3))) & 3) - 1 == t[n, k]
    assert np.array_equal(oracle.unpack(c, 256), t)


def test_pack_rejects_non_ternary():
    t = np.zeros((1, 128), dtype=np.int8)
    t[0, 3] = 2
    with pytest.raises(ValueError):
        oracle.pack(t)


# --------------------------------------------------------------------------
# plane order
# --------------------------------------------------------------------------
def test_plane_order_golden_positions():
    K = 256
    for k, byte, s, pos in (map(int, r) for r in _read_golden("plane_order_positions.txt")):
        assert byte == k >> 2 and s == k & 3
        q = np.zeros((1, K), dtype=np.int8)
        q[0, k] = 7
        qp = oracle.plane_order(q)
        assert np.flatnonzero(qp[0]).tolist() == [pos]
        assert np.array_equal(oracle.natural_order(qp), q)


def test_one_hot_weight_selects_its_activation():
    # Only weight k of the row is +1 (code 2), all others 0 (code 1); then the
    # group dot is exactly q_k and y = q_k * s * ws.
    K = 256
    rng = np.random.default_rng(11)
    x = rng.standard_normal((1, K)).astype(np.float16)
    q, S, T = oracle.quantize(x)
    qp = oracle.plane_order(q)
    ws = np.full((1, K // 128), 0.03125, dtype=np.float16)
    for k in range(K):
        t = np.zeros((1, K), dtype=np.int8)
        t[0, k] = 1
        codes = oracle.pack(t)
        dots = oracle.group_dots(qp, codes)
        g = k // 128
        want = np.zeros(K // 128, dtype=np.int32)
        want[g] = q[0, k]
        assert np.array_equal(dots[0, 0], want)
        y, _ = oracle.matmul(qp, S, codes, ws)
        assert y[0, 0] == float(q[0, k]) * float(S[0, g]) * 0.03125


# --------------------------------------------------------------------------
# identity and special cases
# --------------------------------------------------------------------------
def test_offset_identity_random():
    p = inputs.Problem("t", 3, 384, 9, "uniform", "outliers", 21)
    tern, ws, x = inputs.generate(p)
    qp, S, T = oracle.quantize_act(x)
    codes = oracle.pack(tern)
    d_codes = oracle.codes_dots(qp, codes).astype(np.int64)
    d = oracle.group_dots(qp, codes).astype(np.int64)
    assert np.array_equal(d_codes - T.astype(np.int64)[:, None, :], d)


@pytest.mark.parametrize("code,sign", [(0, -1), (1, 0), (2, 1)])
def test_constant_codes(code, sign):
    M, K, N = 2, 512, 3
    rng = np.random.default_rng(3)
    x = rng.standard_normal((M, K)).astype(np.float16)
    qp, S, T = oracle.quantize_act(x)
    codes = np.full((N, K // 4), sum(code << (2 * s) for s in range(4)), dtype=np.uint8)
    d = oracle.group_dots(qp, codes)
    assert np.array_equal(d, np.broadcast_to(sign * T[:, None, :], d.shape))
    ws = rng.uniform(0.01, 0.05, size=(N, K // 128)).astype(np.float16)
    y, _ = oracle.matmul(qp, S, codes, ws)
    want = sign * np.einsum("mg,mg,ng->mn", T.astype(np.float64), S.astype(np.float64),
                            ws.astype(np.float64))
    if sign == 0:
        assert np.all(y == 0.0)
    else:
        np.testing.assert_allclose(y, want, rtol=1e-13, atol=0)


def test_brute_force_tiny():
    # pure-Python loops over natural-order q and ternary t
    for (M, K, N, seed) in [(1, 128, 1, 0), (2, 128, 5, 1), (3, 256, 4, 2), (1, 256, 5, 3)]:
        p = inputs.Problem("bf", M, K, N, "uniform", "outliers", seed)
        tern, ws, x = inputs.generate(p)
        q, S, T = oracle.quantize(x)
        qp = oracle.plane_order(q)
        codes = oracle.pack(tern)
        dots = oracle.group_dots(qp, codes)
        y, A = oracle.matmul(qp, S, codes, ws)
        G = K // 128
        for m in range(M):
            for n in range(N):
                tot = 0.0
                mag = 0.0
                for g in range(G):
                    d = 0
                    for k in range(g * 128, (g + 1) * 128):
                        d += int(tern[n, k]) * int(q[m, k])
                    assert dots[m, n, g] == d
                    term = d * float(S[m, g]) * float(ws[n, g])
                    tot += term
                    mag += abs(term)
                assert abs(y[m, n] - tot) <= 1e-12 * max(mag, 1e-300)
                assert abs(A[m, n] - mag) <= 1e-12 * max(mag, 1e-300)


def test_unit_scales_is_integer_matmul():
    rng = np.random.default_rng(8)
    M, K, N = 4, 640, 13
    q = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
    t = rng.integers(-1, 2, size=(N, K), dtype=np.int8)
    qp = oracle.plane_order(q)
    codes = oracle.pack(t)
    S = np.ones((M, K // 128), dtype=np.float32)
    ws = np.ones((N, K // 128), dtype=np.float16)
    y, A = oracle.matmul(qp, S, codes, ws)
    ref = q.astype(np.int64) @ t.astype(np.int64).T
    assert np.array_equal(y, ref.astype(np.float64))


def test_entries_match_full():
    p = inputs.Problem("e", 3, 384, 17, "p343", "outliers", 4)
    tern, ws, x = inputs.generate(p)
    qp, S, T = oracle.quantize_act(x)
    codes = oracle.pack(tern)
    y, A = oracle.matmul(qp, S, codes, ws)
    ms = np.array([0, 2, 1, 2])
    ns = np.array([0, 16, 5, 3])
    ye, Ae = oracle.matmul_entries(qp, S, codes, ws, ms, ns)
    assert np.array_equal(ye, y[ms, ns]) and np.array_equal(Ae, A[ms, ns])
    yr, Ar = oracle.matmul(qp, S, codes, ws, rows=(5, 12))
    assert np.array_equal(yr, y[:, 5:12])


# --------------------------------------------------------------------------
# the page's word/plane formulation (independent route to the same y)
# --------------------------------------------------------------------------
def _plane_word_route(qp, S, T, codes, ws):
    """y from 32-bit code words: plane s of word j is (w >> 2s) & 0x03030303,
    four codes aligned with activation bytes s*32 + 4j .. s*32 + 4j + 3 of the
    group; the group's codes-dot minus T, times s, times ws."""
    M, K = qp.shape
    N = codes.shape[0]
    G = K // 128
    w = codes.view("<u4").reshape(N, G, 8).astype(np.int64)
    qb = qp.reshape(M, G, 4, 32).astype(np.int64)      # [m, g, plane, byte]
    y = np.zeros((M, N))
    for s in range(4):
        plane = (w >> (2 * s)) & 0x03030303             # [n, g, j]
        for b in range(4):
            c = (plane >> (8 * b)) & 0xFF               # code of byte 4j+b
            for j in range(8):
                # activation byte s*32 + 4j + b
                y_part = np.einsum("ng,mg->mng", c[:, :, j], qb[:, :, s, 4 * j + b])
                if s == 0 and b == 0 and j == 0:
                    acc = y_part
                else:
                    acc = acc + y_part
    dot = acc - T.astype(np.int64)[:, None, :]
    return np.einsum("mng,mg,ng->mn", dot.astype(np.float64), S.astype(np.float64),
                     ws.astype(np.float64))


def test_word_plane_formulation_agrees():
    for prob in [inputs.Problem("w", 2, 512, 11, "p343", "outliers", 9),
                 inputs.Problem("w2", 1, 1024, 6, "uniform", "normal", 0)]:
        tern, ws, x = inputs.generate(prob)
        qp, S, T = oracle.quantize_act(x)
        codes = oracle.pack(tern)
        y, A = oracle.matmul(qp, S, codes, ws)
        y2 = _plane_word_route(qp, S, T, codes, ws)
        assert np.all(np.abs(y - y2) <= 1e-12 * A + 1e-300)


# --------------------------------------------------------------------------
# quantisation
# --------------------------------------------------------------------------
def test_quant_exact_scale_and_ties():
    # amax = 127 * 2^-3 makes d = 2^-3 exact; x = (k + 1/2) d are exact ties
    d = 0.125
    vals = [127 * d, 0.5 * d, 1.5 * d, 2.5 * d, -0.5 * d, -1.5 * d, -2.5 * d, 3 * d, -127 * d]
    x = np.zeros((1, 128), dtype=np.float16)
    x[0, :len(vals)] = vals
    q, S, T = oracle.quantize(x)
    assert S[0, 0] == np.float32(d)
    want = [127, 0, 2, 2, 0, -2, -2, 3, -127]       # round half to even
    assert q[0, :len(vals)].tolist() == want
    assert np.all(q[0, len(vals):] == 0)
    assert T[0, 0] == sum(want)


def test_quant_zero_group_and_sums():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 384)).astype(np.float16)
    x[1, 128:256] = 0
    q, S, T = oracle.quantize(x)
    assert S[1, 1] == 0 and T[1, 1] == 0 and np.all(q[1, 128:256] == 0)
    assert np.array_equal(T, q.reshape(3, 3, 128).sum(-1, dtype=np.int64).astype(np.int32))


def test_quant_invariants_random():
    x = inputs.generate_x(16, 1024, "outliers", seed=6)
    q, S, T = oracle.quantize(x)
    xf = x.astype(np.float64).reshape(16, 8, 128)
    qf = q.astype(np.float64).reshape(16, 8, 128)
    amax = np.abs(xf).max(-1)
    d = S.astype(np.float64)
    # S is the fp32 rounding of amax / 127
    assert np.array_equal(S, (amax / 127.0).astype(np.float32))
    # the amax element maps to +-127
    idx = np.abs(xf).argmax(-1)
    top = np.take_along_axis(qf, idx[..., None], -1)[..., 0]
    top_sign = np.sign(np.take_along_axis(xf, idx[..., None], -1)[..., 0])
    assert np.array_equal(top, 127 * top_sign)
    # rounding error at most half a step, plus the fp32 rounding of the
    # quotient x/d (relative 2^-24 of |x/d|, i.e. 2^-24 |x| after scaling)
    err = np.abs(xf - qf * d[..., None])
    assert np.all(err <= 0.5 * d[..., None] + np.abs(xf) * 2.0 ** -23)
    assert np.all(np.abs(qf) <= 127)
