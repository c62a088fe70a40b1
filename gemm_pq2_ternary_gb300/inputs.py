"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers: it holds none of the matmul's
arithmetic (no packing, no quantisation, no plane order).  Both the CUDA path
(tests, benchmark) and the CPU oracle (tests) take their inputs from here.

Draw order per problem: ternary weights (as values in {-1,0,+1}), then the
fp16 group scales, then the fp16 activations -- one numpy PCG64 stream per
problem, seeded explicitly.

Distributions (the shapes and value ranges of the workloads the pages
measure; the pages' captured activations are not available, these stand in
for them):
  codes "uniform"  code in {0,1,2} uniform       (ternary -1/0/+1 equally)
  codes "p343"     P(code=0,1,2) = 0.3, 0.4, 0.3
  ws               U[0.01, 0.05], rounded to fp16
  x "normal"       N(0,1), rounded to fp16
  x "outliers"     N(0,1) with each element multiplied by 20 with
                   probability 0.01, rounded to fp16
"""
from dataclasses import dataclass

import numpy as np

_ROW_CHUNK = 1024  # rows drawn per batch (bounds host memory for big N*K)


@dataclass(frozen=True)
class Problem:
    """One synthetic matmul problem: y[M,N] = x[M,K] * W[N,K]^T."""
    name: str
    M: int
    K: int
    N: int
    codes: str = "uniform"     # "uniform" | "p343"
    x: str = "normal"          # "normal" | "outliers"
    seed: int = 0


def draw_ternary(rng: np.random.Generator, N: int, K: int, dist: str) -> np.ndarray:
    out = np.empty((N, K), dtype=np.int8)
    for r0 in range(0, N, _ROW_CHUNK):
        r1 = min(N, r0 + _ROW_CHUNK)
        if dist == "uniform":
            c = rng.integers(0, 3, size=(r1 - r0, K), dtype=np.int8)
        elif dist == "p343":
            u = rng.random(size=(r1 - r0, K), dtype=np.float32)
            c = (u >= 0.3).astype(np.int8) + (u >= 0.7).astype(np.int8)
        else:
            raise ValueError(dist)
        out[r0:r1] = c - 1
    return out


def draw_ws(rng: np.random.Generator, N: int, K: int) -> np.ndarray:
    return rng.uniform(0.01, 0.05, size=(N, K // 128)).astype(np.float16)


def draw_x(rng: np.random.Generator, M: int, K: int, dist: str) -> np.ndarray:
    x = rng.standard_normal(size=(M, K), dtype=np.float32)
    if dist == "outliers":
        mask = rng.random(size=(M, K), dtype=np.float32) < 0.01
        x = np.where(mask, x * 20.0, x)
    elif dist != "normal":
        raise ValueError(dist)
    return x.astype(np.float16)


def generate(p: Problem):
    """-> (tern int8 [N,K] in {-1,0,1}, ws fp16 [N,K/128], x fp16 [M,K])."""
    rng = np.random.default_rng(p.seed)
    tern = draw_ternary(rng, p.N, p.K, p.codes)
    ws = draw_ws(rng, p.N, p.K)
    x = draw_x(rng, p.M, p.K, p.x)
    return tern, ws, x


def generate_x(M: int, K: int, dist: str = "normal", seed: int = 0) -> np.ndarray:
    """Activations alone (e.g. the MLP pair's synthetic intermediate h)."""
    return draw_x(np.random.default_rng(seed), M, K, dist)


# The five workloads (sizes as the pages' projections: o_proj 5120x6144,
# gate/up 5120 -> 2x17408, down 17408 -> 5120).
PR1 = Problem("pr1_gemv_k1024_n256", 1, 1024, 256, "uniform", "normal", 0)
DECODE = Problem("decode_gemv_k6144_n5120", 1, 6144, 5120, "p343", "outliers", 1)


def small_batch(M: int, K: int, N: int) -> Problem:
    return Problem(f"small_m{M}_k{K}_n{N}", M, K, N, "p343", "outliers", 2)


SMALL_SHAPES = [(6144, 5120), (5120, 17408)]
SMALL_MS = [2, 4, 8, 16]


def mlp_gate_up(M: int) -> Problem:
    return Problem(f"mlp_gateup_m{M}", M, 5120, 2 * 17408, "uniform", "normal", 3)


def mlp_down(M: int) -> Problem:
    return Problem(f"mlp_down_m{M}", M, 17408, 5120, "uniform", "normal", 3)


def prefill(M: int) -> Problem:
    return Problem(f"prefill_m{M}", M, 5120, 17408, "uniform", "normal", 4)


# ---------------------------------------------------------------------------
# Device-side draws for the benchmark's many distinct weight sets (too large
# to draw on the host every run).  Same distributions, torch's seeded
# generator; values are compared to the oracle on sampled outputs.
# ---------------------------------------------------------------------------
def draw_ternary_torch(N: int, K: int, dist: str, gen, device):
    import torch
    if dist == "uniform":
        c = torch.randint(0, 3, (N, K), generator=gen, device=device, dtype=torch.int8)
    elif dist == "p343":
        u = torch.rand((N, K), generator=gen, device=device)
        c = (u >= 0.3).to(torch.int8) + (u >= 0.7).to(torch.int8)
    else:
        raise ValueError(dist)
    return c - 1


def draw_ws_torch(N: int, K: int, gen, device):
    import torch
    u = torch.rand((N, K // 128), generator=gen, device=device)
    return (0.01 + 0.04 * u).to(torch.float16)


def draw_x_torch(M: int, K: int, dist: str, gen, device):
    import torch
    x = torch.randn((M, K), generator=gen, device=device)
    if dist == "outliers":
        mask = torch.rand((M, K), generator=gen, device=device) < 0.01
        x = torch.where(mask, x * 20.0, x)
    return x.to(torch.float16)


# ---------------------------------------------------------------------------
# The unquantised bf16 projection (in_proj_ba: 96 output rows, K = 5120, a
# few decode tokens).  Values are float32 draws with the lower 16 bits of
# each dropped, so every value is a bf16 pattern; the arrays hold those
# patterns as uint16.
#   x "normal"    N(0, 1)             (hidden states after the norm)
#   x "integer"   integers in [-4, 4] (exact-arithmetic cases)
#   w "normal"    N(0, 0.02^2)        (a projection's initial scale)
#   w "integer"   integers in [-4, 4]
# Draw order: w, then x, from one PCG64 stream seeded explicitly.
# ---------------------------------------------------------------------------
def _bf16_bits(v: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(v, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _draw_bf16(rng: np.random.Generator, shape, dist: str, sigma: float) -> np.ndarray:
    if dist == "normal":
        return _bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma))
    if dist == "integer":
        return _bf16_bits(rng.integers(-4, 5, size=shape).astype(np.float32))
    raise ValueError(dist)


def generate_bf16(M: int, N: int, K: int, seed: int, x: str = "normal", w: str = "normal"):
    """-> (x_bits [M, K], w_bits [N, K]) uint16."""
    rng = np.random.default_rng(seed)
    wb = _draw_bf16(rng, (N, K), w, 0.02)
    xb = _draw_bf16(rng, (M, K), x, 1.0)
    return xb, wb


def draw_bf16_torch(shape, sigma: float, gen, device):
    """bf16 tensor on `device`: N(0, sigma^2) float32 draws (torch's seeded
    generator) with the lower 16 bits of each dropped."""
    import torch
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * sigma
    return (v.view(torch.int32) >> 16).to(torch.int16).view(torch.bfloat16)
