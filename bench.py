"""Benchmark of the PQ2_0 ternary matmul hot path on GB300.

One JSON line (rank 0).  The default run measures the decode GEMV (the
headline) and then every configuration of SUITE with shorter timing, each
with its own roofline, clocks, end-to-end figure, oracle sample and accuracy,
in the line's `configs` list.  A step is one pass of the hot path over one
batch of synthetic input: for each of R distinct projections (distinct weight sets, so
the step's weights exceed 4x L2 and come from HBM), quantise its fp16
activations (pq2_quantize_act) and run its matmul (pq2_gemv for M = 1,
pq2_gemm_small for M <= 16, pq2_gemm_prefill above).  The R projections are
captured once in a CUDA graph and replayed; times are CUDA events on the
replay stream.

Workloads (--workload):
  decode   M=1, K=6144 -> N=5120 (default; the o_proj-shaped decode GEMV)
  pr1      M=1, K=1024 -> N=256
  small    M=--m (2..16), --shape K,N (6144,5120 or 5120,17408)
  mlp      M=--m (1 or 16): gate/up 5120 -> 34816, quantise the synthetic
           intermediate h, down 17408 -> 5120
  prefill  M=--m (128 or 4096), 5120 -> 17408
  mid      M=--m (17..64), --shape K,N (5120,17408 by default) through
           pq2_gemm_prefill, in GB/s
  lmhead   M=1, K=5120 -> N=248320 (an lm_head-scale decode GEMV)
  mlp_swiglu  M=--m: gate/up 5120 -> 34816, then the down projection straight
           from its output (pq2_mlp_down_swiglu: SwiGLU + quantise, 17408 -> 5120)
  in_proj_ba  M=--m (1..16): the unquantised bf16 projection 5120 -> 96
           (pq2_gemm_bf16_splitk)

--impl reference runs the CPU oracle (the method's plain definition) on the
host cores on a bounded sample of the same workload, as the baseline arm.
"""
import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0
# nominal GB300 figures (context beside the measured peaks): HBM3e ~8 TB/s,
# dense bf16 2.25 PFLOP/s
HBM_NOMINAL_GBS = 8000.0
BF16_NOMINAL_TFLOPS = 2250.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs", HBM_FALLBACK_GBS), d.get("bf16_tflops", BF16_FALLBACK_TFLOPS), \
            d.get("bf16_tflops_sustained", None), "measured"
    return HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, None, "fallback"


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def gemm_bytes(M, N, K):
    """Algorithmic bytes of one matmul call (each byte once): codes, weight
    scales, quantised activations, S and T, fp32 output.  For M = 1 the step
    runs the fused quantise + GEMV kernel, whose inputs are the fp16
    activations instead of the quantised ones."""
    G = K // 128
    if M == 1:
        return N * K // 4 + 2 * N * G + 2 * K + 4 * N
    return N * K // 4 + 2 * N * G + M * K + 8 * M * G + 4 * M * N


def bf16_bytes(M, N, K):
    """Algorithmic bytes of one bf16 projection: w, x and the bf16 y, once
    each."""
    return 2 * (N * K + M * K + M * N)


def is_bf16(proj):
    return proj[3] == "bf16"


def weight_bytes(proj):
    M, K, N = proj[:3]
    return 2 * N * K if is_bf16(proj) else N * K // 4 + 2 * N * (K // 128)


def swiglu_down_bytes(M, N, I):
    """Algorithmic bytes of pq2_mlp_down_swiglu: codes, weight scales, the fp32
    gate/up input [M, 2I] and the fp32 output (the quantised h stays inside)."""
    return N * I // 4 + 2 * N * (I // 128) + 8 * M * I + 4 * M * N


# Workloads whose projection `dst` reads the output of projection `src` of
# the same layer through pq2_mlp_down_swiglu (SwiGLU + quantise + matmul).
SWIGLU_CHAINS = {"mlp_swiglu": (0, 1)}


def chain_of(name):
    for prefix, pair in SWIGLU_CHAINS.items():
        if name.startswith(prefix + "_m"):
            return pair
    return None


def quant_bytes(M, K):
    return 2 * M * K + M * K + 8 * M * (K // 128)


def workload_spec(args):
    """-> (name, list of (M, K, N, code_dist, x_dist) per projection in a
    layer, metric kind)"""
    w = args.workload
    if w == "decode":
        return "decode_gemv_m1_k6144_n5120", [(1, 6144, 5120, "p343", "outliers")], "GB/s"
    if w == "pr1":
        return "pr1_gemv_m1_k1024_n256", [(1, 1024, 256, "uniform", "normal")], "GB/s"
    if w == "small":
        K, N = (int(v) for v in args.shape.split(","))
        return f"small_m{args.m}_k{K}_n{N}", [(args.m, K, N, "p343", "outliers")], "GB/s"
    if w == "mid":
        if not 16 < args.m <= 64:
            raise SystemExit("--workload mid takes 17 <= --m <= 64")
        K, N = (int(v) for v in (args.shape or "5120,17408").split(","))
        return f"mid_m{args.m}_k{K}_n{N}", [(args.m, K, N, "p343", "outliers")], "GB/s"
    if w == "mlp":
        return f"mlp_pair_m{args.m}", [(args.m, 5120, 34816, "uniform", "normal"),
                                       (args.m, 17408, 5120, "uniform", "normal")], "GB/s"
    if w == "mlp_swiglu":
        # the down projection reads the gate/up output (SWIGLU_CHAINS)
        return f"mlp_swiglu_m{args.m}", [(args.m, 5120, 34816, "uniform", "normal"),
                                         (args.m, 17408, 5120, "uniform", "normal")], "GB/s"
    if w == "lmhead":
        return "lmhead_gemv_m1_k5120_n248320", [(1, 5120, 248320, "uniform", "normal")], "GB/s"
    if w == "in_proj_ba":
        return f"in_proj_ba_bf16_m{args.m}_k5120_n96", [(args.m, 5120, 96, "bf16", "normal")], \
            "GB/s"
    if w == "prefill":
        return f"prefill_m{args.m}_k5120_n17408", [(args.m, 5120, 17408, "uniform", "normal")], \
            "TOPS"
    raise SystemExit(f"unknown workload {w}")


# Sources whose compiled code a workload's dominant kernel comes from; the
# DRAM traffic recorded in profiles/dram_traffic.txt is used only while their
# hash matches the one recorded with it.
KERNEL_SOURCES = {
    "gemv": ["pq2_gemv.cu", "pq2_common.cuh"],
    "small": ["pq2_small.cu", "pq2_tokens.cuh", "pq2_common.cuh"],
    "tile": ["pq2_tile.cu", "pq2_tokens.cuh", "pq2_common.cuh"],
    "wtile": ["pq2_wtile.cu", "pq2_tokens.cuh", "pq2_common.cuh"],
    "prefill": ["pq2_prefill.cu", "pq2_tokens.cuh", "pq2_common.cuh"],
    "bf16": ["pq2_bf16.cu", "pq2_common.cuh"],
    "multi": ["pq2_multi.cu", "pq2_common.cuh"],
}


def small_takes_dp4a(M, N, K, num_sms=152):
    """The library's routing of pq2_gemm_small (gemv_multi_supported in
    csrc/pq2_multi.cu): 2-4 tokens on the DP4A kernel where a CTA's terms fit
    its shared memory."""
    if M < 2 or M > 4:
        return False
    mt = 2 if M <= 2 else (4 if M <= 4 else 8)
    G = K // 128
    rows = (N + num_sms - 1) // num_sms
    return G * mt <= 480 and rows * mt * G * 4 <= 160 * 1024


def prefill_takes_wtile(M, N, K, num_sms=152):
    """The library's routing of pq2_gemm_prefill (wtile_default in
    csrc/pq2_wtile.cu): 33-64 tokens on the weights-wide token-tile kernel
    when a CTA gets at most 4 items of 128 weight rows x 4 groups."""
    if M <= 32 or M > 64:
        return False
    items = ((N + 127) // 128) * ((K // 128 + 3) // 4)
    return items <= 4 * min(num_sms, 256)


def kernel_family(layer):
    if is_bf16(layer[0]):
        return "bf16"
    M, K, N = layer[0][:3]
    if small_takes_dp4a(M, N, K):
        return "multi"
    if M == 1:
        return "gemv"
    # the library's routing: small_kernel to 16 tokens, the token-tile kernel
    # to 32 (pq2_gemm_prefill), then the weights-wide token-tile kernel where
    # a CTA gets few items, else the 128-row tile kernels
    if M <= 16:
        return "small"
    if M <= 32:
        return "tile"
    return "wtile" if prefill_takes_wtile(M, N, K) else "prefill"


def sources_hash(family):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, "gemm_pq2_ternary_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, family):
    """DRAM bytes per launch of the dominant kernel from one ncu capture
    (profiles/dram_traffic.txt: workload, kernel family, sources hash, bytes),
    or None when absent or when the kernel's sources changed since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = sources_hash(family)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == workload \
                    and parts[1] == family and parts[2] == want:
                return int(parts[3])
    return None


def per_layer_units(layer, kind, name=""):
    """Algorithmic bytes (GB/s workloads) or int8-equivalent ops (TOPS) of one
    layer."""
    if kind == "TOPS":
        return sum(2.0 * M * N * K for (M, K, N, _, _) in layer)
    chain = chain_of(name)
    total = 0.0
    for j, (M, K, N, cdist, _) in enumerate(layer):
        if cdist == "bf16":
            total += bf16_bytes(M, N, K)
        elif chain and j == chain[1]:
            total += swiglu_down_bytes(M, N, K)
        else:
            total += gemm_bytes(M, N, K)
    return total


def layer_launches(layer, name=""):
    """Kernel launches of one layer (pq2_matmul_ex per projection): the fused
    quantise + GEMV for M = 1; quantise and the DP4A matmul for 2-4 tokens;
    quantise-into-token-tiles and the token-tile matmul wherever a token-tile
    kernel takes the call (up to 16 tokens, and 17-64 on tile_kernel or
    wtile_kernel); quantise, token preparation and matmul for the 128-token
    kernels; SwiGLU-quantise and the matmul (plus its preparation for M > 1)
    for a chained down projection; one split-K launch for a bf16 projection."""
    chain = chain_of(name)
    n = 0
    for j, (M, K, N, cdist, _) in enumerate(layer):
        if cdist == "bf16":
            n += 1
        elif chain and j == chain[1]:
            n += 2 if M == 1 or small_takes_dp4a(M, N, K) else 3
        elif M == 1:
            n += 1
        else:
            n += 2 if kernel_family([(M, K, N, cdist, None)]) in ("small", "multi", "tile", "wtile") \
                else 3
    return n


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
ACC_ROWS = 64       # output rows of the first projection compared with the oracle
ACC_TOKENS = 256    # at most this many token rows of it


def build_layers(args, layer, R, device, name=""):
    """R layers of distinct weight sets.  Each projection type j keeps its
    activations of all R layers in one tensor X[j] [R, M, K] and its outputs
    in Y[j] [R, M, N] (contiguous, so the end-to-end arm copies them in one
    transfer each).  Also returns a host copy of the inputs of layer 0's
    first projection, restricted to its first ACC_ROWS output rows and
    ACC_TOKENS token rows (drawn by torch's generator on the device, like
    every weight here), for the accuracy check against the oracle."""
    import torch
    from gemm_pq2_ternary_gb300 import binding as pq2
    from gemm_pq2_ternary_gb300 import inputs

    X = [torch.empty((R, M, K), dtype=torch.bfloat16 if c == "bf16" else torch.float16,
                     device=device) for (M, K, N, c, _) in layer]
    Y = [torch.empty((R, M, N), dtype=torch.bfloat16 if c == "bf16" else torch.float32,
                     device=device) for (M, K, N, c, _) in layer]
    layers = []
    sample = None
    for r in range(R):
        gen = torch.Generator(device=device)
        gen.manual_seed(1000 + r)
        projs = []
        for j, (M, K, N, cdist, xdist) in enumerate(layer):
            rows, toks = min(N, ACC_ROWS), min(M, ACC_TOKENS)
            if cdist == "bf16":
                w = inputs.draw_bf16_torch((N, K), 0.02, gen, device)
                X[j][r].copy_(inputs.draw_bf16_torch((M, K), 1.0, gen, device))
                projs.append(dict(M=M, K=K, N=N, bf16=True, w=w, x=X[j][r], y=Y[j][r]))
                if r == 0 and j == 0:
                    sample = dict(bf16=True, rows=rows, toks=toks,
                                  w=w[:rows].view(torch.int16).cpu().numpy().view("uint16"),
                                  x=X[j][r][:toks].view(torch.int16).cpu().numpy().view("uint16"))
                continue
            tern = inputs.draw_ternary_torch(N, K, cdist, gen, device)
            ws = inputs.draw_ws_torch(N, K, gen, device)
            codes, ws_p = pq2.pack(tern, ws)
            X[j][r].copy_(inputs.draw_x_torch(M, K, xdist, gen, device))
            if r == 0 and j == 0:
                sample = dict(bf16=False, rows=rows, toks=toks, K=K,
                              tern=tern[:rows].cpu().numpy(), ws=ws[:rows].cpu().numpy(),
                              x=X[j][r][:toks].cpu().numpy())
            del tern
            qp, S, T = pq2.alloc_act(M, K, device)
            op = pq2.PQ2_OP_GEMV if M == 1 else (pq2.PQ2_OP_SMALL if M <= 16 else pq2.PQ2_OP_PREFILL)
            wsp = pq2.alloc_workspace(op, M, N, K, device)
            mmws = pq2.alloc_workspace(pq2.PQ2_OP_MATMUL, M, N, K, device)
            projs.append(dict(M=M, K=K, N=N, codes=codes, ws=ws_p, x=X[j][r], qp=qp, S=S, T=T,
                              y=Y[j][r], op=op, wsp=wsp, mmws=mmws))
        chain = chain_of(name)
        if chain:
            src, dst = projs[chain[0]], projs[chain[1]]
            assert src["N"] == 2 * dst["K"] and src["M"] == dst["M"]
            dst["gu"] = src["y"]
            dst["swws"] = pq2.alloc_workspace(pq2.PQ2_OP_SWIGLU_DOWN, dst["M"], dst["N"],
                                              dst["K"], device)
        layers.append(projs)
    torch.cuda.synchronize()
    return layers, X, Y, sample


def weight_flags(pq2, args):
    """The step's weights are uploaded once and never written again, so the
    calls may declare them static (PQ2_WEIGHTS_STATIC: pq2_matmul_ex for M = 1,
    pq2_gemm_small_ex, pq2_gemm_bf16_splitk) unless --weights default."""
    return pq2.PQ2_WEIGHTS_STATIC if args.weights == "static" else 0


def run_matmul(pq2, p, flags=0):
    if p["op"] == pq2.PQ2_OP_GEMV:
        pq2.pq2_gemv(p["qp"], p["S"], p["T"], p["codes"], p["ws"], p["y"])
    elif p["op"] == pq2.PQ2_OP_SMALL:
        pq2.pq2_gemm_small_ex(p["qp"], p["S"], p["T"], p["codes"], p["ws"], p["y"], flags, p["wsp"])
    else:
        pq2.pq2_gemm_prefill(p["qp"], p["S"], p["T"], p["codes"], p["ws"], p["y"], p["wsp"])


def step_fn(pq2, layers, matmul_only=False, flags=0):
    """One pass: per projection, pq2_matmul_ex (the public call from fp16
    activations: the fused quantise + GEMV kernel for M = 1; for 5-16 tokens
    a kernel that quantises straight into the tensor-core kernel's token
    tiles, then that kernel; otherwise pq2_quantize_act, then the matmul);
    with matmul_only, the matmul entry point alone on activations quantised
    beforehand (its preparation kernel included)."""
    def fn():
        for projs in layers:
            for p in projs:
                if "bf16" in p:
                    pq2.pq2_gemm_bf16_splitk(p["x"], p["w"], p["y"], flags)
                    continue
                if "gu" in p:  # down projection from the gate/up output
                    pq2.pq2_mlp_down_swiglu(p["gu"], p["codes"], p["ws"], p["y"], p["swws"])
                    continue
                if p["M"] == 1 or not matmul_only:
                    pq2.pq2_matmul_ex(p["x"], p["codes"], p["ws"], p["y"], flags, p["mmws"])
                    continue
                run_matmul(pq2, p, flags)
    return fn


def capture(torch, fn, stream):
    with torch.cuda.stream(stream):
        fn()  # eager once (sets kernel attributes, warms caches)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


def timed_steps(torch, graph, reps, steps, stream):
    """`steps` steps of `reps` replays each, back to back on `stream`, with an
    event after each step (events do not synchronise).  Returns (total ms,
    per-step ms list)."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(steps):
            for _ in range(reps):
                graph.replay()
            ev[i + 1].record(stream)
    ev[-1].synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return ev[0].elapsed_time(ev[-1]), per


def timed_replays(torch, graph, n, stream):
    """Replays `graph` n times on `stream`; returns elapsed ms (CUDA events
    recorded on that stream)."""
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(n):
            graph.replay()
        t1.record(stream)
    t1.synchronize()
    return t0.elapsed_time(t1)


def max_over_ranks(x, dist, device):
    """The largest of every rank's x (the job's time is its slowest rank's);
    x itself with no process group.  Any backend: NCCL with device tensors
    on GPUs, gloo with CPU tensors."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank, world, seconds, scale):
    """Aggregate throughput: every rank processes units_per_rank in the same
    (max-over-ranks) time (weak scaling)."""
    return units_per_rank * world / seconds * scale


def metric_name(kind, name, layer):
    if is_bf16(layer[0]):
        return f"bf16 split-K projection {kind} ({name})"
    return f"ternary matmul {kind} ({name})"


def latency_floor(torch, pq2, layer, R, flags, stream, reps):
    """Per-launch time of a chain of empty kernels shaped like the fused
    M = 1 calls of the step (pq2_debug_gemv_floor), captured and replayed
    like the step: what a dependent chain of calls pays before any byte
    moves."""
    M, K, N = layer[0][:3]

    def fn():
        for _ in range(R):
            for (_, k, n, _, _) in layer:
                pq2.pq2_debug_gemv_floor(n, k, flags)
    g = capture(torch, fn, stream)
    timed_replays(torch, g, reps, stream)
    ms = timed_replays(torch, g, reps, stream)
    return ms * 1e3 / (reps * R * len(layer))


def tensor_probe(torch, pq2, device, stream, clk):
    """The measured issue rate of the tensor-core instruction the prefill
    kernels use (tcgen05 kind::f8f6f4, e4m3, M = 128, N = 256, K = 32, back
    to back on every SM: pq2_debug_mma_rate), as int8-equivalent TOPS at the
    SM clock sampled during the timed region (each int8 product is two e4m3
    products, hi and lo, so int8-equivalent operations per second equal e4m3
    multiply-adds per second)."""
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    cycles = torch.zeros(sms, dtype=torch.int64, device=device)
    iters = 4096
    with torch.cuda.stream(stream):
        for _ in range(2):
            pq2.pq2_debug_mma_rate(256, iters, cycles, stream)
    stream.synchronize()
    c = cycles.double().mean().item()
    mac_per_cycle = 128.0 * 256 * 32 * iters / c
    mhz = (clk or {}).get("sm_mhz") or 2070.0
    return {"instr": "tcgen05.mma kind::f8f6f4 e4m3 M=128 N=256 K=32, A in tensor memory",
            "mac_per_cycle_per_sm": round(mac_per_cycle, 1), "sms": sms, "sm_mhz": mhz,
            "int8eq_tops_at_clock": round(mac_per_cycle * sms * mhz * 1e6 * 1e-12, 1)}


def measure(args, wl, rank, world, dist, steps, warmup, target_ms, e2e_passes, floor):
    """Build R layers of the workload, capture the step graph, time `steps`
    steps of `reps` replays (after `warmup` untimed ones), then the dominant
    kernel alone, the latency floor (M = 1, if `floor`) and the end-to-end
    arm.  Returns (bench-line dict, accuracy sample, Y)."""
    import torch
    from gemm_pq2_ternary_gb300 import binding as pq2

    name, layer, kind = wl
    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    layer_weight_bytes = sum(weight_bytes(pr) for pr in layer)
    bf16_proj = is_bf16(layer[0])
    R = args.projections or max(1, math.ceil(4 * l2 / layer_weight_bytes))
    layers, X, Y, sample = build_layers(args, layer, R, device, name)

    stream = torch.cuda.Stream(device)
    flags = weight_flags(pq2, args)
    g_step = capture(torch, step_fn(pq2, layers, flags=flags), stream)
    g_mm = capture(torch, step_fn(pq2, layers, matmul_only=True, flags=flags), stream)
    assert pq2.pq2_last_device_error(stream) == pq2.PQ2_OK

    # A step replays the R-layer graph `reps` times, so that the timed region
    # lasts about target_ms over all steps (long enough for the clock sampler).
    timed_replays(torch, g_step, 3, stream)
    t_rep = timed_replays(torch, g_step, 3, stream) / 3
    reps = args.reps or max(1, math.ceil(target_ms / (steps * t_rep)))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    for _ in range(warmup):
        timed_replays(torch, g_step, reps, stream)
    barrier()
    clocks.start()
    time.sleep(0.25)  # let the sampler attach
    ms_total, per_step = timed_steps(torch, g_step, reps, steps, stream)
    barrier()
    clk = clocks.stop()
    ms_step = max_over_ranks(ms_total / steps, dist, device)

    # dominant kernel (the matmul) alone, same weight sets, for the roofline
    timed_replays(torch, g_mm, reps, stream)
    ms_mm = timed_replays(torch, g_mm, reps * steps, stream)
    mm_per_launch_ms = ms_mm / (reps * steps * R * len(layer))

    units_layer = per_layer_units(layer, kind, name)
    units_step = units_layer * R * reps
    scale = 1e-9 if kind == "GB/s" else 1e-12
    value = whole_job_value(units_step, world, ms_step * 1e-3, scale)

    hbm, bf16, bf16_sus, peak_src = load_peaks()
    per_launch = units_layer / len(layer)
    if kind == "GB/s":
        achieved = per_launch / (mm_per_launch_ms * 1e-3) * 1e-9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4),
                "frac_of_nominal": round(achieved / HBM_NOMINAL_GBS, 4),
                "traffic": recorded_traffic(name, kernel_family(layer)),
                "peak_source": f"{peak_src}: MEASURED_PEAKS.json hbm_gbs (copy)"}
    else:
        achieved = per_launch / (mm_per_launch_ms * 1e-3) * 1e-12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16, "unit": "TFLOP/s",
                "frac": round(achieved / bf16, 4),
                "frac_of_nominal": round(achieved / BF16_NOMINAL_TFLOPS, 4),
                "traffic": recorded_traffic(name, kernel_family(layer)),
                "peak_source": f"{peak_src}: MEASURED_PEAKS.json bf16_tflops (burst)"}

    if kind == "TOPS":
        roof["tensor_probe"] = tensor_probe(torch, pq2, device, stream, clk)
        roof["frac_of_probe"] = round(achieved / roof["tensor_probe"]["int8eq_tops_at_clock"], 4)

    floor_us = None
    if floor and all(M == 1 and not is_bf16(pr) for pr in layer for M in [pr[0]]):
        floor_us = latency_floor(torch, pq2, layer, R, flags, stream, reps)

    library = None
    if bf16_proj:
        library = library_baseline(torch, layers, stream, reps, steps, R * len(layer))

    e2e = None
    if e2e_passes and not args.no_e2e:
        e2e = e2e_arm(torch, pq2, layers, X, Y, flags, stream, kind, units_layer * R, world,
                      dist, device, name, e2e_passes)

    launches = steps * reps * R * layer_launches(layer, name)
    if bf16_proj:
        arith = "bf16 x bf16 products and fp32 sums on the CUDA cores, one rounding to bf16"
        graph = ("one CUDA graph per pass (per projection one pq2_gemm_bf16_splitk launch), "
                 "programmatic dependent launch")
    else:
        arith = "int8 activations x 2-bit ternary codes, int32 group dots, fp32 sums"
        graph = ("one CUDA graph per pass (per projection: fused quantise+GEMV "
                 "for M=1, quantise then matmul otherwise), programmatic dependent launch")
    out = {
        "metric": metric_name(kind, name, layer),
        "value": round(value, 2), "unit": kind, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if bf16_proj else "i8",
        "data": ("synthetic (seeded; bf16 weights and activations drawn on device)" if bf16_proj else
                 "synthetic (seeded; ternary codes, fp16 scales and activations drawn on device)"),
        "config": {"workload": name, "projections_per_pass": R * len(layer),
                   "passes_per_step": reps,
                   "shapes": [{"M": M, "K": K, "N": N} for (M, K, N, _, _) in layer],
                   "l2": (f"inputs larger than L2: {R * layer_weight_bytes / 1e6:.0f} MB of distinct "
                          f"weights per pass vs {l2 / 1e6:.0f} MB L2"
                          if R * layer_weight_bytes > l2 else
                          f"inputs SMALLER than L2 ({R * layer_weight_bytes / 1e6:.1f} MB of weights "
                          f"vs {l2 / 1e6:.0f} MB; --projections set: a profiling case, not a "
                          f"measurement)"),
                   "graph": graph,
                   "arith": arith,
                   "weights": ("static: M = 1, small-batch and bf16 calls pass PQ2_WEIGHTS_STATIC (weights "
                               "uploaded once; each call may read them before the preceding call "
                               "ends)"
                               if args.weights == "static" else "default ordering"),
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "matmul_us_per_launch": round(mm_per_launch_ms * 1e3, 3),
        **({"latency_floor_us": round(floor_us, 3),
            "latency_floor": ("per-launch time of a captured chain of empty kernels with the "
                              "same grid, block, shared memory and dependent-launch attributes "
                              "as the step's calls (pq2_debug_gemv_floor), same run")}
           if floor_us is not None else {}),
        "step_ms_spread": {"min": round(min(per_step), 4),
                           "median": round(float(np.median(per_step)), 4),
                           "max": round(max(per_step), 4), "rank": rank},
        **({"library_baseline": library} if library else {}),
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
    }
    if sample is not None:
        sample["y"] = Y[0][0][:sample["toks"], :sample["rows"]]
        if sample["bf16"]:
            sample["y"] = sample["y"].view(torch.int16).cpu().numpy().view("uint16")
        else:
            sample["y"] = sample["y"].cpu().numpy()
    del layers, X, Y, g_step, g_mm
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out, sample


def library_baseline(torch, layers, stream, reps, steps, calls_per_pass):
    """Context for the bf16 projection: the same calls through torch.matmul
    (cuBLAS) on the same weight sets, captured and replayed the same way."""
    def fn():
        for projs in layers:
            for p in projs:
                torch.matmul(p["x"], p["w"].t(), out=p["y"])
    g = capture(torch, fn, stream)
    timed_replays(torch, g, reps, stream)
    ms = timed_replays(torch, g, reps * steps, stream)
    return {"impl": "torch.matmul (cuBLAS), same graph of calls",
            "us_per_call": round(ms * 1e3 / (reps * steps * calls_per_pass), 3)}


def e2e_arm(torch, pq2, layers, X, Y, flags, stream, kind, units_pass, world, dist, device,
            name, passes):
    """The same metric through pq2_matmul_ex (the public call, eager) with host
    buffers: every pass copies all activations in from pinned host memory
    and all outputs back, inside the timed region (CUDA events on the
    stream).  In a SwiGLU chain the down projection's input is the gate/up
    output on the device, and only the down projection's output is read
    back."""
    chain = chain_of(name)
    if chain:
        X = [x for j, x in enumerate(X) if j != chain[1]]
        Y = [y for j, y in enumerate(Y) if j != chain[0]]
    Xh = [x.cpu().pin_memory() for x in X]
    Yh = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in Y]
    h2d = sum(x.numel() * x.element_size() for x in Xh)
    d2h = sum(y.numel() * y.element_size() for y in Yh)
    projs = [p for layer in layers for p in layer]

    def one_pass():
        for x, xh in zip(X, Xh):
            x.copy_(xh, non_blocking=True)
        for p in projs:
            if "bf16" in p:
                pq2.pq2_gemm_bf16_splitk(p["x"], p["w"], p["y"], flags, stream)
            elif "gu" in p:
                pq2.pq2_mlp_down_swiglu(p["gu"], p["codes"], p["ws"], p["y"], p["swws"], stream)
            else:
                pq2.pq2_matmul_ex(p["x"], p["codes"], p["ws"], p["y"], flags, p["mmws"], stream)
        for y, yh in zip(Y, Yh):
            yh.copy_(y, non_blocking=True)

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(2):
            one_pass()
        stream.synchronize()
        t0.record(stream)
        for _ in range(passes):
            one_pass()
        t1.record(stream)
    t1.synchronize()
    dt = max_over_ranks(t0.elapsed_time(t1) * 1e-3 / passes, dist, device)
    scale = 1e-9 if kind == "GB/s" else 1e-12
    return {"value": round(whole_job_value(units_pass, world, dt, scale), 2), "unit": kind,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(dt * 1e3, 4),
            "step": "one pass over all projections: copy in, the public call each "
                    "(pq2_matmul_ex, pq2_mlp_down_swiglu or pq2_gemm_bf16_splitk), copy out"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline) arm
# ---------------------------------------------------------------------------
def oracle_sample(layer, kind, seconds):
    """Time the oracle on a bounded sample: the first `rows` output rows of
    each projection of one layer, drawn from the seeded host generator.
    Returns (units per second, description, threads)."""
    import oracle
    from gemm_pq2_ternary_gb300 import inputs

    probs = []
    for i, (M, K, N, cdist, xdist) in enumerate(layer):
        rows = min(N, 64)
        if cdist == "bf16":
            xb, wb = inputs.generate_bf16(M, rows, K, seed=100 + i)
            probs.append((M, K, rows, "bf16", (xb, wb)))
            continue
        p = inputs.Problem("sample", M, K, rows, cdist, xdist, 100 + i)
        tern, ws, x = inputs.generate(p)
        qp, S, T = oracle.quantize_act(x)
        codes = oracle.pack(tern)
        probs.append((M, K, rows, "ternary", (qp, S, codes, ws)))

    def run(rows_frac):
        units = 0.0
        t0 = time.perf_counter()
        for pr in probs:
            M, K, rows = pr[:3]
            r = max(1, int(rows * rows_frac))
            if pr[3] == "bf16":
                xb, wb = pr[4]
                ref, _ = oracle.gemm_bf16(xb, wb[:r])
                oracle.f64_to_bf16(ref)
                units += bf16_bytes(M, r, K)
                continue
            qp, S, codes, ws = pr[4]
            oracle.matmul(qp, S, codes[:r], ws[:r])
            units += (gemm_bytes(M, r, K) if kind == "GB/s" else 2.0 * M * r * K)
        return units, time.perf_counter() - t0

    u, dt = run(1.0)
    reps = max(1, int(seconds / max(dt, 1e-6)))
    t0 = time.perf_counter()
    tot = 0.0
    for _ in range(reps):
        tot += run(1.0)[0]
    dt = time.perf_counter() - t0
    scale = 1e-9 if kind == "GB/s" else 1e-12
    desc = (f"{reps} x first {[p[2] for p in probs]} output rows of the "
            f"{[(p[0], p[1]) for p in probs]} (M,K) projections; all M tokens, all K")
    threads = oracle.threads()
    if any(p[3] == "bf16" for p in probs):
        # numpy's float64 matmul: its BLAS may use every host core
        threads = os.cpu_count() or 1
        desc += "; float64 matmul through numpy's BLAS (up to all host cores)"
    return tot / dt * scale, desc, threads, dt


def accuracy(sample):
    """The pages' accuracy measures for the GPU's output rows in `sample`
    (the first output rows and token rows of one projection of the step,
    inputs copied back from the device) against the oracle on the same
    inputs: the relative RMS error ([P1] "One token at a time": rel-RMS of
    the reordered fp32 sum) and the largest elementwise relative error over
    outputs with |ref| > 1e-3 * A, A = sum_g |dot_g * s * ws| (where ref is
    near 0 against A, cancellation makes the relative error meaningless);
    `within_tolerance` applies the parity tests' bound to every sampled
    output."""
    import oracle
    if sample["bf16"]:
        ref, A = oracle.gemm_bf16(sample["x"], sample["w"])
        got = oracle.bf16_to_f64(sample["y"])
        tol = oracle.bf16_gemm_tolerance(ref, A, sample["x"].shape[1])
    else:
        qp, S, _ = oracle.quantize_act(sample["x"])
        ref, A = oracle.matmul(qp, S, oracle.pack(sample["tern"]), sample["ws"])
        got = sample["y"].astype(np.float64)
        tol = oracle.fp32_tolerance(ref, A, sample["K"] // 128)
    err = np.abs(got - ref)
    big = np.abs(ref) > 1e-3 * A
    return {"rel_rms": float(np.sqrt(np.sum(err ** 2) / max(np.sum(ref ** 2), 1e-300))),
            "max_rel_err": float(np.max(err[big] / np.abs(ref[big]))) if big.any() else 0.0,
            "within_tolerance": bool(np.all(err <= tol)),
            "outputs": int(ref.size),
            "sample": f"first {ref.shape[1]} output rows x first {ref.shape[0]} tokens of the "
                      f"first projection, inputs copied from the device"}


def oracle_single_core(layer, kind, seconds):
    """The oracle's C loops on one thread, a shorter sample; None where the
    sample runs through numpy's BLAS, whose threads the oracle does not set."""
    if any(is_bf16(pr) for pr in layer):
        return None
    import oracle
    before = oracle.threads()
    try:
        oracle.set_threads(1)
        v, desc, threads, _ = oracle_sample(layer, kind, seconds)
    finally:
        oracle.set_threads(before)
    return {"value": round(v, 6), "unit": kind, "cores": threads, "sample": desc}


def reference_arm(args, rank, world):
    name, layer, kind = workload_spec(args)
    if rank != 0:
        return None
    vals = []
    t_start = time.perf_counter()
    for i in range(args.warmup + args.steps):
        v, desc, threads, dt = oracle_sample(layer, kind, args.ref_step_seconds)
        if i >= args.warmup:
            vals.append((v, dt))
    value = float(np.median([v for v, _ in vals]))
    ms = float(np.mean([dt for _, dt in vals])) * 1e3
    return {
        "impl": "reference",
        "metric": metric_name(kind, name, layer), "value": round(value, 6), "unit": kind,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64" if is_bf16(layer[0]) else "i8",
        "data": "synthetic (seeded host draws)",
        "config": {"workload": name, "parallelism": "host cores, one process"},
        "cpu_baseline": {"value": round(value, 6), "unit": kind, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": kind, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": round(time.perf_counter() - t_start, 1),
    }


# The configurations of the default run (besides the decode headline), each
# as (workload, M, "K,N"): the PR1 reference shape, the small-batch sweep,
# the MLP pair, prefill, 17-64 tokens, and the next rows (lm_head-scale
# GEMV, the bf16 projection, the SwiGLU-chained MLP).
SUITE = ([("pr1", 1, None)] +
         [("small", m, sh) for m in (2, 4, 8, 16) for sh in ("6144,5120", "5120,17408")] +
         [("mlp", 1, None), ("mlp", 16, None), ("prefill", 128, None), ("prefill", 4096, None),
          ("mid", 32, None), ("mid", 64, None), ("mid", 64, "6144,5120"),
          ("lmhead", 1, None), ("in_proj_ba", 4, None), ("mlp_swiglu", 1, None)])


def suite_entry(args, workload, m, shape, rank, world, dist):
    """One configuration of the default run: short timing, then the oracle on
    a short sample and the accuracy of the GPU's sampled outputs."""
    sub = argparse.Namespace(**vars(args))
    sub.workload, sub.m = workload, m
    if shape:
        sub.shape = shape
    wl = workload_spec(sub)
    line, sample = measure(sub, wl, rank, world, dist, steps=args.config_steps, warmup=3,
                           target_ms=args.config_ms, e2e_passes=3, floor=False)
    keep = ("metric", "value", "unit", "ms_per_step", "roofline", "matmul_us_per_launch",
            "gpu_launches", "clocks", "library_baseline", "steps", "warmup")
    entry = {"workload": wl[0], **{k: line[k] for k in keep if k in line},
             "config": {k: line["config"][k] for k in ("shapes", "projections_per_pass",
                                                       "passes_per_step", "l2")},
             "e2e": line["e2e"] and {k: line["e2e"][k] for k in ("value", "unit",
                                                                  "h2d_bytes_per_step",
                                                                  "d2h_bytes_per_step")}}
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, threads, _ = oracle_sample(wl[1], wl[2], args.config_cpu_seconds)
        entry["cpu_baseline"] = {"value": round(v, 6), "unit": wl[2], "cores": threads,
                                 "kind": "oracle", "sample": desc}
        entry["accuracy"] = accuracy(sample)
    return entry


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pq2", choices=["pq2", "reference"])
    ap.add_argument("--workload", default=None,
                    choices=["decode", "pr1", "small", "mid", "mlp", "mlp_swiglu", "prefill",
                             "lmhead", "in_proj_ba"],
                    help="one workload alone (default: the decode headline plus every "
                         "configuration in `configs`)")
    ap.add_argument("--m", type=int, default=16)
    ap.add_argument("--shape", default="5120,17408")
    ap.add_argument("--projections", type=int, default=0, help="weight sets per step (0: auto)")
    ap.add_argument("--reps", type=int, default=0,
                    help="passes over the R weight sets per step (0: auto, >= 1.5 s timed)")
    ap.add_argument("--weights", default="static", choices=["static", "default"],
                    help="static: M = 1 calls pass PQ2_WEIGHTS_STATIC (weights read before the "
                         "preceding call ends); default: plain pq2_matmul ordering")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="default run: the decode headline only")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-step-seconds", type=float, default=2.0)
    ap.add_argument("--config-steps", type=int, default=5)
    ap.add_argument("--config-ms", type=float, default=400.0,
                    help="timed milliseconds per configuration of the default run")
    ap.add_argument("--config-cpu-seconds", type=float, default=1.0)
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    suite = args.workload is None and not args.no_configs
    if args.workload is None:
        args.workload = "decode"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None

    if args.impl == "reference":
        out = reference_arm(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return

    import torch
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    wl = workload_spec(args)
    out, sample = measure(args, wl, rank, world, dist, steps=args.steps, warmup=args.warmup,
                          target_ms=1500.0, e2e_passes=max(3, min(args.steps, 20)), floor=True)
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, threads, _ = oracle_sample(wl[1], wl[2], args.cpu_seconds)
        out["cpu_baseline"] = {"value": round(v, 6), "unit": wl[2], "cores": threads,
                               "kind": "oracle", "sample": desc}
        single = oracle_single_core(wl[1], wl[2], args.cpu_seconds / 4)
        if single is not None:
            out["cpu_baseline"]["single_core"] = single
        out["accuracy"] = accuracy(sample)
    if suite:
        out["configs"] = [suite_entry(args, w, m, sh, rank, world, dist) for (w, m, sh) in SUITE]
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
