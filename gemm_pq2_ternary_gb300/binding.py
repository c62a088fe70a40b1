"""Thin Python binding of the C ABI in include/pq2.h (argument marshalling only).

Every function has the name of its C entry point, takes torch CUDA tensors,
passes their data pointers and the current CUDA stream, and raises
``PQ2Error`` when the C call returns a non-zero status.  All computation runs
in the CUDA kernels of libpq2.so; there is no other implementation here, and
importing this module fails if the library has not been built.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpq2.so")

PQ2_OK = 0
PQ2_ERR_INVALID_ARG = 1
PQ2_ERR_UNSUPPORTED_SHAPE = 2
PQ2_ERR_MISALIGNED = 3
PQ2_ERR_CUDA = 4
PQ2_ERR_TIMEOUT = 5
PQ2_ERR_WORKSPACE = 6
PQ2_ERR_BOUNDS = 7

PQ2_OP_GEMV = 0
PQ2_OP_SMALL = 1
PQ2_OP_PREFILL = 2
PQ2_OP_MATMUL = 3
PQ2_OP_SWIGLU_DOWN = 4

PQ2_WEIGHTS_STATIC = 1

# kernel variants for pq2_debug_force_kernel
PQ2_VARIANT_DEFAULT = 0
PQ2_VARIANT_GEMV_DIRECT = 1
PQ2_VARIANT_GEMV_RING = 2
PQ2_VARIANT_GEMV_STAGED = 3
PQ2_VARIANT_SMALL_DP4A = 1
PQ2_VARIANT_SMALL_TC = 2
PQ2_VARIANT_SMALL_TILE = 3
PQ2_VARIANT_SMALL_WTILE = 4
PQ2_VARIANT_PREFILL_128 = 1
PQ2_VARIANT_PREFILL_WIDE = 2
PQ2_VARIANT_PREFILL_TILE = 3
PQ2_VARIANT_PREFILL_WTILE = 4

SIZE_MAX = ctypes.c_size_t(-1).value

# Exported names and argument types (every one declared in include/pq2.h).
_P, _I64, _SZ, _I, _U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64
_U32 = ctypes.c_uint32
SIGNATURES = {
    "pq2_status_string": ([_I], ctypes.c_char_p),
    "pq2_version": ([], ctypes.c_char_p),
    "pq2_quantize_act": ([_P, _I64, _I64, _P, _P, _P, _P], _I),
    "pq2_pack_weights": ([_P, _P, _I64, _I64, _P, _P, _P], _I),
    "pq2_gemv": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _P], _I),
    "pq2_gemm_small": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], _I),
    "pq2_gemm_small_ex": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _U32, _P, _SZ, _P], _I),
    "pq2_gemm_prefill": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], _I),
    "pq2_matmul": ([_P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], _I),
    "pq2_matmul_ex": ([_P, _P, _P, _P, _I64, _I64, _I64, _U32, _P, _SZ, _P], _I),
    "pq2_quantize_swiglu": ([_P, _I64, _I64, _P, _P, _P, _P], _I),
    "pq2_gemm_bf16_splitk": ([_P, _P, _P, _I64, _I64, _I64, _U32, _P], _I),
    "pq2_mlp_down_swiglu": ([_P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], _I),
    "pq2_workspace_bytes": ([_I, _I64, _I64, _I64], _SZ),
    "pq2_group_dots": ([_I, _P, _P, _P, _I64, _I64, _I64, _P, _P, _SZ, _P], _I),
    "pq2_last_device_error": ([_P], _I),
    "pq2_debug_set_wait_limit_ns": ([_U64], _I),
    "pq2_debug_skip_stage": ([_I], _I),
    "pq2_bounds_checked": ([], _I),
    "pq2_debug_shrink_bounds": ([_I], _I),
    "pq2_debug_force_kernel": ([_I, _I], _I),
    "pq2_debug_gemv_floor": ([_I64, _I64, _U32, _P], _I),
    "pq2_debug_mma_rate": ([_I, _I, _P, _P], _I),
    "pq2_gemm_small_noalloc": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P], _I),
    "pq2_gemm_small_noalloc_max_scratch": ([], _SZ),
}


def load_library(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = load_library()


class PQ2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.pq2_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def _check(status: int, where: str):
    if status != PQ2_OK:
        raise PQ2Error(status, where)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream  # an int: ctypes passes it as the void* argument


def _ptr(t):
    if t is None:
        return None
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError("expected a contiguous CUDA tensor")
    return t.data_ptr()


def _dtype(t, dt, name):
    if t.dtype != dt:
        raise ValueError(f"{name}: expected {dt}, got {t.dtype}")


def pq2_version() -> str:
    return _lib.pq2_version().decode()


def pq2_status_string(status: int) -> str:
    return _lib.pq2_status_string(status).decode()


def pq2_workspace_bytes(op: int, M: int, N: int, K: int) -> int:
    return int(_lib.pq2_workspace_bytes(op, M, N, K))


def pq2_quantize_act(x, qp, S, T, stream=None):
    """x fp16 [M,K] -> qp int8 [M,K] (plane order), S fp32 [M,G], T int32 [M,G]."""
    _dtype(x, torch.float16, "x")
    _dtype(qp, torch.int8, "qp")
    _dtype(S, torch.float32, "S")
    _dtype(T, torch.int32, "T")
    M, K = x.shape
    _check(_lib.pq2_quantize_act(_ptr(x), M, K, _ptr(qp), _ptr(S), _ptr(T), _stream(stream)),
           "pq2_quantize_act")


def pq2_pack_weights(tern, ws, codes, ws_out, stream=None):
    """tern int8 [N,K] in {-1,0,1} -> codes uint8 [N,K/4]; ws copied to ws_out."""
    _dtype(tern, torch.int8, "tern")
    _dtype(codes, torch.uint8, "codes")
    N, K = tern.shape
    _check(_lib.pq2_pack_weights(_ptr(tern), _ptr(ws), N, K, _ptr(codes), _ptr(ws_out),
                                 _stream(stream)), "pq2_pack_weights")


def _mm_shapes(qp, codes):
    M, K = qp.shape
    N = codes.shape[0]
    if codes.shape[1] * 4 != K:
        raise ValueError("codes must be [N, K/4]")
    return M, N, K


def pq2_gemv(qp, S, T, codes, ws, y, stream=None):
    M, N, K = _mm_shapes(qp, codes)
    _dtype(y, torch.float32, "y")
    _check(_lib.pq2_gemv(_ptr(qp), _ptr(S), _ptr(T), _ptr(codes), _ptr(ws), _ptr(y), N, K,
                         _stream(stream)), "pq2_gemv")


def _ws(workspace):
    if workspace is None:
        return None, 0
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def pq2_gemm_small(qp, S, T, codes, ws, y, workspace=None, stream=None):
    M, N, K = _mm_shapes(qp, codes)
    wp, wb = _ws(workspace)
    _check(_lib.pq2_gemm_small(_ptr(qp), _ptr(S), _ptr(T), _ptr(codes), _ptr(ws), _ptr(y),
                               M, N, K, wp, wb, _stream(stream)), "pq2_gemm_small")


def pq2_gemm_small_ex(qp, S, T, codes, ws, y, flags, workspace=None, stream=None):
    M, N, K = _mm_shapes(qp, codes)
    wp, wb = _ws(workspace)
    _check(_lib.pq2_gemm_small_ex(_ptr(qp), _ptr(S), _ptr(T), _ptr(codes), _ptr(ws), _ptr(y),
                                  M, N, K, flags, wp, wb, _stream(stream)), "pq2_gemm_small_ex")


def pq2_gemm_prefill(qp, S, T, codes, ws, y, workspace=None, stream=None):
    M, N, K = _mm_shapes(qp, codes)
    wp, wb = _ws(workspace)
    _check(_lib.pq2_gemm_prefill(_ptr(qp), _ptr(S), _ptr(T), _ptr(codes), _ptr(ws), _ptr(y),
                                 M, N, K, wp, wb, _stream(stream)), "pq2_gemm_prefill")


def pq2_gemm_small_noalloc(qp, S, T, codes, ws, y, stream=None):
    """pq2_gemm_small without a workspace: its scratch is a fixed device array
    inside the library (for callers that cannot allocate device memory)."""
    M, N, K = _mm_shapes(qp, codes)
    _check(_lib.pq2_gemm_small_noalloc(_ptr(qp), _ptr(S), _ptr(T), _ptr(codes), _ptr(ws), _ptr(y),
                                       M, N, K, _stream(stream)), "pq2_gemm_small_noalloc")


def pq2_gemm_small_noalloc_max_scratch() -> int:
    return int(_lib.pq2_gemm_small_noalloc_max_scratch())


def pq2_matmul(x, codes, ws, y, workspace, stream=None):
    M, K = x.shape
    N = codes.shape[0]
    wp, wb = _ws(workspace)
    _check(_lib.pq2_matmul(_ptr(x), _ptr(codes), _ptr(ws), _ptr(y), M, N, K, wp, wb,
                           _stream(stream)), "pq2_matmul")


def pq2_matmul_ex(x, codes, ws, y, flags, workspace, stream=None):
    M, K = x.shape
    N = codes.shape[0]
    wp, wb = _ws(workspace)
    _check(_lib.pq2_matmul_ex(_ptr(x), _ptr(codes), _ptr(ws), _ptr(y), M, N, K, flags, wp, wb,
                              _stream(stream)), "pq2_matmul_ex")


def pq2_gemm_bf16_splitk(x, w, y, flags=0, stream=None):
    """x [M, K], w [N, K], y [M, N]: torch.bfloat16 (or int16 bit patterns)
    on the device."""
    for t, name in ((x, "x"), (w, "w"), (y, "y")):
        if t.dtype not in (torch.bfloat16, torch.int16):
            raise ValueError(f"{name}: expected torch.bfloat16 (or int16 bit patterns), got {t.dtype}")
    M, K = x.shape
    N, Kw = w.shape
    if Kw != K or tuple(y.shape) != (M, N):
        raise ValueError(f"shapes: x {tuple(x.shape)}, w {tuple(w.shape)}, y {tuple(y.shape)}")
    _check(_lib.pq2_gemm_bf16_splitk(_ptr(x), _ptr(w), _ptr(y), M, N, K, flags,
                                     _stream(stream)), "pq2_gemm_bf16_splitk")


def pq2_quantize_swiglu(gu, qp, S, T, stream=None):
    """gu [M, 2I] fp32 (gate | up) -> qp, S, T of h = fp16(silu(gate) * up)."""
    M, I2 = gu.shape
    _check(_lib.pq2_quantize_swiglu(_ptr(gu), M, I2 // 2, _ptr(qp), _ptr(S), _ptr(T),
                                    _stream(stream)), "pq2_quantize_swiglu")


def pq2_mlp_down_swiglu(gu, codes, ws, y, workspace, stream=None):
    M, I2 = gu.shape
    N = codes.shape[0]
    wp, wb = _ws(workspace)
    _check(_lib.pq2_mlp_down_swiglu(_ptr(gu), _ptr(codes), _ptr(ws), _ptr(y), M, N, I2 // 2,
                                    wp, wb, _stream(stream)), "pq2_mlp_down_swiglu")


def pq2_group_dots(op, qp, T, codes, dots, workspace=None, stream=None):
    M, N, K = _mm_shapes(qp, codes)
    wp, wb = _ws(workspace)
    _check(_lib.pq2_group_dots(op, _ptr(qp), _ptr(T), _ptr(codes), M, N, K, _ptr(dots), wp, wb,
                               _stream(stream)), "pq2_group_dots")


def pq2_last_device_error(stream=None) -> int:
    return int(_lib.pq2_last_device_error(_stream(stream)))


def pq2_debug_set_wait_limit_ns(ns: int):
    _check(_lib.pq2_debug_set_wait_limit_ns(ns), "pq2_debug_set_wait_limit_ns")


def pq2_debug_skip_stage(stage: int):
    _check(_lib.pq2_debug_skip_stage(stage), "pq2_debug_skip_stage")


def pq2_bounds_checked() -> bool:
    return bool(_lib.pq2_bounds_checked())


def pq2_debug_shrink_bounds(elements: int):
    _check(_lib.pq2_debug_shrink_bounds(elements), "pq2_debug_shrink_bounds")


def pq2_debug_force_kernel(op: int, variant: int):
    _check(_lib.pq2_debug_force_kernel(op, variant), "pq2_debug_force_kernel")


def pq2_debug_gemv_floor(N: int, K: int, flags: int = 0, stream=None):
    """One empty launch shaped like a fused M = 1 call (the latency floor)."""
    _check(_lib.pq2_debug_gemv_floor(N, K, flags, _stream(stream)), "pq2_debug_gemv_floor")


def pq2_debug_mma_rate(n: int, iters: int, cycles, stream=None):
    """cycles: int64 CUDA tensor with (at least) one entry per SM."""
    _dtype(cycles, torch.int64, "cycles")
    sms = torch.cuda.get_device_properties(cycles.device).multi_processor_count
    if cycles.numel() < sms:
        raise ValueError(f"cycles: needs {sms} entries, got {cycles.numel()}")
    _check(_lib.pq2_debug_mma_rate(n, iters, _ptr(cycles), _stream(stream)), "pq2_debug_mma_rate")


class forced_kernel:
    """Context manager: calls of `op` run kernel `variant` inside the block
    (pq2_debug_force_kernel), the library's own routing again after it."""

    def __init__(self, op: int, variant: int):
        self.op, self.variant = op, variant

    def __enter__(self):
        pq2_debug_force_kernel(self.op, self.variant)
        return self

    def __exit__(self, *exc):
        pq2_debug_force_kernel(self.op, PQ2_VARIANT_DEFAULT)
        return False


# ---------------------------------------------------------------------------
# Allocation helpers (torch owns the memory; the library never allocates).
# ---------------------------------------------------------------------------
def alloc_act(M: int, K: int, device="cuda"):
    qp = torch.empty((M, K), dtype=torch.int8, device=device)
    S = torch.empty((M, K // 128), dtype=torch.float32, device=device)
    T = torch.empty((M, K // 128), dtype=torch.int32, device=device)
    return qp, S, T


def alloc_workspace(op: int, M: int, N: int, K: int, device="cuda"):
    n = pq2_workspace_bytes(op, M, N, K)
    if n == SIZE_MAX:
        raise PQ2Error(PQ2_ERR_UNSUPPORTED_SHAPE, "pq2_workspace_bytes")
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device)


def pack(tern, ws, stream=None):
    """Convenience: returns (codes, ws_copy) for device tensors tern, ws."""
    N, K = tern.shape
    codes = torch.empty((N, K // 4), dtype=torch.uint8, device=tern.device)
    ws_out = torch.empty_like(ws)
    pq2_pack_weights(tern, ws, codes, ws_out, stream)
    return codes, ws_out


def quantize(x, stream=None):
    M, K = x.shape
    qp, S, T = alloc_act(M, K, x.device)
    pq2_quantize_act(x, qp, S, T, stream)
    return qp, S, T


def matmul_q(qp, S, T, codes, ws, stream=None):
    """Route quantised activations to pq2_gemv / pq2_gemm_small / pq2_gemm_prefill."""
    M, N, K = _mm_shapes(qp, codes)
    y = torch.empty((M, N), dtype=torch.float32, device=qp.device)
    if M == 1:
        pq2_gemv(qp, S, T, codes, ws, y, stream)
    elif M <= 16:
        pq2_gemm_small(qp, S, T, codes, ws, y, alloc_workspace(PQ2_OP_SMALL, M, N, K, qp.device),
                       stream)
    else:
        pq2_gemm_prefill(qp, S, T, codes, ws, y,
                         alloc_workspace(PQ2_OP_PREFILL, M, N, K, qp.device), stream)
    return y
