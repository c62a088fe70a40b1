"""CPU-only checks of the C ABI: the library loads, exports every function
include/pq2.h declares, and rejects bad arguments on the host before any CUDA
call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pq2.h")


@pytest.fixture(scope="module")
def lib():
    from gemm_pq2_ternary_gb300 import _build
    _build.build()
    from gemm_pq2_ternary_gb300 import binding
    return binding._lib


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pq2_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for want in ["pq2_quantize_act", "pq2_pack_weights", "pq2_gemv", "pq2_gemm_small",
                 "pq2_gemm_prefill", "pq2_matmul", "pq2_workspace_bytes", "pq2_group_dots",
                 "pq2_last_device_error", "pq2_status_string"]:
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    from gemm_pq2_ternary_gb300 import binding
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in binding.SIGNATURES, name


def test_version_and_status_strings(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    assert "sm_103a" in b.pq2_version()
    for s in range(8):
        assert b.pq2_status_string(s) not in ("", "unknown status")
    assert b.pq2_status_string(99) == "unknown status"


FAKE = 0x10000          # 16-byte aligned, never dereferenced
ODD = 0x10008           # 8-byte aligned only


def _p(v):
    return ctypes.c_void_p(v)


def test_gemv_rejects_bad_arguments(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    ok = [_p(FAKE)] * 6
    assert lib.pq2_gemv(*ok, 256, 100, None) == b.PQ2_ERR_UNSUPPORTED_SHAPE   # K % 128
    assert lib.pq2_gemv(*ok, 0, 128, None) == b.PQ2_ERR_INVALID_ARG           # N < 1
    assert lib.pq2_gemv(*ok, 1, 0, None) == b.PQ2_ERR_INVALID_ARG             # K < 1
    assert lib.pq2_gemv(*ok, 1, 128 * 4096, None) == b.PQ2_ERR_UNSUPPORTED_SHAPE
    bad = list(ok)
    bad[3] = None
    assert lib.pq2_gemv(*bad, 4, 128, None) == b.PQ2_ERR_INVALID_ARG          # codes null
    bad = list(ok)
    bad[5] = _p(ODD)
    assert lib.pq2_gemv(*bad, 4, 128, None) == b.PQ2_ERR_MISALIGNED           # y misaligned


def test_small_and_prefill_reject_bad_arguments(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    ok = [_p(FAKE)] * 6
    for M in (1, 17, 0):
        st = lib.pq2_gemm_small(*ok, M, 64, 128, None, 0, None)
        assert st in (b.PQ2_ERR_UNSUPPORTED_SHAPE, b.PQ2_ERR_INVALID_ARG)
    assert lib.pq2_gemm_prefill(*ok, 0, 64, 128, None, 0, None) == b.PQ2_ERR_INVALID_ARG
    assert lib.pq2_gemm_prefill(*ok, 64, 64, 200, None, 0, None) == b.PQ2_ERR_UNSUPPORTED_SHAPE


def test_workspace_query(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    assert b.pq2_workspace_bytes(b.PQ2_OP_GEMV, 1, 5120, 6144) == 0
    assert b.pq2_workspace_bytes(b.PQ2_OP_GEMV, 2, 5120, 6144) == b.SIZE_MAX
    assert b.pq2_workspace_bytes(b.PQ2_OP_SMALL, 17, 5120, 6144) == b.SIZE_MAX
    assert b.pq2_workspace_bytes(b.PQ2_OP_SMALL, 4, 5120, 100) == b.SIZE_MAX
    assert b.pq2_workspace_bytes(99, 4, 5120, 6144) == b.SIZE_MAX
    mm = b.pq2_workspace_bytes(b.PQ2_OP_MATMUL, 4, 5120, 6144)
    assert mm >= 4 * 6144 + 2 * 4 * 48 * 4


def test_matmul_rejects_small_workspace(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    st = lib.pq2_matmul(_p(FAKE), _p(FAKE), _p(FAKE), _p(FAKE), 4, 64, 128, _p(FAKE), 16, None)
    assert st == b.PQ2_ERR_WORKSPACE
    st = lib.pq2_matmul(_p(FAKE), _p(FAKE), _p(FAKE), _p(FAKE), 4, 64, 128, None, 1 << 20, None)
    assert st == b.PQ2_ERR_WORKSPACE


def test_matmul_ex_rejects_unknown_flags(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    st = lib.pq2_matmul_ex(_p(FAKE), _p(FAKE), _p(FAKE), _p(FAKE), 1, 64, 128, 2, None, 0, None)
    assert st == b.PQ2_ERR_INVALID_ARG
    st = lib.pq2_matmul_ex(_p(FAKE), _p(FAKE), _p(FAKE), _p(FAKE), 4, 64, 128,
                           b.PQ2_WEIGHTS_STATIC, _p(FAKE), 16, None)
    assert st == b.PQ2_ERR_WORKSPACE


def test_swiglu_entry_points_check_arguments(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    assert 0 < b.pq2_workspace_bytes(b.PQ2_OP_SWIGLU_DOWN, 1, 5120, 17408) < b.SIZE_MAX
    assert b.pq2_workspace_bytes(b.PQ2_OP_SWIGLU_DOWN, 1, 5120, 100) == b.SIZE_MAX
    st = lib.pq2_quantize_swiglu(_p(FAKE), 1, 100, _p(FAKE), _p(FAKE), _p(FAKE), None)
    assert st == b.PQ2_ERR_UNSUPPORTED_SHAPE
    st = lib.pq2_quantize_swiglu(_p(ODD), 1, 128, _p(FAKE), _p(FAKE), _p(FAKE), None)
    assert st == b.PQ2_ERR_MISALIGNED
    st = lib.pq2_mlp_down_swiglu(_p(FAKE), _p(FAKE), _p(FAKE), _p(FAKE), 1, 64, 128, None, 0, None)
    assert st == b.PQ2_ERR_WORKSPACE


def test_group_dots_rejects_bad_op(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    st = lib.pq2_group_dots(7, _p(FAKE), _p(FAKE), _p(FAKE), 1, 8, 128, _p(FAKE), None, 0, None)
    assert st == b.PQ2_ERR_INVALID_ARG
    st = lib.pq2_group_dots(b.PQ2_OP_GEMV, _p(FAKE), _p(FAKE), _p(FAKE), 3, 8, 128, _p(FAKE),
                            None, 0, None)
    assert st == b.PQ2_ERR_UNSUPPORTED_SHAPE


def test_quantize_and_pack_reject_bad_arguments(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    P = _p(FAKE)
    assert lib.pq2_quantize_act(P, 2, 130, P, P, P, None) == b.PQ2_ERR_UNSUPPORTED_SHAPE
    assert lib.pq2_quantize_act(P, -1, 128, P, P, P, None) == b.PQ2_ERR_INVALID_ARG
    assert lib.pq2_quantize_act(P, 0, 128, P, P, P, None) == b.PQ2_OK   # nothing to do
    assert lib.pq2_quantize_act(P, 2, 128, _p(ODD), P, P, None) == b.PQ2_ERR_MISALIGNED
    assert lib.pq2_pack_weights(P, P, 4, 96, P, P, None) == b.PQ2_ERR_UNSUPPORTED_SHAPE
    assert lib.pq2_pack_weights(P, P, 4, 128, P, None, None) == b.PQ2_ERR_INVALID_ARG


def test_bf16_splitk_checks_arguments(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    f = lib.pq2_gemm_bf16_splitk
    assert f(_p(FAKE), _p(FAKE), _p(FAKE), 2, 96, 5124, 0, None) == b.PQ2_ERR_UNSUPPORTED_SHAPE
    assert f(_p(FAKE), _p(FAKE), _p(FAKE), 2, 96, 5120, 2, None) == b.PQ2_ERR_INVALID_ARG
    assert f(_p(FAKE), _p(FAKE), _p(FAKE), -1, 96, 5120, 0, None) == b.PQ2_ERR_INVALID_ARG
    assert f(None, _p(FAKE), _p(FAKE), 2, 96, 5120, 0, None) == b.PQ2_ERR_INVALID_ARG
    assert f(_p(ODD), _p(FAKE), _p(FAKE), 2, 96, 5120, 0, None) == b.PQ2_ERR_MISALIGNED
    assert f(_p(FAKE), _p(ODD), _p(FAKE), 2, 96, 5120, 0, None) == b.PQ2_ERR_MISALIGNED
    assert f(_p(FAKE), _p(FAKE), _p(FAKE + 1), 2, 96, 5120, 0, None) == b.PQ2_ERR_MISALIGNED
    assert f(_p(FAKE), _p(FAKE), _p(FAKE), 1048561, 96, 5120, 0, None) == b.PQ2_ERR_UNSUPPORTED_SHAPE
    # empty problems enqueue nothing, whatever the pointers
    assert f(None, None, None, 0, 96, 5120, 0, None) == b.PQ2_OK
    assert f(None, None, None, 4, 0, 5120, 0, None) == b.PQ2_OK


def test_prefill_workspace_holds_expanded_weights_for_wide_shapes(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    K, N = 5120, 17408
    G = K // 128

    def planes(M):  # token planes hi and lo, (s, t) per group
        return 2 * M * K + M * G * 8

    small = b.pq2_workspace_bytes(b.PQ2_OP_PREFILL, 128, N, K)      # one token tile
    assert planes(128) <= small < planes(128) + N * K
    big = b.pq2_workspace_bytes(b.PQ2_OP_PREFILL, 4096, N, K)       # 32 token tiles
    npad = (N + 255) // 256 * 256
    assert big >= planes(4096) + N * K + G * npad * 4
    # the matmul's workspace for large M includes the prefill's
    assert b.pq2_workspace_bytes(b.PQ2_OP_MATMUL, 4096, N, K) >= big


def test_bf16_binding_checks_dtype_and_shapes(lib):
    import torch
    from gemm_pq2_ternary_gb300 import binding as b
    x = torch.zeros((2, 64), dtype=torch.float32)
    w = torch.zeros((8, 64), dtype=torch.bfloat16)
    y = torch.zeros((2, 8), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="x: expected"):
        b.pq2_gemm_bf16_splitk(x, w, y)
    with pytest.raises(ValueError, match="shapes"):
        b.pq2_gemm_bf16_splitk(x.bfloat16(), w, torch.zeros((2, 9), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA"):   # host tensors never reach the library
        b.pq2_gemm_bf16_splitk(x.bfloat16(), w, y)


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    # 16 tokens at lm_head scale (N = 248320, K = 5120): the split-K partial
    # sums alone need about 16 MB, more than the fixed array holds; the call
    # is refused on the host, before any CUDA call
    from gemm_pq2_ternary_gb300 import binding as b
    P = _p(FAKE)
    assert b.pq2_gemm_small_noalloc_max_scratch() == 4 << 20
    st = lib.pq2_gemm_small_noalloc(P, P, P, P, P, P, 16, 248320, 5120, None)
    assert st == b.PQ2_ERR_WORKSPACE
    st = lib.pq2_gemm_small_noalloc(P, P, P, P, P, P, 17, 5120, 5120, None)
    assert st == b.PQ2_ERR_UNSUPPORTED_SHAPE


def test_force_kernel_checks_its_arguments(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    f = lib.pq2_debug_force_kernel
    assert f(b.PQ2_OP_MATMUL, 1) == b.PQ2_ERR_INVALID_ARG      # not a kernel family
    assert f(b.PQ2_OP_SMALL, 7) == b.PQ2_ERR_INVALID_ARG
    assert f(b.PQ2_OP_PREFILL, -1) == b.PQ2_ERR_INVALID_ARG
    K, N = 5120, 17408
    default = b.pq2_workspace_bytes(b.PQ2_OP_PREFILL, 128, N, K)
    try:
        # the 128 x 256 kernel, forced, needs room for the expanded weights
        assert f(b.PQ2_OP_PREFILL, b.PQ2_VARIANT_PREFILL_WIDE) == b.PQ2_OK
        assert b.pq2_workspace_bytes(b.PQ2_OP_PREFILL, 128, N, K) >= default + N * K
    finally:
        assert f(b.PQ2_OP_PREFILL, b.PQ2_VARIANT_DEFAULT) == b.PQ2_OK
    assert b.pq2_workspace_bytes(b.PQ2_OP_PREFILL, 128, N, K) == default


def test_measurement_hooks_check_their_arguments(lib):
    from gemm_pq2_ternary_gb300 import binding as b
    assert lib.pq2_debug_mma_rate(48, 16, _p(FAKE), None) == b.PQ2_ERR_INVALID_ARG
    assert lib.pq2_debug_mma_rate(256, 0, _p(FAKE), None) == b.PQ2_ERR_INVALID_ARG
    assert lib.pq2_debug_mma_rate(256, 16, None, None) == b.PQ2_ERR_INVALID_ARG
    assert lib.pq2_debug_gemv_floor(5120, 6144, 2, None) == b.PQ2_ERR_INVALID_ARG
    assert lib.pq2_debug_gemv_floor(5120, 100, 0, None) == b.PQ2_ERR_UNSUPPORTED_SHAPE


def test_bounds_checked_build_hooks(lib):
    # the normal library reports 0; the checked one (PQ2_DEBUG=1) 1 and the
    # same exports; the shrink hook takes no negative count
    from gemm_pq2_ternary_gb300 import _build, binding as b
    assert lib.pq2_bounds_checked() == 0
    assert lib.pq2_debug_shrink_bounds(-1) == b.PQ2_ERR_INVALID_ARG
    assert lib.pq2_debug_shrink_bounds(0) == b.PQ2_OK
    dbg = b.load_library(_build.build(debug=True))
    assert dbg.pq2_bounds_checked() == 1
    for name in _declared():
        assert hasattr(dbg, name), name
