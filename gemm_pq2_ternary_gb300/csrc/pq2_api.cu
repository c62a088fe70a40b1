// The C ABI (include/pq2.h): host-side argument checks, per-device set-up,
// routing to the kernels, and the device error word.
#include <atomic>
#include <cstring>
#include <mutex>

#include "../../include/pq2.h"
#include "pq2_internal.h"

// Device error word: bit flags of pq2::DEVERR_*, one per device context.
__device__ unsigned g_pq2_error_word = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
pq2h::DeviceInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices] = {};
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_debug_skip_stage{-1};
std::atomic<int> g_debug_bounds_shrink{0};
// pq2_debug_force_kernel: forced variant per op (GEMV, SMALL, PREFILL)
std::atomic<int> g_force[3] = {{0}, {0}, {0}};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pq2_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return PQ2_OK;
    if (e == pq2h::kUnsupportedVariant) {
        cudaGetLastError();  // (not sticky; clear it all the same)
        return PQ2_ERR_UNSUPPORTED_SHAPE;
    }
    return PQ2_ERR_CUDA;
}

// Common shape checks: K a positive multiple of 128 within the supported
// range, N >= 1.
pq2_status check_nk(int64_t N, int64_t K) {
    if (N < 1 || K < 1) return PQ2_ERR_INVALID_ARG;
    if (K % 128 != 0 || K > PQ2_MAX_K) return PQ2_ERR_UNSUPPORTED_SHAPE;
    if (N > (int64_t(1) << 31) - 1) return PQ2_ERR_UNSUPPORTED_SHAPE;
    return PQ2_OK;
}

struct Ctx {
    pq2h::DeviceInfo dev;
    pq2::DevCtl ctl;
};

pq2_status get_ctx(Ctx* c) {
    if (!pq2h::device_info(&c->dev)) return PQ2_ERR_CUDA;
    if (!pq2h::make_ctl(&c->ctl)) return PQ2_ERR_CUDA;
    return PQ2_OK;
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

namespace pq2h {

int forced_variant(int op) {
    return (op >= PQ2_OP_GEMV && op <= PQ2_OP_PREFILL) ? g_force[op].load() : PQ2_VARIANT_DEFAULT;
}

bool device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_dev_ok[dev]) {
        DeviceInfo d = {};
        d.device = dev;
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess)
            return false;
        if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                   dev) != cudaSuccess)
            return false;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pq2_error_word) != cudaSuccess) return false;
        d.err = static_cast<unsigned*>(p);
        g_dev[dev] = d;
        g_dev_ok[dev] = true;
    }
    *out = g_dev[dev];
    return true;
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}
}  // namespace

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
                    bool swizzle128) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_ctl(pq2::DevCtl* ctl) {
    DeviceInfo d;
    if (!device_info(&d)) return false;
    ctl->err = d.err;
    ctl->wait_limit_ns = g_wait_limit_ns.load();
    ctl->debug_skip_stage = g_debug_skip_stage.load();
    ctl->debug_bounds_shrink = g_debug_bounds_shrink.load();
    return true;
}

}  // namespace pq2h

extern "C" {

const char* pq2_status_string(int status) {
    switch (status) {
        case PQ2_OK: return "ok";
        case PQ2_ERR_INVALID_ARG: return "invalid argument";
        case PQ2_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case PQ2_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case PQ2_ERR_CUDA: return "CUDA error";
        case PQ2_ERR_TIMEOUT: return "device wait timed out";
        case PQ2_ERR_WORKSPACE: return "workspace missing or too small";
        case PQ2_ERR_BOUNDS: return "bounds-checked build: a store outside its buffer";
        default: return "unknown status";
    }
}

const char* pq2_version(void) { return "pq2-gb300 0.1 sm_103a"; }

pq2_status pq2_debug_set_wait_limit_ns(uint64_t ns) {
    if (ns == 0) return PQ2_ERR_INVALID_ARG;
    g_wait_limit_ns.store(ns);
    return PQ2_OK;
}

// Not in the public header: makes every later launch's producer withhold
// stage `stage` (-1 = off), so the consumers' bounded wait runs out.  For the
// timeout test only.
pq2_status pq2_debug_skip_stage(int stage) {
    g_debug_skip_stage.store(stage < 0 ? -1 : stage);
    return PQ2_OK;
}

int pq2_bounds_checked(void) { return PQ2_DEBUG; }

pq2_status pq2_debug_shrink_bounds(int elements) {
    if (elements < 0) return PQ2_ERR_INVALID_ARG;
    g_debug_bounds_shrink.store(elements);
    return PQ2_OK;
}

pq2_status pq2_debug_force_kernel(int op, int variant) {
    int max_variant = -1;
    if (op == PQ2_OP_GEMV) max_variant = PQ2_VARIANT_GEMV_STAGED;
    if (op == PQ2_OP_SMALL) max_variant = PQ2_VARIANT_SMALL_WTILE;
    if (op == PQ2_OP_PREFILL) max_variant = PQ2_VARIANT_PREFILL_WTILE;
    if (variant < 0 || variant > max_variant) return PQ2_ERR_INVALID_ARG;
    g_force[op].store(variant);
    return PQ2_OK;
}

pq2_status pq2_debug_gemv_floor(int64_t N, int64_t K, uint32_t flags, void* stream) {
    if (flags & ~static_cast<uint32_t>(PQ2_WEIGHTS_STATIC)) return PQ2_ERR_INVALID_ARG;
    pq2_status s = check_nk(N, K);
    if (s != PQ2_OK) return s;
    if (!pq2h::gemv_fused_supported(K)) return PQ2_ERR_UNSUPPORTED_SHAPE;
    Ctx c;
    s = get_ctx(&c);
    if (s != PQ2_OK) return s;
    return cuda_status(pq2h::launch_gemv_floor(N, K, (flags & PQ2_WEIGHTS_STATIC) != 0,
                                               static_cast<cudaStream_t>(stream), c.ctl, c.dev));
}

pq2_status pq2_debug_mma_rate(int n, int iters, uint64_t* cycles, void* stream) {
    if ((n != 32 && n != 64 && n != 128 && n != 256) || iters < 1 || iters > (1 << 24))
        return PQ2_ERR_INVALID_ARG;
    if (!cycles) return PQ2_ERR_INVALID_ARG;
    Ctx c;
    pq2_status s = get_ctx(&c);
    if (s != PQ2_OK) return s;
    return cuda_status(pq2h::launch_mma_rate(n, iters,
                                             reinterpret_cast<unsigned long long*>(cycles),
                                             static_cast<cudaStream_t>(stream), c.ctl, c.dev));
}

pq2_status pq2_quantize_act(const void* x_f16, int64_t M, int64_t K, int8_t* qp, float* S,
                            int32_t* T, void* stream) {
    if (M < 0 || K < 1) return PQ2_ERR_INVALID_ARG;
    if (K % 128 != 0 || K > PQ2_MAX_K) return PQ2_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return PQ2_OK;
    if (!x_f16 || !qp || !S || !T) return PQ2_ERR_INVALID_ARG;
    if (!aligned16(x_f16) || !aligned16(qp) || !aligned16(S) || !aligned16(T))
        return PQ2_ERR_MISALIGNED;
    Ctx c;
    pq2_status s = get_ctx(&c);
    if (s != PQ2_OK) return s;
    return cuda_status(pq2h::launch_quantize(static_cast<const __half*>(x_f16), qp, S, T, M, K,
                                             static_cast<cudaStream_t>(stream), c.ctl, c.dev));
}

pq2_status pq2_quantize_swiglu(const float* gu, int64_t M, int64_t I, int8_t* qp, float* S,
                               int32_t* T, void* stream) {
    if (M < 0 || I < 1) return PQ2_ERR_INVALID_ARG;
    if (I % 128 != 0 || I > PQ2_MAX_K) return PQ2_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return PQ2_OK;
    if (!gu || !qp || !S || !T) return PQ2_ERR_INVALID_ARG;
    if (!aligned16(gu) || !aligned16(qp) || !aligned16(S) || !aligned16(T))
        return PQ2_ERR_MISALIGNED;
    Ctx c;
    pq2_status s = get_ctx(&c);
    if (s != PQ2_OK) return s;
    return cuda_status(pq2h::launch_quantize_swiglu(gu, qp, S, T, M, I,
                                                    static_cast<cudaStream_t>(stream), c.ctl,
                                                    c.dev));
}

pq2_status pq2_pack_weights(const int8_t* tern, const void* ws_f16, int64_t N, int64_t K,
                            uint8_t* codes, void* ws_out, void* stream) {
    pq2_status s = check_nk(N, K);
    if (s != PQ2_OK) return s;
    if (!tern || !codes) return PQ2_ERR_INVALID_ARG;
    if ((ws_f16 == nullptr) != (ws_out == nullptr)) return PQ2_ERR_INVALID_ARG;
    if (!aligned16(tern) || !aligned16(codes) || (ws_f16 && (!aligned16(ws_f16) ||
                                                            !aligned16(ws_out))))
        return PQ2_ERR_MISALIGNED;
    Ctx c;
    s = get_ctx(&c);
    if (s != PQ2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = pq2h::launch_pack(tern, codes, N, K, st, c.ctl, c.dev);
    if (e != cudaSuccess) return PQ2_ERR_CUDA;
    if (ws_f16 && ws_out != ws_f16) {
        e = cudaMemcpyAsync(ws_out, ws_f16, static_cast<size_t>(N) * (K / 128) * 2,
                            cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return PQ2_ERR_CUDA;
    }
    return PQ2_OK;
}

static pq2_status check_mm(const int8_t* qp, const float* S, const int32_t* T,
                           const uint8_t* codes, const void* ws, const void* out, int64_t M,
                           int64_t N, int64_t K) {
    pq2_status s = check_nk(N, K);
    if (s != PQ2_OK) return s;
    if (M < 1) return PQ2_ERR_INVALID_ARG;
    if (!qp || !T || !codes || !out) return PQ2_ERR_INVALID_ARG;
    if (!aligned16(qp) || !aligned16(T) || !aligned16(codes) || !aligned16(out))
        return PQ2_ERR_MISALIGNED;
    if (S && !aligned16(S)) return PQ2_ERR_MISALIGNED;
    if (ws && !aligned16(ws)) return PQ2_ERR_MISALIGNED;
    return PQ2_OK;
}

pq2_status pq2_gemv(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                    const void* ws_f16, float* y, int64_t N, int64_t K, void* stream) {
    pq2_status s = check_mm(qp, S, T, codes, ws_f16, y, 1, N, K);
    if (s != PQ2_OK) return s;
    if (!S || !ws_f16) return PQ2_ERR_INVALID_ARG;
    Ctx c;
    s = get_ctx(&c);
    if (s != PQ2_OK) return s;
    return cuda_status(pq2h::launch_gemv(nullptr, qp, S, T, codes,
                                         static_cast<const __half*>(ws_f16), y, nullptr, N, K,
                                         static_cast<cudaStream_t>(stream), c.ctl, c.dev));
}

size_t pq2_workspace_bytes(int op, int64_t M, int64_t N, int64_t K) {
    if (check_nk(N, K) != PQ2_OK || M < 1) return SIZE_MAX;
    switch (op) {
        case PQ2_OP_GEMV: return M == 1 ? 0 : SIZE_MAX;
        case PQ2_OP_SMALL:
            return (M >= 2 && M <= 16) ? pq2h::small_tc_workspace_bytes(M, N, K) : SIZE_MAX;
        case PQ2_OP_PREFILL: return pq2h::prefill_workspace_bytes(M, N, K);
        case PQ2_OP_SWIGLU_DOWN:  // K is the intermediate size I
        case PQ2_OP_MATMUL: {
            if (op == PQ2_OP_MATMUL && M == 1 && pq2h::gemv_fused_supported(K))
                return 0;  // fused, no scratch
            const size_t G = static_cast<size_t>(K / 128);
            const size_t act = align256(static_cast<size_t>(M) * K) +
                               2 * align256(static_cast<size_t>(M) * G * 4);
            const int inner = M == 1 ? PQ2_OP_GEMV : (M <= 16 ? PQ2_OP_SMALL : PQ2_OP_PREFILL);
            const size_t k = pq2_workspace_bytes(inner, M, N, K);
            return k == SIZE_MAX ? SIZE_MAX : act + k;
        }
        default: return SIZE_MAX;
    }
}

// pq2_gemm_small; weights_static: PQ2_WEIGHTS_STATIC of pq2_matmul_ex
static pq2_status gemm_small(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                      const void* ws_f16, float* y, int64_t M, int64_t N, int64_t K,
                      void* workspace, size_t workspace_bytes, void* stream, bool weights_static) {
    pq2_status s = check_mm(qp, S, T, codes, ws_f16, y, M, N, K);
    if (s != PQ2_OK) return s;
    if (!S || !ws_f16) return PQ2_ERR_INVALID_ARG;
    if (M < 2 || M > 16) return PQ2_ERR_UNSUPPORTED_SHAPE;
    const size_t need = pq2_workspace_bytes(PQ2_OP_SMALL, M, N, K);
    if (need > 0 && (!workspace || workspace_bytes < need)) return PQ2_ERR_WORKSPACE;
    Ctx c;
    s = get_ctx(&c);
    if (s != PQ2_OK) return s;
    if (pq2h::gemv_multi_supported(M, N, K, c.dev.num_sms))
        return cuda_status(pq2h::launch_gemv_multi(qp, S, T, codes,
                                                   static_cast<const __half*>(ws_f16), y, nullptr,
                                                   M, N, K, static_cast<cudaStream_t>(stream),
                                                   c.dev, weights_static, c.ctl));
    return cuda_status(pq2h::launch_small_tc(qp, S, T, codes, static_cast<const __half*>(ws_f16), y,
                                          nullptr, M, N, K, workspace,
                                          static_cast<cudaStream_t>(stream), c.ctl, c.dev));
}

pq2_status pq2_gemm_small(const int8_t* qp, const float* S, const int32_t* T,
                          const uint8_t* codes, const void* ws_f16, float* y, int64_t M,
                          int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                          void* stream) {
    return gemm_small(qp, S, T, codes, ws_f16, y, M, N, K, workspace, workspace_bytes, stream,
                      false);
}

pq2_status pq2_gemm_small_ex(const int8_t* qp, const float* S, const int32_t* T,
                             const uint8_t* codes, const void* ws_f16, float* y, int64_t M,
                             int64_t N, int64_t K, uint32_t flags, void* workspace,
                             size_t workspace_bytes, void* stream) {
    if (flags & ~PQ2_WEIGHTS_STATIC) return PQ2_ERR_INVALID_ARG;
    return gemm_small(qp, S, T, codes, ws_f16, y, M, N, K, workspace, workspace_bytes, stream,
                      (flags & PQ2_WEIGHTS_STATIC) != 0);
}

pq2_status pq2_gemm_prefill(const int8_t* qp, const float* S, const int32_t* T,
                            const uint8_t* codes, const void* ws_f16, float* y, int64_t M,
                            int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                            void* stream) {
    pq2_status s = check_mm(qp, S, T, codes, ws_f16, y, M, N, K);
    if (s != PQ2_OK) return s;
    if (!S || !ws_f16) return PQ2_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) - 1) return PQ2_ERR_UNSUPPORTED_SHAPE;
    const size_t need = pq2_workspace_bytes(PQ2_OP_PREFILL, M, N, K);
    if (need > 0 && (!workspace || workspace_bytes < need)) return PQ2_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PQ2_ERR_MISALIGNED;
    Ctx c;
    s = get_ctx(&c);
    if (s != PQ2_OK) return s;
    return cuda_status(pq2h::launch_prefill(qp, S, T, codes, static_cast<const __half*>(ws_f16), y,
                                            nullptr, M, N, K, workspace,
                                            static_cast<cudaStream_t>(stream), c.ctl, c.dev));
}

pq2_status pq2_matmul(const void* x_f16, const uint8_t* codes, const void* ws_f16, float* y,
                      int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                      void* stream) {
    return pq2_matmul_ex(x_f16, codes, ws_f16, y, M, N, K, 0u, workspace, workspace_bytes, stream);
}

pq2_status pq2_matmul_ex(const void* x_f16, const uint8_t* codes, const void* ws_f16, float* y,
                         int64_t M, int64_t N, int64_t K, uint32_t flags, void* workspace,
                         size_t workspace_bytes, void* stream) {
    if (flags & ~PQ2_WEIGHTS_STATIC) return PQ2_ERR_INVALID_ARG;
    pq2_status s = check_nk(N, K);
    if (s != PQ2_OK) return s;
    if (M < 1 || !x_f16 || !codes || !ws_f16 || !y) return PQ2_ERR_INVALID_ARG;
    const size_t need = pq2_workspace_bytes(PQ2_OP_MATMUL, M, N, K);
    if (need == SIZE_MAX) return PQ2_ERR_UNSUPPORTED_SHAPE;
    if (M == 1 && pq2h::gemv_fused_supported(K)) {
        // fused: the GEMV kernel quantises x itself
        if (!aligned16(x_f16) || !aligned16(codes) || !aligned16(ws_f16) || !aligned16(y))
            return PQ2_ERR_MISALIGNED;
        Ctx c;
        s = get_ctx(&c);
        if (s != PQ2_OK) return s;
        return cuda_status(pq2h::launch_gemv(static_cast<const __half*>(x_f16), nullptr, nullptr,
                                             nullptr, codes, static_cast<const __half*>(ws_f16),
                                             y, nullptr, N, K, static_cast<cudaStream_t>(stream),
                                             c.ctl, c.dev, (flags & PQ2_WEIGHTS_STATIC) != 0));
    }
    if (!workspace || workspace_bytes < need) return PQ2_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PQ2_ERR_MISALIGNED;
    const size_t G = static_cast<size_t>(K / 128);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    int8_t* qp = reinterpret_cast<int8_t*>(w);
    w += align256(static_cast<size_t>(M) * K);
    float* S = reinterpret_cast<float*>(w);
    w += align256(static_cast<size_t>(M) * G * 4);
    int32_t* T = reinterpret_cast<int32_t*>(w);
    w += align256(static_cast<size_t>(M) * G * 4);
    const size_t rest = need - static_cast<size_t>(w - static_cast<uint8_t*>(workspace));
    if (M > 1 && M <= pq2h::kTileMaxM) {
        // the token-tile tensor-core kernels: their token tiles straight from
        // x (one launch fewer; y bit-identical to quantise + the matmul)
        Ctx c;
        s = get_ctx(&c);
        if (s != PQ2_OK) return s;
        using pq2h::TokenTile;
        const TokenTile tt =
            M <= 16 ? (pq2h::small_x_supported(M, N, K, c.dev.num_sms) ? TokenTile::kSmall
                                                                       : TokenTile::kNone)
                    : pq2h::prefill_token_tile_kernel(M, N, K, c.dev.num_sms);
        if (tt != TokenTile::kNone) {
            if (!aligned16(x_f16) || !aligned16(codes) || !aligned16(ws_f16) || !aligned16(y))
                return PQ2_ERR_MISALIGNED;
            const int op = M <= 16 ? PQ2_OP_SMALL : PQ2_OP_PREFILL;
            if (rest < pq2_workspace_bytes(op, M, N, K)) return PQ2_ERR_WORKSPACE;
            const __half* xh = static_cast<const __half*>(x_f16);
            const __half* wsh = static_cast<const __half*>(ws_f16);
            const cudaStream_t st = static_cast<cudaStream_t>(stream);
            if (tt == TokenTile::kSmall)
                return cuda_status(pq2h::launch_small_x(xh, codes, wsh, y, M, N, K, w, st, c.ctl,
                                                        c.dev));
            if (tt == TokenTile::kWide)
                return cuda_status(pq2h::launch_wtile_x(xh, codes, wsh, y, M, N, K, w, st, c.ctl,
                                                        c.dev));
            return cuda_status(pq2h::launch_tile_x(xh, codes, wsh, y, M, N, K, w, st, c.ctl, c.dev));
        }
    }
    s = pq2_quantize_act(x_f16, M, K, qp, S, T, stream);
    if (s != PQ2_OK) return s;
    if (M == 1) return pq2_gemv(qp, S, T, codes, ws_f16, y, N, K, stream);
    if (M <= 16)
        return gemm_small(qp, S, T, codes, ws_f16, y, M, N, K, rest ? w : nullptr, rest, stream,
                          (flags & PQ2_WEIGHTS_STATIC) != 0);
    return pq2_gemm_prefill(qp, S, T, codes, ws_f16, y, M, N, K, rest ? w : nullptr, rest,
                            stream);
}

pq2_status pq2_mlp_down_swiglu(const float* gu, const uint8_t* codes, const void* ws_f16, float* y,
                               int64_t M, int64_t N, int64_t I, void* workspace,
                               size_t workspace_bytes, void* stream) {
    pq2_status s = check_nk(N, I);
    if (s != PQ2_OK) return s;
    if (M < 1 || !gu || !codes || !ws_f16 || !y) return PQ2_ERR_INVALID_ARG;
    const size_t need = pq2_workspace_bytes(PQ2_OP_SWIGLU_DOWN, M, N, I);
    if (need == SIZE_MAX) return PQ2_ERR_UNSUPPORTED_SHAPE;
    if (!workspace || workspace_bytes < need) return PQ2_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PQ2_ERR_MISALIGNED;
    const size_t G = static_cast<size_t>(I / 128);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    int8_t* qp = reinterpret_cast<int8_t*>(w);
    w += align256(static_cast<size_t>(M) * I);
    float* S = reinterpret_cast<float*>(w);
    w += align256(static_cast<size_t>(M) * G * 4);
    int32_t* T = reinterpret_cast<int32_t*>(w);
    w += align256(static_cast<size_t>(M) * G * 4);
    const size_t rest = need - static_cast<size_t>(w - static_cast<uint8_t*>(workspace));
    s = pq2_quantize_swiglu(gu, M, I, qp, S, T, stream);
    if (s != PQ2_OK) return s;
    if (M == 1) return pq2_gemv(qp, S, T, codes, ws_f16, y, N, I, stream);
    if (M <= 16)
        return pq2_gemm_small(qp, S, T, codes, ws_f16, y, M, N, I, rest ? w : nullptr, rest,
                              stream);
    return pq2_gemm_prefill(qp, S, T, codes, ws_f16, y, M, N, I, rest ? w : nullptr, rest,
                            stream);
}

pq2_status pq2_gemm_bf16_splitk(const uint16_t* x, const uint16_t* w, uint16_t* y, int64_t M,
                                int64_t N, int64_t K, uint32_t flags, void* stream) {
    if (M < 0 || N < 0 || K < 0) return PQ2_ERR_INVALID_ARG;
    if (flags & ~static_cast<uint32_t>(PQ2_WEIGHTS_STATIC)) return PQ2_ERR_INVALID_ARG;
    if (K % 8 != 0 || K > PQ2_MAX_K || M > PQ2_MAX_M_BF16 || N > PQ2_MAX_N_BF16)
        return PQ2_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || N == 0) return PQ2_OK;
    if (!y || (K > 0 && (!x || !w))) return PQ2_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || (reinterpret_cast<uintptr_t>(y) & 1u))
        return PQ2_ERR_MISALIGNED;
    Ctx c;
    pq2_status s = get_ctx(&c);
    if (s != PQ2_OK) return s;
    return cuda_status(pq2h::launch_bf16_splitk(x, w, y, M, N, K,
                                                (flags & PQ2_WEIGHTS_STATIC) != 0,
                                                static_cast<cudaStream_t>(stream), c.ctl));
}

pq2_status pq2_group_dots(int op, const int8_t* qp, const int32_t* T, const uint8_t* codes,
                          int64_t M, int64_t N, int64_t K, int32_t* dots, void* workspace,
                          size_t workspace_bytes, void* stream) {
    pq2_status s = check_mm(qp, nullptr, T, codes, nullptr, dots, M, N, K);
    if (s != PQ2_OK) return s;
    if (op != PQ2_OP_GEMV && op != PQ2_OP_SMALL && op != PQ2_OP_PREFILL)
        return PQ2_ERR_INVALID_ARG;
    const size_t need = pq2_workspace_bytes(op, M, N, K);
    if (need == SIZE_MAX) return PQ2_ERR_UNSUPPORTED_SHAPE;
    if (need > 0 && (!workspace || workspace_bytes < need)) return PQ2_ERR_WORKSPACE;
    Ctx c;
    s = get_ctx(&c);
    if (s != PQ2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (op == PQ2_OP_GEMV)
        return cuda_status(
            pq2h::launch_gemv(nullptr, qp, nullptr, T, codes, nullptr, nullptr, dots, N, K, st,
                              c.ctl, c.dev));
    if (op == PQ2_OP_SMALL) {
        if (pq2h::gemv_multi_supported(M, N, K, c.dev.num_sms))
            return cuda_status(pq2h::launch_gemv_multi(qp, nullptr, T, codes, nullptr, nullptr,
                                                       dots, M, N, K, st, c.dev, false, c.ctl));
        return cuda_status(pq2h::launch_small_tc(qp, nullptr, T, codes, nullptr, nullptr, dots, M, N,
                                              K, workspace, st, c.ctl, c.dev));
    }
    // the prefill path needs S only to prepare its token planes
    return cuda_status(pq2h::launch_prefill(qp, nullptr, T, codes, nullptr, nullptr, dots, M, N,
                                            K, workspace, st, c.ctl, c.dev));
}

pq2_status pq2_last_device_error(void* stream) {
    Ctx c;
    pq2_status s = get_ctx(&c);
    if (s != PQ2_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return PQ2_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, c.dev.err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PQ2_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpy(c.dev.err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return PQ2_ERR_CUDA;
    if (word & pq2::DEVERR_TIMEOUT) return PQ2_ERR_TIMEOUT;
    if (word & pq2::DEVERR_BOUNDS) return PQ2_ERR_BOUNDS;
    if (word & pq2::DEVERR_BAD_TERNARY) return PQ2_ERR_INVALID_ARG;
    return PQ2_OK;
}

}  // extern "C"
