// pq2_gemm_small_noalloc: the small-batch matmul without a caller-supplied
// workspace, for callers that cannot allocate device memory on their own --
// for example code running inside a captured CUDA graph region or a plugin
// whose host framework owns every allocation and gives it no allocator.
//
// Its split-K partial sums live in one fixed file-scope device array of
// kScratchBytes (4 MiB), which every GPU that loads this library holds until
// the process exits.  Host code cannot use the array's symbol as a device
// address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and keeps it; that first
// call should therefore come before any stream capture.  Nothing here calls
// cudaMalloc, cudaFree or any allocating routine.
//
// All calls share the one array: calls whose kernels can overlap on the GPU
// (different streams without ordering between them) race on it.  The array
// keeps the last call's partial sums; nothing in it needs to start at zero,
// since every partial sum the kernel reads is first written by the same call.
#include <mutex>

#include "../../include/pq2.h"
#include "pq2_internal.h"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_small_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device).  Returns nullptr on a CUDA error.
void* scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_small_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

size_t pq2_gemm_small_noalloc_max_scratch(void) { return kScratchBytes; }

pq2_status pq2_gemm_small_noalloc(const int8_t* qp, const float* S, const int32_t* T,
                                  const uint8_t* codes, const void* ws_f16, float* y, int64_t M,
                                  int64_t N, int64_t K, void* stream) {
    // the argument checks of pq2_gemm_small
    if (M < 1 || N < 1 || K < 1) return PQ2_ERR_INVALID_ARG;
    if (K % 128 != 0 || K > PQ2_MAX_K || N > (int64_t(1) << 31) - 1) return PQ2_ERR_UNSUPPORTED_SHAPE;
    if (M < 2 || M > 16) return PQ2_ERR_UNSUPPORTED_SHAPE;
    if (!qp || !S || !T || !codes || !ws_f16 || !y) return PQ2_ERR_INVALID_ARG;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(qp) || !a16(S) || !a16(T) || !a16(codes) || !a16(ws_f16) || !a16(y))
        return PQ2_ERR_MISALIGNED;
    // Beyond 8 tokens only the tensor-core kernel can take the call, and its
    // scratch grows with the number of 128-row tiles: a shape that does not
    // fit even with a single CTA is refused before the device is touched
    // (e.g. N = 248320 at 16 tokens needs about 16 MB).
    if (M > 8 && pq2h::small_tc_scratch_bytes(M, N, K, 1) > kScratchBytes) return PQ2_ERR_WORKSPACE;
    pq2h::DeviceInfo dev;
    pq2::DevCtl ctl;
    if (!pq2h::device_info(&dev) || !pq2h::make_ctl(&ctl)) return PQ2_ERR_CUDA;
    if (pq2h::gemv_multi_supported(M, N, K, dev.num_sms))  // needs no scratch
        return pq2h::launch_gemv_multi(qp, S, T, codes, static_cast<const __half*>(ws_f16), y,
                                       nullptr, M, N, K, static_cast<cudaStream_t>(stream),
                                       dev, false, ctl) == cudaSuccess
                   ? PQ2_OK
                   : PQ2_ERR_CUDA;
    // scratch this shape needs on this device (split-K partial sums)
    if (pq2h::small_tc_scratch_bytes(M, N, K, dev.num_sms) > kScratchBytes) return PQ2_ERR_WORKSPACE;
    void* scratch = scratch_for_current_device();
    if (!scratch) return PQ2_ERR_CUDA;
    const cudaError_t e = pq2h::launch_small_tc(qp, S, T, codes, static_cast<const __half*>(ws_f16),
                                             y, nullptr, M, N, K, scratch,
                                             static_cast<cudaStream_t>(stream), ctl, dev);
    return e == cudaSuccess ? PQ2_OK : PQ2_ERR_CUDA;
}

}  // extern "C"
