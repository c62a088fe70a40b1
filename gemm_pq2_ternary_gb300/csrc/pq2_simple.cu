// Plain warp-per-output kernel for any M (the first correct CUDA path for
// M > 1).  Same per-group arithmetic as the M = 1 kernel ("Making a ternary
// reasoning model fast in vLLM", page "From CUDA to Triton and Gluon",
// section "One token at a time"): lane l takes groups l, l+32, ... of one
// (m, n) output, reads the 32 code bytes and 128 plane-ordered activation
// bytes of each group straight from global memory, and the warp sums the
// fp32 group terms in a fixed butterfly order.
#include "pq2_internal.h"

namespace {

template <bool DOTS>
__global__ void __launch_bounds__(256) simple_kernel(const int8_t* __restrict__ qp,
                                                     const float* __restrict__ S,
                                                     const int32_t* __restrict__ T,
                                                     const uint8_t* __restrict__ codes,
                                                     const __half* __restrict__ ws,
                                                     float* __restrict__ y,
                                                     int32_t* __restrict__ dots, int64_t M,
                                                     int64_t N, int64_t K, pq2::DevCtl ctl) {
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();
    const int G = static_cast<int>(K / 128);
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t o = warp; o < M * N; o += nwarps) {
        const int64_t m = o / N;
        const int64_t n = o - m * N;
        float acc = 0.0f;
        for (int g = lane; g < G; g += 32) {
            const uint8_t* cp = codes + n * (K / 4) + g * 32;
            const uint4 c0 = pq2::ld_nc_v4(cp), c1 = pq2::ld_nc_v4(cp + 16);
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint32_t q[32];
            const int8_t* qg = qp + m * K + g * 128;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const uint4 t = pq2::ld_nc_v4(qg + 16 * v);
                q[4 * v] = t.x;
                q[4 * v + 1] = t.y;
                q[4 * v + 2] = t.z;
                q[4 * v + 3] = t.w;
            }
            const int dot = pq2::group_codes_dot(w, q) - T[m * G + g];
            if (DOTS)
                dots[(m * N + n) * G + g] = dot;
            else
                acc = fmaf(static_cast<float>(dot) * S[m * G + g], __half2float(ws[n * G + g]),
                           acc);
        }
        if (!DOTS) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) y[m * N + n] = acc;
        }
    }
}

}  // namespace

namespace pq2h {

cudaError_t launch_simple(const int8_t* qp, const float* S, const int32_t* T,
                          const uint8_t* codes, const __half* ws, float* y, int32_t* dots,
                          int64_t M, int64_t N, int64_t K, cudaStream_t st,
                          const pq2::DevCtl& ctl, const DeviceInfo& dev) {
    const int64_t outputs = M * N;
    if (outputs == 0) return cudaSuccess;
    const int64_t want = (outputs + 7) / 8;
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 16;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    if (dots)
        return launch(simple_kernel<true>, dim3(grid), dim3(256), 0, st, true, qp, S, T, codes,
                      ws, y, dots, M, N, K, ctl);
    return launch(simple_kernel<false>, dim3(grid), dim3(256), 0, st, true, qp, S, T, codes, ws,
                  y, dots, M, N, K, ctl);
}

}  // namespace pq2h
