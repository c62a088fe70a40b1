// Activation quantisation + plane reorder, and weight packing.
//
// Quantise ("Making a ternary reasoning model fast in vLLM", page "From CUDA
// to Triton and Gluon", section "Prompt processing": one quantize kernel
// emits q [m,k] int8, s [m,G] fp32, t [m,G] int32; section "One token at a
// time": q in plane order).  Eight lanes per 128-value group, four groups per
// warp (grid-stride); the per-group step is shared with the fused M = 1 path
// (quantize_group8).
//
// Pack (same page, "One token at a time": codes 0,1,2 for -1,0,+1, four to a
// byte, weight 4*byte+s in bits 2s).  One thread per 16 ternary values.
#include "pq2_internal.h"

namespace {

__global__ void __launch_bounds__(256) quantize_kernel(const __half* __restrict__ x,
                                                       int8_t* __restrict__ qp,
                                                       float* __restrict__ S,
                                                       int32_t* __restrict__ T, int64_t groups,
                                                       pq2::DevCtl ctl) {
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int j = lane & 7;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t g0 = warp * 4; g0 < groups; g0 += nwarps * 4) {
        const int64_t g = g0 + (lane >> 3);
        const bool valid = g < groups;
        const int64_t gl = valid ? g : g0;
        const uint4* src = reinterpret_cast<const uint4*>(x + gl * 128 + 16 * j);
        const uint4 h[2] = {pq2::ld_nc_v4(src), pq2::ld_nc_v4(src + 1)};
        pq2::quantize_group8(h, j, valid, qp + gl * 128, S + gl, T + gl);
    }
}

__global__ void __launch_bounds__(256) pack_kernel(const int8_t* __restrict__ tern,
                                                   uint8_t* __restrict__ codes, int64_t chunks,
                                                   pq2::DevCtl ctl) {
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < chunks;
         i += stride) {
        const uint4 v = *reinterpret_cast<const uint4*>(tern + i * 16);
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        uint32_t out = 0;
        bool bad = false;
#pragma unroll
        for (int b = 0; b < 4; ++b) {      // output byte b <- input word b
            uint32_t byte = 0;
#pragma unroll
            for (int s = 0; s < 4; ++s) {  // weight 4*b+s, bits 2s
                const int t = static_cast<int8_t>((in[b] >> (8 * s)) & 0xFFu);
                uint32_t code = static_cast<uint32_t>(t + 1);
                if (t < -1 || t > 1) {
                    bad = true;
                    code = 3u;
                }
                byte |= code << (2 * s);
            }
            out |= byte << (8 * b);
        }
        *reinterpret_cast<uint32_t*>(codes + i * 4) = out;
        if (bad) atomicOr(ctl.err, pq2::DEVERR_BAD_TERNARY);
    }
}

}  // namespace

namespace pq2h {

cudaError_t launch_quantize(const __half* x, int8_t* qp, float* S, int32_t* T, int64_t M,
                            int64_t K, cudaStream_t st, const pq2::DevCtl& ctl,
                            const DeviceInfo& dev) {
    const int64_t groups = M * (K / 128);
    if (groups == 0) return cudaSuccess;
    const int64_t want = (groups + 31) / 32;  // 8 warps x 4 groups per block
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    return launch(quantize_kernel, dim3(grid), dim3(256), 0, st, true, x, qp, S, T, groups, ctl);
}

cudaError_t launch_pack(const int8_t* tern, uint8_t* codes, int64_t N, int64_t K,
                        cudaStream_t st, const pq2::DevCtl& ctl, const DeviceInfo& dev) {
    const int64_t chunks = N * K / 16;
    if (chunks == 0) return cudaSuccess;
    const int64_t want = (chunks + 255) / 256;
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 16;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    return launch(pack_kernel, dim3(grid), dim3(256), 0, st, true, tern, codes, chunks, ctl);
}

}  // namespace pq2h
