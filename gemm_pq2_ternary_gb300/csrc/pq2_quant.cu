// Activation quantisation + plane reorder, and weight packing.
//
// Quantise ("Making a ternary reasoning model fast in vLLM", page "From CUDA
// to Triton and Gluon", section "Prompt processing": one quantize kernel
// emits q [m,k] int8, s [m,G] fp32, t [m,G] int32; section "One token at a
// time": q in plane order).  One warp per 128-value group: lane b holds the
// four values of code byte b (weights 4b..4b+3), so plane s of the group is
// written by the 32 lanes as 32 consecutive bytes at s*32.
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
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t gi = warp; gi < groups; gi += nwarps) {
        // group gi covers x[gi*128 .. gi*128+127] (row-major [M,K], K = 128*G)
        const uint2 raw = *reinterpret_cast<const uint2*>(x + gi * 128 + 4 * lane);
        const __half2 h01 = *reinterpret_cast<const __half2*>(&raw.x);
        const __half2 h23 = *reinterpret_cast<const __half2*>(&raw.y);
        float v[4] = {__low2float(h01), __high2float(h01), __low2float(h23), __high2float(h23)};
        float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float d = __fdiv_rn(amax, 127.0f);
        int sum = 0;
        int8_t* dst = qp + gi * 128 + lane;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            int q = 0;
            if (amax != 0.0f) {
                q = __float2int_rn(__fdiv_rn(v[s], d));  // round half to even
                q = max(-127, min(127, q));
            }
            sum += q;
            dst[s * 32] = static_cast<int8_t>(q);  // weight 4*lane+s -> s*32+lane
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) {
            S[gi] = (amax != 0.0f) ? d : 0.0f;
            T[gi] = sum;
        }
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
    const int64_t want = (groups + 7) / 8;
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
