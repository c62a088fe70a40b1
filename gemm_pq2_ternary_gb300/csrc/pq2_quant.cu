// Activation quantisation + plane reorder, and weight packing.
//
// Quantise ("Making a ternary reasoning model fast in vLLM", page "From CUDA
// to Triton and Gluon", section "Prompt processing": one quantize kernel
// emits q [m,k] int8, s [m,G] fp32, t [m,G] int32; section "One token at a
// time": q in plane order).  Eight lanes per 128-value group, four groups per
// warp (grid-stride); the per-group step is shared with the fused M = 1 path
// (quantize_group8).
//
// SwiGLU + quantise (an assumed activation between the MLP projections; see
// swiglu_quantize_kernel).
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

// ---------------------------------------------------------------------------
// SwiGLU + quantise: h = silu(gate) * up of a gate/up output, rounded to fp16
// (saturating at +-65504), then quantised exactly like an fp16 activation.
// The pages do not define the MLP's activation; this is the plain reading
// h = silu(g) * u, silu(g) = g / (1 + exp(-g)), every step one IEEE fp32
// operation.  exp follows a stated method, Cody and Waite's argument
// reduction (W. J. Cody, W. Waite, "Software Manual for the Elementary
// Functions", 1980): n = rint(x log2 e); r = x - n ln2 with ln2 split into two
// fp32 parts (one fused multiply-add each); the degree-7 Taylor polynomial of
// e^r (coefficients 1/i!, Horner with fused multiply-adds); times 2^n (exact).
// x is clamped to [-87, 88] first.  Written with explicit round-to-nearest
// intrinsics so that no step is contracted or approximated.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float exp_cw(float x) {
    x = fminf(fmaxf(x, -87.0f), 88.0f);
    const float n = rintf(__fmul_rn(x, 0x1.715476p+0f));   // log2 e
    float r = __fmaf_rn(-n, 0x1.62e430p-1f, x);            // ln2, high part
    r = __fmaf_rn(-n, -0x1.05c610p-29f, r);                // ln2, low part
    float p = __fmaf_rn(0x1.a01a02p-13f, r, 0x1.6c16c2p-10f);  // 1/7!, 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);                   // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);                   // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);                   // 1/3!
    p = __fmaf_rn(p, r, 0x1.0p-1f);                        // 1/2!
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    // 2^n with n in [-126, 127]: a normal power of two, so the product is exact
    return __fmul_rn(p, __int_as_float((static_cast<int>(n) + 127) << 23));
}

__device__ __forceinline__ float swiglu1(float g, float u) {
    const float s = __fdiv_rn(g, __fadd_rn(1.0f, exp_cw(-g)));
    const float h = __fmul_rn(s, u);
    return fminf(fmaxf(h, -65504.0f), 65504.0f);  // saturate to the fp16 range
}

__device__ __forceinline__ uint32_t half2_bits(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float4 ld_nc_f4(const float* p) {
    const uint4 v = pq2::ld_nc_v4(p);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                       __uint_as_float(v.w));
}

// gu [M, 2I] fp32 (gate | up) -> qp, S, T of h [M, I].  Eight lanes per
// group of 128 h values (lane j: values 16j..16j+15), four groups per warp.
__global__ void __launch_bounds__(256) swiglu_quantize_kernel(const float* __restrict__ gu,
                                                              int8_t* __restrict__ qp,
                                                              float* __restrict__ S,
                                                              int32_t* __restrict__ T,
                                                              int64_t groups, int64_t G,
                                                              int64_t I, pq2::DevCtl ctl) {
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int j = lane & 7;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t g0 = warp * 4; g0 < groups; g0 += nwarps * 4) {
        const int64_t gi = g0 + (lane >> 3);
        const bool valid = gi < groups;
        const int64_t gl = valid ? gi : g0;
        const int64_t m = gl / G, g = gl - m * G;
        const float* gate = gu + m * 2 * I + g * 128 + 16 * j;
        const float* up = gate + I;
        uint32_t hw[8];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const float4 a = ld_nc_f4(gate + 4 * v), b = ld_nc_f4(up + 4 * v);
            hw[2 * v] = half2_bits(swiglu1(a.x, b.x), swiglu1(a.y, b.y));
            hw[2 * v + 1] = half2_bits(swiglu1(a.z, b.z), swiglu1(a.w, b.w));
        }
        const uint4 h[2] = {make_uint4(hw[0], hw[1], hw[2], hw[3]),
                            make_uint4(hw[4], hw[5], hw[6], hw[7])};
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

cudaError_t launch_quantize_swiglu(const float* gu, int8_t* qp, float* S, int32_t* T, int64_t M,
                                   int64_t I, cudaStream_t st, const pq2::DevCtl& ctl,
                                   const DeviceInfo& dev) {
    const int64_t G = I / 128;
    const int64_t groups = M * G;
    if (groups == 0) return cudaSuccess;
    const int64_t want = (groups + 31) / 32;  // 8 warps x 4 groups per block
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    return launch(swiglu_quantize_kernel, dim3(grid), dim3(256), 0, st, true, gu, qp, S, T, groups,
                  G, I, ctl);
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
