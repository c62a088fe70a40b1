// Token tiles of the tensor-core matmul kernels written straight from the
// fp16 activations (the x -> y entry points).
//
// The tensor-core kernels meet the int8 activations q as two exact e4m3
// values, 16h and l with q = 16h + l, h = floor(q / 16) ("Making a ternary
// reasoning model fast in vLLM", page "From CUDA to Triton and Gluon",
// section "Prompt processing: check configuration and launch costs": the
// prompt-side kernels take the same plane-ordered int8 q as the M = 1 path).
// Their preparation kernels read q, s and t written by pq2_quantize_act.  On
// pq2_matmul's path the kernel below quantises x itself, with the same
// per-group step as pq2_quantize_act (quantize_group8), and writes the token
// tiles, the (s, t) table and the zeroed split-K counters in one launch; q,
// s and t never reach global memory.  The tiles are therefore bit-identical
// to the two-step path's.
#pragma once

#include "pq2_common.cuh"

namespace pq2 {

// e4m3 bytes (round to nearest, saturating) of four floats, v0 in byte 0.
__device__ __forceinline__ uint32_t e4m3_word(float v0, float v1, float v2, float v3) {
    uint32_t lo, hi;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(lo) : "f"(v0), "f"(v1));
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(hi) : "f"(v2), "f"(v3));
    return lo | (hi << 16);
}

// The e4m3 words of 16 * floor(q / 16) and q - 16 * floor(q / 16) for the
// four int8 q of `qw` (both exact in e4m3).
__device__ __forceinline__ void hi_lo_words(uint32_t qw, uint32_t& hw, uint32_t& lw) {
    float h[4], l[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int q = static_cast<int8_t>((qw >> (8 * b)) & 0xFFu);
        h[b] = static_cast<float>(16 * (q >> 4));
        l[b] = static_cast<float>(q & 15);
    }
    hw = e4m3_word(h[0], h[1], h[2], h[3]);
    lw = e4m3_word(l[0], l[1], l[2], l[3]);
}

// Token tiles from x [M][K] fp16 for a kernel whose layout L gives:
//   L::MT                    token rows of a tile (16, 32 or 64)
//   L::row_hi(m), row_lo(m)  the tile rows of token m's hi and lo parts
//   L::kGroupWords           32-bit words of one group's tile (rows * 32)
//   L::put_st(st, g, m, s, t) the (s, t) table entry of (group g, token m)
// tok [G4][kGroupWords] and the table get zeros for tokens >= M and groups
// >= G; counters [n_tiles] are zeroed.  Eight lanes take one (group, token)
// pair, four pairs a warp; 256 threads a block.
template <class L>
__global__ void __launch_bounds__(256) quant_tiles_kernel(const __half* __restrict__ x,
                                                          uint32_t* __restrict__ tok,
                                                          void* __restrict__ st,
                                                          unsigned* __restrict__ counters,
                                                          int64_t M, int64_t K, int64_t G4,
                                                          int n_tiles) {
    __shared__ __align__(16) int8_t qslot[8][4][128];  // [warp][team] one group's q
    __shared__ float sslot[8][4];
    __shared__ int32_t tslot[8][4];
    pdl_wait();
    pdl_launch_dependents();
    const int64_t G = K / 128;
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int team = lane >> 3;
    const int j = lane & 7;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t pairs = G4 * L::MT;  // (group, token), token-minor
    int8_t* qs = qslot[wib][team];
    for (int64_t i0 = warp * 4; i0 < pairs; i0 += nwarps * 4) {
        const int64_t i = i0 + team;
        const int64_t g = i / L::MT;
        const int m = static_cast<int>(i - g * L::MT);
        const bool valid = i < pairs && m < M && g < G;
        // every lane takes part in the team's shuffles; a team without a
        // valid pair reads token 0's group 0 and stores nothing
        const uint4* src = reinterpret_cast<const uint4*>(
            x + (valid ? static_cast<int64_t>(m) * K + g * 128 : 0) + 16 * j);
        const uint4 h[2] = {ld_nc_v4(src), ld_nc_v4(src + 1)};
        float s_all;
        int t_all;
        quantize_group8(h, j, valid, qs, &sslot[wib][team], &tslot[wib][team], s_all, t_all);
        if (i >= pairs) continue;
        uint32_t* tg = tok + g * L::kGroupWords;
        const int rh = L::row_hi(m), rl = L::row_lo(m);
        // this lane's plane words (bytes 4j..4j+3 of plane sp): its own stores
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) {
            uint32_t hw = 0, lw = 0;
            if (valid) hi_lo_words(*reinterpret_cast<const uint32_t*>(qs + sp * 32 + 4 * j), hw, lw);
            tg[rh * 32 + sp * 8 + j] = hw;
            tg[rl * 32 + sp * 8 + j] = lw;
        }
        if (j == 0) L::put_st(st, g, m, valid ? s_all : 0.0f, valid ? static_cast<float>(t_all) : 0.0f);
    }
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t k = tid; k < n_tiles; k += nthreads) counters[k] = 0u;
}

// Blocks for quant_tiles_kernel over `pairs` (group, token) pairs.
inline unsigned quant_tiles_grid(int64_t pairs, int num_sms) {
    const int64_t want = (pairs + 31) / 32;  // 8 warps x 4 pairs per block
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    return static_cast<unsigned>(want < cap ? want : cap);
}

}  // namespace pq2
