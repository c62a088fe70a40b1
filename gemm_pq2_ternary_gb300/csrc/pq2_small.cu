// Small-batch matmul, 2 <= M <= 16 token rows (pq2_gemm_small).
//
// The pages' small-batch kernels ("Making a ternary reasoning model fast in
// vLLM", page "From CUDA to Triton and Gluon", sections "Small batches: make
// the register layout explicit", "Use a ring buffer for longer rows",
// "Extend the kernels to sixteen token rows") load code bytes straight into
// the A fragments of an m16n8k32 tensor-core MMA and extract each plane with
// a shift and a mask; K splits are summed in the fixed order 0, 1, 2, ...
// (section "Choose the configuration with the proxy").
//
// GB300 design.  The int8 tensor path is a fraction of the fp8 one on this
// part, so the MMA is m16n8k32 with e4m3 operands and an fp32 accumulator,
// and stays exact:
//  * A = 16 weight rows x 32 code bytes of one plane.  A code byte masked in
//    place, w & 0x03030303 or w & 0x0C0C0C0C, read as e4m3 is the subnormal
//    c * 2^-9 or the value 4c * 2^-9 (e4m3 bytes below 16 are exactly
//    byte * 2^-9).  Planes 0,1 are masked in place, planes 2,3 after one
//    shift by 4: five integer ops per code word.
//  * B = 8 tokens x 32 activations of that plane.  An int8 q is split as
//    q = 16h + l (h in [-8,7], l in [0,15]); 16h and l (planes 0,2) or 4h and
//    l/4 (planes 1,3, which compensates the 4x of A) are exact e4m3 values.
//    Two MMAs (high, low) per plane accumulate into the same fp32 D, so
//    D = 2^-9 * sum(code * q) exactly (all partial sums are small integer
//    multiples of 2^-9).
//  * The k order inside an MMA is free as long as A and B agree: lane
//    (gid, tid) holds code words 2tid, 2tid+1 of its rows (one 8-byte load)
//    and the activation words 2tid, 2tid+1 of the same plane.
//  * Per group: dot = D*512 - sum(q) (exact in fp32), then
//    acc += dot * s * ws in fp32, as the M = 1 path.
//
// Work split: the K groups are cut into KS splits and the 16-row tiles of
// each split are shared out evenly over num_SMs/KS persistent CTAs.  A CTA
// streams, per stage, the code bytes of all its rows for a few groups (one
// 1-D bulk copy per row segment) plus the prepared B fragments of those
// groups (one bulk copy) through a shared-memory ring; four consumer warps
// own its tiles, keep each group's B fragments in registers across their
// tiles, and accumulate over the whole split in registers.  KS > 1 writes
// partial sums that a second kernel adds in split order.
#include "pq2_internal.h"

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kTilesPerWarp = 3;                       // register accumulators per warp
constexpr int kBatchTiles = kConsumerWarps * kTilesPerWarp;
constexpr int kFragBytesPerGroupTile = 4 * 2 * 32 * 8;  // planes x (hi,lo) x lanes x 8 B

__device__ __forceinline__ uint32_t pack_e4m3x4(float v0, float v1, float v2, float v3) {
    uint32_t lo, hi;
    // cvt ... e4m3x2.f32 d, a, b packs a into the upper byte, b into the lower
    asm("{\n\t.reg .b16 t;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\t"
        "cvt.u32.u16 %0, t;\n\t}"
        : "=r"(lo)
        : "f"(v0), "f"(v1));
    asm("{\n\t.reg .b16 t;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\t"
        "cvt.u32.u16 %0, t;\n\t}"
        : "=r"(hi)
        : "f"(v2), "f"(v3));
    return lo | (hi << 16);
}

// One activation word (4 int8 q, same plane s) -> its high and low e4m3
// fragment words: q = 16h + l; planes 0,2 take (16h, l), planes 1,3 take
// (4h, l/4).  All of these values are exact in e4m3.
__device__ __forceinline__ void split_word(uint32_t qw, bool quarter, uint32_t* hiw,
                                           uint32_t* low) {
    float hv[4], lv[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int q = static_cast<int8_t>((qw >> (8 * b)) & 0xFFu);
        const int hq = q >> 4;  // floor(q / 16)
        const int lq = q & 15;  // q - 16 * hq
        hv[b] = static_cast<float>(quarter ? 4 * hq : 16 * hq);
        lv[b] = quarter ? 0.25f * static_cast<float>(lq) : static_cast<float>(lq);
    }
    *hiw = pack_e4m3x4(hv[0], hv[1], hv[2], hv[3]);
    *low = pack_e4m3x4(lv[0], lv[1], lv[2], lv[3]);
}

// ---------------------------------------------------------------------------
// main kernel
// ---------------------------------------------------------------------------
struct SmallParams {
    CUtensorMap tm_codes;  // uint32 [N][K/16], box {GC*8, box_rows}
    CUtensorMap tm_qp;     // uint32 [M][K/4],  box {GC*32, 16}
    const __half* ws;
    const float* S;
    const int32_t* T;
    float* out;      // y (KS == 1) or partials [KS][M][N]
    int32_t* dots;   // debug: per-group integer dots [M][N][G]
    int M, N, K, G;
    int KS;
    int ctas_per_ks;
    int n_tiles;
    int GC;          // groups per stage
    int stages;
    int batch_rows;  // rows per batch (<= 16 * kBatchTiles)
    int box_rows;    // rows per codes box (batch_rows or half of it)
    uint32_t stage_bytes;
    uint32_t codes_stage_bytes;  // batch_rows * GC * 32
    uint32_t qp_stage_bytes;     // 16 * GC * 128
    int max_groups_per_split;
    int swizzle;     // codes tiles stored with the 128-byte TMA swizzle (GC == 4)
    pq2::DevCtl ctl;
};

__device__ __forceinline__ void mma_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int NT, bool DOTS>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, 1)
    small_kernel(const __grid_constant__ SmallParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + p.stages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + p.stages);
    const int st_off = 16 * p.stages + 16;
    float2* st_sm = reinterpret_cast<float2*>(smem + st_off);  // [groups][16] (s, t)
    const int ws_off = st_off + p.max_groups_per_split * 16 * 8;
    __half* ws_sm = reinterpret_cast<__half*>(smem + ws_off);  // [batch_rows][groups]
    // stages start on 1024-byte boundaries (the swizzle pattern follows the
    // shared-memory address bits)
    const uint32_t base_addr = pq2::smem_u32(smem);
    const uint32_t ring_addr =
        (base_addr + ws_off + p.batch_rows * p.max_groups_per_split * 2 + 1023) & ~1023u;
    uint8_t* ring = smem + (ring_addr - base_addr);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int ks = blockIdx.x / p.ctas_per_ks;
    const int cj = blockIdx.x - ks * p.ctas_per_ks;
    const int t0 = static_cast<int>((static_cast<long long>(p.n_tiles) * cj) / p.ctas_per_ks);
    const int t1 = static_cast<int>((static_cast<long long>(p.n_tiles) * (cj + 1)) / p.ctas_per_ks);
    const int g0 = (p.G * ks) / p.KS;
    const int g1 = (p.G * (ks + 1)) / p.KS;
    if (t0 >= t1 || g0 >= g1) return;
    const int n_groups = g1 - g0;
    const int n_gstages = (n_groups + p.GC - 1) / p.GC;
    const int batch_tiles = p.batch_rows / 16;
    const int n_batches = (t1 - t0 + batch_tiles - 1) / batch_tiles;
    const int total_stages = n_batches * n_gstages;

    if (tid == 0) {
        for (int i = 0; i < p.stages; ++i) {
            pq2::mbar_init(&full[i], 1);
            pq2::mbar_init(&empty[i], kConsumerWarps);
        }
        *abort_flag = 0;
        pq2::fence_mbar_init();
    }
    __syncthreads();
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane != 0) return;
        const int n_boxes = p.batch_rows / p.box_rows;
        const uint32_t tx = p.codes_stage_bytes + p.qp_stage_bytes;
        int issued_end = 0;
        for (int i = 0; i < total_stages; ++i) {
            const int slot = i % p.stages;
            if (i >= p.stages &&
                !pq2::mbar_wait_bounded(&empty[slot], ((i / p.stages) - 1) & 1, p.ctl, abort_flag))
                break;
            issued_end = i + 1;
            if (i == p.ctl.debug_skip_stage) continue;
            const int b = i / n_gstages;
            const int gs = i - b * n_gstages;
            const int row0 = (t0 + b * batch_tiles) * 16;
            const int ga = g0 + gs * p.GC;
            uint8_t* cdst = ring + static_cast<size_t>(slot) * p.stage_bytes;
            pq2::mbar_arrive_expect_tx(&full[slot], tx);
            for (int bx = 0; bx < n_boxes; ++bx)
                pq2::tma_load_2d(cdst + static_cast<size_t>(bx) * p.box_rows * p.GC * 32,
                                 &p.tm_codes, ga * 8, row0 + bx * p.box_rows, &full[slot]);
            pq2::tma_load_2d(cdst + p.codes_stage_bytes, &p.tm_qp, ga * 32, 0, &full[slot]);
        }
        for (int s = 0; s < p.stages; ++s) {
            if (issued_end <= s) continue;
            int last = s + ((issued_end - 1 - s) / p.stages) * p.stages;
            if (last == p.ctl.debug_skip_stage) last -= p.stages;
            if (last >= 0) pq2::mbar_wait_bounded(&full[s], (last / p.stages) & 1, p.ctl);
        }
        return;
    }

    // -------------------------------- consumers -------------------------------
    constexpr int kCT = kConsumerWarps * 32;
    for (int i = tid; i < n_groups * 16; i += kCT) {
        const int gl = i >> 4, m = i & 15;
        float2 v = make_float2(0.0f, 0.0f);
        if (m < p.M) {
            const size_t idx = static_cast<size_t>(m) * p.G + g0 + gl;
            v = make_float2(DOTS ? 0.0f : p.S[idx], static_cast<float>(p.T[idx]));
        }
        st_sm[i] = v;
    }

    const int gid = lane >> 2;
    const int tq = lane & 3;
    bool failed = false;
    for (int b = 0; b < n_batches; ++b) {
        const int tb0 = t0 + b * batch_tiles;
        const int ntile = min(batch_tiles, t1 - tb0);
        // this batch's weight scales, [row][group of the split]
        if (!DOTS) {
            pq2::named_bar_sync(1, kCT);  // previous batch done with ws_sm
            // one warp per row, lanes over the split's groups, 4 rows in flight
            const int rows = ntile * 16;
            for (int r0 = warp * 4; r0 < rows; r0 += kConsumerWarps * 4)
                for (int c0 = 0; c0 < n_groups; c0 += 32) {
                    const int gl = c0 + lane;
                    __half v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int n = tb0 * 16 + r0 + u;
                        v[u] = (r0 + u < rows && n < p.N && gl < n_groups)
                                   ? p.ws[static_cast<size_t>(n) * p.G + g0 + gl]
                                   : __float2half(0.0f);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (r0 + u < rows && gl < n_groups)
                            ws_sm[(r0 + u) * p.max_groups_per_split + gl] = v[u];
                }
        }
        pq2::named_bar_sync(1, kCT);
        float acc[kTilesPerWarp][NT][4];
#pragma unroll
        for (int j = 0; j < kTilesPerWarp; ++j)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[j][nt][e] = 0.0f;

        for (int gs = 0; gs < n_gstages; ++gs) {
            const int i = b * n_gstages + gs;
            const int slot = i % p.stages;
            if (!failed &&
                !pq2::mbar_wait_bounded(&full[slot], (i / p.stages) & 1, p.ctl, abort_flag)) {
                failed = true;
                *abort_flag = 1;
            }
            uint8_t* cst = ring + static_cast<size_t>(slot) * p.stage_bytes;
            const uint8_t* qst = cst + p.codes_stage_bytes;
            uint32_t* fst = reinterpret_cast<uint32_t*>(cst + p.codes_stage_bytes + p.qp_stage_bytes);
            const int ga = g0 + gs * p.GC;
            const int gcs = min(p.GC, g1 - ga);
            if (!failed) {
                // B fragments of this stage's groups from the staged activations:
                // frag word ((((gl*NT + nt)*4 + s)*2 + h)*32 + lane)*2 + r
                // one thread per activation word, in the staged row-major order
                // qst[m][gl*32 + s*8 + 2*tid + r] (conflict-free reads)
                const int words_per_row = p.GC * 32;
                const int nwords = NT * 8 * words_per_row;
                for (int w = tid; w < nwords; w += kCT) {
                    const int m = w / words_per_row;
                    const int c = w - m * words_per_row;
                    const int gl = c >> 5;
                    if (gl >= gcs) continue;
                    const int s = (c >> 3) & 3;
                    const int tq2 = (c >> 1) & 3;
                    const int r = c & 1;
                    const uint32_t qw = reinterpret_cast<const uint32_t*>(qst)[w];
                    uint32_t hw, lw;
                    split_word(qw, (s & 1) != 0, &hw, &lw);
                    const int nt = m >> 3;
                    const int ln = ((m & 7) << 2) | tq2;
                    const int base = (((gl * NT + nt) * 4 + s) * 2) * 64 + ln * 2 + r;
                    fst[base] = hw;
                    fst[base + 64] = lw;
                }
            }
            const bool any_fail = pq2::named_bar_any(1, kCT, failed);
            if (any_fail) {
                failed = true;
            } else {
                for (int gl = 0; gl < gcs; ++gl) {
                    const int g = ga + gl;
                    uint32_t bf[NT][4][2][2];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int s = 0; s < 4; ++s)
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const uint2 v = reinterpret_cast<const uint2*>(
                                    fst + (((gl * NT + nt) * 4 + s) * 2 + h) * 64)[lane];
                                bf[nt][s][h][0] = v.x;
                                bf[nt][s][h][1] = v.y;
                            }
                    float s_tok[NT][2], t_tok[NT][2];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const float4 st = *reinterpret_cast<const float4*>(
                            &st_sm[(g - g0) * 16 + nt * 8 + 2 * tq]);
                        s_tok[nt][0] = st.x;
                        t_tok[nt][0] = st.y;
                        s_tok[nt][1] = st.z;
                        t_tok[nt][1] = st.w;
                    }
                    // A fragments of this warp's tiles for this group
                    uint32_t a[kTilesPerWarp][4][4];
                    bool tv[kTilesPerWarp];
#pragma unroll
                    for (int j = 0; j < kTilesPerWarp; ++j) {
                        const int tb = warp + kConsumerWarps * j;
                        tv[j] = tb < ntile;
                        const int ra = (tv[j] ? tb : 0) * 16 + gid;
                        uint32_t oa = static_cast<uint32_t>(ra) * p.GC * 32 + gl * 32 + 8 * tq;
                        uint32_t ob = oa + 8u * p.GC * 32;
                        if (p.swizzle) {  // 16-byte chunk index ^= row % 8
                            oa ^= ((oa >> 7) & 7u) << 4;
                            ob ^= ((ob >> 7) & 7u) << 4;
                        }
                        const uint2 c0 = *reinterpret_cast<const uint2*>(cst + oa);
                        const uint2 c1 = *reinterpret_cast<const uint2*>(cst + ob);
                        const uint32_t s0x = c0.x >> 4, s0y = c0.y >> 4, s1x = c1.x >> 4,
                                       s1y = c1.y >> 4;
                        a[j][0][0] = c0.x & 0x03030303u; a[j][0][1] = c1.x & 0x03030303u;
                        a[j][0][2] = c0.y & 0x03030303u; a[j][0][3] = c1.y & 0x03030303u;
                        a[j][1][0] = c0.x & 0x0C0C0C0Cu; a[j][1][1] = c1.x & 0x0C0C0C0Cu;
                        a[j][1][2] = c0.y & 0x0C0C0C0Cu; a[j][1][3] = c1.y & 0x0C0C0C0Cu;
                        a[j][2][0] = s0x & 0x03030303u;  a[j][2][1] = s1x & 0x03030303u;
                        a[j][2][2] = s0y & 0x03030303u;  a[j][2][3] = s1y & 0x03030303u;
                        a[j][3][0] = s0x & 0x0C0C0C0Cu;  a[j][3][1] = s1x & 0x0C0C0C0Cu;
                        a[j][3][2] = s0y & 0x0C0C0C0Cu;  a[j][3][3] = s1y & 0x0C0C0C0Cu;
                    }
                    // MMAs issued tile-interleaved: consecutive MMAs are independent
                    float d[kTilesPerWarp][NT][4];
#pragma unroll
                    for (int j = 0; j < kTilesPerWarp; ++j)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) d[j][nt][e] = 0.0f;
#pragma unroll
                    for (int s = 0; s < 4; ++s)
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int j = 0; j < kTilesPerWarp; ++j)
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
                                    if (tv[j]) mma_e4m3(d[j][nt], a[j][s], bf[nt][s][h][0], bf[nt][s][h][1]);
#pragma unroll
                    for (int j = 0; j < kTilesPerWarp; ++j) {
                        if (!tv[j]) continue;
                        const int ra = (warp + kConsumerWarps * j) * 16 + gid;
                        float wsa = 0.0f, wsb = 0.0f;
                        if (!DOTS) {
                            wsa = __half2float(ws_sm[ra * p.max_groups_per_split + (g - g0)]);
                            wsb = __half2float(ws_sm[(ra + 8) * p.max_groups_per_split + (g - g0)]);
                        }
                        const int na = tb0 * 16 + ra;  // global rows
                        const int nb = na + 8;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            // exact integer group dots, then the fp32 group term
                            const float dot0 = fmaf(d[j][nt][0], 512.0f, -t_tok[nt][0]);
                            const float dot1 = fmaf(d[j][nt][1], 512.0f, -t_tok[nt][1]);
                            const float dot2 = fmaf(d[j][nt][2], 512.0f, -t_tok[nt][0]);
                            const float dot3 = fmaf(d[j][nt][3], 512.0f, -t_tok[nt][1]);
                            if (DOTS) {
                                const int m0 = nt * 8 + 2 * tq;
                                const size_t G = p.G;
                                if (m0 < p.M && na < p.N)
                                    p.dots[(static_cast<size_t>(m0) * p.N + na) * G + g] = static_cast<int>(dot0);
                                if (m0 + 1 < p.M && na < p.N)
                                    p.dots[(static_cast<size_t>(m0 + 1) * p.N + na) * G + g] = static_cast<int>(dot1);
                                if (m0 < p.M && nb < p.N)
                                    p.dots[(static_cast<size_t>(m0) * p.N + nb) * G + g] = static_cast<int>(dot2);
                                if (m0 + 1 < p.M && nb < p.N)
                                    p.dots[(static_cast<size_t>(m0 + 1) * p.N + nb) * G + g] = static_cast<int>(dot3);
                            } else {
                                acc[j][nt][0] = fmaf(dot0 * s_tok[nt][0], wsa, acc[j][nt][0]);
                                acc[j][nt][1] = fmaf(dot1 * s_tok[nt][1], wsa, acc[j][nt][1]);
                                acc[j][nt][2] = fmaf(dot2 * s_tok[nt][0], wsb, acc[j][nt][2]);
                                acc[j][nt][3] = fmaf(dot3 * s_tok[nt][1], wsb, acc[j][nt][3]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) pq2::mbar_arrive(&empty[slot]);
        }
        if (failed) continue;  // keep the barrier schedule; nothing is written
        if (!DOTS) {
            float* out = p.out + static_cast<size_t>(ks) * p.M * p.N;
#pragma unroll
            for (int j = 0; j < kTilesPerWarp; ++j) {
                const int tb = warp + kConsumerWarps * j;
                if (tb >= ntile) break;
                const int na = (tb0 + tb) * 16 + gid;
                const int nb = na + 8;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int m0 = nt * 8 + 2 * tq;
                    if (m0 < p.M) {
                        if (na < p.N) out[static_cast<size_t>(m0) * p.N + na] = acc[j][nt][0];
                        if (nb < p.N) out[static_cast<size_t>(m0) * p.N + nb] = acc[j][nt][2];
                    }
                    if (m0 + 1 < p.M) {
                        if (na < p.N) out[static_cast<size_t>(m0 + 1) * p.N + na] = acc[j][nt][1];
                        if (nb < p.N) out[static_cast<size_t>(m0 + 1) * p.N + nb] = acc[j][nt][3];
                    }
                }
            }
        }
    }
}

// y[i] = sum over splits in order 0, 1, ..., KS-1 of P[split][i]
__global__ void __launch_bounds__(256) reduce_splits_kernel(const float* __restrict__ P,
                                                            float* __restrict__ y, int64_t n,
                                                            int KS) {
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        float s = P[i];
        for (int k = 1; k < KS; ++k) s += P[static_cast<int64_t>(k) * n + i];
        y[i] = s;
    }
}

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

struct SmallPlan {
    int NT, KS, ctas_per_ks, n_tiles, GC, stages, batch_rows, box_rows, swizzle;
    uint32_t stage_bytes, codes_stage_bytes, qp_stage_bytes;
    int max_groups_per_split;
    size_t smem;
    size_t partial_bytes;
};

SmallPlan plan_small(int64_t M, int64_t N, int64_t K, int num_sms) {
    SmallPlan pl = {};
    const int G = static_cast<int>(K / 128);
    pl.NT = M <= 8 ? 1 : 2;
    pl.n_tiles = static_cast<int>((N + 15) / 16);
    // fewest K splits (<= 8) that still give every CTA >= 12 tiles of work
    int KS = 1;
    while (KS < 8 && static_cast<long long>(pl.n_tiles) * KS < 12LL * num_sms && G / (2 * KS) >= 2)
        KS *= 2;
    if (KS > G) KS = G;
    pl.KS = KS;
    pl.ctas_per_ks = num_sms / KS > 0 ? num_sms / KS : 1;
    pl.max_groups_per_split = (G + KS - 1) / KS;
    const int tiles_per_cta = (pl.n_tiles + pl.ctas_per_ks - 1) / pl.ctas_per_ks;
    const int bt = tiles_per_cta < kBatchTiles ? tiles_per_cta : kBatchTiles;
    pl.batch_rows = bt * 16;
    // a TMA box holds at most 256 rows: one box, or two equal halves
    pl.box_rows = pl.batch_rows <= 256 ? pl.batch_rows : pl.batch_rows / 2;
    int GC = 4;
    if (GC > pl.max_groups_per_split) GC = pl.max_groups_per_split;
    pl.GC = GC;
    pl.swizzle = GC == 4 ? 1 : 0;
    pl.codes_stage_bytes = static_cast<uint32_t>(pl.batch_rows * GC * 32);
    pl.qp_stage_bytes = static_cast<uint32_t>(16 * GC * 128);
    pl.stage_bytes = (pl.codes_stage_bytes + pl.qp_stage_bytes +
                      static_cast<uint32_t>(GC * pl.NT * kFragBytesPerGroupTile) + 1023u) & ~1023u;
    auto head = [&](int stages) {
        return (16 * static_cast<size_t>(stages) + 16 +
                static_cast<size_t>(pl.max_groups_per_split) * 16 * 8 +
                static_cast<size_t>(pl.batch_rows) * pl.max_groups_per_split * 2 + 127) &
               ~static_cast<size_t>(127);
    };
    int stages = static_cast<int>((206 * 1024 - head(4)) / pl.stage_bytes);
    if (stages > 4) stages = 4;
    if (stages < 2) stages = 2;
    pl.stages = stages;
    pl.smem = head(stages) + 1024 + static_cast<size_t>(stages) * pl.stage_bytes;
    pl.partial_bytes = KS > 1 ? align256(static_cast<size_t>(KS) * M * N * 4) : 0;
    return pl;
}

template <int NT, bool DOTS>
cudaError_t launch_main(const SmallParams& p, const SmallPlan& pl, cudaStream_t st) {
    auto kern = small_kernel<NT, DOTS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(pl.smem));
    if (e != cudaSuccess) return e;
    return pq2h::launch(kern, dim3(pl.KS * pl.ctas_per_ks), dim3((kConsumerWarps + 1) * 32), pl.smem,
                        st, true, p);
}

}  // namespace

namespace pq2h {

// Exact scratch (split-K partial sums) for this shape on a device with
// num_sms multiprocessors.
size_t small_scratch_bytes(int64_t M, int64_t N, int64_t K, int num_sms) {
    return plan_small(M, N, K, num_sms).partial_bytes;
}

// Device-independent upper bound: partial sums for the largest split count
// the planner uses (8).
size_t small_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    (void)K;
    return align256(static_cast<size_t>(8) * M * N * 4);
}

cudaError_t launch_small(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                         const __half* ws, float* y, int32_t* dots, int64_t M, int64_t N,
                         int64_t K, void* workspace, cudaStream_t st, const pq2::DevCtl& ctl,
                         const DeviceInfo& dev) {
    const SmallPlan pl = plan_small(M, N, K, dev.num_sms);
    if (pl.smem > static_cast<size_t>(dev.max_smem_optin)) return cudaErrorInvalidConfiguration;
    float* partial = static_cast<float*>(workspace);
    SmallParams p = {};
    if (!encode_tmap_2d(&p.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, codes,
                        static_cast<uint64_t>(K / 16), static_cast<uint64_t>(N),
                        static_cast<uint64_t>(K / 4), static_cast<uint32_t>(pl.GC * 8),
                        static_cast<uint32_t>(pl.box_rows), pl.swizzle != 0))
        return cudaErrorInvalidValue;
    if (!encode_tmap_2d(&p.tm_qp, CU_TENSOR_MAP_DATA_TYPE_UINT32, qp, static_cast<uint64_t>(K / 4),
                        static_cast<uint64_t>(M), static_cast<uint64_t>(K),
                        static_cast<uint32_t>(pl.GC * 32), 16u, false))
        return cudaErrorInvalidValue;
    p.ws = ws;
    p.S = S;
    p.T = T;
    p.out = (pl.KS > 1 && !dots) ? partial : y;
    p.dots = dots;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.G = static_cast<int>(K / 128);
    p.KS = pl.KS;
    p.ctas_per_ks = pl.ctas_per_ks;
    p.n_tiles = pl.n_tiles;
    p.GC = pl.GC;
    p.stages = pl.stages;
    p.batch_rows = pl.batch_rows;
    p.box_rows = pl.box_rows;
    p.stage_bytes = pl.stage_bytes;
    p.codes_stage_bytes = pl.codes_stage_bytes;
    p.qp_stage_bytes = pl.qp_stage_bytes;
    p.max_groups_per_split = pl.max_groups_per_split;
    p.swizzle = pl.swizzle;
    p.ctl = ctl;
    cudaError_t e;
    if (pl.NT == 1)
        e = dots ? launch_main<1, true>(p, pl, st) : launch_main<1, false>(p, pl, st);
    else
        e = dots ? launch_main<2, true>(p, pl, st) : launch_main<2, false>(p, pl, st);
    if (e != cudaSuccess || dots || pl.KS == 1) return e;
    const int64_t n = M * N;
    const int64_t want = (n + 255) / 256;
    const int grid = static_cast<int>(want < dev.num_sms * 8 ? want : dev.num_sms * 8);
    return launch(reduce_splits_kernel, dim3(grid), dim3(256), 0, st, true,
                  static_cast<const float*>(partial), y, n, pl.KS);
}

}  // namespace pq2h
