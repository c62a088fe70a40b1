// Small-batch matmul, 2 <= M <= 16 tokens (pq2_gemm_small), on the
// 5th-generation tensor cores (tcgen05, operands and accumulators in tensor
// memory).
//
// The method is the pages' small-batch kernels ("Making a ternary reasoning
// model fast in vLLM", page "From CUDA to Triton and Gluon", sections "Small
// batches: make the register layout explicit" and "Extend the kernels to
// sixteen token rows"): the planes of the code bytes go straight to the
// tensor cores, which meet them with the int8 activations of all token rows
// at once, one exact integer dot per (row, token, group); then the same
// per-group -sum(q) correction and fp32 dequantise-accumulate as the M = 1
// path.  Split partial sums are combined in a fixed order (section "Choose
// the configuration with the proxy").
//
// GB300 design.  tcgen05 has no int8 kind on sm_103a; kind::f8f6f4 with e4m3
// operands is exact here (as in the prefill kernel):
//  * weights = A operand (M = 128 rows per tile), kept in TENSOR MEMORY: each
//    thread owns one weight row (one TMEM lane) and writes plane s of its
//    code words, (w >> 2s) & 0x03030303, as e4m3 bytes (bytes below 16 are
//    exactly byte * 2^-9) with tcgen05.st.  No shared-memory round trip for
//    the expanded weights;
//  * tokens = B operand: q = 16h + l, with 16h and l exact e4m3 values.  A
//    per-call preparation kernel writes, per group, one 32 x 128-byte tile
//    holding the hi and the lo parts of tokens 0..15 (zero past M).  So one
//    MMA with N = 32 per k-step gives the hi and lo partial dots side by side
//    in D, and D_hi + D_lo = 2^-9 * dot(codes, q) exactly;
//  * per group, 4 k-steps: the k order inside a group is the plane order of
//    the activations, so k-step s is plane s (8 A columns);
//  * epilogue: dot = (D_hi + D_lo) * 512 - t (an exact integer), then
//    acc += dot * s * ws in registers (the integer-dot debug output writes
//    dot itself); the 16 tokens of a weight row split over four warps.  The
//    B rows are ordered [hi of tokens 0-3, lo of tokens 0-3, hi 4-7, lo 4-7,
//    ...], so a warp's 4 tokens are 8 adjacent D columns.
//
// Items are (row tile, quad of 4 groups): one item's codes are a 128-row x
// 128-byte box (whole lines for the TMA engine, 128-byte swizzle) and its
// token tiles one 128-row box of the prepared tensor.  The items are cut
// into contiguous, balanced ranges, one per CTA (one CTA per SM).  A CTA
// flushes its accumulators at each row-tile boundary of its range: a tile
// owned by a single CTA is written straight to y; otherwise each contributor
// writes its partial sums and bumps the tile's counter, and the last one to
// arrive sums the partials of all contributors in CTA order and writes y
// (deterministic: the order is fixed, not the arrival order).
//
// Per CTA:
//   warp 0      producer: per item, TMA loads of the code box and the token
//               tiles, one bulk copy of the tokens' (s, t); its 32 lanes load
//               the 128 rows' weight scales (two items ahead) into the stage
//   warp 1      TMEM allocation; MMA issuer (one thread)
//   warp 2      second MMA issuer (one thread): the item's groups are split
//               between the two
//   warps 3-18  workers: expansion of item i (codes -> A in TMEM; the four
//               warps of a lane quadrant take one group each), then the
//               epilogue of item i-1 (the four warps take 4 tokens each)
// Every mbarrier wait is bounded (device error word on expiry).
#include "pq2_internal.h"
#include "pq2_tokens.cuh"

namespace {

constexpr int kRows = 128;            // weight rows per tile (MMA M)
constexpr int kTok = 16;              // token rows of B per plane (hi, lo)
constexpr int kGQ = 4;                // groups per item
constexpr int kStages = 4;            // TMA ring
constexpr int kBufs = 2;              // A and D buffers in TMEM, per item
constexpr int kWorkerWarps = 16;      // four per TMEM lane quadrant
#ifndef PQ2_SMALL_ISSUERS
#define PQ2_SMALL_ISSUERS 2
#endif
constexpr int kIssuers = PQ2_SMALL_ISSUERS;  // MMA-issuing warps (1, 2 or 4), groups split among them
constexpr int kWorker0 = 1 + kIssuers;       // first worker warp
constexpr int kTokPerWarp = 4;        // epilogue tokens per worker warp
constexpr int kWorkerThreads = kWorkerWarps * 32;
constexpr int kThreads = (kWorker0 + kWorkerWarps) * 32;
constexpr uint32_t kTmemCols = 512;   // A: 2 items x 4 groups x 32; D: 2 x 4 x 32
constexpr uint32_t kGCols = 32;       // TMEM columns per group (A: K = 128 e4m3; D: N = 32 fp32)
constexpr uint32_t kDCol0 = kBufs * kGQ * kGCols;  // 256
constexpr int kMaxGrid = 256;         // CTAs per call at most (bounds the partial-sum slots)
constexpr int kWsAhead = 2;           // items ahead the producer loads weight scales
constexpr int kFlushBatch = 8;        // contributors whose partials the last one loads at once

constexpr uint32_t kCodesBytes = kRows * 128;          // 4 groups x 32 B per row, swizzled
constexpr uint32_t kTokGroupBytes = 2 * kTok * 128;    // 32 rows x 128 B per group
constexpr uint32_t kTokOff = kCodesBytes;
constexpr uint32_t kStOff = kTokOff + kGQ * kTokGroupBytes;  // (s, t): 4 groups x 16 tokens
constexpr uint32_t kWsOff = kStOff + kGQ * kTok * 8;         // ws: 4 groups x 128 rows, fp32
constexpr uint32_t kTmaBytes = kStOff + kGQ * kTok * 8;      // bytes the TMA engine brings
constexpr uint32_t kStageBytes = 35840;                      // multiple of 1024
static_assert(kWsOff + kGQ * kRows * 4 <= kStageBytes, "stage layout");

struct SmallParams {
    CUtensorMap tm_codes;  // uint8 [N][K/4], box {128, 128}, 128B swizzle
    CUtensorMap tm_tok;    // uint8 [G4 * 32][128], box {128, 128}, 128B swizzle
    const float2* st16;    // [G4][16] (s, t) pairs, zero past M and past G
    const __half* ws;      // [N][G]
    float* y;              // [M][N]
    int32_t* dots;         // debug: [M][N][G]
    float* partial;        // [grid + n_tiles][M][128]
    unsigned* counters;    // [n_tiles], zero on entry
    int M, N, K, G;
    int Q;                 // quads per row tile: ceil(G / 4)
    int n_tiles;
    int grid;
    long long items;       // n_tiles * Q
    pq2::DevCtl ctl;
};

// First item of CTA c; CTA owning item i (the inverse of the split).
__host__ __device__ __forceinline__ long long range_begin(long long c, long long items, int grid) {
    return c * items / grid;
}
__host__ __device__ __forceinline__ int owner_of(long long i, long long items, int grid) {
    return static_cast<int>(((i + 1) * grid - 1) / items);
}

// ---------------------------------------------------------------------------
// per-call preparation: token tiles, (s, t) table, tile counters
// ---------------------------------------------------------------------------
// tok [G4][32][128]: token m's e4m3(16h) in row 8*(m/4) + m%4 and its
// e4m3(l) in row 8*(m/4) + 4 + m%4 (q = 16h + l, h = floor(q/16)); zero for
// tokens >= M and groups >= G.  st16 [G4][16]: (s, t), or (0, t) when S is
// null (the integer-dot debug output); zero likewise.
__global__ void __launch_bounds__(256) small_prep_kernel(const int8_t* __restrict__ qp,
                                                         const float* __restrict__ S,
                                                         const int32_t* __restrict__ T,
                                                         uint32_t* __restrict__ tok,
                                                         float2* __restrict__ st16,
                                                         unsigned* __restrict__ counters,
                                                         int64_t M, int64_t K, int64_t G4,
                                                         int n_tiles) {
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();
    const int64_t G = K / 128;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    // one index = one 4-byte word of one token of one group (hi and lo together)
    const int64_t words = G4 * kTok * 32;
    for (int64_t i = i0; i < words; i += stride) {
        const int64_t g = i / (kTok * 32);
        const int m = static_cast<int>((i / 32) % kTok);
        const int wq = static_cast<int>(i % 32);
        uint32_t hw = 0, lw = 0;
        if (m < M && g < G) {
            const uint32_t qw = reinterpret_cast<const uint32_t*>(qp + m * K + g * 128)[wq];
            pq2::hi_lo_words(qw, hw, lw);  // e4m3 of 16 * floor(q / 16), q mod 16
        }
        uint32_t* tg = tok + g * (2 * kTok * 32);
        const int rh = 8 * (m / 4) + (m % 4);
        tg[rh * 32 + wq] = hw;
        tg[(rh + 4) * 32 + wq] = lw;
    }
    for (int64_t i = i0; i < G4 * kTok; i += stride) {
        const int64_t g = i / kTok, m = i - g * kTok;
        float2 v = make_float2(0.0f, 0.0f);
        if (m < M && g < G) {
            const float t = static_cast<float>(T[m * G + g]);
            v = make_float2(S ? S[m * G + g] : 0.0f, t);
        }
        st16[i] = v;
    }
    for (int64_t i = i0; i < n_tiles; i += stride) counters[i] = 0u;
}

// Layout of the token tiles for quant_tiles_kernel (pq2_matmul's path: the
// same tiles, (s, t) table and counters straight from the fp16 activations).
struct SmallTok {
    static constexpr int MT = kTok;
    static constexpr int kGroupWords = 2 * kTok * 32;
    __device__ static int row_hi(int m) { return 8 * (m / 4) + (m % 4); }
    __device__ static int row_lo(int m) { return 8 * (m / 4) + (m % 4) + 4; }
    __device__ static void put_st(void* st, int64_t g, int m, float s, float t) {
        static_cast<float2*>(st)[g * kTok + m] = make_float2(s, t);
    }
};

// ---------------------------------------------------------------------------
// tcgen05 helpers
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1) << 16;          // leading offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;  // stride offset
    d |= static_cast<uint64_t>(1) << 46;          // descriptor version
    d |= static_cast<uint64_t>(2) << 61;          // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f8f6f4: D f32, A and B e4m3, K-major,
// M = 128, N = 32 (the hi and lo token rows of one group).
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) |
                            (static_cast<uint32_t>((2 * kTok) >> 3) << 17) |
                            (static_cast<uint32_t>(kRows >> 4) << 24);

// D (tensor memory) += A (tensor memory) x B (shared memory descriptor).
__device__ __forceinline__ void mma_f8_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(kIdesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            pq2::smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]));
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float ld_cg(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// main kernel
// ---------------------------------------------------------------------------
template <bool DOTS>
__global__ void __launch_bounds__(kThreads, 1) small_kernel(const __grid_constant__ SmallParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t full[kStages];    // stage landed: TMA bytes + the producer's 32 lanes
    __shared__ uint64_t sfree[kStages];   // stage consumed: 8 worker warps, after the item's
                                          // epilogue (so after its MMAs, which read the tokens)
    __shared__ uint64_t aready[kBufs];    // expanded weights written to TMEM (8 worker warps)
    __shared__ uint64_t dfull[kBufs];     // the item's MMAs are done (commit): D holds its dots
                                          // and its A buffer may be rewritten
    __shared__ uint64_t dfree[kBufs];     // epilogue done reading a D buffer (8 worker warps)
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ int last_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t base = pq2::smem_u32(smem);
    uint8_t* stage0 = smem + ((1024 - (base & 1023)) & 1023);
    const uint32_t stage0_s = pq2::smem_u32(stage0);

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            pq2::mbar_init(&full[i], 1 + 32);
            pq2::mbar_init(&sfree[i], kWorkerWarps);
        }
        for (int i = 0; i < kBufs; ++i) {
            pq2::mbar_init(&aready[i], kWorkerWarps);
            pq2::mbar_init(&dfull[i], kIssuers);  // one commit per issuer
            pq2::mbar_init(&dfree[i], kWorkerWarps);
        }
        abort_flag = 0;
        pq2::fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         pq2::smem_u32(&tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();

    const uint32_t tmem = tmem_base;
    const int G = p.G, Q = p.Q;
    const long long w0 = range_begin(blockIdx.x, p.items, p.grid);
    const long long w1 = range_begin(blockIdx.x + 1, p.items, p.grid);
    const int n = static_cast<int>(w1 - w0);
    // (tile, quad) of the first item; later items advance it incrementally
    // (a 64-bit division per item costs hundreds of cycles)
    const int t_first = static_cast<int>(w0 / Q);
    const int q_first = static_cast<int>(w0 - static_cast<long long>(t_first) * Q);
    volatile int* abort_v = &abort_flag;

    if (warp == 0) {
        // -------------------------------- producer --------------------------------
        // Weight scales of rows 4*lane .. 4*lane+3 of an item's tile, its 4
        // groups, are read kWsAhead items before they are stored into the
        // item's stage, so the loads' latency overlaps (raw fp16 registers;
        // the loop is unrolled so that each slot is a fixed register set:
        // moving a register whose load is in flight would wait for it).
        unsigned short wraw[kWsAhead][16];
        auto load_ws = [&](int i, int t, int q, unsigned short (&v)[16]) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0;
            if (DOTS || i >= n) return;
            const unsigned short* wsu = reinterpret_cast<const unsigned short*>(p.ws);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int row = t * kRows + 4 * lane + j;
                if (row >= p.N) continue;
#pragma unroll
                for (int gq = 0; gq < kGQ; ++gq) {
                    const int g = q * kGQ + gq;
                    if (g < G) v[4 * gq + j] = wsu[static_cast<size_t>(row) * G + g];
                }
            }
        };
        int tl = t_first, ql = q_first;  // item of the next weight-scale load
        int tp = t_first, qi = q_first;  // item being issued
#pragma unroll
        for (int k = 0; k < kWsAhead; ++k) {
            load_ws(k, tl, ql, wraw[k]);
            if (++ql == Q) { ql = 0; ++tl; }
        }
        int s = 0;
        uint32_t ph = 0;
        int issued = 0;
        bool stop = false;
        for (int it0 = 0; it0 < n && !stop; it0 += kWsAhead) {
#pragma unroll
            for (int k = 0; k < kWsAhead; ++k) {
                const int it = it0 + k;
                if (it >= n) break;
                bool ok = true;
                if (it >= kStages) ok = pq2::mbar_wait_warp(&sfree[s], ph ^ 1u, p.ctl, abort_v);
                if (!ok) {
                    stop = true;
                    break;
                }
                issued = it + 1;
                const int t = tp, q = qi;
                if (++qi == Q) { qi = 0; ++tp; }
                uint8_t* st = stage0 + static_cast<size_t>(s) * kStageBytes;
                if (lane == 0 && it != p.ctl.debug_skip_stage) {
                    pq2::mbar_arrive_expect_tx(&full[s], kTmaBytes);
                    pq2::tma_load_2d(st, &p.tm_codes, q * 128, t * kRows, &full[s]);
                    pq2::tma_load_2d(st + kTokOff, &p.tm_tok, 0, q * kGQ * 2 * kTok, &full[s]);
                    pq2::bulk_g2s(st + kStOff, p.st16 + static_cast<size_t>(q) * kGQ * kTok,
                                  kGQ * kTok * 8, &full[s]);
                }
                if (!DOTS) {
                    // ws area: [group][row] fp32
                    float* wss = reinterpret_cast<float*>(st + kWsOff);
#pragma unroll
                    for (int gq = 0; gq < kGQ; ++gq)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            wss[gq * kRows + 4 * lane + j] =
                                __half2float(__ushort_as_half(wraw[k][4 * gq + j]));
                }
                if (it != p.ctl.debug_skip_stage) pq2::mbar_arrive(&full[s]);
                load_ws(it + kWsAhead, tl, ql, wraw[k]);
                if (++ql == Q) { ql = 0; ++tl; }
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        // drain: every armed stage must have landed before exit
        if (lane == 0) {
            for (int k = 0; k < kStages; ++k) {
                if (issued <= k) continue;
                int last = k + ((issued - 1 - k) / kStages) * kStages;
                if (last == p.ctl.debug_skip_stage) last -= kStages;
                if (last >= 0) pq2::mbar_wait_bounded(&full[k], (last / kStages) & 1, p.ctl);
            }
        }
    } else if (warp < kWorker0) {
        // ------------------------------ MMA issuers ------------------------------
        // Each issuer takes kGQ / kIssuers of the item's groups: a warp that
        // issues tcgen05.mma is held for tens of cycles per instruction, far
        // longer than a small (N = 32) MMA keeps the tensor pipe busy.
        const int gq0 = (warp - 1) * (kGQ / kIssuers);
        if (lane == 0) {
            int s = 0, b = 0;
            uint32_t ps = 0, pb = 0;
            int done = 0;
            for (int it = 0; it < n; ++it) {
                if (!pq2::mbar_spin_bounded(&full[s], ps, p.ctl, abort_v) ||
                    !pq2::mbar_spin_bounded(&aready[b], pb, p.ctl, abort_v) ||
                    (it >= kBufs && !pq2::mbar_spin_bounded(&dfree[b], pb ^ 1u, p.ctl, abort_v))) {
                    *abort_v = 1;
                    break;
                }
                tc_fence_after();
                // descriptor of the stage's first token tile; the start
                // address field (bits 0..13, address >> 4) of the others is
                // this one's plus the offset >> 4 (no carry: addresses < 256 KB)
                const uint64_t desc0 = sw128_desc(stage0_s + s * kStageBytes + kTokOff);
                // k-step outer, group inner: consecutive MMAs write different
                // accumulators, so they do not wait on one another
#pragma unroll
                for (int k = 0; k < 4; ++k) {
#pragma unroll
                    for (int gq = gq0; gq < gq0 + kGQ / kIssuers; ++gq)
                        mma_f8_ta(tmem + kDCol0 + (b * kGQ + gq) * kGCols,
                                  tmem + (b * kGQ + gq) * kGCols + 8 * k,
                                  desc0 + ((gq * kTokGroupBytes + 32 * k) >> 4), k > 0);
                }
                mma_commit(&dfull[b]);
                done = it + 1;
                if (++s == kStages) { s = 0; ps ^= 1u; }
                if (++b == kBufs) { b = 0; pb ^= 1u; }
            }
            // no MMA may still be running when tensor memory is released
            if (done > 0)
                pq2::mbar_wait_bounded(&dfull[(done - 1) % kBufs], ((done - 1) / kBufs) & 1, p.ctl);
        }
    } else {
        // -------------------------------- workers --------------------------------
        const int wi = warp - kWorker0;   // 0..15
        const int quad = warp & 3;        // TMEM lane quadrant of this warp
        const int wq = wi >> 2;           // 0..3: the group it expands, its tokens 4wq..4wq+3
        const int r = quad * 32 + lane;   // weight row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const int lead = (wi == 0);       // warp 2: counters and flags
        bool failed = false;
        float acc[kTokPerWarp];
#pragma unroll
        for (int j = 0; j < kTokPerWarp; ++j) acc[j] = 0.0f;
        int xs = 0, xb = 0;               // expansion: stage, buffer
        uint32_t xps = 0;
        int es = 0, eb = 0;               // epilogue: stage, buffer
        uint32_t epb = 0;
        int te = t_first, qe = q_first;   // epilogue item

        for (int step = 0; step <= n; ++step) {
            // ---- expansion of group wq of item `step` ----
            if (step < n) {
                // warp-uniform waits: the tensor-memory accesses below are .sync.aligned
                if (!failed && !pq2::mbar_spin_warp(&full[xs], xps, p.ctl, abort_v)) {
                    failed = true;
                    *abort_v = 1;
                }
                // A buffer xb was last read by the MMAs of item step-2, which
                // this warp's own epilogue of that item (one step ago) already
                // waited for: no further wait before rewriting it
                if (!failed) {
                    // 16-byte chunks 2wq, 2wq+1 of the row, 128-byte swizzled
                    const uint32_t crow = stage0_s + xs * kStageBytes + r * 128;
                    const uint4 lo4 = pq2::lds_v4(crow + (((2 * wq) ^ (r & 7)) << 4));
                    const uint4 hi4 = pq2::lds_v4(crow + (((2 * wq + 1) ^ (r & 7)) << 4));
                    const uint32_t w[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
                    // plane s of word j -> column 8s + j of the group's 32
                    uint32_t v0[16], v1[16];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        v0[j] = w[j] & 0x03030303u;
                        v0[8 + j] = (w[j] >> 2) & 0x03030303u;
                        v1[j] = (w[j] >> 4) & 0x03030303u;
                        v1[8 + j] = (w[j] >> 6) & 0x03030303u;
                    }
                    const uint32_t acol = tmem + lane_off + (xb * kGQ + wq) * kGCols;
                    tmem_st16(acol, v0);
                    tmem_st16(acol + 16, v1);
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) pq2::mbar_arrive(&aready[xb]);
                if (++xs == kStages) { xs = 0; xps ^= 1u; }
                if (++xb == kBufs) xb = 0;
            }

            // ---- epilogue of item `step - 1`, tokens 4wq..4wq+3 ----
            const int e = step - 1;
            if (e < 0) continue;
            const int t = te, q = qe;
            const bool tile_end = (qe + 1 == Q);
            if (++qe == Q) { qe = 0; ++te; }
            if (!failed && !pq2::mbar_spin_warp(&dfull[eb], epb, p.ctl, abort_v)) {
                failed = true;
                *abort_v = 1;
            }
            // D columns 8wq .. 8wq+7 of each group: hi of the 4 tokens, then lo.
            // A warp whose 4 tokens are all past M loads and adds nothing (its
            // tensor-memory reads would only slow the MMAs down).
            float dv[kGQ][8];
            const bool live = 4 * wq < p.M;  // warp-uniform
            if (!failed && live) {
                tc_fence_after();
#pragma unroll
                for (int gq = 0; gq < kGQ; ++gq)
                    tmem_ld8(tmem + lane_off + kDCol0 + (eb * kGQ + gq) * kGCols + 8 * wq, dv[gq]);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int gq = 0; gq < kGQ; ++gq)
#pragma unroll
                    for (int j = 0; j < 8; ++j) dv[gq][j] = 0.0f;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) pq2::mbar_arrive(&dfree[eb]);
            if (++eb == kBufs) { eb = 0; epb ^= 1u; }
            const uint32_t es_s = stage0_s + es * kStageBytes;
            const int row = t * kRows + r;
            if (!failed && live) {
#pragma unroll
                for (int gq = 0; gq < kGQ; ++gq) {
                    // (s, t) of the 4 tokens (dots: (0, t)), weight scale of this row
                    const uint32_t sta = es_s + kStOff + gq * kTok * 8 + wq * 32;
                    const uint4 st01 = pq2::lds_v4(sta), st23 = pq2::lds_v4(sta + 16);
                    const float sv[4] = {__uint_as_float(st01.x), __uint_as_float(st01.z),
                                         __uint_as_float(st23.x), __uint_as_float(st23.z)};
                    const float tv[4] = {__uint_as_float(st01.y), __uint_as_float(st01.w),
                                         __uint_as_float(st23.y), __uint_as_float(st23.w)};
                    const float wsv =
                        DOTS ? 0.0f : pq2::lds_f32(es_s + kWsOff + 4 * (gq * kRows + r));
                    const int g = q * kGQ + gq;
#pragma unroll
                    for (int j = 0; j < kTokPerWarp; ++j) {
                        // D_hi + D_lo = 2^-9 dot(codes, q): exact (both multiples of 2^-9)
                        const float d = dv[gq][j] + dv[gq][4 + j];
                        if (DOTS) {
                            const int m = 4 * wq + j;
                            const float dot = fmaf(d, 512.0f, -tv[j]);  // exact integer
                            if (m < p.M && row < p.N && g < G &&
                                pq2::store_ok(p.ctl, (static_cast<long long>(m) * p.N + row) * G + g, 1,
                                              static_cast<long long>(p.M) * p.N * G))
                                p.dots[(static_cast<size_t>(m) * p.N + row) * G + g] =
                                    static_cast<int>(dot);
                        } else {
                            // the exact integer dot first, then its scales (an
                            // fma with a rounded s t could cancel catastrophically
                            // when t is much larger than dot(codes, q) - t)
                            const float dot = fmaf(d, 512.0f, -tv[j]);
                            acc[j] = fmaf(dot * sv[j], wsv, acc[j]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) pq2::mbar_arrive(&sfree[es]);  // the item's stage is consumed
            if (++es == kStages) es = 0;

            // ---- end of this CTA's part of row tile t: flush ----
            const bool seg_end = (e == n - 1) || tile_end;
            if (!seg_end) continue;
            if (pq2::named_bar_any(1, kWorkerThreads, failed)) {
                if (lead && lane == 0) *abort_v = 1;
                break;
            }
            if (!DOTS) {
                const int c_lo = owner_of(static_cast<long long>(t) * Q, p.items, p.grid);
                const int c_hi = owner_of(static_cast<long long>(t + 1) * Q - 1, p.items, p.grid);
                if (c_lo == c_hi) {
                    // the whole tile is this CTA's: straight to y
                    if (row < p.N) {
#pragma unroll
                        for (int j = 0; j < kTokPerWarp; ++j) {
                            const int m = 4 * wq + j;
                            if (m < p.M &&
                                pq2::store_ok(p.ctl, static_cast<long long>(m) * p.N + row, 1, static_cast<long long>(p.M) * p.N))
                                p.y[static_cast<size_t>(m) * p.N + row] = acc[j];
                        }
                    }
                } else {
                    float* part = p.partial + static_cast<size_t>(blockIdx.x + t) * p.M * kRows;
#pragma unroll
                    for (int j = 0; j < kTokPerWarp; ++j) {
                        const int m = 4 * wq + j;
                        if (m < p.M &&
                            pq2::store_ok(p.ctl, static_cast<long long>(blockIdx.x + t) * p.M * kRows +
                                                     static_cast<long long>(m) * kRows + r,
                                          1, static_cast<long long>(p.grid + p.n_tiles) * p.M * kRows))
                            part[static_cast<size_t>(m) * kRows + r] = acc[j];
                    }
                    pq2::named_bar_sync(2, kWorkerThreads);
                    if (lead && lane == 0) {
                        const unsigned old = pq2::atom_add_acq_rel_gpu(&p.counters[t], 1u);
                        last_flag = (old == static_cast<unsigned>(c_hi - c_lo)) ? 1 : 0;
                    }
                    pq2::named_bar_sync(2, kWorkerThreads);
                    if (last_flag) {
                        // the contributors' partials added in CTA order; the
                        // loads of kFlushBatch contributors are in flight
                        // together (one L2 round trip per batch)
                        float sum[kTokPerWarp];
#pragma unroll
                        for (int j = 0; j < kTokPerWarp; ++j) sum[j] = 0.0f;
                        for (int c0 = c_lo; c0 <= c_hi; c0 += kFlushBatch) {
                            float v[kFlushBatch][kTokPerWarp];
#pragma unroll
                            for (int b = 0; b < kFlushBatch; ++b) {
                                const int c = c0 + b;
                                const float* pc =
                                    p.partial + static_cast<size_t>(c + t) * p.M * kRows + r;
#pragma unroll
                                for (int j = 0; j < kTokPerWarp; ++j) {
                                    const int m = 4 * wq + j;
                                    v[b][j] = (c <= c_hi && m < p.M)
                                                  ? ld_cg(pc + static_cast<size_t>(m) * kRows)
                                                  : 0.0f;
                                }
                            }
#pragma unroll
                            for (int b = 0; b < kFlushBatch; ++b)
                                if (c0 + b <= c_hi) {
#pragma unroll
                                    for (int j = 0; j < kTokPerWarp; ++j) sum[j] += v[b][j];
                                }
                        }
                        if (row < p.N) {
#pragma unroll
                            for (int j = 0; j < kTokPerWarp; ++j) {
                                const int m = 4 * wq + j;
                                if (m < p.M &&
                                    pq2::store_ok(p.ctl, static_cast<long long>(m) * p.N + row, 1, static_cast<long long>(p.M) * p.N))
                                    p.y[static_cast<size_t>(m) * p.N + row] = sum[j];
                            }
                        }
                    }
                    // last_flag is rewritten at the next flush only after
                    // every worker has passed the first barrier there
                }
#pragma unroll
                for (int j = 0; j < kTokPerWarp; ++j) acc[j] = 0.0f;
            }
        }
    }

    // teardown: every role is done with tensor memory
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
}

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

struct SmallLayout {
    int grid, n_tiles, Q;
    long long items;
    int64_t G4;
    size_t tok, st16, counters, partial, total;  // byte offsets / total
};

SmallLayout layout_small(int64_t M, int64_t N, int64_t K, int num_sms) {
    SmallLayout l = {};
    const int64_t G = K / 128;
    l.Q = static_cast<int>((G + kGQ - 1) / kGQ);
    l.G4 = static_cast<int64_t>(l.Q) * kGQ;
    l.n_tiles = static_cast<int>((N + kRows - 1) / kRows);
    l.items = static_cast<long long>(l.n_tiles) * l.Q;
    long long grid = num_sms < kMaxGrid ? num_sms : kMaxGrid;
    if (grid > l.items) grid = l.items;
    l.grid = static_cast<int>(grid);
    size_t off = 0;
    l.tok = off;
    off += align256(static_cast<size_t>(l.G4) * kTokGroupBytes);
    l.st16 = off;
    off += align256(static_cast<size_t>(l.G4) * kTok * 8);
    l.counters = off;
    off += align256(static_cast<size_t>(l.n_tiles) * 4);
    l.partial = off;
    // one [M][128] slot per (CTA c, tile t) pair, at index c + t
    off += align256(static_cast<size_t>(l.grid + l.n_tiles) * M * kRows * 4);
    l.total = off;
    return l;
}

}  // namespace

namespace pq2h {

size_t small_scratch_bytes(int64_t M, int64_t N, int64_t K, int num_sms) {
    return layout_small(M, N, K, num_sms).total;
}

// Device-independent: the size for the largest grid any device gets.
size_t small_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    return small_scratch_bytes(M, N, K, kMaxGrid);
}

}  // namespace pq2h

namespace {

// small_kernel on token tiles, (s, t) and counters already prepared in the
// workspace (layout l).
cudaError_t launch_small_main(const SmallLayout& l, uint8_t* w, const uint8_t* codes,
                              const __half* ws, float* y, int32_t* dots, int64_t M, int64_t N,
                              int64_t K, cudaStream_t st, const pq2::DevCtl& ctl) {
    using namespace pq2h;
    uint32_t* tok = reinterpret_cast<uint32_t*>(w + l.tok);
    float2* st16 = reinterpret_cast<float2*>(w + l.st16);
    unsigned* counters = reinterpret_cast<unsigned*>(w + l.counters);
    SmallParams p = {};
    if (!encode_tmap_2d(&p.tm_tok, CU_TENSOR_MAP_DATA_TYPE_UINT8, tok, 128u,
                        static_cast<uint64_t>(l.G4) * 2 * kTok, 128u, 128u, kRows, true) ||
        !encode_tmap_2d(&p.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes,
                        static_cast<uint64_t>(K / 4), static_cast<uint64_t>(N),
                        static_cast<uint64_t>(K / 4), 128u, kRows, true))
        return cudaErrorInvalidValue;
    p.st16 = st16;
    p.ws = ws;
    p.y = y;
    p.dots = dots;
    p.partial = reinterpret_cast<float*>(w + l.partial);
    p.counters = counters;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.G = static_cast<int>(K / 128);
    p.Q = l.Q;
    p.n_tiles = l.n_tiles;
    p.grid = l.grid;
    p.items = l.items;
    p.ctl = ctl;
    const size_t smem = 1024 + static_cast<size_t>(kStages) * kStageBytes;
    auto kern = dots ? small_kernel<true> : small_kernel<false>;
    static SmemLimit lim[2];
    cudaError_t e = ensure_smem(lim[dots ? 1 : 0], kern, smem);
    if (e != cudaSuccess) return e;
    return launch(kern, dim3(l.grid), dim3(kThreads), smem, st, true, p);
}

}  // namespace

namespace pq2h {

cudaError_t launch_small(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                         const __half* ws, float* y, int32_t* dots, int64_t M, int64_t N,
                         int64_t K, void* workspace, cudaStream_t st, const pq2::DevCtl& ctl,
                         const DeviceInfo& dev) {
    if (M < 1 || M > kTok) return cudaErrorInvalidValue;
    // (the DP4A kernel, when forced, takes every shape it can; this is not one)
    if (forced_variant(PQ2_OP_SMALL) == PQ2_VARIANT_SMALL_DP4A) return kUnsupportedVariant;
    const SmallLayout l = layout_small(M, N, K, dev.num_sms);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    {
        const int64_t words = l.G4 * kTok * 32;
        const int64_t want = (words + 255) / 256;
        const int grid = static_cast<int>(want < dev.num_sms * 4 ? want : dev.num_sms * 4);
        cudaError_t e = launch(small_prep_kernel, dim3(grid), dim3(256), 0, st, true, qp, S, T,
                               reinterpret_cast<uint32_t*>(w + l.tok),
                               reinterpret_cast<float2*>(w + l.st16),
                               reinterpret_cast<unsigned*>(w + l.counters), M, K, l.G4, l.n_tiles);
        if (e != cudaSuccess) return e;
    }
    return launch_small_main(l, w, codes, ws, y, dots, M, N, K, st, ctl);
}

bool small_x_supported(int64_t M, int64_t N, int64_t K, int num_sms) {
    if (M < 2 || M > kTok) return false;
    const int force = forced_variant(PQ2_OP_SMALL);
    if (force == PQ2_VARIANT_SMALL_TC) return true;
    return force == PQ2_VARIANT_DEFAULT && !gemv_multi_supported(M, N, K, num_sms);
}

cudaError_t launch_small_x(const __half* x, const uint8_t* codes, const __half* ws, float* y,
                           int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                           const pq2::DevCtl& ctl, const DeviceInfo& dev) {
    if (M < 1 || M > kTok) return cudaErrorInvalidValue;
    const SmallLayout l = layout_small(M, N, K, dev.num_sms);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    {
        cudaError_t e = launch(pq2::quant_tiles_kernel<SmallTok>,
                               dim3(pq2::quant_tiles_grid(l.G4 * kTok, dev.num_sms)), dim3(256), 0,
                               st, true, x, reinterpret_cast<uint32_t*>(w + l.tok),
                               static_cast<void*>(w + l.st16),
                               reinterpret_cast<unsigned*>(w + l.counters), M, K, l.G4, l.n_tiles);
        if (e != cudaSuccess) return e;
    }
    return launch_small_main(l, w, codes, ws, y, nullptr, M, N, K, st, ctl);
}

// The tensor-core kernel of pq2_gemm_small: small_kernel by default, the
// token-tile kernel when forced (PQ2_VARIANT_SMALL_TILE).  Measured on GB300
// at 16 tokens, us per call (5120 -> 17408, 6144 -> 5120): small_kernel 22.7
// and 15.5 against 23.9 and 18.3; at 8 tokens 22.3 and 15.2 against 23.2 and
// 17.0.  The workspace covers either.
size_t small_tc_scratch_bytes(int64_t M, int64_t N, int64_t K, int num_sms) {
    const int force = forced_variant(PQ2_OP_SMALL);
    if (force == PQ2_VARIANT_SMALL_WTILE) return wtile_scratch_bytes(M, N, K, num_sms);
    return force == PQ2_VARIANT_SMALL_TILE
               ? tile_scratch_bytes(M, N, K, num_sms)
               : small_scratch_bytes(M, N, K, num_sms);
}

size_t small_tc_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    const size_t a = small_workspace_bytes(M, N, K), b0 = tile_workspace_bytes(M, N, K);
    const size_t b1 = wtile_workspace_bytes(M, N, K), b = b0 > b1 ? b0 : b1;
    return a > b ? a : b;
}

cudaError_t launch_small_tc(const int8_t* qp, const float* S, const int32_t* T,
                            const uint8_t* codes, const __half* ws, float* y, int32_t* dots,
                            int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                            const pq2::DevCtl& ctl, const DeviceInfo& dev) {
    if (forced_variant(PQ2_OP_SMALL) == PQ2_VARIANT_SMALL_TILE)
        return launch_tile(qp, S, T, codes, ws, y, dots, M, N, K, workspace, st, ctl, dev);
    if (forced_variant(PQ2_OP_SMALL) == PQ2_VARIANT_SMALL_WTILE)
        return launch_wtile(qp, S, T, codes, ws, y, dots, M, N, K, workspace, st, ctl, dev);
    return launch_small(qp, S, T, codes, ws, y, dots, M, N, K, workspace, st, ctl, dev);
}

}  // namespace pq2h
