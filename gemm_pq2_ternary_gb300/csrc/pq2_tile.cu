// Weights-stationary token-tile matmul for 5 to 64 token rows, on the
// 5th-generation tensor cores (tcgen05, operands and accumulators in tensor
// memory).
//
// The method is the pages' small-batch kernels ("Making a ternary reasoning
// model fast in vLLM", page "From CUDA to Triton and Gluon", sections "Small
// batches: make the register layout explicit" and "Extend the kernels to
// sixteen token rows"): the planes of the code bytes meet the int8
// activations of all token rows at once, one exact integer dot per (row,
// token, group), then the per-group -sum(q) correction and the fp32
// dequantise-accumulate of the M = 1 path.  The same page names the gap this
// kernel closes ("Limits of the port": 17 to 64 tokens).  Split partial sums
// are combined in a fixed order (section "Choose the configuration with the
// proxy").
//
// GB300 design.  tcgen05 has no int8 kind on sm_103a; kind::f8f6f4 with e4m3
// operands is exact here:
//  * weights = A operand (M = 128 rows per tile), kept in TENSOR MEMORY: each
//    expansion thread owns one weight row (one TMEM lane) and writes plane s
//    of its code words, (w >> 2s) & 0x03030303, as e4m3 bytes (bytes below
//    16 are exactly byte * 2^-9) with tcgen05.st;
//  * tokens = B operand, from shared memory: q = 16h + l with 16h and l
//    exact e4m3 values, prepared once per call;
//  * up to 32 tokens (MT = 16, 32) the hi and lo parts of a token are two
//    rows of B, so one MMA with N = 2 MT per k-step gives both partial dots
//    side by side in D (a single-thread MMA issue costs about 46 cycles
//    whatever N up to 64, so wide MMAs are cheap); for 64 tokens they
//    accumulate into the same D with two MMAs of N = 64 per k-step (the
//    tensor pipe is busy either way, and D and the epilogue halve);
//  * per group, 4 k-steps: the k order inside a group is the plane order of
//    the activations, so k-step s is plane s (8 A columns);
//  * epilogue: dot = D_sum * 512 - t (an exact integer), then
//    acc += dot * s * ws in registers, two tokens per fp32x2 instruction.
//
// Tensor memory holds two A slots of one item each (4 groups x 32 columns;
// barriers: A written, aready; MMAs of the item done, afree) and a ring of
// NS D slots of one group each (NC columns; MMAs done, dfull; D read,
// dfree).
// Shared memory is a ring of stages, one per item (row tile, 4 groups): the
// 128-row x 128-byte code box, the token tiles of the 4 groups, their (s, t)
// and the rows' weight scales.
//
// Items are cut into contiguous, balanced ranges, one CTA per SM.  A CTA
// flushes its accumulators at each row-tile boundary of its range: a tile
// owned by a single CTA is written straight to y; otherwise each contributor
// writes its partial sums and bumps the tile's counter, and the last one to
// arrive sums the partials of all contributors in CTA order and writes y.
//
// Per CTA (warp roles):
//   warp 0        producer: TMA of the code box and token tiles, one bulk copy
//                 of (s, t); its lanes copy the rows' weight scales into the
//                 stage with cp.async
//   warp 1        TMEM allocation; MMA issuer of the even groups
//   warp 2        MMA issuer of the odd groups (each issue holds its warp for
//                 tens of cycles: two issuers keep the tensor pipe fed)
//   warp 3        idle (keeps the later roles aligned to TMEM lane quadrants)
//   warps 4-11    expansion: lane quadrant warp % 4, the even or the odd items
//   then          epilogue: lane quadrant warp % 4, a block of 16 tokens, and
//                 (up to 32 tokens) the even or the odd groups; the two
//                 group parities are added at the flush (even + odd)
// Every mbarrier wait is bounded (device error word on expiry).
#include "pq2_internal.h"
#include "pq2_tokens.cuh"

namespace {

constexpr int kRows = 128;                    // weight rows per tile (MMA M)
constexpr int kGQ = 4;                        // groups per item
constexpr int kMaxGrid = 256;                 // CTAs per call at most (bounds the partial-sum slots)
constexpr uint32_t kCodesBytes = kRows * 128;  // 4 groups x 32 bytes per row, 128B swizzle

template <int MT>
struct Cfg {
    static constexpr int HL = MT <= 32 ? 2 : 1;             // 2: hi and lo side by side in D
    static constexpr int NC = HL == 2 ? 2 * MT : MT;         // D columns per group (MMA N)
    static constexpr int NB = 2 * MT;                        // token-tile rows per group
    static constexpr int AS = 2;                             // A slots, one item (4 groups) each
    static constexpr uint32_t D0 = AS * kGQ * 32;            // first D column (A: 128 per slot)
    static constexpr int NS = (512 - D0) / NC;               // D slots, one group each
    static constexpr int STAGES = MT == 16 ? 4 : (MT == 32 ? 3 : 2);
    static constexpr int GP = MT <= 32 ? 2 : 1;              // epilogue group parities
    static constexpr int TBLK = MT / 16;                     // 16-token blocks
    static constexpr int PW = 4 * GP * TBLK;                 // epilogue warps
    static constexpr int EH = AS;                            // expansion warps per lane quadrant
    static constexpr int EW0 = 4;                            // first expansion warp
    static constexpr int PW0 = EW0 + 4 * EH;                 // first epilogue warp
    static constexpr int THREADS = (PW0 + PW) * 32;
    static constexpr uint32_t TOK_OFF = kCodesBytes;
    static constexpr uint32_t TOK_GROUP = NB * 128;          // bytes of one group's token tile
    static constexpr uint32_t ST_OFF = TOK_OFF + kGQ * TOK_GROUP;
    static constexpr uint32_t ST_BYTES = kGQ * 2 * MT * 4;   // per group: s[MT], t[MT]
    static constexpr uint32_t WS_OFF = ST_OFF + ST_BYTES;    // ws: [128 rows][4 groups] fp16
    static constexpr uint32_t TMA_BYTES = WS_OFF;            // what the bulk copies bring
    static constexpr uint32_t STAGE = (WS_OFF + kRows * kGQ * 2 + 1023) / 1024 * 1024;
    static constexpr uint32_t COMB_BYTES = GP == 2 ? kRows * MT * 4 : 0;
    static constexpr size_t SMEM = 1024 + static_cast<size_t>(STAGES) * STAGE + COMB_BYTES;
    static constexpr uint32_t TOK_BOX = kGQ * NB <= 256 ? kGQ * NB : 256;  // rows per TMA box
    static constexpr int TOK_BOXES = kGQ * NB / TOK_BOX;
    // kind::f8f6f4: D f32, A and B e4m3, both K-major, M = 128, N = NC
    static constexpr uint32_t IDESC = (1u << 4) | (static_cast<uint32_t>(NC >> 3) << 17) |
                                      (static_cast<uint32_t>(kRows >> 4) << 24);
    static_assert(D0 + NS * NC <= 512 && NS >= 2, "tensor memory");
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(TOK_OFF % 1024 == 0 && TOK_GROUP % 1024 == 0, "swizzled tiles on 1 KB");
    static_assert(HL == 2 || (MT * 128) % 1024 == 0, "lo half of a token tile on 1 KB");
};

struct TileParams {
    CUtensorMap tm_codes;  // uint8 [N][K/4], box {128, 128}, 128B swizzle
    CUtensorMap tm_tok;    // uint8 [G4 * NB][128], box {128, TOK_BOX}, 128B swizzle
    const float* st;       // [G4][2][MT]: s then t, zero past M and past G
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

__host__ __device__ __forceinline__ long long range_begin(long long c, long long items, int grid) {
    return c * items / grid;
}
__host__ __device__ __forceinline__ int owner_of(long long i, long long items, int grid) {
    return static_cast<int>(((i + 1) * grid - 1) / items);
}

// ---------------------------------------------------------------------------
// per-call preparation: token tiles, (s, t), tile counters
// ---------------------------------------------------------------------------
// tok [G4][NB][128]: token m's e4m3(16h) and e4m3(l) (q = 16h + l,
// h = floor(q/16)) in rows hi(m), lo(m) of its group: 8(m/4) + m%4 and 4 rows
// further (hi and lo side by side in D), or m and MT + m (same D).  Zero for
// tokens >= M and groups >= G.  st [G4][2][MT]: s then t (s = 0 for the
// integer-dot debug output, where S is null).
template <int MT>
__global__ void __launch_bounds__(256) tile_prep_kernel(const int8_t* __restrict__ qp,
                                                        const float* __restrict__ S,
                                                        const int32_t* __restrict__ T,
                                                        uint32_t* __restrict__ tok,
                                                        float* __restrict__ st,
                                                        unsigned* __restrict__ counters,
                                                        int64_t M, int64_t K, int64_t G4,
                                                        int n_tiles) {
    using C = Cfg<MT>;
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();
    const int64_t G = K / 128;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    // one index = one 4-byte word of one token of one group (hi and lo together)
    const int64_t words = G4 * MT * 32;
    for (int64_t i = i0; i < words; i += stride) {
        const int64_t g = i / (MT * 32);
        const int m = static_cast<int>((i / 32) % MT);
        const int wq = static_cast<int>(i % 32);
        uint32_t hw = 0, lw = 0;
        if (m < M && g < G) {
            const uint32_t qw = reinterpret_cast<const uint32_t*>(qp + m * K + g * 128)[wq];
            pq2::hi_lo_words(qw, hw, lw);  // e4m3 of 16 * floor(q / 16), q mod 16
        }
        uint32_t* tg = tok + g * (C::NB * 32);
        const int rh = C::HL == 2 ? 8 * (m / 4) + (m % 4) : m;
        const int rl = C::HL == 2 ? rh + 4 : MT + m;
        tg[rh * 32 + wq] = hw;
        tg[rl * 32 + wq] = lw;
    }
    for (int64_t i = i0; i < G4 * MT; i += stride) {
        const int64_t g = i / MT, m = i - g * MT;
        float s = 0.0f, t = 0.0f;
        if (m < M && g < G) {
            s = S ? S[m * G + g] : 0.0f;
            t = static_cast<float>(T[m * G + g]);
        }
        st[(g * 2) * MT + m] = s;
        st[(g * 2 + 1) * MT + m] = t;
    }
    for (int64_t i = i0; i < n_tiles; i += stride) counters[i] = 0u;
}

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

// D (tensor memory) += A (tensor memory) x B (shared memory descriptor).
template <uint32_t IDESC>
__device__ __forceinline__ void mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(IDESC), "r"(acc));
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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Two-wide fp32 arithmetic (one instruction, two IEEE round-to-nearest
// operations: the same bits as two scalar ones).
__device__ __forceinline__ unsigned long long f2pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// 8-byte asynchronous copy global -> shared (both 8-byte aligned).
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(pq2::smem_u32(dst)), "l"(src)
                 : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival counts towards the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(pq2::smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ float ld_cg(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// main kernel
// ---------------------------------------------------------------------------
template <int MT, bool DOTS>
__global__ void __launch_bounds__(Cfg<MT>::THREADS, 1) tile_kernel(const __grid_constant__ TileParams p) {
    using C = Cfg<MT>;
    constexpr int NS = C::NS;
    constexpr int ST = C::STAGES;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t full[ST];     // stage landed: TMA bytes + the producer's 32 lanes
    __shared__ uint64_t sfree[ST];    // stage consumed: every epilogue warp, after the item
    __shared__ uint64_t aready[C::AS];  // A of an item written (4 expansion warps)
    __shared__ uint64_t afree[C::AS];   // MMAs of an item done, A free (a commit per issuer)
    __shared__ uint64_t dfull[NS];      // MMAs of a group done: D complete (commit)
    __shared__ uint64_t dfree[NS];      // D of a group read (every epilogue warp of its parity)
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ int last_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t base = pq2::smem_u32(smem);
    uint8_t* stage0 = smem + ((1024 - (base & 1023)) & 1023);
    const uint32_t stage0_s = pq2::smem_u32(stage0);
    float* comb = reinterpret_cast<float*>(stage0 + static_cast<size_t>(ST) * C::STAGE);

    if (tid == 0) {
        for (int i = 0; i < ST; ++i) {
            pq2::mbar_init(&full[i], 1 + 32);
            pq2::mbar_init(&sfree[i], C::PW);
        }
        for (int i = 0; i < C::AS; ++i) {
            pq2::mbar_init(&aready[i], 4);
            pq2::mbar_init(&afree[i], 2);
        }
        for (int i = 0; i < NS; ++i) {
            pq2::mbar_init(&dfull[i], 1);
            pq2::mbar_init(&dfree[i], C::PW / C::GP);
        }
        abort_flag = 0;
        pq2::fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         pq2::smem_u32(&tmem_base)),
                     "r"(512));
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
    const int n = static_cast<int>(w1 - w0);  // items of this CTA
    const int ng = n * kGQ;                   // groups of this CTA
    // (tile, quad) of the first item; later items advance it incrementally
    const int t_first = static_cast<int>(w0 / Q);
    const int q_first = static_cast<int>(w0 - static_cast<long long>(t_first) * Q);
    volatile int* abort_v = &abort_flag;

    if (warp == 0) {
        // -------------------------------- producer --------------------------------
        // Weight scales: lane l copies rows 4l .. 4l + 3 of the item's tile, the
        // item's 4 groups (8 bytes of fp16 per row), into the stage with
        // cp.async; the copies arrive on the stage's full barrier when they
        // land, so no register waits for them.  A lane with a row past N, or
        // any lane when a row's 4 scales are not 8-byte aligned (G % 4 != 0),
        // reads its rows with plain loads instead (zero past N and past G).
        const bool ws_async = (G & 3) == 0;
        const unsigned short* wsu = reinterpret_cast<const unsigned short*>(p.ws);
        int tp = t_first, qi = q_first;  // item being issued
        int s = 0;
        uint32_t ph = 0;
        int issued = 0;
        for (int it = 0; it < n; ++it) {
            if (it >= ST && !pq2::mbar_suspend_warp(&sfree[s], ph ^ 1u, p.ctl, abort_v)) break;
            issued = it + 1;
            const int t = tp, q = qi;
            if (++qi == Q) { qi = 0; ++tp; }
            uint8_t* stg = stage0 + static_cast<size_t>(s) * C::STAGE;
            if (lane == 0 && it != p.ctl.debug_skip_stage) {
                pq2::mbar_arrive_expect_tx(&full[s], C::TMA_BYTES);
                pq2::tma_load_2d(stg, &p.tm_codes, q * 128, t * kRows, &full[s]);
#pragma unroll
                for (int b = 0; b < C::TOK_BOXES; ++b)
                    pq2::tma_load_2d(stg + C::TOK_OFF + b * C::TOK_BOX * 128, &p.tm_tok, 0,
                                     q * kGQ * C::NB + b * C::TOK_BOX, &full[s]);
                pq2::bulk_g2s(stg + C::ST_OFF, p.st + static_cast<size_t>(q) * kGQ * 2 * MT,
                              C::ST_BYTES, &full[s]);
            }
            bool lane_async = false;
            if (!DOTS) {
                const int row0 = t * kRows + 4 * lane;
                uint8_t* dst = stg + C::WS_OFF + 4 * lane * 8;  // [row][4 groups] fp16
                lane_async = ws_async && row0 + 3 < p.N;
                if (lane_async) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        cp_async8(dst + 8 * j, wsu + static_cast<size_t>(row0 + j) * G + q * kGQ);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        unsigned short v[kGQ];
#pragma unroll
                        for (int gq = 0; gq < kGQ; ++gq) {
                            const int g = q * kGQ + gq;
                            v[gq] = (row0 + j < p.N && g < G)
                                        ? wsu[static_cast<size_t>(row0 + j) * G + g]
                                        : static_cast<unsigned short>(0);
                        }
                        *reinterpret_cast<uint2*>(dst + 8 * j) =
                            make_uint2(v[0] | (static_cast<uint32_t>(v[1]) << 16),
                                       v[2] | (static_cast<uint32_t>(v[3]) << 16));
                    }
                }
            }
            if (it != p.ctl.debug_skip_stage) {
                if (lane_async)
                    cp_async_arrive_noinc(&full[s]);  // arrives when this lane's copies land
                else
                    pq2::mbar_arrive(&full[s]);
            }
            if (++s == ST) {
                s = 0;
                ph ^= 1u;
            }
        }
        // no copy of this lane may still be in flight at exit
        asm volatile("cp.async.wait_all;" ::: "memory");
        // drain: every armed stage must have landed before exit
        if (lane == 0) {
            for (int k = 0; k < ST; ++k) {
                if (issued <= k) continue;
                int last = k + ((issued - 1 - k) / ST) * ST;
                if (last == p.ctl.debug_skip_stage) last -= ST;
                if (last >= 0) pq2::mbar_wait_bounded(&full[k], (last / ST) & 1, p.ctl);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------ MMA issuers ------------------------------
        // Issuer p takes groups p and p + 2 of every item; after its groups of
        // an item it commits to the item's afree barrier (the A slot may be
        // rewritten once both issuers' MMAs have read it).
        const int parity = warp - 1;
        if (lane == 0) {
            int last = -1;
            bool ok = true;
            for (int item = 0; item < n && ok; ++item) {
                const int as = item % C::AS;
                if (!pq2::mbar_spin_bounded(&aready[as], (item / C::AS) & 1, p.ctl, abort_v)) {
                    *abort_v = 1;
                    break;
                }
                const uint32_t tok0 = stage0_s + (item % ST) * C::STAGE + C::TOK_OFF;
                for (int gq = parity; gq < kGQ; gq += 2) {
                    const int gi = item * kGQ + gq;
                    const int slot = gi % NS;
                    // busy polling: this thread is on the critical path
                    if (gi >= NS &&
                        !pq2::mbar_spin_bounded(&dfree[slot], ((gi / NS) - 1) & 1, p.ctl, abort_v)) {
                        *abort_v = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t b0 = sw128_desc(tok0 + gq * C::TOK_GROUP);
                    const uint32_t d_tmem = tmem + C::D0 + slot * C::NC;
                    const uint32_t a_tmem = tmem + (as * kGQ + gq) * 32;
                    // descriptor start addresses advance by (offset >> 4) without
                    // a carry out of the 14-bit field: shared addresses < 256 KB
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        mma_ta<C::IDESC>(d_tmem, a_tmem + 8 * k, b0 + ((32 * k) >> 4), k > 0);
                        if (C::HL == 1)
                            mma_ta<C::IDESC>(d_tmem, a_tmem + 8 * k,
                                             b0 + ((MT * 128 + 32 * k) >> 4), 1);
                    }
                    mma_commit(&dfull[slot]);
                    last = gi;
                }
                if (ok) mma_commit(&afree[as]);
            }
            // no MMA may still be running when tensor memory is released
            if (last >= 0)
                pq2::mbar_wait_bounded(&dfull[last % NS], (last / NS) & 1, p.ctl);
        }
    } else if (warp >= C::EW0 && warp < C::PW0) {
        // -------------------------------- expansion --------------------------------
        // Warp (quadrant, half) expands items half, half + AS, ... into A slot
        // `half`: the four groups of its 32 rows, then one wait for the stores
        // and one arrival (the per-group hand-off cost more than the work).
        const int quad = warp & 3;              // TMEM lane quadrant
        const int half = (warp - C::EW0) >> 2;  // A slot
        const int r = quad * 32 + lane;         // weight row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        bool failed = false;
        for (int item = half; item < n; item += C::AS) {
            const int stg = item % ST;
            // warp-uniform waits: the tensor-memory stores below are .sync.aligned
            if (!failed && !pq2::mbar_suspend_warp(&full[stg], (item / ST) & 1, p.ctl, abort_v))
                failed = true;
            // the slot's previous item has been read by both issuers' MMAs
            if (!failed && item >= C::AS &&
                !pq2::mbar_suspend_warp(&afree[half], ((item / C::AS) - 1) & 1, p.ctl, abort_v))
                failed = true;
            if (failed) *abort_v = 1;
            if (!failed) {
                tc_fence_after();
                const uint32_t crow = stage0_s + stg * C::STAGE + r * 128;
#pragma unroll 1
                for (int gq = 0; gq < kGQ; ++gq) {
                    // 16-byte chunks 2gq, 2gq+1 of the row, 128-byte swizzled
                    const uint4 lo4 = pq2::lds_v4(crow + (((2 * gq) ^ (r & 7)) << 4));
                    const uint4 hi4 = pq2::lds_v4(crow + (((2 * gq + 1) ^ (r & 7)) << 4));
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
                    const uint32_t acol = tmem + lane_off + (half * kGQ + gq) * 32;
                    tmem_st16(acol, v0);
                    tmem_st16(acol + 16, v1);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) pq2::mbar_arrive(&aready[half]);
        }
    } else if (warp >= C::PW0) {
        // -------------------------------- epilogue --------------------------------
        const int e = warp - C::PW0;
        const int quad = warp & 3;               // TMEM lane quadrant
        const int eb = e >> 2;                   // 0 .. GP * TBLK - 1
        const int par = eb % C::GP;              // group parity (0 when GP == 1)
        const int tb = eb / C::GP;               // token block: tokens 16 tb .. 16 tb + 15
        const int r = quad * 32 + lane;          // weight row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const bool flusher = par == 0;           // adds the odd parity's sums and flushes
        constexpr uint32_t kFlushThreads = 4 * C::TBLK * 32;
        bool failed = false;
        unsigned long long acc[8];  // tokens 16 tb + 2i, + 2i + 1
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0ull;
        const unsigned long long k512 = f2pack(512.0f, 512.0f);
        int te = t_first, qe = q_first;  // item being finished
        for (int item = 0; item < n; ++item) {
            const int stg = item % ST;
            const uint32_t stg_s = stage0_s + stg * C::STAGE;
            const int t = te, q = qe;
            const bool tile_end = (qe + 1 == Q);
            if (++qe == Q) { qe = 0; ++te; }
            const int row = t * kRows + r;
            for (int gq = par; gq < kGQ; gq += C::GP) {
                const int gi = item * kGQ + gq;
                const int slot = gi % NS;
                if (!failed &&
                    !pq2::mbar_suspend_warp(&dfull[slot], (gi / NS) & 1, p.ctl, abort_v)) {
                    failed = true;
                    *abort_v = 1;
                }
                float d[32];
                if (!failed) {
                    tc_fence_after();
                    const uint32_t dcol = tmem + lane_off + C::D0 + slot * C::NC;
                    if (C::HL == 2) {
                        tmem_ld16(dcol + 32 * tb, d);
                        tmem_ld16(dcol + 32 * tb + 16, d + 16);
                    } else {
                        tmem_ld16(dcol + 16 * tb, d);
                    }
                    tmem_wait_ld();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) pq2::mbar_arrive(&dfree[slot]);
                if (failed) continue;
                // (s, t) of the block's 16 tokens, this row's weight scale
                const uint32_t sa = stg_s + C::ST_OFF + gq * (2 * MT * 4) + 16 * tb * 4;
                const uint32_t ta = sa + MT * 4;
                const float wsv =
                    DOTS ? 0.0f
                         : __half2float(__ushort_as_half(static_cast<unsigned short>(
                               pq2::lds_u16(stg_s + C::WS_OFF + 2 * (r * kGQ + gq)))));
                const unsigned long long ws2 = f2pack(wsv, wsv);
                const int g = q * kGQ + gq;
#pragma unroll
                for (int v = 0; v < 4; ++v) {  // tokens 16 tb + 4v .. + 4v + 3
                    const uint4 s4 = pq2::lds_v4(sa + 16 * v);
                    const uint4 t4 = pq2::lds_v4(ta + 16 * v);
                    // D of the 4 tokens: hi then lo (side by side), or the sum
                    unsigned long long sum2[2];
                    if (C::HL == 2) {
                        sum2[0] = add2(f2pack(d[8 * v], d[8 * v + 1]), f2pack(d[8 * v + 4], d[8 * v + 5]));
                        sum2[1] = add2(f2pack(d[8 * v + 2], d[8 * v + 3]), f2pack(d[8 * v + 6], d[8 * v + 7]));
                    } else {
                        sum2[0] = f2pack(d[4 * v], d[4 * v + 1]);
                        sum2[1] = f2pack(d[4 * v + 2], d[4 * v + 3]);
                    }
                    // exact integer dots: D_sum = 2^-9 dot(codes, q), so
                    // D_sum * 512 - t is dot(codes, q) - sum(q) exactly
                    const unsigned long long negt0 = f2pack(-__uint_as_float(t4.x), -__uint_as_float(t4.y));
                    const unsigned long long negt1 = f2pack(-__uint_as_float(t4.z), -__uint_as_float(t4.w));
                    const unsigned long long dot0 = fma2(sum2[0], k512, negt0);
                    const unsigned long long dot1 = fma2(sum2[1], k512, negt1);
                    if (DOTS) {
                        float e0, e1, e2, e3;
                        f2unpack(dot0, e0, e1);
                        f2unpack(dot1, e2, e3);
                        const float ev[4] = {e0, e1, e2, e3};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int m = 16 * tb + 4 * v + j;
                            if (m < p.M && row < p.N && g < G &&
                                pq2::store_ok(p.ctl, (static_cast<long long>(m) * p.N + row) * G + g, 1,
                                              static_cast<long long>(p.M) * p.N * G))
                                p.dots[(static_cast<size_t>(m) * p.N + row) * G + g] =
                                    static_cast<int>(ev[j]);
                        }
                    } else {
                        // the exact integer dot first, then its scales
                        const unsigned long long s0 = f2pack(__uint_as_float(s4.x), __uint_as_float(s4.y));
                        const unsigned long long s1 = f2pack(__uint_as_float(s4.z), __uint_as_float(s4.w));
                        acc[2 * v] = fma2(mul2(dot0, s0), ws2, acc[2 * v]);
                        acc[2 * v + 1] = fma2(mul2(dot1, s1), ws2, acc[2 * v + 1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) pq2::mbar_arrive(&sfree[stg]);  // the item's stage is consumed

            // ---- end of this CTA's part of row tile t: flush ----
            if (!(item == n - 1 || tile_end)) continue;
            if (pq2::named_bar_any(1, C::PW * 32, failed)) {
                *abort_v = 1;
                break;
            }
            if (DOTS) continue;
            float a[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) f2unpack(acc[i], a[2 * i], a[2 * i + 1]);
            if (C::GP == 2) {
                // the odd parity hands its sums to the even one: even + odd
                // (comb is [token][row]: consecutive lanes, consecutive words)
                float* cb = comb + 16 * tb * kRows + r;
                if (!flusher) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) cb[i * kRows] = a[i];
                }
                pq2::named_bar_sync(1, C::PW * 32);
                if (flusher) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) a[i] += cb[i * kRows];
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0ull;
            if (!flusher) continue;
            const int c_lo = owner_of(static_cast<long long>(t) * Q, p.items, p.grid);
            const int c_hi = owner_of(static_cast<long long>(t + 1) * Q - 1, p.items, p.grid);
            if (c_lo == c_hi) {
                // the whole tile is this CTA's: straight to y
                if (row < p.N) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int m = 16 * tb + i;
                        if (m < p.M &&
                            pq2::store_ok(p.ctl, static_cast<long long>(m) * p.N + row, 1, static_cast<long long>(p.M) * p.N))
                            p.y[static_cast<size_t>(m) * p.N + row] = a[i];
                    }
                }
            } else {
                float* part = p.partial + static_cast<size_t>(blockIdx.x + t) * p.M * kRows;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int m = 16 * tb + i;
                    if (m < p.M &&
                        pq2::store_ok(p.ctl, static_cast<long long>(blockIdx.x + t) * p.M * kRows +
                                                 static_cast<long long>(m) * kRows + r,
                                      1, static_cast<long long>(p.grid + p.n_tiles) * p.M * kRows))
                        part[static_cast<size_t>(m) * kRows + r] = a[i];
                }
                pq2::named_bar_sync(2, kFlushThreads);
                if (e == 0 && lane == 0) {
                    const unsigned old = pq2::atom_add_acq_rel_gpu(&p.counters[t], 1u);
                    last_flag = (old == static_cast<unsigned>(c_hi - c_lo)) ? 1 : 0;
                }
                pq2::named_bar_sync(2, kFlushThreads);
                if (last_flag) {
                    // the contributors' partials added in CTA order, two
                    // contributors' loads in flight together
                    float sum[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) sum[i] = 0.0f;
                    for (int c0 = c_lo; c0 <= c_hi; c0 += 2) {
                        const bool two = c0 + 1 <= c_hi;
                        const float* pa = p.partial + static_cast<size_t>(c0 + t) * p.M * kRows + r;
                        const float* pb = pa + static_cast<size_t>(p.M) * kRows;  // contributor c0 + 1
                        float va[16], vb[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int m = 16 * tb + i;
                            va[i] = m < p.M ? ld_cg(pa + static_cast<size_t>(m) * kRows) : 0.0f;
                            vb[i] = (two && m < p.M) ? ld_cg(pb + static_cast<size_t>(m) * kRows) : 0.0f;
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            sum[i] += va[i];
                            if (two) sum[i] += vb[i];
                        }
                    }
                    if (row < p.N) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int m = 16 * tb + i;
                            if (m < p.M &&
                                pq2::store_ok(p.ctl, static_cast<long long>(m) * p.N + row, 1, static_cast<long long>(p.M) * p.N))
                                p.y[static_cast<size_t>(m) * p.N + row] = sum[i];
                        }
                    }
                }
                // last_flag is rewritten at the next flush only after every
                // flushing warp has passed the first barrier there
            }
        }
    }

    // teardown: every role is done with tensor memory
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
}

// ---------------------------------------------------------------------------
// measurement: the issue rate of back-to-back tcgen05 e4m3 MMAs
// ---------------------------------------------------------------------------
// One CTA per SM; one thread issues `iters` MMAs of M = 128, N, K = 32 (A in
// tensor memory, B in shared memory, all into one accumulator), commits, and
// waits (bounded) for them; cycles[blockIdx.x] = clock64 cycles from the
// first issue to the completion.  The operands are constant (e4m3 2^-9).
template <int N>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int iters, unsigned long long* cycles,
                                                          pq2::DevCtl ctl) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t done;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5;
    uint8_t* b = smem + ((1024 - (pq2::smem_u32(smem) & 1023)) & 1023);
    for (int i = tid; i < N * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(b)[i] = 0x01010101u;
    if (tid == 0) {
        pq2::mbar_init(&done, 1);
        pq2::fence_mbar_init();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         pq2::smem_u32(&tmem_base)),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    {  // A: columns 256..287 (4 k-steps of 8), each warp its lane quadrant
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0x01010101u;
        const uint32_t a = tmem + (static_cast<uint32_t>(warp * 32) << 16) + 256;
        tmem_st16(a, v);
        tmem_st16(a + 16, v);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        constexpr uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
                                   (static_cast<uint32_t>(kRows >> 4) << 24);
        const uint64_t b0 = sw128_desc(pq2::smem_u32(b));
        const long long c0 = clock64();
        for (int i = 0; i < iters; ++i) {
            const int k = i & 3;
            mma_ta<idesc>(tmem, tmem + 256 + 8 * k, b0 + ((32 * k) >> 4), i > 0);
        }
        mma_commit(&done);
        const bool ok = pq2::mbar_wait_bounded(&done, 0, ctl);
        const long long c1 = clock64();
        cycles[blockIdx.x] = ok ? static_cast<unsigned long long>(c1 - c0) : 0ull;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
}

template <int N>
cudaError_t launch_mma_rate(int iters, unsigned long long* cycles, cudaStream_t st,
                            const pq2::DevCtl& ctl, const pq2h::DeviceInfo& dev) {
    const size_t smem = 1024 + static_cast<size_t>(N) * 128;
    static pq2h::SmemLimit lim;
    const cudaError_t e = pq2h::ensure_smem(lim, mma_rate_kernel<N>, smem);
    if (e != cudaSuccess) return e;
    return pq2h::launch(mma_rate_kernel<N>, dim3(dev.num_sms), dim3(128), smem, st, false, iters,
                        cycles, ctl);
}

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

struct TileLayout {
    int grid, n_tiles, Q, mt;
    long long items;
    int64_t G4;
    size_t tok, st, counters, partial, total;  // byte offsets / total
};

int tile_tokens(int64_t M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

TileLayout layout_tile(int64_t M, int64_t N, int64_t K, int num_sms) {
    TileLayout l = {};
    l.mt = tile_tokens(M);
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
    off += align256(static_cast<size_t>(l.G4) * 2 * l.mt * 128);
    l.st = off;
    off += align256(static_cast<size_t>(l.G4) * 2 * l.mt * 4);
    l.counters = off;
    off += align256(static_cast<size_t>(l.n_tiles) * 4);
    l.partial = off;
    // one [M][128] slot per (CTA c, tile t) pair, at index c + t
    off += align256(static_cast<size_t>(l.grid + l.n_tiles) * M * kRows * 4);
    l.total = off;
    return l;
}

// Layout of the token tiles for quant_tiles_kernel (pq2_matmul's path: the
// same tiles, (s, t) table and counters straight from the fp16 activations).
template <int T>
struct TileTok {
    static constexpr int MT = T;
    static constexpr int kGroupWords = Cfg<T>::NB * 32;
    __device__ static int row_hi(int m) { return Cfg<T>::HL == 2 ? 8 * (m / 4) + (m % 4) : m; }
    __device__ static int row_lo(int m) {
        return Cfg<T>::HL == 2 ? 8 * (m / 4) + (m % 4) + 4 : T + m;
    }
    __device__ static void put_st(void* st, int64_t g, int m, float s, float t) {
        float* f = static_cast<float*>(st);
        f[(g * 2) * T + m] = s;
        f[(g * 2 + 1) * T + m] = t;
    }
};

template <int MT>
cudaError_t launch_mt(const __half* x, const int8_t* qp, const float* S, const int32_t* T,
                      const uint8_t* codes,
                      const __half* ws, float* y, int32_t* dots, int64_t M, int64_t N, int64_t K,
                      const TileLayout& l, uint8_t* w, cudaStream_t st, const pq2::DevCtl& ctl,
                      const pq2h::DeviceInfo& dev) {
    using C = Cfg<MT>;
    uint32_t* tok = reinterpret_cast<uint32_t*>(w + l.tok);
    float* stv = reinterpret_cast<float*>(w + l.st);
    unsigned* counters = reinterpret_cast<unsigned*>(w + l.counters);
    if (x) {
        // pq2_matmul's path: the tiles straight from the fp16 activations
        cudaError_t e = pq2h::launch(pq2::quant_tiles_kernel<TileTok<MT>>,
                                     dim3(pq2::quant_tiles_grid(l.G4 * MT, dev.num_sms)), dim3(256),
                                     0, st, true, x, tok, static_cast<void*>(stv), counters, M, K,
                                     l.G4, l.n_tiles);
        if (e != cudaSuccess) return e;
    } else {
        const int64_t words = l.G4 * MT * 32;
        const int64_t want = (words + 255) / 256;
        const int grid = static_cast<int>(want < dev.num_sms * 4 ? want : dev.num_sms * 4);
        cudaError_t e = pq2h::launch(tile_prep_kernel<MT>, dim3(grid), dim3(256), 0, st, true, qp,
                                     S, T, tok, stv, counters, M, K, l.G4, l.n_tiles);
        if (e != cudaSuccess) return e;
    }
    TileParams p = {};
    if (!pq2h::encode_tmap_2d(&p.tm_tok, CU_TENSOR_MAP_DATA_TYPE_UINT8, tok, 128u,
                              static_cast<uint64_t>(l.G4) * C::NB, 128u, 128u, C::TOK_BOX, true) ||
        !pq2h::encode_tmap_2d(&p.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes,
                              static_cast<uint64_t>(K / 4), static_cast<uint64_t>(N),
                              static_cast<uint64_t>(K / 4), 128u, kRows, true))
        return cudaErrorInvalidValue;
    p.st = stv;
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
    auto kern = dots ? tile_kernel<MT, true> : tile_kernel<MT, false>;
    static pq2h::SmemLimit lim[2];
    cudaError_t e = pq2h::ensure_smem(lim[dots ? 1 : 0], kern, C::SMEM);
    if (e != cudaSuccess) return e;
    return pq2h::launch(kern, dim3(l.grid), dim3(C::THREADS), C::SMEM, st, true, p);
}

// x != nullptr: the token tiles straight from x (qp, S, T unused)
cudaError_t launch_tile_any(const __half* x, const int8_t* qp, const float* S, const int32_t* T,
                           const uint8_t* codes, const __half* ws, float* y, int32_t* dots,
                           int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                           const pq2::DevCtl& ctl, const pq2h::DeviceInfo& dev) {
    if (M < 1 || M > pq2h::kTileMaxM) return cudaErrorInvalidValue;
    const TileLayout l = layout_tile(M, N, K, dev.num_sms);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    if (l.mt == 16)
        return launch_mt<16>(x, qp, S, T, codes, ws, y, dots, M, N, K, l, w, st, ctl, dev);
    if (l.mt == 32)
        return launch_mt<32>(x, qp, S, T, codes, ws, y, dots, M, N, K, l, w, st, ctl, dev);
    return launch_mt<64>(x, qp, S, T, codes, ws, y, dots, M, N, K, l, w, st, ctl, dev);
}

}  // namespace

namespace pq2h {

size_t tile_scratch_bytes(int64_t M, int64_t N, int64_t K, int num_sms) {
    return layout_tile(M, N, K, num_sms).total;
}

size_t tile_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    return tile_scratch_bytes(M, N, K, kMaxGrid);
}

cudaError_t launch_tile(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                        const __half* ws, float* y, int32_t* dots, int64_t M, int64_t N, int64_t K,
                        void* workspace, cudaStream_t st, const pq2::DevCtl& ctl,
                        const DeviceInfo& dev) {
    return launch_tile_any(nullptr, qp, S, T, codes, ws, y, dots, M, N, K, workspace, st, ctl, dev);
}

cudaError_t launch_tile_x(const __half* x, const uint8_t* codes, const __half* ws, float* y,
                          int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                          const pq2::DevCtl& ctl, const DeviceInfo& dev) {
    return launch_tile_any(x, nullptr, nullptr, nullptr, codes, ws, y, nullptr, M, N, K, workspace,
                          st, ctl, dev);
}

cudaError_t launch_mma_rate(int n, int iters, unsigned long long* cycles, cudaStream_t st,
                            const pq2::DevCtl& ctl, const DeviceInfo& dev) {
    switch (n) {
        case 32: return ::launch_mma_rate<32>(iters, cycles, st, ctl, dev);
        case 64: return ::launch_mma_rate<64>(iters, cycles, st, ctl, dev);
        case 128: return ::launch_mma_rate<128>(iters, cycles, st, ctl, dev);
        case 256: return ::launch_mma_rate<256>(iters, cycles, st, ctl, dev);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pq2h
