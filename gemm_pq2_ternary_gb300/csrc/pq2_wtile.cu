// Weights-wide token-tile matmul for 5 to 64 token rows, on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
// pq2_gemm_prefill runs it by default for 33 to 64 tokens where a CTA gets
// few items (wtile_default); 5 to 64 tokens when forced.
//
// The method is the pages' small-batch and prefill arithmetic ("Making a
// ternary reasoning model fast in vLLM", page "From CUDA to Triton and
// Gluon", sections "Small batches: make the register layout explicit",
// "Extend the kernels to sixteen token rows" and "Prompt processing": one
// exact integer dot per (token, weight row, group), the per-group -sum(q)
// correction, then the fp32 dequantise-accumulate of the M = 1 path), for the
// token counts the same page names as the gap of its port ("Limits of the
// port": 17 to 64 tokens).  Split partial sums are combined in a fixed order
// (section "Choose the configuration with the proxy").
//
// GB300 design.  tcgen05 has no int8 kind on sm_103a; kind::f8f6f4 with e4m3
// operands is exact here.  The operand with many rows is the weights:
//  * B = weights, N = 128 rows per tile, in shared memory in the MMA's
//    K-major 128-byte-swizzled layout; expansion warps write plane s of each
//    code word, (w >> 2s) & 0x03030303, as e4m3 bytes (exactly code * 2^-9);
//  * A = tokens, M = 128 rows from shared memory (TMA): token m's exact e4m3
//    parts 16h and l (q = 16h + l) on rows 2m and 2m + 1 (zero for tokens
//    past the call's), so one A tile holds up to 64 tokens; the rows past
//    the tile's 2 x 16, 32 or 64 only reach D rows that are never read;
//  * per group, 4 MMAs of M = 128, N = 128, K = 32 (k-step s = plane s): as
//    many instructions per code byte as the 128 x 32 small-batch tile, for up
//    to 64 tokens instead of 16.
//    A group's completion reaches its mbarrier about 1400 cycles after the
//    commit, MMAs or not, so tensor memory holds 4 D buffers of 128 columns
//    and shared memory 5-6 expanded-weight slots: groups in flight;
//  * epilogue: D rows 2m and 2m + 1 sit on adjacent lanes, one shuffle adds
//    them (exact), then dot = D_sum * 512 - t (an exact integer) and
//    acc += dot * s * ws.
// Items are (128-row tile, 4 groups), cut into contiguous balanced ranges, one
// CTA per SM; a tile shared by several CTAs is finished by the last
// contributor, which sums all partials in CTA order.
//
// Per CTA (warp roles; a warp may read only its own TMEM lane quadrant,
// warp % 4, so the epilogue warps are the warps w < 16 whose quadrant holds
// token rows, and the other roles take the remaining warps in order):
//   epilogue      TMEM lane quadrant w % 4 x 32 columns (block w / 4)
//   producer      TMA of the item's code box and of each group's token tile
//   MMA issuer    also allocates tensor memory (4 D buffers of 128 columns)
//   expansion     8 warps at 16 tokens (two planes of a row per thread), else
//                 4 (a whole row); they also stage each group's fp32 weight
//                 scales and the tokens' (s, t) for the epilogue
// Every mbarrier wait is bounded (device error word on expiry).
#include "pq2_internal.h"
#include "pq2_tokens.cuh"

namespace {

constexpr int kBN = 128;                      // weight rows per tile (MMA N)
constexpr int kCB = kBN / 4;                  // columns per epilogue warp (4 column blocks)
constexpr int kWsRows = kBN / 32;             // weight rows whose scales each producer lane copies
constexpr int kGQ = 4;                        // groups per item
constexpr int kMaxGrid = 256;                 // CTAs per call at most (bounds the partial slots)
constexpr uint32_t kCodesBytes = kBN * 128;   // an item's code box: kBN rows x 4 groups
constexpr uint32_t kBTile = kBN * 128;        // a group's expanded weights
constexpr int kCStages = 3;                   // code boxes in flight (items)
constexpr int kMaxASlots = 16;                // token tiles (groups) in flight at most
constexpr int kMaxBSlots = 8;                 // expanded weights (groups) in flight at most
constexpr int kDSlots = 512 / kBN;            // D buffers in tensor memory (groups)
constexpr int kESlots = 8;                    // epilogue inputs (groups)
constexpr int kNL = kCB / 16;                 // 16-column tensor-memory loads per group
constexpr int kAcc = 8 * kNL;                 // accumulators per epilogue lane
static_assert(kNL % 2 == 0, "the last contributor sums 16 columns at a time");
// kind::f8f6f4: D f32, A and B e4m3, both K-major, M = 128, N = kBN
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(kBN >> 3) << 17) |
                            (static_cast<uint32_t>(128 >> 4) << 24);

template <int MT>
struct WCfg {
    static constexpr int AROWS = 2 * MT;           // token rows written per group
    static constexpr int QA = AROWS / 32;          // TMEM lane quadrants holding tokens
    static constexpr int EACT = 4 * QA;            // epilogue warps (4 column blocks each)
    // epilogue warps are the warps w < 16 with w % 4 < QA (quadrant w % 4,
    // column block w / 4); the other warps, in order, are the producer, the
    // MMA issuer and XW expansion warps: 8 at 16 tokens, else 4 (no more than
    // 4 warps share an SM sub-partition at 32 tokens: 128 registers a thread)
    static constexpr int XW = MT == 16 ? 8 : 4;
    // an expansion unit is one weight row's two planes 2 hp, 2 hp + 1 (unit
    // u: row u % kBN, hp = u / kBN); each expansion thread takes UPT units
    static constexpr int UPT = 2 * kBN / (32 * XW);
    static constexpr int WARPS = QA == 4 ? 16 + 2 + XW : 14;
    // expanded-weight slots: the expansion of group g waits for the MMAs of
    // group g - BSLOTS
    static constexpr int BSLOTS = MT == 64 ? 5 : 6;
    static constexpr int THREADS = WARPS * 32;
    // epilogue inputs of a group: weight scales [kBN] fp32, then s[MT], t[MT]
    static constexpr uint32_t E_S = kBN * 4;
    static constexpr uint32_t E_T = E_S + MT * 4;
    static constexpr uint32_t ESLOT = (E_T + MT * 4 + 127) / 128 * 128;
    // code stage (an item): code box | weight scales [kBN rows][4 groups]
    // fp16 | (s, t) [4 groups][2][MT] fp32
    static constexpr uint32_t WS_OFF = kCodesBytes;
    static constexpr uint32_t ST_OFF = WS_OFF + kBN * kGQ * 2;
    static constexpr uint32_t ST_BYTES = kGQ * 2 * MT * 4;
    static constexpr uint32_t CSTAGE = (ST_OFF + ST_BYTES + 1023) / 1024 * 1024;
    // token tiles: the MMA reads 128 rows from a slot, of which only the
    // first AROWS are written; the rest (the next slots' rows, or the pad after
    // the last slot) only reach D rows no epilogue warp reads, so slots sit
    // AROWS rows apart and more groups' tiles are in flight at few tokens
    static constexpr uint32_t ASLOT = AROWS * 128;
    static constexpr int ASLOTS = MT == 16 ? 12 : (MT == 32 ? 6 : 4);
    static constexpr uint32_t OFF_A = kCStages * CSTAGE;
    static constexpr uint32_t OFF_B = OFF_A + ASLOTS * ASLOT + (128 - AROWS) * 128;
    static constexpr uint32_t OFF_E = OFF_B + BSLOTS * kBTile;
    static constexpr size_t SMEM = 1024 + OFF_E + kESlots * ESLOT;
    static_assert(MT == 16 || MT == 32 || MT == 64, "token tile");
    static_assert(ASLOTS <= kMaxASlots && ASLOT % 1024 == 0, "token tile slots");
    static_assert(BSLOTS <= kMaxBSlots && UPT >= 1 && 32 * XW * UPT == 2 * kBN, "expansion");
    static_assert(2 * MT <= 32 * XW, "one thread per token scale");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct WTileParams {
    CUtensorMap tm_codes;  // uint8 [N][K/4], box {128, kBN}, 128B swizzle
    CUtensorMap tm_tok;    // uint8 [G4 * AROWS][128], box {128, AROWS}, 128B swizzle
    const float* st;       // [G4][2][MT]: s then t, zero past M and past G
    const __half* ws;      // [N][G]
    float* y;              // [M][N]
    int32_t* dots;         // debug: [M][N][G]
    float* partial;        // [grid + n_tiles][M][kBN]
    unsigned* counters;    // [n_tiles], zero on entry
    int M, N, K, G;
    int Q;                 // quads per tile: ceil(G / 4)
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
// tok [G4][2 MT][128]: row 2m = e4m3(16h), row 2m + 1 = e4m3(l) of token m
// (q = 16h + l, h = floor(q / 16)), zero for tokens >= M and groups >= G;
// st [G4][2][MT]: s then t (s = 0 for the integer-dot output, where S is null).
template <int MT>
__global__ void __launch_bounds__(256) wtile_prep_kernel(const int8_t* __restrict__ qp,
                                                         const float* __restrict__ S,
                                                         const int32_t* __restrict__ T,
                                                         uint32_t* __restrict__ tok,
                                                         float* __restrict__ st,
                                                         unsigned* __restrict__ counters,
                                                         int64_t M, int64_t K, int64_t G4,
                                                         int n_tiles) {
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
        uint32_t* tg = tok + g * (2 * MT * 32);
        tg[(2 * m) * 32 + wq] = hw;
        tg[(2 * m + 1) * 32 + wq] = lw;
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

// D (tensor memory) += A (shared memory) x B (shared memory).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kIdesc), "r"(acc));
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

// 8-byte asynchronous copy global -> shared (both 8-byte aligned).
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(pq2::smem_u32(dst)), "l"(src)
                 : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(pq2::smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ float4 ld_cg4(const float* p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// main kernel
// ---------------------------------------------------------------------------
enum WRole { kProducer, kIssuer, kExpand, kEpilogue, kIdle };

// Role of warp w (idx: the expansion warp's index or the epilogue warp's
// column block).
__device__ __forceinline__ WRole wrole(int w, int qa, int xw, int& idx) {
    if (w < 16 && (w & 3) < qa) {
        idx = w >> 2;
        return kEpilogue;
    }
    // rank = the warps below w that are not epilogue warps
    const int rank = w < 16 ? w - (w >> 2) * qa - ((w & 3) < qa ? (w & 3) : qa) : w - 4 * qa;
    idx = rank - 2;
    return rank == 0 ? kProducer : (rank == 1 ? kIssuer : (rank < 2 + xw ? kExpand : kIdle));
}

template <int MT, bool DOTS>
__global__ void __launch_bounds__(WCfg<MT>::THREADS, 1) wtile_kernel(const __grid_constant__ WTileParams p) {
    using C = WCfg<MT>;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t cfull[kCStages];   // an item's code box landed (TMA)
    __shared__ uint64_t cfree[kCStages];   // the box's codes were expanded (expansion warps)
    __shared__ uint64_t afull[kMaxASlots];  // a group's token tile landed (TMA)
    __shared__ uint64_t afree[kMaxASlots];  // its MMAs are done (commit)
    __shared__ uint64_t bready[kMaxBSlots];  // a group's weights expanded (expansion warps)
    __shared__ uint64_t bfree[kMaxBSlots];   // its MMAs are done (commit)
    __shared__ uint64_t efull[kESlots];    // a group's scales, s and t staged (expansion warps)
    __shared__ uint64_t efree[kESlots];    // the epilogue read them (epilogue warps)
    __shared__ uint64_t dfull[kDSlots];    // a group's D complete (commit)
    __shared__ uint64_t dfree[kDSlots];    // its D read (epilogue warps)
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ int last_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t base = pq2::smem_u32(smem);
    uint8_t* sm = smem + ((1024 - (base & 1023)) & 1023);
    const uint32_t sm_s = pq2::smem_u32(sm);

    if (tid == 0) {
        for (int i = 0; i < kCStages; ++i) {
            pq2::mbar_init(&cfull[i], 1 + 32);  // the TMA bytes + the producer's 32 lanes
            pq2::mbar_init(&cfree[i], C::XW);
        }
        for (int i = 0; i < C::ASLOTS; ++i) {
            pq2::mbar_init(&afull[i], 1);
            pq2::mbar_init(&afree[i], 1);
        }
        for (int i = 0; i < C::BSLOTS; ++i) {
            pq2::mbar_init(&bready[i], C::XW);
            pq2::mbar_init(&bfree[i], 1);
        }
        for (int i = 0; i < kDSlots; ++i) {
            pq2::mbar_init(&dfull[i], 1);
            pq2::mbar_init(&dfree[i], C::EACT);
        }
        for (int i = 0; i < kESlots; ++i) {
            pq2::mbar_init(&efull[i], C::XW);
            pq2::mbar_init(&efree[i], C::EACT);
        }
        abort_flag = 0;
        pq2::fence_mbar_init();
    }
    int ridx = 0;
    const WRole role = wrole(warp, C::QA, C::XW, ridx);
    if (role == kIssuer) {
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

    if (role == kProducer) {
        // -------------------------------- producer --------------------------------
        // Lane 0 issues the TMA of the item's code box and token tiles and one
        // bulk copy of its (s, t).  Lane l copies the weight scales of its
        // kWsRows rows (the item's 4 groups: 8 bytes of fp16 a row) with
        // cp.async, which arrive on the stage's barrier when they land; rows
        // past N, or every row when a row's 4 scales are not 8-byte aligned
        // (G % 4 != 0), are read with plain loads (zero past N and past G).
        const bool ws_async = (G & 3) == 0;
        const unsigned short* wsu = reinterpret_cast<const unsigned short*>(p.ws);
        int tp = t_first, qi = q_first;
        int c_issued = 0, a_issued = 0;
        for (int it = 0; it < n; ++it) {
            const int t = tp, q = qi;
            if (++qi == Q) { qi = 0; ++tp; }
            const int cs = it % kCStages;
            if (it >= kCStages &&
                !pq2::mbar_suspend_warp(&cfree[cs], ((it / kCStages) - 1) & 1, p.ctl, abort_v))
                break;
            c_issued = it + 1;
            uint8_t* stg = sm + cs * C::CSTAGE;
            if (lane == 0 && it != p.ctl.debug_skip_stage) {
                pq2::mbar_arrive_expect_tx(&cfull[cs], kCodesBytes + C::ST_BYTES);
                pq2::tma_load_2d(stg, &p.tm_codes, q * 128, t * kBN, &cfull[cs]);
                pq2::bulk_g2s(stg + C::ST_OFF, p.st + static_cast<size_t>(q) * kGQ * 2 * MT,
                              C::ST_BYTES, &cfull[cs]);
            }
            bool lane_async = false;
            if (!DOTS) {
                const int row0 = t * kBN + kWsRows * lane;
                uint8_t* dst = stg + C::WS_OFF + kWsRows * lane * 8;  // [row][4 groups] fp16
                lane_async = ws_async && row0 + kWsRows - 1 < p.N;
                if (lane_async) {
#pragma unroll
                    for (int j = 0; j < kWsRows; ++j)
                        cp_async8(dst + 8 * j, wsu + static_cast<size_t>(row0 + j) * G + q * kGQ);
                } else {
#pragma unroll
                    for (int j = 0; j < kWsRows; ++j) {
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
                    cp_async_arrive_noinc(&cfull[cs]);  // arrives when this lane's copies land
                else
                    pq2::mbar_arrive(&cfull[cs]);
            }
            bool ok = true;
            if (lane == 0) {
                for (int gq = 0; gq < kGQ; ++gq) {
                    const int gi = it * kGQ + gq;
                    const int as = gi % C::ASLOTS;
                    if (gi >= C::ASLOTS &&
                        !pq2::mbar_wait_bounded(&afree[as], ((gi / C::ASLOTS) - 1) & 1, p.ctl, abort_v)) {
                        ok = false;
                        break;
                    }
                    a_issued = gi + 1;
                    pq2::mbar_arrive_expect_tx(&afull[as], C::AROWS * 128);
                    pq2::tma_load_2d(sm + C::OFF_A + as * C::ASLOT, &p.tm_tok, 0,
                                     (q * kGQ + gq) * C::AROWS, &afull[as]);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        }
        // no copy of this lane may still be in flight at exit
        asm volatile("cp.async.wait_all;" ::: "memory");
        // drain: every armed copy must have landed before exit
        if (lane == 0) {
            for (int k = 0; k < kCStages; ++k) {
                if (c_issued <= k) continue;
                int last = k + ((c_issued - 1 - k) / kCStages) * kCStages;
                if (last == p.ctl.debug_skip_stage) last -= kCStages;
                if (last >= 0) pq2::mbar_wait_bounded(&cfull[k], (last / kCStages) & 1, p.ctl);
            }
            for (int k = 0; k < C::ASLOTS; ++k) {
                if (a_issued <= k) continue;
                const int last = k + ((a_issued - 1 - k) / C::ASLOTS) * C::ASLOTS;
                pq2::mbar_wait_bounded(&afull[k], (last / C::ASLOTS) & 1, p.ctl);
            }
        }
    } else if (role == kIssuer) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            int last = -1;
            for (int gi = 0; gi < ng; ++gi) {
                const int as = gi % C::ASLOTS, bs = gi % C::BSLOTS, ds = gi % kDSlots;
                // busy polling: this thread is on the critical path
                if (!pq2::mbar_spin_bounded(&afull[as], (gi / C::ASLOTS) & 1, p.ctl, abort_v) ||
                    !pq2::mbar_spin_bounded(&bready[bs], (gi / C::BSLOTS) & 1, p.ctl, abort_v) ||
                    (gi >= kDSlots &&
                     !pq2::mbar_spin_bounded(&dfree[ds], ((gi / kDSlots) - 1) & 1, p.ctl, abort_v))) {
                    *abort_v = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = sm_s + C::OFF_A + as * C::ASLOT;
                const uint32_t b0 = sm_s + C::OFF_B + bs * kBTile;
                const uint32_t d_tmem = tmem + ds * kBN;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss(d_tmem, sw128_desc(a0 + 32 * k), sw128_desc(b0 + 32 * k), k > 0);
                mma_commit(&afree[as]);
                mma_commit(&bfree[bs]);
                mma_commit(&dfull[ds]);
                last = gi;
            }
            // no MMA may still be running when tensor memory is released
            if (last >= 0)
                pq2::mbar_wait_bounded(&dfull[last % kDSlots], (last / kDSlots) & 1, p.ctl);
        }
    } else if (role == kExpand) {
        // -------------------------------- expansion --------------------------------
        // Thread x expands units x + 32 XW j (j < UPT) of the tile into the
        // group's B slot: unit u is planes 2 hp and 2 hp + 1 of weight row
        // u % kBN, hp = u / kBN.  The thread whose unit is a row's hp = 0 also
        // writes the row's fp32 weight scale, and thread x < 2 MT one of the
        // tokens' s or t, into the group's epilogue slot.
        const int x = ridx * 32 + lane;
        bool failed = false;
        for (int it = 0; it < n; ++it) {
            const int cs = it % kCStages;
            if (!failed && !pq2::mbar_suspend_warp(&cfull[cs], (it / kCStages) & 1, p.ctl, abort_v))
                failed = true;
            const uint32_t cbox = sm_s + cs * C::CSTAGE;
#pragma unroll 1
            for (int gq = 0; gq < kGQ; ++gq) {
                const int gi = it * kGQ + gq;
                const int bs = gi % C::BSLOTS, es = gi % kESlots;
                // the weight scales of this thread's hp = 0 rows and (for x <
                // 2 MT) s or t of a token, from the stage (zero past N, M and G)
                float wsv[C::UPT], stv = 0.0f;
#pragma unroll
                for (int j = 0; j < C::UPT; ++j) wsv[j] = 0.0f;
                if (!failed) {
#pragma unroll
                    for (int j = 0; j < C::UPT; ++j) {
                        const int u = x + 32 * C::XW * j;
                        if (!DOTS && u < kBN)
                            wsv[j] = __half2float(__ushort_as_half(static_cast<unsigned short>(
                                pq2::lds_u16(cbox + C::WS_OFF + 2 * (u * kGQ + gq)))));
                    }
                    if (x < 2 * MT) stv = pq2::lds_f32(cbox + C::ST_OFF + 4 * (gq * 2 * MT + x));
                }
                if (!failed && gi >= C::BSLOTS &&
                    !pq2::mbar_suspend_warp(&bfree[bs], ((gi / C::BSLOTS) - 1) & 1, p.ctl, abort_v))
                    failed = true;
                if (!failed && gi >= kESlots &&
                    !pq2::mbar_suspend_warp(&efree[es], ((gi / kESlots) - 1) & 1, p.ctl, abort_v))
                    failed = true;
                if (failed) *abort_v = 1;
                if (!failed) {
                    uint8_t* bslot = sm + C::OFF_B + bs * kBTile;
                    float* eslot = reinterpret_cast<float*>(sm + C::OFF_E + es * C::ESLOT);
#pragma unroll
                    for (int j = 0; j < C::UPT; ++j) {
                        const int u = x + 32 * C::XW * j;
                        const int r = u % kBN, hp = u / kBN;  // row within the tile, plane pair
                        // code box row r: 16-byte chunks 2gq, 2gq + 1, 128-byte swizzled
                        const uint32_t crow = cbox + r * 128;
                        const uint4 lo4 = pq2::lds_v4(crow + (((2 * gq) ^ (r & 7)) << 4));
                        const uint4 hi4 = pq2::lds_v4(crow + (((2 * gq + 1) ^ (r & 7)) << 4));
                        const uint32_t w[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
                        uint8_t* brow = bslot + r * 128;
#pragma unroll
                        for (int pp = 0; pp < 2; ++pp) {
                            const int pl = 2 * hp + pp;
#pragma unroll
                            for (int hc = 0; hc < 2; ++hc) {  // 16-byte chunk 2 pl + hc of the row
                                uint4 v;
                                v.x = (w[4 * hc + 0] >> (2 * pl)) & 0x03030303u;
                                v.y = (w[4 * hc + 1] >> (2 * pl)) & 0x03030303u;
                                v.z = (w[4 * hc + 2] >> (2 * pl)) & 0x03030303u;
                                v.w = (w[4 * hc + 3] >> (2 * pl)) & 0x03030303u;
                                *reinterpret_cast<uint4*>(brow + 16 * ((2 * pl + hc) ^ (r & 7))) = v;
                            }
                        }
                        if (u < kBN) eslot[r] = wsv[j];
                    }
                    if (x < 2 * MT) eslot[kBN + x] = stv;  // s[m] at kBN + m, t[m] at kBN + MT + m
                    // the B tile is read by the tensor cores (async proxy)
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                __syncwarp();
                if (lane == 0) {
                    pq2::mbar_arrive(&bready[bs]);
                    pq2::mbar_arrive(&efull[es]);
                }
            }
            __syncwarp();
            if (lane == 0) pq2::mbar_arrive(&cfree[cs]);
        }
    } else if (role == kEpilogue) {
        // -------------------------------- epilogue --------------------------------
        const int quad = warp & 3;               // TMEM lane quadrant
        const int cb = ridx;                     // column block: kCB cb .. kCB (cb + 1) - 1
        const int h = lane & 1;                  // 0: the hi row of the token, 1: the lo row
        const int m = (quad * 32 + lane) >> 1;   // token
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        constexpr uint32_t kEpiThreads = C::EACT * 32;
        bool failed = false;
        float acc[kAcc];  // this lane's columns: kCB cb + 16 c + 8 h + i, at acc[8 c + i]
#pragma unroll
        for (int i = 0; i < kAcc; ++i) acc[i] = 0.0f;
        int te = t_first, qe = q_first;  // item being finished
        for (int it = 0; it < n; ++it) {
            const int t = te, q = qe;
            const bool tile_end = (qe + 1 == Q);
            if (++qe == Q) { qe = 0; ++te; }
            for (int gq = 0; gq < kGQ; ++gq) {
                const int gi = it * kGQ + gq;
                const int ds = gi % kDSlots, es = gi % kESlots;
                const int g = q * kGQ + gq;
                // busy polling for D: the next MMAs into this buffer wait for its
                // release, and a suspended try_wait can resume well after the
                // phase completes
                if (!failed &&
                    (!pq2::mbar_spin_warp(&dfull[ds], (gi / kDSlots) & 1, p.ctl, abort_v) ||
                     !pq2::mbar_spin_warp(&efull[es], (gi / kESlots) & 1, p.ctl, abort_v))) {
                    failed = true;
                    *abort_v = 1;
                }
                const float* eslot = reinterpret_cast<const float*>(sm + C::OFF_E + es * C::ESLOT);
                const float sv = failed ? 0.0f : eslot[kBN + m];
                const float tv = failed ? 0.0f : eslot[kBN + MT + m];
                if (!failed) tc_fence_after();
                // Up to 32 tokens 32 columns per wait, at 64 tokens (fewer
                // registers a thread) 16; D is released after the last wait, before
                // the arithmetic on those columns.
                constexpr int kLoads = C::QA <= 2 ? 2 : 1;  // 16-column loads per wait
#pragma unroll
                for (int cl = 0; cl < kNL; cl += kLoads) {
                    float v[16 * kLoads];
                    if (!failed) {
#pragma unroll
                        for (int l = 0; l < kLoads; ++l)
                            tmem_ld16(tmem + lane_off + ds * kBN + kCB * cb + 16 * (cl + l), v + 16 * l);
                        tmem_wait_ld();
                    }
                    if (cl + kLoads == kNL) {
                        // every column of the group is in registers: D is free
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) pq2::mbar_arrive(&dfree[ds]);
                    }
                    if (failed) continue;
#pragma unroll
                    for (int l = 0; l < kLoads; ++l) {
                    const int c = cl + l;
                    const float* vc = v + 16 * l;
                    // rows 2m (hi) and 2m + 1 (lo) are lanes 2j, 2j + 1: each lane
                    // keeps 8 of the 16 columns (8 h .. 8 h + 7) and takes its
                    // partner's values of them; the sum is exact
                    float sum[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float keep = h ? vc[8 + i] : vc[i];
                        const float give = h ? vc[i] : vc[8 + i];
                        sum[i] = keep + __shfl_xor_sync(0xffffffffu, give, 1);
                    }
                    const int c0 = kCB * cb + 16 * c + 8 * h;  // first column of this lane
                    if (DOTS) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int col = t * kBN + c0 + i;
                            const float dot = fmaf(sum[i], 512.0f, -tv);  // exact integer
                            if (m < p.M && col < p.N && g < G &&
                                pq2::store_ok(p.ctl, (static_cast<long long>(m) * p.N + col) * G + g, 1,
                                              static_cast<long long>(p.M) * p.N * G))
                                p.dots[(static_cast<size_t>(m) * p.N + col) * G + g] =
                                    static_cast<int>(dot);
                        }
                        continue;
                    }
                    const float4* wsp = reinterpret_cast<const float4*>(eslot + c0);
#pragma unroll
                    for (int i4 = 0; i4 < 2; ++i4) {
                        const float4 w4 = wsp[i4];
                        const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int i = 4 * i4 + j;
                            // the exact integer dot first, then its scales
                            const float dot = fmaf(sum[i], 512.0f, -tv);
                            acc[8 * c + i] = fmaf(dot * sv, wv[j], acc[8 * c + i]);
                        }
                    }
                    }
                }
                __syncwarp();
                if (lane == 0) pq2::mbar_arrive(&efree[es]);
            }

            // ---- end of this CTA's part of tile t: flush ----
            if (!(it == n - 1 || tile_end)) continue;
            if (pq2::named_bar_any(1, kEpiThreads, failed)) {
                *abort_v = 1;
                break;
            }
            if (DOTS) continue;
            const int c_lo = owner_of(static_cast<long long>(t) * Q, p.items, p.grid);
            const int c_hi = owner_of(static_cast<long long>(t + 1) * Q - 1, p.items, p.grid);
            // acc[8 c + i] is column colb + 16 c + i: kNL runs of 8 columns,
            // written and read as float4 j = 2 c + (i >> 2)
            const int colb = t * kBN + kCB * cb + 8 * h;
            const bool y_vec = (p.N & 3) == 0;  // 16-byte aligned rows of y
            if (c_lo == c_hi) {
                // the whole tile is this CTA's: straight to y
                if (m < p.M) {
                    float* yr = p.y + static_cast<size_t>(m) * p.N;
#pragma unroll
                    for (int j = 0; j < 2 * kNL; ++j) {
                        const int col = colb + 16 * (j >> 1) + 4 * (j & 1);
                        const long long yi = static_cast<long long>(m) * p.N + col;
                        if (y_vec && col + 3 < p.N) {
                            if (pq2::store_ok(p.ctl, yi, 4, static_cast<long long>(p.M) * p.N))
                                *reinterpret_cast<float4*>(yr + col) = make_float4(
                                    acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (col + e < p.N && pq2::store_ok(p.ctl, yi + e, 1, static_cast<long long>(p.M) * p.N))
                                    yr[col + e] = acc[4 * j + e];
                        }
                    }
                }
            } else {
                float* part = p.partial + static_cast<size_t>(blockIdx.x + t) * p.M * kBN;
                if (m < p.M) {
                    float* pr = part + static_cast<size_t>(m) * kBN + (colb - t * kBN);
#pragma unroll
                    for (int j = 0; j < 2 * kNL; ++j) {
                        float* dst = pr + 16 * (j >> 1) + 4 * (j & 1);
                        if (pq2::store_ok(p.ctl, dst - p.partial, 4,
                                          static_cast<long long>(p.grid + p.n_tiles) * p.M * kBN))
                            *reinterpret_cast<float4*>(dst) = make_float4(
                                acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
                    }
                }
                pq2::named_bar_sync(2, kEpiThreads);
                if (warp == 0 && lane == 0) {  // quadrant 0, column block 0
                    const unsigned old = pq2::atom_add_acq_rel_gpu(&p.counters[t], 1u);
                    last_flag = (old == static_cast<unsigned>(c_hi - c_lo)) ? 1 : 0;
                }
                pq2::named_bar_sync(2, kEpiThreads);
                if (last_flag && m < p.M) {
                    // the contributors' partials added in CTA order, 16 columns
                    // at a time, two contributors' loads in flight together
                    float* yr = p.y + static_cast<size_t>(m) * p.N;
                    const size_t roff = static_cast<size_t>(m) * kBN + (colb - t * kBN);
#pragma unroll 1
                    for (int hb = 0; hb < kNL / 2; ++hb) {  // float4 j = 4 hb .. 4 hb + 3
                        float4 sum[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) sum[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        for (int c = c_lo; c <= c_hi; c += 2) {
                            const bool two = c + 1 <= c_hi;
                            float4 a[4], b[4];
                            const float* pa = p.partial + static_cast<size_t>(c + t) * p.M * kBN + roff;
                            const float* pb = pa + static_cast<size_t>(p.M) * kBN;  // contributor c + 1
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int o = 16 * ((4 * hb + j) >> 1) + 4 * (j & 1);
                                a[j] = ld_cg4(pa + o);
                                b[j] = two ? ld_cg4(pb + o) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                            }
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                sum[j].x += a[j].x; sum[j].y += a[j].y;
                                sum[j].z += a[j].z; sum[j].w += a[j].w;
                                if (two) {
                                    sum[j].x += b[j].x; sum[j].y += b[j].y;
                                    sum[j].z += b[j].z; sum[j].w += b[j].w;
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int jj = 4 * hb + j;
                            const int col = colb + 16 * (jj >> 1) + 4 * (jj & 1);
                            const long long yi = static_cast<long long>(m) * p.N + col;
                            if (y_vec && col + 3 < p.N) {
                                if (pq2::store_ok(p.ctl, yi, 4, static_cast<long long>(p.M) * p.N))
                                    *reinterpret_cast<float4*>(yr + col) = sum[j];
                            } else {
                                const float e4[4] = {sum[j].x, sum[j].y, sum[j].z, sum[j].w};
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    if (col + e < p.N && pq2::store_ok(p.ctl, yi + e, 1, static_cast<long long>(p.M) * p.N))
                                        yr[col + e] = e4[e];
                            }
                        }
                    }
                }
                // last_flag is rewritten at the next flush only after every
                // flushing warp has passed the first barrier there
            }
#pragma unroll
            for (int i = 0; i < kAcc; ++i) acc[i] = 0.0f;
        }
    }

    // teardown: every role is done with tensor memory
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (role == kIssuer)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
}

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

struct WTileLayout {
    int grid, n_tiles, Q, mt;
    long long items;
    int64_t G4;
    size_t tok, st, counters, partial, total;  // byte offsets / total
};

int wtile_tokens(int64_t M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

WTileLayout layout_wtile(int64_t M, int64_t N, int64_t K, int num_sms) {
    WTileLayout l = {};
    l.mt = wtile_tokens(M);
    const int64_t G = K / 128;
    l.Q = static_cast<int>((G + kGQ - 1) / kGQ);
    l.G4 = static_cast<int64_t>(l.Q) * kGQ;
    l.n_tiles = static_cast<int>((N + kBN - 1) / kBN);
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
    // one [M][kBN] slot per (CTA c, tile t) pair, at index c + t
    off += align256(static_cast<size_t>(l.grid + l.n_tiles) * M * kBN * 4);
    l.total = off;
    return l;
}

// Layout of the token tiles for quant_tiles_kernel (pq2_matmul's path: the
// same tiles, (s, t) table and counters straight from the fp16 activations).
template <int T>
struct WTileTok {
    static constexpr int MT = T;
    static constexpr int kGroupWords = 2 * T * 32;
    __device__ static int row_hi(int m) { return 2 * m; }
    __device__ static int row_lo(int m) { return 2 * m + 1; }
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
                      const WTileLayout& l, uint8_t* w, cudaStream_t st, const pq2::DevCtl& ctl,
                      const pq2h::DeviceInfo& dev) {
    using C = WCfg<MT>;
    uint32_t* tok = reinterpret_cast<uint32_t*>(w + l.tok);
    float* stv = reinterpret_cast<float*>(w + l.st);
    unsigned* counters = reinterpret_cast<unsigned*>(w + l.counters);
    if (x) {
        // pq2_matmul's path: the tiles straight from the fp16 activations
        cudaError_t e = pq2h::launch(pq2::quant_tiles_kernel<WTileTok<MT>>,
                                     dim3(pq2::quant_tiles_grid(l.G4 * MT, dev.num_sms)), dim3(256),
                                     0, st, true, x, tok, static_cast<void*>(stv), counters, M, K,
                                     l.G4, l.n_tiles);
        if (e != cudaSuccess) return e;
    } else {
        const int64_t words = l.G4 * MT * 32;
        const int64_t want = (words + 255) / 256;
        const int grid = static_cast<int>(want < dev.num_sms * 4 ? want : dev.num_sms * 4);
        cudaError_t e = pq2h::launch(wtile_prep_kernel<MT>, dim3(grid), dim3(256), 0, st, true, qp,
                                     S, T, tok, stv, counters, M, K, l.G4, l.n_tiles);
        if (e != cudaSuccess) return e;
    }
    WTileParams p = {};
    if (!pq2h::encode_tmap_2d(&p.tm_tok, CU_TENSOR_MAP_DATA_TYPE_UINT8, tok, 128u,
                              static_cast<uint64_t>(l.G4) * C::AROWS, 128u, 128u, C::AROWS, true) ||
        !pq2h::encode_tmap_2d(&p.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes,
                              static_cast<uint64_t>(K / 4), static_cast<uint64_t>(N),
                              static_cast<uint64_t>(K / 4), 128u, kBN, true))
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
    auto kern = dots ? wtile_kernel<MT, true> : wtile_kernel<MT, false>;
    static pq2h::SmemLimit lim[2];
    cudaError_t e = pq2h::ensure_smem(lim[dots ? 1 : 0], kern, C::SMEM);
    if (e != cudaSuccess) return e;
    return pq2h::launch(kern, dim3(l.grid), dim3(C::THREADS), C::SMEM, st, true, p);
}

// x != nullptr: the token tiles straight from x (qp, S, T unused)
cudaError_t launch_wtile_any(const __half* x, const int8_t* qp, const float* S, const int32_t* T,
                           const uint8_t* codes, const __half* ws, float* y, int32_t* dots,
                           int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                           const pq2::DevCtl& ctl, const pq2h::DeviceInfo& dev) {
    if (M < 1 || M > pq2h::kTileMaxM) return cudaErrorInvalidValue;
    const WTileLayout l = layout_wtile(M, N, K, dev.num_sms);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    if (l.mt == 16)
        return launch_mt<16>(x, qp, S, T, codes, ws, y, dots, M, N, K, l, w, st, ctl, dev);
    if (l.mt == 32)
        return launch_mt<32>(x, qp, S, T, codes, ws, y, dots, M, N, K, l, w, st, ctl, dev);
    return launch_mt<64>(x, qp, S, T, codes, ws, y, dots, M, N, K, l, w, st, ctl, dev);
}

}  // namespace

namespace pq2h {

bool wtile_default(int64_t M, int64_t N, int64_t K, int num_sms) {
    if (M <= kWTileDefaultMinM || M > kTileMaxM) return false;
    const WTileLayout l = layout_wtile(M, N, K, num_sms);
    const long long cap = num_sms < kMaxGrid ? num_sms : kMaxGrid;
    return l.items <= kWTileDefaultItemsPerCta * cap;
}

size_t wtile_scratch_bytes(int64_t M, int64_t N, int64_t K, int num_sms) {
    return layout_wtile(M, N, K, num_sms).total;
}

size_t wtile_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    return wtile_scratch_bytes(M, N, K, kMaxGrid);
}

cudaError_t launch_wtile(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                        const __half* ws, float* y, int32_t* dots, int64_t M, int64_t N, int64_t K,
                        void* workspace, cudaStream_t st, const pq2::DevCtl& ctl,
                        const DeviceInfo& dev) {
    return launch_wtile_any(nullptr, qp, S, T, codes, ws, y, dots, M, N, K, workspace, st, ctl, dev);
}

cudaError_t launch_wtile_x(const __half* x, const uint8_t* codes, const __half* ws, float* y,
                          int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                          const pq2::DevCtl& ctl, const DeviceInfo& dev) {
    return launch_wtile_any(x, nullptr, nullptr, nullptr, codes, ws, y, nullptr, M, N, K, workspace,
                          st, ctl, dev);
}

}  // namespace pq2h
