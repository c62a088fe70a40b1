// Prompt-processing matmul, any M (pq2_gemm_prefill), on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// The method is the pages' prefill kernel ("Making a ternary reasoning model
// fast in vLLM", page "From CUDA to Triton and Gluon", section "Prompt
// processing: check configuration and launch costs"): 2-D output tiles,
// per-group integer products from the planes of the codes, the -sum(q)
// correction and the same per-group fp32 dequantise-accumulate order as the
// M = 1 path.
//
// GB300 design.  tcgen05 has no int8 kind on sm_103a; kind::f8f6f4 with e4m3
// operands is exact here:
//  * weights (B operand, N = 128 rows per tile): plane s of code byte b is
//    (byte >> 2s) & 3, stored as the e4m3 byte itself = c * 2^-9 (e4m3 bytes
//    below 16 are exactly byte * 2^-9);
//  * tokens (A operand, M = 128 rows per tile): q = 16h + l with h in
//    [-8,7], l in [0,15]; 16h and l are exact e4m3 values, prepared once per
//    call in two planes (hi, lo) by a small kernel;
//  * two MMAs per k-step (hi, lo) accumulate into the same fp32 D in tensor
//    memory: D = 2^-9 * sum(code * q), an exact small multiple of 2^-9.
//  The k order inside a group is the plane order of the activations: k-step
//  s of a group (32 values) is plane s, so a weight row of B is
//  [plane0 bytes 0..31 | plane1 | plane2 | plane3], written by the expansion
//  warps straight into the 128-byte-swizzled K-major shared layout.
//
// Per CTA (persistent over 128x128 output tiles, one per SM):
//   warp 0      TMA producer: per group, the hi and lo token tiles
//               (128 x 128 B, 128B swizzle) and the code tile (128 x 32 B)
//   warps 1, 14 MMA issuers (one thread each; warp 1 the even groups, warp 14
//               the odd ones): 4 k-steps x (hi, lo) per group into one of
//               four D buffers, then tcgen05.commit.  A warp that issues
//               tcgen05.mma is held for tens of cycles per instruction; two
//               issuers keep the tensor pipe fed.  Even and odd groups use
//               disjoint stages and D buffers, so the two share no barrier.
//   warps 2-5   expansion: one weight row per thread, codes -> e4m3 B tile;
//               also the group's weight scales for the epilogue (a ring of
//               their own, released by the epilogue, so the expansion never
//               waits for the epilogue of the previous group)
//   warps 6-13  epilogue: per group, dot = D*512 - t (exact), then
//               acc += dot * s * ws with the running fp32 accumulator in
//               registers (64 columns per thread); finally acc -> y.
// Four D buffers (all 512 columns of tensor memory) give the MMAs three
// groups of slack on the epilogue.
//
// prefill_wide_kernel (below) runs the same arithmetic on 128 x 256 tiles
// from weights expanded once per call by the preparation kernel; it is the
// default from 8 token tiles on, once its tiles fill every SM.
// Every mbarrier wait is bounded (device error word on expiry).
#include "pq2_internal.h"
#include "pq2_tokens.cuh"

namespace {

constexpr int kTileM = 128;  // tokens per tile (MMA M)
constexpr int kTileN = 128;  // weight rows per tile (MMA N)
constexpr int kStages = 4;
constexpr int kDBufs = 4;            // D buffers in tensor memory, 128 columns each
constexpr int kEpiWarp0 = 6;
constexpr int kIssuer2 = 14;         // second MMA issuer (odd groups)
static_assert(kStages % 2 == 0 && kDBufs % 2 == 0,
              "even and odd groups must use disjoint stages and D buffers");
constexpr int kThreads = 15 * 32;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kATileBytes = kTileM * 128;   // one group of 128 token rows
constexpr uint32_t kBTileBytes = kTileN * 128;   // expanded weight rows
constexpr uint32_t kCTileBytes = kTileN * 32;    // raw code rows
constexpr uint32_t kStageBytes = 2 * kATileBytes + kBTileBytes + kCTileBytes;  // 53248

struct PrefillParams {
    CUtensorMap tm_ahi;    // e4m3 [M][K], box {128, 128}, 128B swizzle
    CUtensorMap tm_alo;
    CUtensorMap tm_codes;  // uint8 [N][K/4], box {32, 128}
    const float2* st;      // [G][M] (s, t)
    const __half* ws;      // [N][G]
    float* y;              // [M][N]
    int32_t* dots;         // debug: [M][N][G]
    int M, N, K, G;
    int m_tiles, n_tiles;
    pq2::DevCtl ctl;
};

// ---------------------------------------------------------------------------
// token planes: q = 16h + l -> e4m3(16h), e4m3(l); (s, t) transposed to [G][M]
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) token_planes_kernel(const int8_t* __restrict__ qp,
                                                           const float* __restrict__ S,
                                                           const int32_t* __restrict__ T,
                                                           uint32_t* __restrict__ ahi,
                                                           uint32_t* __restrict__ alo,
                                                           float2* __restrict__ st, int64_t M,
                                                           int64_t K,
                                                           const uint8_t* __restrict__ codes,
                                                           const __half* __restrict__ ws,
                                                           uint8_t* __restrict__ wexp,
                                                           float* __restrict__ wst, int64_t N,
                                                           int64_t Npad) {
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();
    const int64_t words = M * K / 4;
    const int64_t G = K / 128;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < words;
         i += stride) {
        const uint32_t qw = reinterpret_cast<const uint32_t*>(qp)[i];
        uint32_t hw, lw;  // e4m3 of 16 * floor(q / 16) and q - 16 * floor(q / 16)
        pq2::hi_lo_words(qw, hw, lw);
        ahi[i] = hw;
        alo[i] = lw;
    }
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < M * G;
         i += stride) {
        const int64_t m = i / G, g = i - m * G;
        st[g * M + m] = make_float2(S ? S[i] : 0.0f, static_cast<float>(T[i]));
    }
    if (!wexp) return;
    // wide kernel: the weights' e4m3 planes, row n of group g being
    // [plane 0 bytes 0..31 | plane 1 | plane 2 | plane 3] (plane s of code
    // byte b = (byte >> 2s) & 3, the e4m3 byte c = c * 2^-9), 16 code bytes
    // per index
    const int cpr = static_cast<int>(K / 64);  // 16-byte code chunks per row
    for (int64_t n = blockIdx.x; n < N; n += gridDim.x) {
        for (int c = threadIdx.x; c < cpr; c += blockDim.x) {
            const int g = c >> 1, half = c & 1;
            const uint4 w = *reinterpret_cast<const uint4*>(codes + n * (K / 4) + g * 32 + half * 16);
            uint8_t* dst = wexp + n * K + g * 128 + half * 16;
#pragma unroll
            for (int pl = 0; pl < 4; ++pl) {
                const uint4 v = make_uint4(
                    (w.x >> (2 * pl)) & 0x03030303u, (w.y >> (2 * pl)) & 0x03030303u,
                    (w.z >> (2 * pl)) & 0x03030303u, (w.w >> (2 * pl)) & 0x03030303u);
                *reinterpret_cast<uint4*>(dst + 32 * pl) = v;
            }
        }
    }
    // and the weight scales as fp32 [G][Npad], zero past N
    for (int64_t g = 0; g < G; ++g)
        for (int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; n < Npad;
             n += stride)
            wst[g * Npad + n] = (ws && n < N) ? __half2float(ws[n * G + g]) : 0.0f;
}

// ---------------------------------------------------------------------------
// tcgen05 helpers
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1) << 16;             // leading offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;     // stride offset
    d |= static_cast<uint64_t>(1) << 46;             // descriptor version
    d |= static_cast<uint64_t>(2) << 61;             // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f8f6f4: D f32, A and B e4m3, both K-major.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) |
                            (static_cast<uint32_t>(kTileN >> 3) << 17) |
                            (static_cast<uint32_t>(kTileM >> 4) << 24);

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
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

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
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

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// main kernel
// ---------------------------------------------------------------------------
template <bool DOTS>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t full[kStages];   // TMA bytes of a stage landed
    __shared__ uint64_t bready[kStages]; // expanded weight tile written (4 warps)
    __shared__ uint64_t empty[kStages];  // MMAs of the stage done (commit)
    __shared__ uint64_t wsfree[kStages]; // epilogue done with a slot of ws_sm (8 warps)
    __shared__ uint64_t dfull[kDBufs];   // D buffer holds a finished group (commit)
    __shared__ uint64_t dempty[kDBufs];  // epilogue done with a D buffer (8 warps)
    __shared__ __align__(16) float ws_sm[kStages][kTileN];  // weight scales per stage
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t base = pq2::smem_u32(smem);
    uint8_t* stage0 = smem + ((1024 - (base & 1023)) & 1023);

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            pq2::mbar_init(&full[i], 1);
            pq2::mbar_init(&bready[i], 4);
            pq2::mbar_init(&empty[i], 1);
            pq2::mbar_init(&wsfree[i], 8);
        }
        for (int i = 0; i < kDBufs; ++i) {
            pq2::mbar_init(&dfull[i], 1);
            pq2::mbar_init(&dempty[i], 8);
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
    const int G = p.G;
    const int n_tiles_total = p.m_tiles * p.n_tiles;
    volatile int* abort_v = &abort_flag;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            int it = 0;  // global group counter (stage = it % kStages)
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles_total && ok; tile += gridDim.x) {
                const int mt = tile % p.m_tiles, nt = tile / p.m_tiles;
                for (int g = 0; g < G; ++g, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages &&
                        !pq2::mbar_wait_bounded(&empty[s], ((it / kStages) - 1) & 1, p.ctl, abort_v)) {
                        ok = false;
                        break;
                    }
                    if (it == p.ctl.debug_skip_stage) continue;
                    uint8_t* st = stage0 + static_cast<size_t>(s) * kStageBytes;
                    pq2::mbar_arrive_expect_tx(&full[s], kStageBytes - kBTileBytes);
                    pq2::tma_load_2d(st, &p.tm_ahi, g * 128, mt * kTileM, &full[s]);
                    pq2::tma_load_2d(st + kATileBytes, &p.tm_alo, g * 128, mt * kTileM, &full[s]);
                    pq2::tma_load_2d(st + 2 * kATileBytes + kBTileBytes, &p.tm_codes, g * 32,
                                     nt * kTileN, &full[s]);
                }
            }
            // drain: every armed stage must have landed before exit
            const int issued = it;
            for (int s = 0; s < kStages; ++s) {
                if (issued <= s) continue;
                int last = s + ((issued - 1 - s) / kStages) * kStages;
                if (last == p.ctl.debug_skip_stage) last -= kStages;
                if (last >= 0) pq2::mbar_wait_bounded(&full[s], (last / kStages) & 1, p.ctl);
            }
        }
    } else if (warp == 1 || warp == kIssuer2) {
        // ------------------------------ MMA issuers ------------------------------
        const int parity = warp == 1 ? 0 : 1;
        if (lane == 0) {
            int it = 0;
            int last = -1;  // last group this issuer committed
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles_total && ok; tile += gridDim.x) {
                for (int g = 0; g < G; ++g, ++it) {
                    if ((it & 1) != parity) continue;
                    const int s = it % kStages;
                    const int db = it % kDBufs;
                    // busy polling: this thread is on the critical path (a
                    // sleeping poller wakes up hundreds of cycles late)
                    if (!pq2::mbar_spin_bounded(&bready[s], (it / kStages) & 1, p.ctl, abort_v) ||
                        (it >= kDBufs &&
                         !pq2::mbar_spin_bounded(&dempty[db], ((it / kDBufs) - 1) & 1, p.ctl,
                                                 abort_v))) {
                        ok = false;
                        *abort_v = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = pq2::smem_u32(stage0 + static_cast<size_t>(s) * kStageBytes);
                    const uint32_t d_tmem = tmem + db * 128;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t bdesc = sw128_desc(st + 2 * kATileBytes + 32 * k);
                        mma_f8(d_tmem, sw128_desc(st + 32 * k), bdesc, k > 0);
                        mma_f8(d_tmem, sw128_desc(st + kATileBytes + 32 * k), bdesc, 1);
                    }
                    mma_commit(&empty[s]);
                    mma_commit(&dfull[db]);
                    last = it;
                }
            }
            // no MMA may still be running when tensor memory is released
            if (last >= 0)
                pq2::mbar_wait_bounded(&dfull[last % kDBufs], (last / kDBufs) & 1, p.ctl);
        }
    } else if (warp < kEpiWarp0) {  // warps 2-5
        // ------------------------------ expansion ------------------------------
        const int r = (warp - 2) * 32 + lane;  // weight row within the tile
        const int half = (lane >> 2) & 1;      // conflict-free order of the 2 loads
        int it = 0;
        bool failed = false;
        for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x) {
            const int nt = tile / p.m_tiles;
            const int n = nt * kTileN + r;
            for (int g = 0; g < G; ++g, ++it) {
                const int s = it % kStages;
                // weight scale of this row for the epilogue (prefetched before the waits)
                const float wsv = (!DOTS && n < p.N) ? __half2float(p.ws[static_cast<size_t>(n) * G + g]) : 0.0f;
                // ws_sm[s] was last read by the epilogue of group it - kStages
                if (!failed &&
                    (!pq2::mbar_wait_bounded(&full[s], (it / kStages) & 1, p.ctl, abort_v) ||
                     (it >= kStages &&
                      !pq2::mbar_wait_bounded(&wsfree[s], ((it / kStages) - 1) & 1, p.ctl,
                                              abort_v)))) {
                    failed = true;
                    *abort_v = 1;
                }
                if (!failed) {
                    uint8_t* st = stage0 + static_cast<size_t>(s) * kStageBytes;
                    const uint8_t* crow = st + 2 * kATileBytes + kBTileBytes + r * 32;
                    const uint4 ca = *reinterpret_cast<const uint4*>(crow + 16 * half);
                    const uint4 cb = *reinterpret_cast<const uint4*>(crow + 16 * (half ^ 1));
                    const uint32_t w[8] = {half ? cb.x : ca.x, half ? cb.y : ca.y,
                                           half ? cb.z : ca.z, half ? cb.w : ca.w,
                                           half ? ca.x : cb.x, half ? ca.y : cb.y,
                                           half ? ca.z : cb.z, half ? ca.w : cb.w};
                    uint8_t* brow = st + 2 * kATileBytes + r * 128;
#pragma unroll
                    for (int pl = 0; pl < 4; ++pl) {
#pragma unroll
                        for (int hc = 0; hc < 2; ++hc) {  // 16-byte chunk 2*pl + hc
                            uint4 v;
                            v.x = (w[4 * hc + 0] >> (2 * pl)) & 0x03030303u;
                            v.y = (w[4 * hc + 1] >> (2 * pl)) & 0x03030303u;
                            v.z = (w[4 * hc + 2] >> (2 * pl)) & 0x03030303u;
                            v.w = (w[4 * hc + 3] >> (2 * pl)) & 0x03030303u;
                            const int chunk = (2 * pl + hc) ^ (r & 7);
                            *reinterpret_cast<uint4*>(brow + 16 * chunk) = v;
                        }
                    }
                    ws_sm[s][r] = wsv;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                __syncwarp();
                if (lane == 0) pq2::mbar_arrive(&bready[s]);
            }
        }
    } else if (warp < kIssuer2) {
        // ------------------------------ epilogue ------------------------------
        const int ew = warp - kEpiWarp0;  // 0..7
        const int quad = warp & 3;        // TMEM lane quadrant of this warp
        const int col0 = (ew >> 2) * 64;  // two warps per quadrant: columns [0,64), [64,128)
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        int it = 0;
        bool failed = false;
        for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x) {
            const int mt = tile % p.m_tiles, nt = tile / p.m_tiles;
            const int m = mt * kTileM + quad * 32 + lane;  // token row of this thread
            const bool mvalid = m < p.M;
            // accumulators as pairs of adjacent columns (two-wide fp32 ops)
            unsigned long long acc2[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc2[j] = 0ull;
            float2 stv = (mvalid && !failed) ? p.st[m] : make_float2(0.0f, 0.0f);  // group 0
            for (int g = 0; g < G; ++g, ++it) {
                const int s = it % kStages;
                const int db = it % kDBufs;
                // prefetch next group's (s, t) for this token
                float2 st_next = make_float2(0.0f, 0.0f);
                if (mvalid && g + 1 < G) st_next = p.st[static_cast<size_t>(g + 1) * p.M + m];
                if (!failed &&
                    !pq2::mbar_wait_bounded(&dfull[db], (it / kDBufs) & 1, p.ctl, abort_v)) {
                    failed = true;
                    *abort_v = 1;
                }
                // warp-uniform from here: the tensor-memory loads below are
                // executed by all 32 lanes or none
                failed = __any_sync(0xffffffffu, failed);
                if (!failed) {
                    tc_fence_after();
                    // the 64 weight scales of this thread's columns: 16-byte
                    // broadcast loads (every lane reads the same address)
                    const ulonglong2* ws2 = reinterpret_cast<const ulonglong2*>(ws_sm[s] + col0);
                    const unsigned long long k512 = f2pack(512.0f, 512.0f);
                    const unsigned long long negt = f2pack(-stv.y, -stv.y);
                    const unsigned long long sv2 = f2pack(stv.x, stv.x);
#pragma unroll
                    for (int c = 0; c < 64; c += 32) {
                        float d[32];
                        tmem_ld32(tmem + lane_off + db * 128 + col0 + c, d);
                        tmem_wait_ld();
                        if (DOTS) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const float dot = fmaf(d[j], 512.0f, -stv.y);  // exact integer
                                const int n = nt * kTileN + col0 + c + j;
                                if (mvalid && n < p.N &&
                                    pq2::store_ok(p.ctl, (static_cast<long long>(m) * p.N + n) * G + g,
                                                  1, static_cast<long long>(p.M) * p.N * G))
                                    p.dots[(static_cast<size_t>(m) * p.N + n) * G + g] =
                                        static_cast<int>(dot);
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; j += 2) {
                                // exact integer dots of columns j, j + 1, then the
                                // scales; the first group's term seeds the sum (0 + x
                                // would turn a -0 term into +0)
                                const unsigned long long dot2 =
                                    fma2(f2pack(d[j], d[j + 1]), k512, negt);
                                const unsigned long long term2 = mul2(dot2, sv2);
                                const ulonglong2 w4 = ws2[(c + j) >> 2];
                                const unsigned long long w2 = ((j >> 1) & 1) ? w4.y : w4.x;
                                const int a = (c + j) >> 1;
                                acc2[a] = g > 0 ? fma2(term2, w2, acc2[a]) : mul2(term2, w2);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    pq2::mbar_arrive(&dempty[db]);
                    pq2::mbar_arrive(&wsfree[s]);
                }
                stv = st_next;
            }
            float acc[64];
#pragma unroll
            for (int j = 0; j < 32; ++j) f2unpack(acc2[j], acc[2 * j], acc[2 * j + 1]);
            // tile done: acc -> y
            if (!DOTS && !failed && mvalid) {
                const int nb = nt * kTileN + col0;
                float* yrow = p.y + static_cast<size_t>(m) * p.N + nb;
                const long long yi = static_cast<long long>(m) * p.N + nb;
                if (nb + 64 <= p.N && (p.N & 3) == 0) {
#pragma unroll
                    for (int j = 0; j < 64; j += 4)
                        if (pq2::store_ok(p.ctl, yi + j, 4, static_cast<long long>(p.M) * p.N))
                            *reinterpret_cast<float4*>(yrow + j) =
                                make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        if (nb + j < p.N && pq2::store_ok(p.ctl, yi + j, 1, static_cast<long long>(p.M) * p.N))
                            yrow[j] = acc[j];
                }
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

// ---------------------------------------------------------------------------
// wide variant: 128 tokens x 256 weight rows per tile
// ---------------------------------------------------------------------------
// The same arithmetic as prefill_kernel (bit-identical y) with twice the MMA
// work per group: every barrier round trip of the per-group protocol and
// every MMA instruction covers 256 weight rows, and each tensor-core read of
// the token tile serves twice the products.  The weights' e4m3 planes and
// the weight scales (fp32, [G][Npad]) are written once per call by the
// preparation kernel, so the TMA engine brings the B tile in the MMA's
// layout and no warp writes shared memory per group: shared-memory
// bandwidth, which the tensor cores' operand reads share with every warp's
// loads, stores and barrier polls, was the limit with expansion warps.
// Tensor memory holds two D buffers of 256 columns; three stages of 64 KB
// (token hi and lo planes, expanded weights) fill shared memory, and a ring
// of kWsSlots weight-scale rows (1 KB each, bulk copies) feeds the epilogue.
//   warp 0        TMA producer
//   warp 1        TMEM allocation, the MMA issuer (one thread; an N = 256
//                 MMA keeps the pipe busy for longer than it holds the warp)
//   warps 2-3     idle
//   warps 4-11    epilogue: a TMEM lane quadrant and 128 columns each, the
//                 fp32 accumulator (128 columns) in registers
// Registers: warpgroup 0 gives its back (setmaxnreg.dec to kRegsLow),
// warpgroups 1-2 take them (setmaxnreg.inc to kRegsHigh).  The launch
// checks that the kernel's register allocation covers the split.
constexpr int kWTileN = 256;
constexpr int kWStages = 3;
constexpr int kWsSlots = 6;
constexpr int kWThreads = 12 * 32;
constexpr int kWEpi0 = 4;             // first epilogue warp
constexpr int kRegsLow = 64;
constexpr int kRegsHigh = 216;
constexpr int kWRegsNeeded = 128 * kRegsLow + 2 * 128 * kRegsHigh;  // 63488
constexpr uint32_t kWBTileBytes = kWTileN * 128;
constexpr uint32_t kWStageBytes = 2 * kATileBytes + kWBTileBytes;  // 65536
constexpr uint32_t kWsRowBytes = kWTileN * 4;
static_assert(kWStageBytes % 1024 == 0, "stages on 1024-byte boundaries");
static_assert(kWRegsNeeded <= 65536, "register split");

constexpr uint32_t kWIdesc = (1u << 4) | (0u << 7) | (0u << 10) |
                             (static_cast<uint32_t>(kWTileN >> 3) << 17) |
                             (static_cast<uint32_t>(kTileM >> 4) << 24);

struct PrefillWideParams {
    CUtensorMap tm_ahi;    // e4m3 [M][K], box {128, 128}, 128B swizzle
    CUtensorMap tm_alo;
    CUtensorMap tm_b;      // e4m3 planes of the weights [N][K], box {128, 256}, 128B swizzle
    const float2* st;      // [G][M] (s, t)
    const float* wst;      // [G][Npad] weight scales, zero past N
    float* y;              // [M][N]
    int32_t* dots;         // debug: [M][N][G]
    int M, N, K, G, Npad;
    int m_tiles, n_tiles;
    pq2::DevCtl ctl;
};

__device__ __forceinline__ void mma_f8_wide(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kWIdesc), "r"(acc));
}

template <bool DOTS>
__global__ void __launch_bounds__(kWThreads, 1) prefill_wide_kernel(const __grid_constant__ PrefillWideParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t full[kWStages];    // TMA bytes of a stage landed
    __shared__ uint64_t empty[kWStages];   // MMAs of the stage done (commit)
    __shared__ uint64_t wsfull[kWsSlots];  // a weight-scale row landed
    __shared__ uint64_t wsfree[kWsSlots];  // epilogue done with a weight-scale row (8 warps)
    __shared__ uint64_t dfull[2];          // D buffer holds a finished group (commit)
    __shared__ uint64_t dempty[2];         // epilogue done with a D buffer (8 warps)
    __shared__ __align__(16) float ws_ring[kWsSlots][kWTileN];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t base = pq2::smem_u32(smem);
    uint8_t* stage0 = smem + ((1024 - (base & 1023)) & 1023);

    if (tid == 0) {
        for (int i = 0; i < kWStages; ++i) {
            pq2::mbar_init(&full[i], 1);
            pq2::mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < kWsSlots; ++i) {
            pq2::mbar_init(&wsfull[i], 1);
            pq2::mbar_init(&wsfree[i], 8);
        }
        for (int i = 0; i < 2; ++i) {
            pq2::mbar_init(&dfull[i], 1);
            pq2::mbar_init(&dempty[i], 8);
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
    const int G = p.G;
    const int n_tiles_total = p.m_tiles * p.n_tiles;
    volatile int* abort_v = &abort_flag;

    // Each role's code follows its own setmaxnreg, so that the compiler
    // allocates its registers to the new limit.
    if (warp < kWEpi0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
        if (warp == 0 && lane == 0) {
            // ------------------------------ TMA producer ------------------------------
            int it = 0;  // global group counter
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles_total && ok; tile += gridDim.x) {
                const int mt = tile % p.m_tiles, nt = tile / p.m_tiles;
                for (int g = 0; g < G; ++g, ++it) {
                    const int s = it % kWStages;
                    const int w = it % kWsSlots;
                    if ((it >= kWStages &&
                         !pq2::mbar_wait_bounded(&empty[s], ((it / kWStages) - 1) & 1, p.ctl,
                                                 abort_v)) ||
                        (it >= kWsSlots &&
                         !pq2::mbar_wait_bounded(&wsfree[w], ((it / kWsSlots) - 1) & 1, p.ctl,
                                                 abort_v))) {
                        ok = false;
                        break;
                    }
                    if (it == p.ctl.debug_skip_stage) continue;
                    uint8_t* st = stage0 + static_cast<size_t>(s) * kWStageBytes;
                    pq2::mbar_arrive_expect_tx(&full[s], kWStageBytes);
                    pq2::tma_load_2d(st, &p.tm_ahi, g * 128, mt * kTileM, &full[s]);
                    pq2::tma_load_2d(st + kATileBytes, &p.tm_alo, g * 128, mt * kTileM, &full[s]);
                    pq2::tma_load_2d(st + 2 * kATileBytes, &p.tm_b, g * 128, nt * kWTileN, &full[s]);
                    pq2::mbar_arrive_expect_tx(&wsfull[w], kWsRowBytes);
                    pq2::bulk_g2s(ws_ring[w],
                                  p.wst + static_cast<size_t>(g) * p.Npad +
                                      static_cast<size_t>(nt) * kWTileN,
                                  kWsRowBytes, &wsfull[w]);
                }
            }
            // drain: every armed copy must have landed before exit
            const int issued = it;
            for (int s = 0; s < kWStages; ++s) {
                if (issued <= s) continue;
                int last = s + ((issued - 1 - s) / kWStages) * kWStages;
                if (last == p.ctl.debug_skip_stage) last -= kWStages;
                if (last >= 0) pq2::mbar_wait_bounded(&full[s], (last / kWStages) & 1, p.ctl);
            }
            for (int w = 0; w < kWsSlots; ++w) {
                if (issued <= w) continue;
                int last = w + ((issued - 1 - w) / kWsSlots) * kWsSlots;
                if (last == p.ctl.debug_skip_stage) last -= kWsSlots;
                if (last >= 0) pq2::mbar_wait_bounded(&wsfull[w], (last / kWsSlots) & 1, p.ctl);
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------ MMA issuer ------------------------------
            int it = 0;
            int last = -1;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles_total && ok; tile += gridDim.x) {
                for (int g = 0; g < G; ++g, ++it) {
                    const int s = it % kWStages;
                    const int db = it & 1;
                    if (!pq2::mbar_spin_bounded(&full[s], (it / kWStages) & 1, p.ctl, abort_v) ||
                        (it >= 2 &&
                         !pq2::mbar_spin_bounded(&dempty[db], ((it >> 1) - 1) & 1, p.ctl, abort_v))) {
                        ok = false;
                        *abort_v = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = pq2::smem_u32(stage0 + static_cast<size_t>(s) * kWStageBytes);
                    const uint32_t d_tmem = tmem + db * kWTileN;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t bdesc = sw128_desc(st + 2 * kATileBytes + 32 * k);
                        mma_f8_wide(d_tmem, sw128_desc(st + 32 * k), bdesc, k > 0);
                        mma_f8_wide(d_tmem, sw128_desc(st + kATileBytes + 32 * k), bdesc, 1);
                    }
                    mma_commit(&empty[s]);
                    mma_commit(&dfull[db]);
                    last = it;
                }
            }
            // no MMA may still be running when tensor memory is released
            if (last >= 0) pq2::mbar_wait_bounded(&dfull[last & 1], (last >> 1) & 1, p.ctl);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ------------------------------ epilogue ------------------------------
        const int ew = warp - kWEpi0;      // 0..7
        const int quad = warp & 3;         // TMEM lane quadrant of this warp
        const int col0 = (ew >> 2) * 128;  // two warps per quadrant: columns [0,128), [128,256)
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        int it = 0;
        bool failed = false;
        for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x) {
            const int mt = tile % p.m_tiles, nt = tile / p.m_tiles;
            const int m = mt * kTileM + quad * 32 + lane;  // token row of this thread
            const bool mvalid = m < p.M;
            unsigned long long acc2[64];  // columns 2j, 2j + 1
#pragma unroll
            for (int j = 0; j < 64; ++j) acc2[j] = 0ull;
            float2 stv = (mvalid && !failed) ? p.st[m] : make_float2(0.0f, 0.0f);  // group 0
            for (int g = 0; g < G; ++g, ++it) {
                const int db = it & 1;
                const int w = it % kWsSlots;
                float2 st_next = make_float2(0.0f, 0.0f);
                if (mvalid && g + 1 < G) st_next = p.st[static_cast<size_t>(g + 1) * p.M + m];
                if (!failed &&
                    (!pq2::mbar_wait_bounded(&dfull[db], (it >> 1) & 1, p.ctl, abort_v) ||
                     !pq2::mbar_wait_bounded(&wsfull[w], (it / kWsSlots) & 1, p.ctl, abort_v))) {
                    failed = true;
                    *abort_v = 1;
                }
                // warp-uniform from here: the tensor-memory loads and the
                // warp barriers below are executed by all 32 lanes or none
                failed = __any_sync(0xffffffffu, failed);
                if (!failed) {
                    tc_fence_after();
                    const ulonglong2* ws2 = reinterpret_cast<const ulonglong2*>(ws_ring[w] + col0);
                    const unsigned long long k512 = f2pack(512.0f, 512.0f);
                    const unsigned long long negt = f2pack(-stv.y, -stv.y);
                    const unsigned long long sv2 = f2pack(stv.x, stv.x);
                    // 64 columns per tensor-memory round trip (two loads, one wait)
#pragma unroll
                    for (int c = 0; c < 128; c += 64) {
                        float d[64];
                        tmem_ld32(tmem + lane_off + db * kWTileN + col0 + c,
                                  *reinterpret_cast<float(*)[32]>(&d[0]));
                        tmem_ld32(tmem + lane_off + db * kWTileN + col0 + c + 32,
                                  *reinterpret_cast<float(*)[32]>(&d[32]));
                        tmem_wait_ld();
                        if (c == 64) {
                            // every column is in registers: the D buffer is free
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) pq2::mbar_arrive(&dempty[db]);
                        }
                        if (DOTS) {
#pragma unroll
                            for (int j = 0; j < 64; ++j) {
                                const float dot = fmaf(d[j], 512.0f, -stv.y);  // exact integer
                                const int n = nt * kWTileN + col0 + c + j;
                                if (mvalid && n < p.N &&
                                    pq2::store_ok(p.ctl, (static_cast<long long>(m) * p.N + n) * G + g,
                                                  1, static_cast<long long>(p.M) * p.N * G))
                                    p.dots[(static_cast<size_t>(m) * p.N + n) * G + g] =
                                        static_cast<int>(dot);
                            }
                            continue;
                        }
#pragma unroll
                        for (int j = 0; j < 64; j += 2) {
                            // exact integer dots of two columns, then the scales;
                            // the first group's term seeds the sum
                            const unsigned long long dot2 = fma2(f2pack(d[j], d[j + 1]), k512, negt);
                            const unsigned long long term2 = mul2(dot2, sv2);
                            const ulonglong2 w4 = ws2[(c + j) >> 2];
                            const unsigned long long w2 = ((j >> 1) & 1) ? w4.y : w4.x;
                            const int a = (c + j) >> 1;
                            acc2[a] = g > 0 ? fma2(term2, w2, acc2[a]) : mul2(term2, w2);
                        }
                    }
                } else {
                    // (the failed path never reached the early release)
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) pq2::mbar_arrive(&dempty[db]);
                }
                __syncwarp();
                if (lane == 0) pq2::mbar_arrive(&wsfree[w]);
                stv = st_next;
            }
            // tile done: acc -> y
            if (!DOTS && !failed && mvalid) {
                const int nb = nt * kWTileN + col0;
                float* yrow = p.y + static_cast<size_t>(m) * p.N + nb;
                const long long yi = static_cast<long long>(m) * p.N + nb;
                if (nb + 128 <= p.N && (p.N & 3) == 0) {
#pragma unroll
                    for (int j = 0; j < 64; j += 2) {
                        float a0, a1, a2, a3;
                        f2unpack(acc2[j], a0, a1);
                        f2unpack(acc2[j + 1], a2, a3);
                        if (pq2::store_ok(p.ctl, yi + 2 * j, 4, static_cast<long long>(p.M) * p.N))
                            *reinterpret_cast<float4*>(yrow + 2 * j) = make_float4(a0, a1, a2, a3);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        float a0, a1;
                        f2unpack(acc2[j], a0, a1);
                        if (nb + 2 * j < p.N && pq2::store_ok(p.ctl, yi + 2 * j, 1, static_cast<long long>(p.M) * p.N))
                            yrow[2 * j] = a0;
                        if (nb + 2 * j + 1 < p.N && pq2::store_ok(p.ctl, yi + 2 * j + 1, 1, static_cast<long long>(p.M) * p.N))
                            yrow[2 * j + 1] = a1;
                    }
                }
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

// setmaxnreg.inc draws on the registers the block was launched with: the
// wide kernel runs only if its compiled allocation covers the split (else
// the raising warps would wait forever).
template <bool DOTS>
bool wide_kernel_fits() {
    static const bool ok = [] {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, prefill_wide_kernel<DOTS>) != cudaSuccess) return false;
        return fa.numRegs * kWThreads >= kWRegsNeeded;
    }();
    return ok;
}

// Workspace: token planes hi, lo [M][K]; (s, t) [G][M]; and, for shapes the
// wide kernel may take, the weights' e4m3 planes [N][K] and the weight
// scales [G][Npad] fp32 (Npad = N rounded up to 256).  The wide kernel
// needs at least kWideMinMTiles token tiles (the expansion pass writes N*K
// bytes once per call: measured at N = 17408, M = 512 it only ties the
// 128 x 128 kernel, 662 against 659 TOPS, and M = 1024 gains 778 against
// 685) and at least kWideMinTiles tiles, a bound below the SM count of the
// GPUs this library is built for; forcing the variant
// (pq2_debug_force_kernel) gives it room at any shape.  The size depends on
// the shape (and the forced variant) only, not on the device.
constexpr int kTileDefaultMaxM = 32;
constexpr int kWideMinTiles = 128;
constexpr int kWideMinMTiles = 8;
struct WsLayout {
    size_t ahi, alo, st, wexp, wst, total;
    size_t wexp_bytes;
    int64_t npad;
};
WsLayout ws_layout(int64_t M, int64_t N, int64_t K) {
    WsLayout l = {};
    const int64_t G = K / 128;
    const int64_t m_tiles = (M + kTileM - 1) / kTileM;
    const int64_t wide_tiles = m_tiles * ((N + kWTileN - 1) / kWTileN);
    const int force = pq2h::forced_variant(PQ2_OP_PREFILL);
    const bool room = force == PQ2_VARIANT_PREFILL_WIDE ||
                      (force == PQ2_VARIANT_DEFAULT && m_tiles >= kWideMinMTiles &&
                       wide_tiles >= kWideMinTiles);
    l.npad = (N + kWTileN - 1) / kWTileN * kWTileN;
    size_t off = 0;
    l.ahi = off;
    off += align256(static_cast<size_t>(M) * K);
    l.alo = off;
    off += align256(static_cast<size_t>(M) * K);
    l.st = off;
    off += align256(static_cast<size_t>(M) * G * 8);
    if (room) {
        l.wexp = off;
        l.wexp_bytes = static_cast<size_t>(N) * K;
        off += align256(l.wexp_bytes);
        l.wst = off;
        off += align256(static_cast<size_t>(G) * l.npad * 4);
    }
    l.total = off;
    return l;
}

}  // namespace

namespace pq2h {

// Up to kTileMaxM tokens the token-tile kernel runs by default; the
// workspace covers it and the 128-row tile kernels (either may be forced).
size_t prefill_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    const WsLayout l = ws_layout(M, N, K);
    if (M > kTileMaxM) return l.total;
    size_t t = tile_workspace_bytes(M, N, K);
    const size_t u = wtile_workspace_bytes(M, N, K);
    if (u > t) t = u;
    return t > l.total ? t : l.total;
}

// The token-tile kernel pq2_gemm_prefill would run (the routing of
// launch_prefill below).
TokenTile prefill_token_tile_kernel(int64_t M, int64_t N, int64_t K, int num_sms) {
    if (M < 1 || M > kTileMaxM) return TokenTile::kNone;
    const int force = forced_variant(PQ2_OP_PREFILL);
    if (force == PQ2_VARIANT_PREFILL_WTILE ||
        (force == PQ2_VARIANT_DEFAULT && wtile_default(M, N, K, num_sms)))
        return TokenTile::kWide;
    if (force == PQ2_VARIANT_PREFILL_TILE ||
        (force == PQ2_VARIANT_DEFAULT && M <= kTileDefaultMaxM))
        return TokenTile::kTile;
    return TokenTile::kNone;
}

cudaError_t launch_prefill(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                           const __half* ws, float* y, int32_t* dots, int64_t M, int64_t N,
                           int64_t K, void* workspace, cudaStream_t st, const pq2::DevCtl& ctl,
                           const DeviceInfo& dev) {
    // Up to kTileDefaultMaxM tokens the token-tile kernel by default (measured
    // at 5120 -> 17408, us per call: 17 tokens 33.3 against 39.4 for the
    // 128 x 128 tile kernel, 32 tokens 34.2 against 34.4; at 64 tokens the
    // 128 x 128 tiles are ahead, 35.8 against 37.3).
    // From 33 to 64 tokens, where a CTA gets few items, the weights-wide
    // token-tile kernel (wtile_default).
    const int force = forced_variant(PQ2_OP_PREFILL);
    if (force == PQ2_VARIANT_PREFILL_WTILE ||
        (force == PQ2_VARIANT_DEFAULT && wtile_default(M, N, K, dev.num_sms))) {
        if (M > kTileMaxM) return kUnsupportedVariant;
        return launch_wtile(qp, S, T, codes, ws, y, dots, M, N, K, workspace, st, ctl, dev);
    }
    if (force == PQ2_VARIANT_PREFILL_TILE ||
        (force == PQ2_VARIANT_DEFAULT && M <= kTileDefaultMaxM)) {
        if (M > kTileMaxM) return kUnsupportedVariant;
        return launch_tile(qp, S, T, codes, ws, y, dots, M, N, K, workspace, st, ctl, dev);
    }
    const WsLayout l = ws_layout(M, N, K);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    uint8_t* ahi = w + l.ahi;
    uint8_t* alo = w + l.alo;
    float2* stv = reinterpret_cast<float2*>(w + l.st);
    const int G = static_cast<int>(K / 128);
    const int m_tiles = static_cast<int>((M + kTileM - 1) / kTileM);
    const int wide_tiles = m_tiles * static_cast<int>((N + kWTileN - 1) / kWTileN);
    // The wide tiles (128 x 256) where the workspace has room for the
    // expanded weights (ws_layout) and the tiles fill every SM at least once
    // (below one wave the wide tiles leave SMs idle).  The integer-dot debug
    // output takes the same kernel as y.
    const bool fits = dots ? wide_kernel_fits<true>() : wide_kernel_fits<false>();
    const bool wide = l.wexp_bytes > 0 && fits &&
                      (force == PQ2_VARIANT_PREFILL_WIDE ||
                       (force == PQ2_VARIANT_DEFAULT && wide_tiles >= dev.num_sms));
    if (force == PQ2_VARIANT_PREFILL_WIDE && !wide) return kUnsupportedVariant;
    uint8_t* wexp = wide ? w + l.wexp : nullptr;
    float* wst = wide ? reinterpret_cast<float*>(w + l.wst) : nullptr;
    {
        const int64_t words = M * K / 4 + (wide ? N * K / 64 : 0);
        const int64_t want = (words + 255) / 256;
        const int grid = static_cast<int>(want < dev.num_sms * 16 ? want : dev.num_sms * 16);
        cudaError_t e = launch(token_planes_kernel, dim3(grid), dim3(256), 0, st, true, qp, S, T,
                               reinterpret_cast<uint32_t*>(ahi), reinterpret_cast<uint32_t*>(alo),
                               stv, M, K, codes, ws, wexp, wst, N, l.npad);
        if (e != cudaSuccess) return e;
    }
    if (wide) {
        PrefillWideParams p = {};
        if (!encode_tmap_2d(&p.tm_ahi, CU_TENSOR_MAP_DATA_TYPE_UINT8, ahi, static_cast<uint64_t>(K),
                            static_cast<uint64_t>(M), static_cast<uint64_t>(K), 128u, kTileM, true) ||
            !encode_tmap_2d(&p.tm_alo, CU_TENSOR_MAP_DATA_TYPE_UINT8, alo, static_cast<uint64_t>(K),
                            static_cast<uint64_t>(M), static_cast<uint64_t>(K), 128u, kTileM, true) ||
            !encode_tmap_2d(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, wexp, static_cast<uint64_t>(K),
                            static_cast<uint64_t>(N), static_cast<uint64_t>(K), 128u, kWTileN, true))
            return cudaErrorInvalidValue;
        p.st = stv;
        p.wst = wst;
        p.y = y;
        p.dots = dots;
        p.M = static_cast<int>(M);
        p.N = static_cast<int>(N);
        p.K = static_cast<int>(K);
        p.G = G;
        p.Npad = static_cast<int>(l.npad);
        p.m_tiles = m_tiles;
        p.n_tiles = static_cast<int>((N + kWTileN - 1) / kWTileN);
        p.ctl = ctl;
        const int grid = wide_tiles < dev.num_sms ? wide_tiles : dev.num_sms;
        const size_t smem = 1024 + static_cast<size_t>(kWStages) * kWStageBytes;
        auto kern = dots ? prefill_wide_kernel<true> : prefill_wide_kernel<false>;
        static SmemLimit lim_wide[2];
        cudaError_t e = ensure_smem(lim_wide[dots ? 1 : 0], kern, smem);
        if (e != cudaSuccess) return e;
        return launch(kern, dim3(grid), dim3(kWThreads), smem, st, true, p);
    }
    PrefillParams p = {};
    if (!encode_tmap_2d(&p.tm_ahi, CU_TENSOR_MAP_DATA_TYPE_UINT8, ahi, static_cast<uint64_t>(K),
                        static_cast<uint64_t>(M), static_cast<uint64_t>(K), 128u, kTileM, true) ||
        !encode_tmap_2d(&p.tm_alo, CU_TENSOR_MAP_DATA_TYPE_UINT8, alo, static_cast<uint64_t>(K),
                        static_cast<uint64_t>(M), static_cast<uint64_t>(K), 128u, kTileM, true) ||
        !encode_tmap_2d(&p.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes,
                        static_cast<uint64_t>(K / 4), static_cast<uint64_t>(N),
                        static_cast<uint64_t>(K / 4), 32u, kTileN, false))
        return cudaErrorInvalidValue;
    p.st = stv;
    p.ws = ws;
    p.y = y;
    p.dots = dots;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.G = G;
    p.m_tiles = m_tiles;
    p.n_tiles = static_cast<int>((N + kTileN - 1) / kTileN);
    p.ctl = ctl;
    const int tiles = p.m_tiles * p.n_tiles;
    const int grid = tiles < dev.num_sms ? tiles : dev.num_sms;
    const size_t smem = 1024 + static_cast<size_t>(kStages) * kStageBytes;
    auto kern = dots ? prefill_kernel<true> : prefill_kernel<false>;
    static SmemLimit lim[2];
    cudaError_t e = ensure_smem(lim[dots ? 1 : 0], kern, smem);
    if (e != cudaSuccess) return e;
    return launch(kern, dim3(grid), dim3(kThreads), smem, st, true, p);
}

}  // namespace pq2h
