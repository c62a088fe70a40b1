// M = 1 decode matmul (pq2_gemv).
//
// The arithmetic is the pages' single-token algorithm ("Making a ternary
// reasoning model fast in vLLM", page "From CUDA to Triton and Gluon",
// section "One token at a time: plain Triton is enough"): activations in
// plane order, plane s of a code word lined up with four activation bytes and
// fed to DP4A, sum(q) subtracted once per 128-weight group, fp32 accumulation
// of dot * s * ws; and, from page "Chasing llama.cpp at batch one", section
// "The win: a program just for one token": no token dimension at all.
//
// GB300 layout of the work (not the pages' tiling):
//  * Persistent CTAs (up to two per SM) each own a contiguous range of output
//    rows.  Rows are contiguous in memory (codes [N, K/4] row-major), so a
//    stage of R rows is ONE contiguous chunk: a single 1-D bulk copy (TMA
//    engine) per stage streams it into a shared-memory ring, completion
//    tracked by an mbarrier.  One elected producer thread keeps the ring full.
//  * Consumer thread (rp, gi) always works on the same 128-weight group gi of
//    the rows it handles, so the group's 128 activation bytes, s and t live
//    in registers for the whole kernel.  Two rows are processed at once for
//    instruction-level parallelism.
//  * Per group: two 16-byte shared loads of codes, 32 mask + 32 DP4A (plane
//    s masked in place is 4^s times the codes; the four plane sums are
//    rescaled exactly by shifts), the -sum(q) correction, one fp32 multiply
//    and one FMA.
//  * Each consumer warp releases a ring slot on its own (mbarrier arrive);
//    per-thread group terms go to a shared array and are summed per row, in
//    a fixed order, once per chunk of rows (one named barrier per chunk).
//  * Every mbarrier wait is bounded; on expiry the block sets the device
//    error word, stops, and the producer waits for its copies in flight.
#include <cstdlib>

#include "pq2_internal.h"

namespace {

struct GemvParams {
    const __half* x;   // fused path: fp16 activations [K] (qp, S, T unused)
    const int8_t* qp;
    const float* S;
    const int32_t* T;
    const uint8_t* codes;
    const __half* ws;
    float* y;
    int32_t* dots;     // debug: per-group integer dots [N, G] instead of y
    int N, K, G;
    int GT;            // threads per row (each owns GPT groups)
    int RP;            // rows handled side by side
    int TC;            // consumer threads (multiple of 32)
    int R;             // rows per stage (multiple of 2*RP)
    int stages;
    int chunk_stages;  // stages per row-sum chunk
    int rows_per_cta;
    uint32_t stage_bytes;      // ring slot size (codes + ws, 16-aligned)
    uint32_t codes_row_bytes;  // K / 4
    int prefetch;              // issue an L2 prefetch of the CTA's weights first
    pq2::DevCtl ctl;
};

__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

constexpr int kMaxThreads = 512 + 32;  // consumers (<= 512) + producer warp

// The group's 32 code bytes are read as two 16-byte halves, half `h` first
// (h alternates every 4 lanes, which makes each 8-lane phase of the shared
// loads hit 8 distinct bank groups).  The thread's activation words were
// permuted the same way when they were loaded, so word i of `w` still meets
// its own activation word.
template <bool WS_SMEM, bool DOTS>
__device__ __forceinline__ float group_term(const uint8_t* crow, const uint8_t* wsrow_smem,
                                            const __half* wsrow_gmem, int32_t* dotrow, int g,
                                            const uint32_t* q, int t, float s, int h) {
    const uint4* cw = reinterpret_cast<const uint4*>(crow + g * 32);
    const uint4 c0 = cw[h], c1 = cw[h ^ 1];
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const int dot = pq2::group_codes_dot(w, q) - t;
    if (DOTS) {
        dotrow[g] = dot;
        return 0.0f;
    }
    const __half wsh = WS_SMEM ? reinterpret_cast<const __half*>(wsrow_smem)[g] : wsrow_gmem[g];
    return static_cast<float>(dot) * s * __half2float(wsh);
}

template <int GPT, bool WS_SMEM, bool DOTS, bool FUSED>
__global__ void __launch_bounds__(kMaxThreads, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + p.stages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + p.stages);
    float* red = reinterpret_cast<float*>(smem + 16 * p.stages + 16);
    const int chunk_rows = p.chunk_stages * p.R;
    const int red_stride = chunk_rows * p.GT;  // floats per buffer
    // fused path: the quantised activations live in shared memory
    const int act_off = (16 * p.stages + 16 + 8 * red_stride + 127) & ~127;
    int8_t* qsm = reinterpret_cast<int8_t*>(smem + act_off);
    float* ssm = reinterpret_cast<float*>(smem + act_off + p.K);
    int32_t* tsm = reinterpret_cast<int32_t*>(smem + act_off + p.K + 4 * p.G);
    const int ring_off = FUSED ? ((act_off + p.K + 8 * p.G + 127) & ~127) : act_off;
    uint8_t* ring = smem + ring_off;

    const int n_begin = blockIdx.x * p.rows_per_cta;
    const int n_end = min(p.N, n_begin + p.rows_per_cta);
    if (n_begin >= n_end) return;
    const int nst = (n_end - n_begin + p.R - 1) / p.R;
    const int tid = threadIdx.x;
    const int nwarps = p.TC >> 5;

    if (tid == 0) {
        for (int i = 0; i < p.stages; ++i) {
            pq2::mbar_init(&full[i], 1);
            pq2::mbar_init(&empty[i], nwarps);
        }
        *abort_flag = 0;
        pq2::fence_mbar_init();
    }
    if (tid == p.TC && p.prefetch) {
        // Start the weight stream before waiting for the preceding kernel.
        // The weights are not its output in normal use, and even if they
        // were, a prefetch into L2 (the coherence point) cannot return stale
        // data to the copies issued after the wait.
        const uint8_t* src = p.codes + static_cast<size_t>(n_begin) * p.codes_row_bytes;
        uint32_t left = static_cast<uint32_t>(n_end - n_begin) * p.codes_row_bytes;
        while (left > 0) {
            const uint32_t b = left < 65536u ? left : 65536u;
            bulk_prefetch_l2(src, b);
            src += b;
            left -= b;
        }
    }
    __syncthreads();
    // Activations, scales and (possibly) weights may come from the preceding
    // kernel: wait for it before reading any of them.
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();

    if (tid >= p.TC) {
        // ------------------------------ producer ------------------------------
        if (tid != p.TC) return;
        const uint64_t policy = pq2::policy_evict_first();
        int issued_end = 0;  // stages [0, issued_end) were armed, except a withheld one
        for (int i = 0; i < nst; ++i) {
            const int slot = i % p.stages;
            if (i >= p.stages) {
                if (!pq2::mbar_wait_bounded(&empty[slot], ((i / p.stages) - 1) & 1, p.ctl,
                                            abort_flag))
                    break;
            }
            issued_end = i + 1;
            if (i == p.ctl.debug_skip_stage) continue;  // withheld (timeout test)
            const int row0 = n_begin + i * p.R;
            const int rows = min(p.R, n_end - row0);
            const uint32_t cbytes = static_cast<uint32_t>(rows) * p.codes_row_bytes;
            const uint32_t wbytes = WS_SMEM ? static_cast<uint32_t>(rows * p.G * 2) : 0u;
            uint8_t* dst = ring + static_cast<size_t>(slot) * p.stage_bytes;
            pq2::mbar_arrive_expect_tx(&full[slot], cbytes + wbytes);
            pq2::bulk_g2s_hint(dst, p.codes + static_cast<size_t>(row0) * p.codes_row_bytes,
                               cbytes, &full[slot], policy);
            if (WS_SMEM)
                pq2::bulk_g2s(dst + static_cast<size_t>(p.R) * p.codes_row_bytes,
                              p.ws + static_cast<size_t>(row0) * p.G, wbytes, &full[slot]);
        }
        // Drain: no copy may still be landing when the block exits.  The last
        // armed stage of each slot is the latest i < issued_end on that slot
        // (skipping a withheld stage).
        for (int s = 0; s < p.stages; ++s) {
            if (issued_end <= s) continue;
            int last = s + ((issued_end - 1 - s) / p.stages) * p.stages;
            if (last == p.ctl.debug_skip_stage) last -= p.stages;
            if (last >= 0) pq2::mbar_wait_bounded(&full[s], (last / p.stages) & 1, p.ctl);
        }
        return;
    }

    // -------------------------------- consumers -------------------------------
    const int rp = tid / p.GT;
    const int gi = tid - rp * p.GT;
    const bool active = rp < p.RP;
    const int RI = p.R / p.RP;  // even
    const int hswap = (tid >> 2) & 1;  // which 16-byte half of a group to read first

    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int8_t* qsrc = p.qp;
    const float* ssrc = p.S;
    const int32_t* tsrc = p.T;
    if (FUSED) {
        // quantise the fp16 activations once per CTA (while the producer's
        // first weight copies are in flight)
        pq2::quantize_row_warps(p.x, p.G, warp, nwarps, lane, qsm, ssm, tsm);
        pq2::named_bar_sync(2, p.TC);
        qsrc = qsm;
        ssrc = ssm;
        tsrc = tsm;
    }

    uint32_t qreg[GPT][32];
    float sg[GPT];
    int tg[GPT];
    bool gval[GPT];
#pragma unroll
    for (int j = 0; j < GPT; ++j) {
        const int g = gi + j * p.GT;
        gval[j] = active && g < p.G;
        const int gl = gval[j] ? g : 0;
        const uint4* src = reinterpret_cast<const uint4*>(qsrc + static_cast<size_t>(gl) * 128);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            // plane v/2, words 4*(v&1)..+3; stored at the half this thread reads first
            const uint4 w = src[v ^ hswap];
            qreg[j][4 * v + 0] = w.x;
            qreg[j][4 * v + 1] = w.y;
            qreg[j][4 * v + 2] = w.z;
            qreg[j][4 * v + 3] = w.w;
        }
        sg[j] = DOTS ? 0.0f : ssrc[gl];
        tg[j] = tsrc[gl];
    }

    bool failed = false;

    for (int c0 = 0; c0 < nst; c0 += p.chunk_stages) {
        const int c1 = min(nst, c0 + p.chunk_stages);
        float* redb = red + ((c0 / p.chunk_stages) & 1) * red_stride;
        for (int i = c0; i < c1; ++i) {
            const int slot = i % p.stages;
            if (!failed) {
                if (!pq2::mbar_wait_bounded(&full[slot], (i / p.stages) & 1, p.ctl, abort_flag)) {
                    failed = true;
                    *abort_flag = 1;
                }
            }
            if (!failed && active) {
                const int row0 = n_begin + i * p.R;
                const int rows = min(p.R, n_end - row0);
                const uint8_t* stage = ring + static_cast<size_t>(slot) * p.stage_bytes;
                const uint8_t* wsm = stage + static_cast<size_t>(p.R) * p.codes_row_bytes;
                for (int t = 0; t < RI; t += 2) {
                    const int ra = rp + t * p.RP;
                    const int rb = ra + p.RP;
                    if (ra >= rows) break;
                    const bool hb = rb < rows;
                    const int rbs = hb ? rb : ra;  // recompute row a when b is past the end
                    const uint8_t* ca = stage + static_cast<size_t>(ra) * p.codes_row_bytes;
                    const uint8_t* cb = stage + static_cast<size_t>(rbs) * p.codes_row_bytes;
                    float acc_a = 0.0f, acc_b = 0.0f;
#pragma unroll
                    for (int j = 0; j < GPT; ++j) {
                        if (!gval[j]) continue;
                        const int g = gi + j * p.GT;
                        acc_a += group_term<WS_SMEM, DOTS>(
                            ca, wsm + ra * p.G * 2, p.ws + static_cast<size_t>(row0 + ra) * p.G,
                            p.dots + static_cast<size_t>(row0 + ra) * p.G, g, qreg[j], tg[j],
                            sg[j], hswap);
                        acc_b += group_term<WS_SMEM, DOTS>(
                            cb, wsm + rbs * p.G * 2, p.ws + static_cast<size_t>(row0 + rbs) * p.G,
                            p.dots + static_cast<size_t>(row0 + rbs) * p.G, g, qreg[j], tg[j],
                            sg[j], hswap);
                    }
                    if (!DOTS) {
                        const int la = (i - c0) * p.R + ra;
                        redb[la * p.GT + gi] = acc_a;
                        if (hb) redb[(la + p.RP) * p.GT + gi] = acc_b;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) pq2::mbar_arrive(&empty[slot]);
        }
        // all consumers have written this chunk's terms; agree on stopping
        const bool any_fail = pq2::named_bar_any(1, p.TC, failed);
        if (any_fail) {
            if (tid == 0) *abort_flag = 1;
            break;
        }
        if (!DOTS) {
            const int crow0 = n_begin + c0 * p.R;
            const int crows = min(n_end, n_begin + c1 * p.R) - crow0;
            for (int r = warp; r < crows; r += nwarps) {
                float s = 0.0f;
                for (int c = lane; c < p.GT; c += 32) s += redb[r * p.GT + c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == 0) p.y[crow0 + r] = s;
            }
        }
    }
}

template <int GPT, bool WS_SMEM, bool DOTS, bool FUSED>
cudaError_t launch_variant(const GemvParams& p, int grid, size_t smem, cudaStream_t st) {
    auto kern = gemv_kernel<GPT, WS_SMEM, DOTS, FUSED>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return pq2h::launch(kern, dim3(grid), dim3(p.TC + 32), smem, st, true, p);
}

template <int GPT>
cudaError_t launch_gpt(const GemvParams& p, int grid, size_t smem, bool ws_smem, bool dots,
                       cudaStream_t st) {
    if (dots) return launch_variant<GPT, false, true, false>(p, grid, smem, st);
    if (p.x) {
        if (ws_smem) return launch_variant<GPT, true, false, true>(p, grid, smem, st);
        return launch_variant<GPT, false, false, true>(p, grid, smem, st);
    }
    if (ws_smem) return launch_variant<GPT, true, false, false>(p, grid, smem, st);
    return launch_variant<GPT, false, false, false>(p, grid, smem, st);
}

// Tuning knobs (environment, read once): PQ2_GEMV_CTAS_PER_SM (default 2),
// PQ2_GEMV_RING_KB (default 64), PQ2_GEMV_THREADS (target consumer threads,
// default 256), PQ2_GEMV_STAGE_KB (default 4), PQ2_GEMV_PREFETCH (1 = on,
// default 1; 2 = off).
int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    if (!v || !*v) return dflt;
    const int x = std::atoi(v);
    return x > 0 ? x : dflt;
}

struct Tuning {
    int ctas_per_sm, ring_kb, threads, stage_kb, prefetch;
};

const Tuning& tuning() {
    static const Tuning t = {env_int("PQ2_GEMV_CTAS_PER_SM", 2), env_int("PQ2_GEMV_RING_KB", 64),
                             env_int("PQ2_GEMV_THREADS", 256), env_int("PQ2_GEMV_STAGE_KB", 4),
                             env_int("PQ2_GEMV_PREFETCH", 1) == 1 ? 1 : 0};
    return t;
}

size_t smem_bytes(const GemvParams& p) {
    const int red_floats = 2 * p.chunk_stages * p.R * p.GT;
    size_t head = (16 * p.stages + 16 + 4 * red_floats + 127) & ~127;
    if (p.x) head = (head + p.K + 8 * p.G + 127) & ~static_cast<size_t>(127);
    return head + static_cast<size_t>(p.stages) * p.stage_bytes;
}

}  // namespace

namespace pq2h {

cudaError_t launch_gemv(const __half* x, const int8_t* qp, const float* S, const int32_t* T,
                        const uint8_t* codes, const __half* ws, float* y, int32_t* dots, int64_t N,
                        int64_t K, cudaStream_t st, const pq2::DevCtl& ctl, const DeviceInfo& dev) {
    const Tuning& tu = tuning();
    GemvParams p = {};
    p.x = dots ? nullptr : x;
    p.qp = qp;
    p.S = S;
    p.T = T;
    p.codes = codes;
    p.ws = ws;
    p.y = y;
    p.dots = dots;
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.G = static_cast<int>(K / 128);
    const int gpt = p.G <= 512 ? 1 : (p.G <= 1024 ? 2 : 4);
    p.GT = (p.G + gpt - 1) / gpt;
    const int target = tu.threads < 32 ? 32 : (tu.threads > 512 ? 512 : tu.threads);
    p.RP = target / p.GT > 0 ? target / p.GT : 1;
    p.TC = ((p.RP * p.GT + 31) / 32) * 32;
    p.codes_row_bytes = static_cast<uint32_t>(K / 4);
    const bool ws_smem = (dots == nullptr) && (p.G % 8 == 0);
    const int row_bytes = static_cast<int>(p.codes_row_bytes) + (ws_smem ? 2 * p.G : 0);
    const int per_pair = 2 * p.RP * row_bytes;  // rows come in pairs per thread
    int pairs = (tu.stage_kb * 1024 + per_pair / 2) / per_pair;
    if (pairs < 1) pairs = 1;
    p.R = 2 * p.RP * pairs;
    p.stage_bytes = static_cast<uint32_t>(((p.R * row_bytes) + 15) & ~15);
    int stages = tu.ring_kb * 1024 / static_cast<int>(p.stage_bytes);
    p.stages = stages > 16 ? 16 : (stages < 2 ? 2 : stages);
    const int64_t slots = static_cast<int64_t>(dev.num_sms) * tu.ctas_per_sm;
    const int rows_per_cta = static_cast<int>((N + slots - 1) / slots);
    p.rows_per_cta = rows_per_cta;
    // ~64 rows per row-sum chunk, never more than the CTA owns
    int cs = (64 + p.R - 1) / p.R;
    const int cta_stages = (rows_per_cta + p.R - 1) / p.R;
    if (cs > cta_stages) cs = cta_stages;
    p.chunk_stages = cs < 1 ? 1 : cs;
    const int grid = static_cast<int>((N + rows_per_cta - 1) / rows_per_cta);
    p.ctl = ctl;
    p.prefetch = tu.prefetch;
    size_t smem = smem_bytes(p);
    while (smem > static_cast<size_t>(dev.max_smem_optin) && p.stages > 2) {
        --p.stages;
        smem = smem_bytes(p);
    }
    if (smem > static_cast<size_t>(dev.max_smem_optin)) return cudaErrorInvalidConfiguration;
    if (gpt == 1) return launch_gpt<1>(p, grid, smem, ws_smem, dots != nullptr, st);
    if (gpt == 2) return launch_gpt<2>(p, grid, smem, ws_smem, dots != nullptr, st);
    return launch_gpt<4>(p, grid, smem, ws_smem, dots != nullptr, st);
}

}  // namespace pq2h
