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
//  * One persistent CTA per SM owns a contiguous range of output rows.  Rows
//    are contiguous in memory (codes [N, K/4] row-major), so a stage of R
//    rows is ONE contiguous chunk: a single 1-D bulk copy (TMA engine) per
//    stage streams it into a shared-memory ring, completion tracked by an
//    mbarrier.  One elected producer thread keeps `stages` copies in flight,
//    enough bytes to cover HBM latency with no register cost.
//  * Consumer thread (rp, gi) always works on the same 128-weight groups
//    gi, gi+GT, ... of every row it handles, so its 128 activation bytes per
//    group, s and t live in registers for the whole kernel: activations cost
//    no shared-memory traffic.  RP rows are processed side by side.
//  * Per group: two 16-byte shared loads of codes, 32 mask + 32 DP4A (plane
//    s masked in place as 4^s * code, rescaled exactly by shifts), the
//    -sum(q) correction, one fp32 multiply and one FMA.
//  * Row sums: per-thread partials go to a double-buffered shared array and
//    a warp sums each row in a fixed order (deterministic), one named
//    barrier per stage (which also ORs the consumers' wait failures, so all
//    of them stop at the same stage).
//  * Every mbarrier wait is bounded; on expiry the block sets the device
//    error word, stops, and the producer waits for its copies in flight.
#include "pq2_internal.h"

namespace {

struct GemvParams {
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
    int R;             // rows per stage (multiple of RP)
    int stages;
    int rows_per_cta;
    uint32_t stage_bytes;      // ring slot size (codes + ws, 16-aligned)
    uint32_t codes_row_bytes;  // K / 4
    pq2::DevCtl ctl;
};

constexpr int kRingBudget = 160 * 1024;
constexpr int kTargetConsumers = 256;
constexpr int kMaxThreads = 512 + 32;  // consumers (<= 512) + producer warp

template <int GPT, bool WS_SMEM, bool DOTS>
__global__ void __launch_bounds__(kMaxThreads, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + p.stages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + p.stages);
    float* red = reinterpret_cast<float*>(smem + 16 * p.stages + 16);
    const int red_stride = p.R * p.GT;  // floats per buffer
    uint8_t* ring = smem + ((16 * p.stages + 16 + 8 * red_stride + 127) & ~127);

    const int n_begin = blockIdx.x * p.rows_per_cta;
    const int n_end = min(p.N, n_begin + p.rows_per_cta);
    if (n_begin >= n_end) return;
    const int nst = (n_end - n_begin + p.R - 1) / p.R;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            pq2::mbar_init(&full[i], 1);
            pq2::mbar_init(&empty[i], 1);
        }
        *abort_flag = 0;
        pq2::fence_mbar_init();
    }
    __syncthreads();
    // Every input may have been written by the preceding kernel.
    pq2::pdl_wait();
    pq2::pdl_launch_dependents();

    const int tid = threadIdx.x;
    if (tid >= p.TC) {
        // ------------------------------ producer ------------------------------
        if (tid != p.TC) return;
        const uint64_t policy = pq2::policy_evict_first();
        int issued_end = 0;  // stages [0, issued_end) were armed, except the withheld one
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
    const int RI = p.R / p.RP;

    uint32_t qreg[GPT][32];
    float sg[GPT];
    int tg[GPT];
    bool gval[GPT];
#pragma unroll
    for (int j = 0; j < GPT; ++j) {
        const int g = gi + j * p.GT;
        gval[j] = active && g < p.G;
        const int gl = gval[j] ? g : 0;
        const uint4* src = reinterpret_cast<const uint4*>(p.qp + static_cast<size_t>(gl) * 128);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const uint4 w = src[v];
            qreg[j][4 * v + 0] = w.x;
            qreg[j][4 * v + 1] = w.y;
            qreg[j][4 * v + 2] = w.z;
            qreg[j][4 * v + 3] = w.w;
        }
        sg[j] = DOTS ? 0.0f : p.S[gl];
        tg[j] = p.T[gl];
    }

    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = p.TC >> 5;

    for (int i = 0; i < nst; ++i) {
        const int slot = i % p.stages;
        const bool ok = pq2::mbar_wait_bounded(&full[slot], (i / p.stages) & 1, p.ctl, abort_flag);
        if (!ok) *abort_flag = 1;
        const int row0 = n_begin + i * p.R;
        const int rows = min(p.R, n_end - row0);
        const uint8_t* stage = ring + static_cast<size_t>(slot) * p.stage_bytes;
        float* redb = red + (i & 1) * red_stride;
        if (ok && active) {
            for (int t = 0; t < RI; ++t) {
                const int r = rp + t * p.RP;
                if (r >= rows) break;
                const uint8_t* crow = stage + static_cast<size_t>(r) * p.codes_row_bytes;
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < GPT; ++j) {
                    if (!gval[j]) continue;
                    const int g = gi + j * p.GT;
                    const uint4* cw = reinterpret_cast<const uint4*>(crow + g * 32);
                    const uint4 c0 = cw[0], c1 = cw[1];
                    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    const int dot = pq2::group_codes_dot(w, qreg[j]) - tg[j];
                    if (DOTS) {
                        p.dots[static_cast<size_t>(row0 + r) * p.G + g] = dot;
                    } else {
                        __half wsh;
                        if (WS_SMEM)
                            wsh = reinterpret_cast<const __half*>(
                                stage + static_cast<size_t>(p.R) * p.codes_row_bytes)[r * p.G + g];
                        else
                            wsh = p.ws[static_cast<size_t>(row0 + r) * p.G + g];
                        acc = fmaf(static_cast<float>(dot) * sg[j], __half2float(wsh), acc);
                    }
                }
                if (!DOTS) redb[r * p.GT + gi] = acc;
            }
        }
        // all consumers are done with this slot; agree on whether to stop
        const bool any_fail = pq2::named_bar_any(1, p.TC, !ok);
        if (tid == 0) {
            pq2::mbar_arrive(&empty[slot]);
            if (any_fail) *abort_flag = 1;
        }
        if (any_fail) break;
        if (!DOTS) {
            for (int r = warp; r < rows; r += nwarps) {
                float s = 0.0f;
                for (int c = lane; c < p.GT; c += 32) s += redb[r * p.GT + c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == 0) p.y[row0 + r] = s;
            }
        }
    }
}

template <int GPT, bool WS_SMEM, bool DOTS>
cudaError_t launch_variant(const GemvParams& p, int grid, size_t smem, cudaStream_t st,
                           const pq2h::DeviceInfo& dev) {
    auto kern = gemv_kernel<GPT, WS_SMEM, DOTS>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return pq2h::launch(kern, dim3(grid), dim3(p.TC + 32), smem, st, true, p);
}

template <int GPT>
cudaError_t launch_gpt(const GemvParams& p, int grid, size_t smem, bool ws_smem, bool dots,
                       cudaStream_t st, const pq2h::DeviceInfo& dev) {
    if (dots) return launch_variant<GPT, false, true>(p, grid, smem, st, dev);
    if (ws_smem) return launch_variant<GPT, true, false>(p, grid, smem, st, dev);
    return launch_variant<GPT, false, false>(p, grid, smem, st, dev);
}

}  // namespace

namespace pq2h {

cudaError_t launch_gemv(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                        const __half* ws, float* y, int32_t* dots, int64_t N, int64_t K,
                        cudaStream_t st, const pq2::DevCtl& ctl, const DeviceInfo& dev) {
    GemvParams p = {};
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
    p.RP = kTargetConsumers / p.GT > 0 ? kTargetConsumers / p.GT : 1;
    p.TC = ((p.RP * p.GT + 31) / 32) * 32;
    p.codes_row_bytes = static_cast<uint32_t>(K / 4);
    const bool ws_smem = (dots == nullptr) && (p.G % 8 == 0);
    const int row_bytes = static_cast<int>(p.codes_row_bytes) + (ws_smem ? 2 * p.G : 0);
    const int per_rp = p.RP * row_bytes;
    int ri = (12 * 1024 + per_rp / 2) / per_rp;
    if (ri < 1) ri = 1;
    p.R = p.RP * ri;
    p.stage_bytes = static_cast<uint32_t>(((p.R * row_bytes) + 15) & ~15);
    int stages = kRingBudget / static_cast<int>(p.stage_bytes);
    if (stages > 16) stages = 16;
    if (stages < 2) stages = 2;
    p.stages = stages;
    const int rows_per_cta = static_cast<int>((N + dev.num_sms - 1) / dev.num_sms);
    p.rows_per_cta = rows_per_cta;
    const int grid = static_cast<int>((N + rows_per_cta - 1) / rows_per_cta);
    p.ctl = ctl;
    const size_t head = ((16 * p.stages + 16 + 8 * p.R * p.GT + 127) & ~127);
    const size_t smem = head + static_cast<size_t>(p.stages) * p.stage_bytes;
    if (smem > static_cast<size_t>(dev.max_smem_optin)) return cudaErrorInvalidConfiguration;
    if (gpt == 1) return launch_gpt<1>(p, grid, smem, ws_smem, dots != nullptr, st, dev);
    if (gpt == 2) return launch_gpt<2>(p, grid, smem, ws_smem, dots != nullptr, st, dev);
    return launch_gpt<4>(p, grid, smem, ws_smem, dots != nullptr, st, dev);
}

}  // namespace pq2h
