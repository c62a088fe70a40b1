// Small-batch matmul for a few tokens (pq2_gemm_small with 2 <= M <= 4 by
// default, where the shape allows): the M = 1 DP4A algorithm with each code word reused by
// every token row ("Making a ternary reasoning model fast in vLLM", page
// "From CUDA to Triton and Gluon", sections "One token at a time: plain
// Triton is enough" for the per-group arithmetic and "Small batches: make the
// register layout explicit" for sharing one weight load among the token rows).
//
// Layout of the work.  One CTA per SM owns a contiguous range of output rows,
// as the direct M = 1 kernel does.  A thread is (row slot rp, group gi, token
// mt), with the MT tokens of a (row, group) on adjacent lanes: they issue the
// same 16-byte code loads, which a warp serves as one broadcast request, and
// each keeps its own token's 128 activation bytes, s and t in registers for
// the whole kernel.  Code words of the next four rows are requested ahead of
// their dots into fixed register slots.  Per group: two 16-byte loads, the
// plane masks and 32 DP4A against the token's activations, the exact
// 64 * (dot - sum(q)), then dot * s * ws in fp32; the terms of a (row, token)
// are summed in the fixed order of the M = 1 kernels (8 lanes over a stride,
// then a 3-step butterfly), so each token's y equals pq2_gemv on that token
// bit for bit.
// Weights declared static (PQ2_WEIGHTS_STATIC) are requested before the
// dependency wait: the first look-ahead rows into registers and, for slices
// up to 64 KB, an L2 prefetch of the CTA's whole slice of code rows and
// weight scales.  The activations are still read only after the wait.

#include "pq2_internal.h"

namespace {

constexpr int kMultiConsumers = 480;     // consumer threads at most
constexpr int kMultiLookahead = 4;       // rows of code loads in flight per thread
constexpr size_t kMultiMaxSmem = 160 * 1024;
constexpr uint32_t kMultiPrefetchMax = 64 * 1024;  // bytes of a CTA's code slice

struct MultiParams {
    const int8_t* qp;       // [M][K] plane order
    const float* S;         // [M][G]
    const int32_t* T;       // [M][G]
    const uint8_t* codes;   // [N][K/4]
    const __half* ws;       // [N][G]
    float* y;               // [M][N]
    int32_t* dots;          // debug: [M][N][G] instead of y
    int M, N, K, G;
    int GT;                 // threads per (row, token): one group each
    int RP;                 // row slots side by side
    int TC;                 // consumer threads (multiple of 32)
    int rows_per_cta;
    uint32_t codes_row_bytes;
    pq2::DevCtl ctl;
};

template <int MT, bool DOTS, bool STATIC>
__global__ void __launch_bounds__(kMultiConsumers, 1) gemv_multi_kernel(const MultiParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    float* red = reinterpret_cast<float*>(smem);  // [rows][MT][GT] group terms

    const int n_begin = blockIdx.x * p.rows_per_cta;
    const int rows = min(p.N, n_begin + p.rows_per_cta) - n_begin;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = p.TC >> 5;
    // the slice's L2 prefetch only where it is small: a large one competes
    // with the preceding call's own weight stream (measured slower at
    // 5120 -> 17408, 148 KB per CTA; faster at 6144 -> 5120, 52 KB)
    if (STATIC && rows > 0 && tid == 0 &&
        static_cast<uint32_t>(rows) * p.codes_row_bytes <= kMultiPrefetchMax) {
        pq2::bulk_prefetch_l2(p.codes + static_cast<size_t>(n_begin) * p.codes_row_bytes,
                              static_cast<uint32_t>(rows) * p.codes_row_bytes);
        if ((p.G & 7) == 0)  // 16-byte aligned slices of the scales
            pq2::bulk_prefetch_l2(p.ws + static_cast<size_t>(n_begin) * p.G,
                                  static_cast<uint32_t>(rows) * p.G * 2u);
    }
    // codes and activations may come from the preceding kernel (the codes not
    // when declared static: their first rows are requested below, before the wait)
    if (!STATIC) {
        pq2::pdl_wait();
        pq2::pdl_launch_dependents();
        if (rows <= 0) return;
    }

    const int mt = tid % MT;
    const int u = tid / MT;
    const int rp = u / p.GT;
    const int gi = u - rp * p.GT;
    const bool active = rp < p.RP;
    // which 16-byte half of the group's codes a thread reads first; shared by
    // the MT lanes of a (row, group), so their loads are identical
    const int hswap = (u >> 2) & 1;
    const int nk = active && rp < rows ? (rows - rp + p.RP - 1) / p.RP : 0;  // my rows
    const uint8_t* cbase =
        p.codes + static_cast<size_t>(n_begin + rp) * p.codes_row_bytes + gi * 32;
    const size_t cstep = static_cast<size_t>(p.RP) * p.codes_row_bytes;
    const unsigned short* wbase =
        reinterpret_cast<const unsigned short*>(p.ws) + static_cast<size_t>(n_begin + rp) * p.G + gi;
    const size_t wstep = static_cast<size_t>(p.RP) * p.G;
    // fixed register slots (loops unrolled by the look-ahead: a register
    // whose load is in flight is never moved)
    uint4 c0[kMultiLookahead], c1[kMultiLookahead];
    unsigned short wr[kMultiLookahead];
#pragma unroll
    for (int j = 0; j < kMultiLookahead; ++j) {
        c0[j] = make_uint4(0u, 0u, 0u, 0u);
        c1[j] = c0[j];
        wr[j] = 0;
        if (j < nk) {
            const uint8_t* cw = cbase + j * cstep;
            c0[j] = pq2::ld_nc_v4(cw + 16 * hswap);
            c1[j] = pq2::ld_nc_v4(cw + 16 * (hswap ^ 1));
            if (!DOTS) wr[j] = wbase[j * wstep];
        }
    }
    if (STATIC) {
        pq2::pdl_wait();
        pq2::pdl_launch_dependents();
        if (rows <= 0) return;
    }

    // this thread's token: its group's activations (zero past M)
    const bool mvalid = active && mt < p.M;
    const int gl = active ? gi : 0;
    uint32_t q[32];
    {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.qp + (static_cast<size_t>(mvalid ? mt : 0) * p.K + static_cast<size_t>(gl) * 128));
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            // plane v/2, words 4*(v&1)..+3; stored at the half this thread reads first
            const uint4 w = mvalid ? src[v ^ hswap] : make_uint4(0u, 0u, 0u, 0u);
            q[4 * v + 0] = w.x;
            q[4 * v + 1] = w.y;
            q[4 * v + 2] = w.z;
            q[4 * v + 3] = w.w;
        }
    }
    const size_t sg = static_cast<size_t>(mvalid ? mt : 0) * p.G + gl;
    const float s64 = (DOTS || !mvalid) ? 0.0f : p.S[sg] * 0.015625f;  // exact scaling by 2^-6
    const int t64 = mvalid ? -64 * p.T[sg] : 0;

    // rows rp, rp + RP, ...: the dot of row k, then the loads of row k + look-ahead
    const uint32_t red_s = pq2::smem_u32(red);
    for (int k0 = 0; k0 < nk; k0 += kMultiLookahead) {
#pragma unroll
        for (int j = 0; j < kMultiLookahead; ++j) {
            const int k = k0 + j;
            if (k >= nk) break;
            const uint32_t w[8] = {c0[j].x, c0[j].y, c0[j].z, c0[j].w,
                                   c1[j].x, c1[j].y, c1[j].z, c1[j].w};
            const int dot64 = pq2::group_codes_dot64(w, q, t64);
            const int r = rp + k * p.RP;
            if (DOTS) {
                if (mvalid &&
                    pq2::store_ok(p.ctl, (static_cast<long long>(mt) * p.N + n_begin + r) * p.G + gi,
                                  1, static_cast<long long>(p.M) * p.N * p.G))
                    p.dots[(static_cast<size_t>(mt) * p.N + n_begin + r) * p.G + gi] =
                        dot64 >> 6;  // exact
            } else {
                // float(dot64) exactly (|dot64| < 2^22) by the 1.5 * 2^23 bit trick
                const float dotf = __fsub_rn(__int_as_float(0x4B400000 + dot64), 12582912.0f);
                pq2::sts_f32(red_s + 4u * ((r * MT + mt) * p.GT + gi),
                             dotf * s64 * __half2float(__ushort_as_half(wr[j])));
            }
            if (k + kMultiLookahead < nk) {
                const uint8_t* cw = cbase + (k + kMultiLookahead) * cstep;
                c0[j] = pq2::ld_nc_v4(cw + 16 * hswap);
                c1[j] = pq2::ld_nc_v4(cw + 16 * (hswap ^ 1));
                if (!DOTS) wr[j] = wbase[(k + kMultiLookahead) * wstep];
            }
        }
    }
    if (DOTS) return;
    pq2::named_bar_sync(1, p.TC);
    // sums per (row, token): 8 lanes each over a fixed stride of the terms,
    // then a fixed 3-step butterfly (the order of the M = 1 kernels)
    const int sub = lane & 7;
    const int pairs = rows * MT;
    for (int pb = warp * 4; pb < pairs; pb += nwarps * 4) {
        const int pr = pb + (lane >> 3);
        float sum = 0.0f;
        if (pr < pairs)
            for (int c = sub; c < p.GT; c += 8) sum += pq2::lds_f32(red_s + 4u * (pr * p.GT + c));
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        const int r = pr / MT, m = pr - r * MT;
        if (sub == 0 && pr < pairs && m < p.M &&
            pq2::store_ok(p.ctl, static_cast<long long>(m) * p.N + n_begin + r, 1, static_cast<long long>(p.M) * p.N))
            p.y[static_cast<size_t>(m) * p.N + n_begin + r] = sum;
    }
}

template <int MT, bool DOTS, bool STATIC = false>
cudaError_t launch_mt(const MultiParams& p, int grid, size_t smem, cudaStream_t st) {
    auto kern = gemv_multi_kernel<MT, DOTS, STATIC>;
    static pq2h::SmemLimit lim;
    cudaError_t e = pq2h::ensure_smem(lim, kern, smem);
    if (e != cudaSuccess) return e;
    return pq2h::launch(kern, dim3(grid), dim3(p.TC), smem, st, true, p);
}

int tokens_per_pass(int64_t M) { return M <= 2 ? 2 : (M <= 4 ? 4 : 8); }

}  // namespace

namespace pq2h {

// The most tokens this kernel takes by default: 4.  Measured on GB300
// against the tensor-core small-batch kernel, GB/s, 6144 -> 5120 and
// 5120 -> 17408: M = 2 1056 / 1900 against 537 / 1049; M = 4 774 / 1256
// against 519 / 1028; M = 8 523 / 624 against 501 / 1003 (at 8 tokens the
// DP4A work per code word outweighs the shared loads).  Forcing the variant
// (pq2_debug_force_kernel) extends the range to 8 tokens.
constexpr int kMultiDefaultMaxM = 4;
constexpr int kMultiMaxM = 8;

bool gemv_multi_supported(int64_t M, int64_t N, int64_t K, int num_sms) {
    const int force = forced_variant(PQ2_OP_SMALL);
    if (force != PQ2_VARIANT_DEFAULT && force != PQ2_VARIANT_SMALL_DP4A) return false;
    const int max_m = force == PQ2_VARIANT_SMALL_DP4A ? kMultiMaxM : kMultiDefaultMaxM;
    if (M < 2 || M > max_m) return false;
    const int mt = tokens_per_pass(M);
    const int64_t G = K / 128;
    if (G * mt > kMultiConsumers) return false;
    const int64_t rows_per_cta = (N + num_sms - 1) / num_sms;
    return static_cast<size_t>(rows_per_cta) * mt * G * 4 <= kMultiMaxSmem;
}

cudaError_t launch_gemv_multi(const int8_t* qp, const float* S, const int32_t* T,
                              const uint8_t* codes, const __half* ws, float* y, int32_t* dots,
                              int64_t M, int64_t N, int64_t K, cudaStream_t st,
                              const DeviceInfo& dev, bool weights_static, const pq2::DevCtl& ctl) {
    if (!gemv_multi_supported(M, N, K, dev.num_sms)) return cudaErrorInvalidValue;
    const int mt = tokens_per_pass(M);
    MultiParams p = {};
    p.ctl = ctl;
    p.qp = qp;
    p.S = S;
    p.T = T;
    p.codes = codes;
    p.ws = ws;
    p.y = y;
    p.dots = dots;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.G = static_cast<int>(K / 128);
    p.GT = p.G;
    p.RP = kMultiConsumers / (p.GT * mt);
    p.TC = ((p.RP * p.GT * mt + 31) / 32) * 32;
    p.codes_row_bytes = static_cast<uint32_t>(K / 4);
    p.rows_per_cta = static_cast<int>((N + dev.num_sms - 1) / dev.num_sms);
    const int grid = static_cast<int>((N + p.rows_per_cta - 1) / p.rows_per_cta);
    const size_t smem = static_cast<size_t>(p.rows_per_cta) * mt * p.GT * 4;
    if (dots) {
        if (mt == 2) return launch_mt<2, true>(p, grid, smem, st);
        if (mt == 4) return launch_mt<4, true>(p, grid, smem, st);
        return launch_mt<8, true>(p, grid, smem, st);
    }
    if (weights_static) {
        if (mt == 2) return launch_mt<2, false, true>(p, grid, smem, st);
        if (mt == 4) return launch_mt<4, false, true>(p, grid, smem, st);
        return launch_mt<8, false, true>(p, grid, smem, st);
    }
    if (mt == 2) return launch_mt<2, false>(p, grid, smem, st);
    if (mt == 4) return launch_mt<4, false>(p, grid, smem, st);
    return launch_mt<8, false>(p, grid, smem, st);
}

}  // namespace pq2h
