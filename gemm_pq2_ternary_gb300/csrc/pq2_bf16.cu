// Small unquantised bf16 projection, y[M, N] = bf16(x[M, K] . w[N, K]^T), as a
// split-K GEMM with a deterministic, fixed-order reduction ("Making a ternary
// reasoning model fast in vLLM", page "From CUDA to Triton and Gluon", section
// "Speed up a small unquantised projection": the 96 x 5120 in_proj_ba of a
// decode step, a few tokens at a time).
//
// The page's kernel writes one fp32 partial per K split to a buffer and sums
// the splits in order in a second pass.  Here the K splits of one output tile
// form a thread-block cluster of kSplits CTAs and the partials never leave
// the chip: each CTA reduces its lanes' partials inside each warp, sums its
// warps (in increasing K) through shared memory, and stores its partial of
// every output straight into the shared memory of the cluster rank that owns
// that output (distributed shared memory).  After one cluster barrier each
// rank sums the kSplits partials of its outputs in increasing-K order from
// its own shared memory and rounds each sum once to bf16.  One launch, no
// workspace, the same bits on every run.
//
// The work is bound by the bytes of w (983,040 for 96 x 5120) and by latency,
// not by arithmetic (16 x 96 x 5120 multiply-adds at most), so the products
// run as fp32 FMAs on the CUDA cores; every bf16 x bf16 product is exact in
// fp32.
#include <algorithm>

#include <cuda_bf16.h>

#include "pq2_common.cuh"
#include "pq2_internal.h"

namespace pq2 {
namespace {

constexpr int kSplits = 8;          // CTAs (K splits) per cluster
constexpr int kMaxThreads = 256;
constexpr int kMaxWarps = kMaxThreads / 32;
constexpr int kMaxOut = 64;         // outputs per tile, largest shape

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Cluster barrier, split: arrive (relaxed: orders nothing) and wait.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// Full cluster barrier whose arrive releases this thread's earlier stores
// (distributed shared memory included) and whose wait acquires everyone's.
__device__ __forceinline__ void cluster_sync_release_acquire() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// L2 prefetch of [src, src + bytes): both 16-byte multiples, bytes <= 64 KiB.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Round to nearest even, fp32 -> bf16 bits (the value is finite or a
// propagated inf/nan; nan keeps a quiet payload).
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    const __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<const uint16_t*>(&b);
}

struct Bf16Params {
    const uint16_t* x;   // [M, K] bf16, row-major
    const uint16_t* w;   // [N, K] bf16, row-major
    uint16_t* y;         // [M, N] bf16, row-major
    int M, N, K;
    int kv_per_split;    // column vectors (kVK values of K) per cluster rank
    int weights_static;  // w may be read before the preceding kernel ends
    DevCtl ctl;
};

// A column vector: kVK consecutive bf16 values of one row (kVK = 8: 16
// bytes; kVK = 4: 8 bytes), as 32-bit words of two values each.
template <int kVK>
struct ColVec {
    uint32_t w[kVK / 2];
};

template <int kVK>
__device__ __forceinline__ ColVec<kVK> load_vec(const uint16_t* base, size_t idx) {
    ColVec<kVK> v;
    if constexpr (kVK == 8) {
        const uint4 u = ld_nc_v4(reinterpret_cast<const uint4*>(base) + idx);
        v.w[0] = u.x, v.w[1] = u.y, v.w[2] = u.z, v.w[3] = u.w;
    } else {
        static_assert(kVK == 4, "column vectors of 4 or 8 values");
        uint2 u;
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                     : "=r"(u.x), "=r"(u.y)
                     : "l"(reinterpret_cast<const uint2*>(base) + idx));
        v.w[0] = u.x, v.w[1] = u.y;
    }
    return v;
}

template <int kVK>
__device__ __forceinline__ ColVec<kVK> zero_vec() {
    ColVec<kVK> v;
#pragma unroll
    for (int i = 0; i < kVK / 2; ++i) v.w[i] = 0;
    return v;
}

// Loads the kNT weight vectors of column vector kv (zeros past N).
template <int kNT, int kVK>
__device__ __forceinline__ void load_w(const Bf16Params& p, int n0, int kv,
                                       ColVec<kVK> (&wv)[kNT]) {
    const size_t row = static_cast<size_t>(p.K) / kVK;
#pragma unroll
    for (int n = 0; n < kNT; ++n)
        wv[n] = (n0 + n < p.N) ? load_vec<kVK>(p.w, static_cast<size_t>(n0 + n) * row + kv)
                               : zero_vec<kVK>();
}

// One CTA: a tile of kMT tokens x kNT output rows over one K split.  Each
// thread owns column vectors kv (kVK values of K each) and accumulates all
// kMT x kNT products of its vectors, k ascending.
template <int kMT, int kNT, int kVK>
__global__ void __launch_bounds__(kMaxThreads, 1) bf16_splitk_kernel(Bf16Params p) {
    constexpr int kOut = kMT * kNT;
    constexpr int kPerLane = kOut / 32;
    constexpr int kOutPerRank = kOut / kSplits;
    static_assert(kOut % 32 == 0 && kOut <= kMaxOut, "the warp reduce-scatter wants 32 | kOut");
    static_assert(kOut % kSplits == 0, "each cluster rank finishes an equal share");
    __shared__ __align__(16) float wsum[kMaxWarps][kOut];        // this CTA's warps
    __shared__ __align__(16) float red[kSplits][kOutPerRank];    // from every rank

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t rank = cluster_ctarank();
    const int n0 = blockIdx.x * kNT;
    const int m0 = blockIdx.z * kMT;
    const int kv_total = p.K / kVK;
    const int kv0 = static_cast<int>(rank) * p.kv_per_split;
    const int kv1 = min(kv0 + p.kv_per_split, kv_total);

    float acc[kOut];
#pragma unroll
    for (int i = 0; i < kOut; ++i) acc[i] = 0.0f;

    int kv = kv0 + tid;
    ColVec<kVK> wv[kNT];
    // x may still be in flight from the preceding kernel: an L2 prefetch is
    // only a hint (L2 is where that kernel's writes land), the loads come
    // after the wait.  Splits start and end on 16-byte boundaries.
    if (tid < kMT && m0 + tid < p.M && kv1 > kv0)
        prefetch_l2(p.x + static_cast<size_t>(m0 + tid) * p.K +
                             static_cast<size_t>(kv0) * kVK,
                         static_cast<uint32_t>(kv1 - kv0) * kVK * 2);
    if (!p.weights_static) pdl_wait();
    if (kv < kv1) load_w<kNT, kVK>(p, n0, kv, wv);
    if (p.weights_static) pdl_wait();
    pdl_launch_dependents();
    // first phase of the cluster barrier: this CTA has started (a rank may
    // store into another's shared memory only once that one runs)
    cluster_arrive_relaxed();

    const size_t xrow = static_cast<size_t>(p.K) / kVK;
    for (bool first = true; kv < kv1; kv += blockDim.x, first = false) {
        if (!first) load_w<kNT, kVK>(p, n0, kv, wv);
        ColVec<kVK> xv[kMT];
#pragma unroll
        for (int m = 0; m < kMT; ++m)
            xv[m] = (m0 + m < p.M) ? load_vec<kVK>(p.x, static_cast<size_t>(m0 + m) * xrow + kv)
                                   : zero_vec<kVK>();
        // k ascending inside the vector: kVK products per (m, n)
#pragma unroll
        for (int j = 0; j < kVK; ++j) {
            float wf[kNT];
#pragma unroll
            for (int n = 0; n < kNT; ++n) {
                const uint32_t word = wv[n].w[j >> 1];
                wf[n] = (j & 1) ? bf16_hi(word) : bf16_lo(word);
            }
#pragma unroll
            for (int m = 0; m < kMT; ++m) {
                const uint32_t word = xv[m].w[j >> 1];
                const float xf = (j & 1) ? bf16_hi(word) : bf16_lo(word);
#pragma unroll
                for (int n = 0; n < kNT; ++n) acc[m * kNT + n] = fmaf(xf, wf[n], acc[m * kNT + n]);
            }
        }
    }

    // Reduce-scatter across the warp: after the step of offset 16 >> s each
    // lane keeps (16 kPerLane >> s) sums; lane l ends with outputs
    // kPerLane l ... kPerLane l + kPerLane - 1.
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const int off = 16 >> s, half = (16 * kPerLane) >> s;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? acc[i] : acc[half + i];
            const float keep = upper ? acc[half + i] : acc[i];
            acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) wsum[warp][kPerLane * lane + j] = acc[j];
    __syncthreads();
    // one partial per output and CTA (its warps in increasing K), stored
    // into the owning rank's shared memory
    cluster_wait();  // every rank of the cluster has started
    if (tid < kOut) {
        float part = 0.0f;
        for (int w = 0; w < nwarps; ++w) part += wsum[w][tid];
        const uint32_t owner = static_cast<uint32_t>(tid / kOutPerRank);
        st_cluster_f32(map_to_rank(smem_u32(&red[rank][tid % kOutPerRank]), owner), part);
    }
    cluster_sync_release_acquire();  // all partials of this rank's outputs have landed

    if (tid < kOutPerRank) {
        // the sum in increasing K: source rank by source rank
        float sum = 0.0f;
#pragma unroll
        for (int r = 0; r < kSplits; ++r) sum += red[r][tid];
        const int o = static_cast<int>(rank) * kOutPerRank + tid;
        const int m = m0 + o / kNT, n = n0 + o % kNT;
        if (m < p.M && n < p.N &&
            store_ok(p.ctl, static_cast<long long>(m) * p.N + n, 1, static_cast<long long>(p.M) * p.N))
            p.y[static_cast<size_t>(m) * p.N + n] = f32_to_bf16_rn(sum);
    }
}

}  // namespace
}  // namespace pq2

namespace pq2h {

cudaError_t launch_bf16_splitk(const uint16_t* x, const uint16_t* w, uint16_t* y, int64_t M,
                               int64_t N, int64_t K, bool weights_static, cudaStream_t stream,
                               const pq2::DevCtl& ctl) {
    using namespace pq2;
    Bf16Params p = {};
    p.ctl = ctl;
    p.x = x;
    p.w = w;
    p.y = y;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    // tile shape by token count (as few padded tokens as the reduce-scatter
    // allows); column vectors of 4 values while a split's vectors fit the
    // block, of 8 beyond
    const bool narrow = (K / 4 + kSplits - 1) / kSplits <= kMaxThreads;
    const int vk = narrow ? 4 : 8;
    void (*kern)(Bf16Params);
    int mt, nt;
    if (M <= 8) {
        kern = narrow ? bf16_splitk_kernel<4, 8, 4> : bf16_splitk_kernel<4, 8, 8>;
        mt = 4, nt = 8;
    } else {
        kern = narrow ? bf16_splitk_kernel<8, 4, 4> : bf16_splitk_kernel<8, 4, 8>;
        mt = 8, nt = 4;
    }
    const int kv_total = static_cast<int>(K / vk);
    // splits of whole 16-byte pieces (K % 8 == 0, so kv_total is even for vk = 4)
    p.kv_per_split = (kv_total + kSplits - 1) / kSplits;
    if (vk == 4) p.kv_per_split = (p.kv_per_split + 1) & ~1;
    p.weights_static = weights_static ? 1 : 0;
    const int threads = std::min(kMaxThreads, std::max(32, (p.kv_per_split + 31) / 32 * 32));

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((N + nt - 1) / nt), kSplits,
                       static_cast<unsigned>((M + mt - 1) / mt));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = kSplits;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace pq2h
