// Shared device helpers of the PQ2 CUDA library (sm_103a only).
//
// Inline PTX wrappers for mbarriers, 1-D bulk async copies (TMA engine),
// programmatic dependent launch, a bounded barrier wait, and the launch
// parameters every kernel gets (device error word, wait limit).
#pragma once

#include <atomic>

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "this library is built for sm_103a only"
#endif

namespace pq2 {

// Bits of the device error word.
enum : unsigned {
    DEVERR_TIMEOUT = 1u,      // a bounded wait ran out
    DEVERR_BAD_TERNARY = 2u,  // pack met a value outside {-1,0,1}
    DEVERR_BOUNDS = 4u,       // bounds-checked build: a store outside its buffer (skipped)
};

// Passed by value to every kernel.
struct DevCtl {
    unsigned* err;          // device error word (never null)
    unsigned long long wait_limit_ns;
    int debug_skip_stage;   // >= 0: producer withholds that stage (timeout tests)
    int debug_bounds_shrink;  // bounds-checked build: the checks treat the last
                              // elements of every buffer as outside (test hook)
};

// Bounds-checked build (compiled with PQ2_DEBUG=1; a separate library): every
// store to an output or scratch buffer first asks store_ok whether its w
// elements i .. i + w - 1 lie inside the buffer's n elements (less
// ctl.debug_bounds_shrink).  If not, the error word gets DEVERR_BOUNDS and the
// store is skipped, so an indexing mistake is reported instead of corrupting
// memory.  In the normal build store_ok is the constant true.
#ifndef PQ2_DEBUG
#define PQ2_DEBUG 0
#endif
__device__ __forceinline__ bool store_ok(const DevCtl& ctl, long long i, int w, long long n) {
#if PQ2_DEBUG
    if (i >= 0 && i + w <= n - ctl.debug_bounds_shrink) return true;
    atomicOr(ctl.err, DEVERR_BOUNDS);
    return false;
#else
    (void)ctl;
    (void)i;
    (void)w;
    (void)n;
    return true;
#endif
}

// ----------------------------------------------------------------------------
// small PTX wrappers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// try_wait: the thread may be suspended for a system-dependent time until
// the phase completes.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of a phase (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed, at most
// `limit_ns` of wall time (polling, with a short sleep between polls after
// the first few).  Returns false (and sets the device error word)
// if the limit ran out.  `abort_flag` (shared memory, may be null): give up
// early, without error, once another thread of the block has set it.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  const DevCtl& ctl,
                                                  volatile int* abort_flag = nullptr) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        // after a few polls, yield the scheduler between polls: a polling
        // warp otherwise takes issue slots from the warps it waits for
        if (i >= 8) __nanosleep(32);
        if ((i & 3u) == 0) {
            if (abort_flag && *abort_flag) return false;
            if (globaltimer_ns() - t0 > ctl.wait_limit_ns) {
                atomicOr(ctl.err, DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Warp-wide wait: lane 0 polls the barrier (bounded) and the warp then
// synchronises, which orders the other lanes after lane 0's acquire.  One
// poller per warp instead of 32 keeps the barrier unit free for the other
// waiters.  All 32 lanes must call it; the result is warp-uniform.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, const DevCtl& ctl,
                                               volatile int* abort_flag = nullptr) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, ctl, abort_flag);
    __syncwarp();
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Same bound, busy-polling with test_wait: for a single thread on the
// critical path (a suspended try_wait can resume well after the phase
// completes).
__device__ __forceinline__ bool mbar_spin_bounded(uint64_t* bar, uint32_t parity,
                                                  const DevCtl& ctl,
                                                  volatile int* abort_flag = nullptr) {
    if (mbar_test_wait(bar, parity)) return true;
    unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (abort_flag && *abort_flag) return false;
            if (globaltimer_ns() - t0 > ctl.wait_limit_ns) {
                atomicOr(ctl.err, DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Same bound, waiting in try_wait alone: the thread is suspended in hardware
// until the phase completes (or a system-dependent time passes), so a
// waiting warp takes no issue slots from the warps that do the work -- with
// several roles per SM sub-partition, polling warps slow the working ones
// down severalfold.
__device__ __forceinline__ bool mbar_suspend_bounded(uint64_t* bar, uint32_t parity,
                                                     const DevCtl& ctl,
                                                     volatile int* abort_flag = nullptr) {
    if (mbar_test_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag && *abort_flag) return false;
        if (globaltimer_ns() - t0 > ctl.wait_limit_ns) {
            atomicOr(ctl.err, DEVERR_TIMEOUT);
            return false;
        }
    }
}

// Warp-wide suspending wait (lane 0 waits in try_wait, the warp then
// synchronises).  All 32 lanes must call it; the result is warp-uniform.
__device__ __forceinline__ bool mbar_suspend_warp(uint64_t* bar, uint32_t parity,
                                                  const DevCtl& ctl,
                                                  volatile int* abort_flag = nullptr) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_suspend_bounded(bar, parity, ctl, abort_flag);
    __syncwarp();
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Warp-wide busy-polling wait (lane 0 spins with test_wait, the warp then
// synchronises): for warps on the critical path of a pipeline, where a
// sleeping poller would wake up late.  All 32 lanes must call it.
__device__ __forceinline__ bool mbar_spin_warp(uint64_t* bar, uint32_t parity, const DevCtl& ctl,
                                               volatile int* abort_flag = nullptr) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_spin_bounded(bar, parity, ctl, abort_flag);
    __syncwarp();
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// L2 prefetch of a global range (a hint: nothing is written, no completion).
// src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 eviction-priority policy (from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 2-D tiled TMA load of box (x, y) of `map` (a __grid_constant__ kernel
// parameter) into shared memory.  x * element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch: wait for the preceding grid's memory, and
// allow the next grid to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier over `count` threads that also ORs a predicate across them:
// every participant gets the same answer.
__device__ __forceinline__ bool named_bar_any(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Split-K hand-off counter: fetch-and-add at gpu scope with acquire-release
// semantics, by one thread right after a barrier of the threads that wrote
// partial sums.  The release half publishes those writes (ordered before
// this thread by the barrier) before the add; the acquire half orders the
// reads after it -- and, through the next barrier, the other threads' reads
// -- after every write released by earlier adds on the same counter.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

// d = c + sum_i a.u8[i] * b.s8[i]   (a unsigned bytes, b signed bytes)
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Shared-memory accesses by 32-bit shared address (explicit ld/st.shared, so
// the hot loops never go through generic addressing).  Volatile: they keep
// their order relative to the mbarrier waits and barriers.
__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v));
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Quotients for the quantiser, each a product with a reciprocal corrected
// once by its exact remainder r = x - q0*d (one fused multiply-add; the
// correction step of Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  They are
// used only on the quantiser's own domain and were checked exhaustively on
// the GPU against IEEE division there:
//   * d = amax / 127 from the fp32 value nearest 1/127: bit-identical to the
//     correctly rounded quotient for all 31,743 positive finite fp16 amax;
//   * x / d from the hardware reciprocal approximation of d: the same integer
//     after round-half-even as the correctly rounded quotient, for every fp16
//     amax and every fp16 x with |x| <= amax (503,856,639 pairs; negative x
//     mirror positive ones).
__device__ __forceinline__ float div_corrected(float x, float d, float y) {
    const float q0 = __fmul_rn(x, y);
    const float r = __fmaf_rn(-q0, d, x);
    return __fmaf_rn(r, y, q0);
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr uint32_t kRcp127Bits = 0x3C010204u;  // fp32 nearest 1/127

// Two-wide fp32 arithmetic (one instruction, two IEEE round-to-nearest
// operations): the same bits as two scalar operations.
__device__ __forceinline__ unsigned long long f32x2_pack(float lo, float hi) {
    unsigned long long v;
    asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
    return v;
}
__device__ __forceinline__ void f32x2_unpack(unsigned long long v, uint32_t& lo, uint32_t& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f32x2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f32x2_fma(unsigned long long a, unsigned long long b,
                                                        unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f32x2_add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
#ifndef PQ2_QUANT_X2
#define PQ2_QUANT_X2 1
#endif

// Quantise one 128-value group with 8 consecutive lanes of a warp ("Making a
// ternary reasoning model fast in vLLM", page "From CUDA to Triton and
// Gluon", section "Prompt processing": q int8, s fp32, t int32 per group;
// section "One token at a time": plane order).  All 32 lanes call it, four
// groups at a time; lane j (0..7) of a group holds its values 16j..16j+15 as
// fp16 (h[0] the first eight), i.e. code bytes 4j..4j+3, and writes plane s
// of them as one 32-bit word at qg + s*32 + 4j.
//   amax = max |x| (exact in fp16); d = RN(amax / 127); q = RN-even(x / d)
// (both divisions by div_corrected, exact on this domain).
// No clamp is needed: |x| <= amax and d >= (amax/127)(1 - 2^-24) keep
// |x / d| below 127.5.  T = sum q.  An all-zero group gives d = 0, q = 0.
// Nothing is written unless `store`; lane j == 0 writes s and t.
__device__ __forceinline__ void quantize_group8(const uint4 (&h)[2], int j, bool store,
                                                int8_t* qg, float* s_out, int32_t* t_out,
                                                float& s_all, int& t_all) {
    const __half2* hv = reinterpret_cast<const __half2*>(h);
    __half2 m = __habs2(hv[0]);
#pragma unroll
    for (int k = 1; k < 8; ++k) m = __hmax2(m, __habs2(hv[k]));
    float amax = fmaxf(__low2float(m), __high2float(m));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const bool zero = amax == 0.0f;
    const float d = div_corrected(amax, 127.0f, __uint_as_float(kRcp127Bits));  // RN(amax/127)
    const float y = rcp_approx(d);  // d is 0 (unused) or a normal number
    // q by adding 1.5 * 2^23: the sum lies in [2^23, 2^24), where the add
    // itself rounds to an integer, half to even, and the low byte of its bit
    // pattern is q as an int8 (|x / d| < 127.5).
    uint32_t qb[16];
#if PQ2_QUANT_X2
    // the quotients of div_corrected two at a time: q0 = x*y,
    // r = q0*(-d) + x (= x - q0*d, one rounding), q = r*y + q0.  An all-zero
    // group runs with y = 0: every x is +-0 there and every q comes out +0,
    // as the scalar path's explicit zero does.
    {
        const float yz = zero ? 0.0f : y;
        const unsigned long long y2 = f32x2_pack(yz, yz);
        const unsigned long long nd2 = f32x2_pack(-d, -d);
        const unsigned long long mg2 = f32x2_pack(12582912.0f, 12582912.0f);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float2 v = __half22float2(hv[k]);
            const unsigned long long v2 = f32x2_pack(v.x, v.y);
            const unsigned long long q0 = f32x2_mul(v2, y2);
            const unsigned long long r = f32x2_fma(q0, nd2, v2);
            const unsigned long long q = f32x2_fma(r, y2, q0);
            f32x2_unpack(f32x2_add(q, mg2), qb[2 * k], qb[2 * k + 1]);
        }
    }
#else
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float v = (i & 1) ? __high2float(hv[i >> 1]) : __low2float(hv[i >> 1]);
        const float qf = zero ? 0.0f : div_corrected(v, d, y);
        qb[i] = __float_as_uint(__fadd_rn(qf, 12582912.0f));
    }
#endif
    int t = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        // bytes 4j..4j+3 of plane s are values s, s+4, s+8, s+12
        const uint32_t lo = __byte_perm(qb[s], qb[s + 4], 0x0040);
        const uint32_t hi = __byte_perm(qb[s + 8], qb[s + 12], 0x0040);
        const uint32_t w = __byte_perm(lo, hi, 0x5410);
        if (store) *reinterpret_cast<uint32_t*>(qg + s * 32 + 4 * j) = w;
        t = __dp4a(static_cast<int>(w), 0x01010101, t);
    }
    t += __shfl_xor_sync(0xffffffffu, t, 4);
    t += __shfl_xor_sync(0xffffffffu, t, 2);
    t += __shfl_xor_sync(0xffffffffu, t, 1);
    if (store && j == 0) {
        *s_out = zero ? 0.0f : d;
        *t_out = t;
    }
    s_all = zero ? 0.0f : d;  // the same in all eight lanes
    t_all = t;
}

__device__ __forceinline__ void quantize_group8(const uint4 (&h)[2], int j, bool store,
                                                int8_t* qg, float* s_out, int32_t* t_out) {
    float s_all;
    int t_all;
    quantize_group8(h, j, store, qg, s_out, t_out, s_all, t_all);
}

// Codes-dot of one 128-weight group: 8 code words against the 32 plane-ordered
// activation words q[s*8 + j] (plane s, word j).  Plane s of word w is
// w & (3 << 2s) per byte, i.e. 4^s times the codes; the four plane sums are
// rescaled exactly with arithmetic shifts (each is a multiple of 4^s).
__device__ __forceinline__ int group_codes_dot(const uint32_t (&w)[8], const uint32_t* q) {
    int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        a0 = dp4a_us(w[j] & 0x03030303u, q[0 * 8 + j], a0);
        a1 = dp4a_us(w[j] & 0x0C0C0C0Cu, q[1 * 8 + j], a1);
        a2 = dp4a_us(w[j] & 0x30303030u, q[2 * 8 + j], a2);
        a3 = dp4a_us(w[j] & 0xC0C0C0C0u, q[3 * 8 + j], a3);
    }
    return a0 + (a1 >> 2) + (a2 >> 4) + (a3 >> 6);
}

// The same group dot times 64, with 64*bias added: the plane sums are
// combined as ((a0*4 + a1)*4 + a2)*4 + a3 (three shift-adds, exact: plane s
// is 4^s times its codes) and the bias enters as the start value of the
// plane-3 sum.  |result| < 2^22 for int8 activations.
__device__ __forceinline__ int group_codes_dot64(const uint32_t (&w)[8], const uint32_t* q,
                                                 int bias64) {
    int a0 = 0, a1 = 0, a2 = 0, a3 = bias64;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        a0 = dp4a_us(w[j] & 0x03030303u, q[0 * 8 + j], a0);
        a1 = dp4a_us(w[j] & 0x0C0C0C0Cu, q[1 * 8 + j], a1);
        a2 = dp4a_us(w[j] & 0x30303030u, q[2 * 8 + j], a2);
        a3 = dp4a_us(w[j] & 0xC0C0C0C0u, q[3 * 8 + j], a3);
    }
    return ((a0 * 4 + a1) * 4 + a2) * 4 + a3;
}

}  // namespace pq2

// ----------------------------------------------------------------------------
// Host-side launch helpers shared by the translation units.
// ----------------------------------------------------------------------------
namespace pq2h {

struct DeviceInfo {
    int device;
    int num_sms;
    int max_smem_optin;
    unsigned* err;  // device address of the error word on this device
};

// Per-device info (queried once per device).  Returns false on CUDA error.
bool device_info(DeviceInfo* out);

// Fills the launch control block for the current device.
bool make_ctl(pq2::DevCtl* ctl);

// Raises a kernel's dynamic shared-memory limit to at least `smem` on the
// current device, calling the driver only the first time a larger size is
// needed (the attribute call costs microseconds, a launch a few).  One
// SmemLimit per kernel instantiation (a function-local static).
constexpr int kSmemLimitDevices = 64;
struct SmemLimit {
    std::atomic<int> bytes[kSmemLimitDevices];
};

template <typename Kern>
cudaError_t ensure_smem(SmemLimit& lim, Kern kern, size_t smem) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSmemLimitDevices)
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
    const int want = static_cast<int>(smem);
    if (lim.bytes[dev].load(std::memory_order_acquire) >= want) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (e != cudaSuccess) return e;
    int cur = lim.bytes[dev].load(std::memory_order_relaxed);
    while (cur < want && !lim.bytes[dev].compare_exchange_weak(cur, want, std::memory_order_release))
        ;
    return cudaSuccess;
}

// Launches are done with cudaLaunchKernelEx, with programmatic stream
// serialisation allowed (the kernels call griddepcontrol.wait before
// touching memory an earlier kernel may write).
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace pq2h
