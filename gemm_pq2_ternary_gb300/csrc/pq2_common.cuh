// Shared device helpers of the PQ2 CUDA library (sm_103a only).
//
// Inline PTX wrappers for mbarriers, 1-D bulk async copies (TMA engine),
// programmatic dependent launch, a bounded barrier wait, and the launch
// parameters every kernel gets (device error word, wait limit).
#pragma once

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
};

// Passed by value to every kernel.
struct DevCtl {
    unsigned* err;          // device error word (never null)
    unsigned long long wait_limit_ns;
    unsigned wait_hint_ns;  // suspend-time hint of mbarrier try_wait (0 = none)
    int debug_skip_stage;   // >= 0: producer withholds that stage (timeout tests)
};

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

// try_wait; with a non-zero suspend-time hint the thread may sleep until the
// phase completes or the hint (ns) passes.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, unsigned hint_ns) {
    uint32_t ok;
    if (hint_ns) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
    }
    return ok != 0;
}

// Wait until the phase with the given parity has completed, at most
// `limit_ns` of wall time.  Returns false (and sets the device error word)
// if the limit ran out.  `abort_flag` (shared memory, may be null): give up
// early, without error, once another thread of the block has set it.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  const DevCtl& ctl,
                                                  volatile int* abort_flag = nullptr) {
    if (mbar_try_wait(bar, parity, ctl.wait_hint_ns)) return true;
    unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity, ctl.wait_hint_ns)) return true;
        if ((i & 3u) == 0) {
            if (abort_flag && *abort_flag) return false;
            if (globaltimer_ns() - t0 > ctl.wait_limit_ns) {
                atomicOr(ctl.err, DEVERR_TIMEOUT);
                return false;
            }
        }
    }
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

// d = c + sum_i a.u8[i] * b.s8[i]   (a unsigned bytes, b signed bytes)
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Quantise one 128-value group with one warp ("Making a ternary reasoning
// model fast in vLLM", page "From CUDA to Triton and Gluon", section "Prompt
// processing": q int8, s fp32, t int32 per group; section "One token at a
// time": plane order).  Lane b holds the four values of code byte b
// (weights 4b..4b+3) and writes plane s at qg[s*32 + b].  amax/127 and x/d
// are IEEE divisions rounded to nearest, q rounds half to even and is clamped
// to [-127,127]; an all-zero group gives s = 0, q = 0.
__device__ __forceinline__ void quantize_group_loaded(uint2 raw, int lane, int8_t* qg,
                                                      float* s_out, int32_t* t_out) {
    const __half2 h01 = *reinterpret_cast<const __half2*>(&raw.x);
    const __half2 h23 = *reinterpret_cast<const __half2*>(&raw.y);
    const float v[4] = {__low2float(h01), __high2float(h01), __low2float(h23), __high2float(h23)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    int sum = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        int q = 0;
        if (amax != 0.0f) {
            q = __float2int_rn(__fdiv_rn(v[s], d));
            q = max(-127, min(127, q));
        }
        sum += q;
        qg[s * 32 + lane] = static_cast<int8_t>(q);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
        *s_out = (amax != 0.0f) ? d : 0.0f;
        *t_out = sum;
    }
}

__device__ __forceinline__ void quantize_group_warp(const __half* xg, int lane, int8_t* qg,
                                                    float* s_out, int32_t* t_out) {
    quantize_group_loaded(*reinterpret_cast<const uint2*>(xg + 4 * lane), lane, qg, s_out, t_out);
}

// All G groups of one activation row by `nwarps` warps (this one is `warp`):
// the loads of up to 8 groups per warp are issued together before any of
// them is quantised, so their latencies overlap.
__device__ __forceinline__ void quantize_row_warps(const __half* x, int G, int warp, int nwarps,
                                                   int lane, int8_t* q, float* s, int32_t* t) {
    for (int g0 = warp; g0 < G; g0 += 8 * nwarps) {
        uint2 raw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int g = g0 + i * nwarps;
            if (g < G) raw[i] = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(g) * 128 + 4 * lane);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int g = g0 + i * nwarps;
            if (g < G) quantize_group_loaded(raw[i], lane, q + g * 128, s + g, t + g);
        }
    }
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
