// Host-side prototypes shared by the translation units of the library.
// Every launcher validates nothing (pq2_api.cu does) and returns the CUDA
// error of its launch.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/pq2.h"
#include "pq2_common.cuh"

namespace pq2h {

// The variant pq2_debug_force_kernel set for `op` (PQ2_VARIANT_DEFAULT when
// none).  A launcher asked for a variant that cannot take the call returns
// kUnsupportedVariant, which the C ABI reports as PQ2_ERR_UNSUPPORTED_SHAPE.
int forced_variant(int op);
constexpr cudaError_t kUnsupportedVariant = cudaErrorNotSupported;

// 2-D tiled tensor map (zero fill out of range): dims {inner, outer}
// elements, row pitch in bytes, box {box_inner, box_outer}; swizzle128 =
// 128-byte swizzle (box rows of exactly 128 bytes), else none.  The driver's
// encoder is reached through the runtime's entry-point query.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
                    bool swizzle128);

cudaError_t launch_quantize(const __half* x, int8_t* qp, float* S, int32_t* T, int64_t M,
                            int64_t K, cudaStream_t st, const pq2::DevCtl& ctl,
                            const DeviceInfo& dev);

// gu [M, 2I] fp32 (gate | up) -> quantised h = fp16(silu(gate) * up), as
// launch_quantize does for fp16 activations.
cudaError_t launch_quantize_swiglu(const float* gu, int8_t* qp, float* S, int32_t* T, int64_t M,
                                   int64_t I, cudaStream_t st, const pq2::DevCtl& ctl,
                                   const DeviceInfo& dev);

// y = bf16(x . w^T), bf16 operands as 16-bit patterns, split-K over a
// cluster of CTAs with a fixed-order reduction (pq2_bf16.cu).
cudaError_t launch_bf16_splitk(const uint16_t* x, const uint16_t* w, uint16_t* y, int64_t M,
                               int64_t N, int64_t K, bool weights_static, cudaStream_t stream,
                               const pq2::DevCtl& ctl);

cudaError_t launch_pack(const int8_t* tern, uint8_t* codes, int64_t N, int64_t K,
                        cudaStream_t st, const pq2::DevCtl& ctl, const DeviceInfo& dev);

// M == 1.  dots != nullptr selects the integer-dot debug output instead of y.
// x != nullptr selects the fused path: the kernel quantises the fp16
// activations itself (qp, S, T unused); only for K where
// gemv_fused_supported(K).  weights_static (fused path only): codes and ws
// are not written by the work preceding the launch on `st`, so the kernel may
// read them before its dependency wait.
bool gemv_fused_supported(int64_t K);
cudaError_t launch_gemv(const __half* x, const int8_t* qp, const float* S, const int32_t* T,
                        const uint8_t* codes, const __half* ws, float* y, int32_t* dots, int64_t N,
                        int64_t K, cudaStream_t st, const pq2::DevCtl& ctl, const DeviceInfo& dev,
                        bool weights_static = false);

// An empty kernel (dependency wait, early launch of the next grid) with the
// grid, block and shared memory a fused M == 1 call of this shape gets.
cudaError_t launch_gemv_floor(int64_t N, int64_t K, bool weights_static, cudaStream_t st,
                              const pq2::DevCtl& ctl, const DeviceInfo& dev);

// 2 <= M <= 16: tcgen05 kernel with the weights expanded into tensor memory,
// split-K partial sums reduced in a fixed order.
// workspace: small_workspace_bytes(M, N, K) bytes.
size_t small_workspace_bytes(int64_t M, int64_t N, int64_t K);
size_t small_scratch_bytes(int64_t M, int64_t N, int64_t K, int num_sms);
// A few tokens (2 <= M <= 4 by default, at most 8) on the DP4A path
// (pq2_multi.cu), where the shape allows: the code words are shared by the
// token rows.  No workspace.
bool gemv_multi_supported(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_gemv_multi(const int8_t* qp, const float* S, const int32_t* T,
                              const uint8_t* codes, const __half* ws, float* y, int32_t* dots,
                              int64_t M, int64_t N, int64_t K, cudaStream_t st,
                              const DeviceInfo& dev, bool weights_static, const pq2::DevCtl& ctl);

cudaError_t launch_small(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                         const __half* ws, float* y, int32_t* dots, int64_t M, int64_t N,
                         int64_t K, void* workspace, cudaStream_t st, const pq2::DevCtl& ctl,
                         const DeviceInfo& dev);
// pq2_matmul's path for the calls pq2_gemm_small sends to small_kernel
// (small_x_supported): one kernel quantises the fp16 activations straight
// into small_kernel's token tiles and (s, t) table (no qp, S, T), then
// small_kernel; y is bit-identical to pq2_quantize_act + pq2_gemm_small.
// workspace: small_workspace_bytes(M, N, K) bytes.
bool small_x_supported(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_small_x(const __half* x, const uint8_t* codes, const __half* ws, float* y,
                           int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                           const pq2::DevCtl& ctl, const DeviceInfo& dev);

// 1 <= M <= kTileMaxM: the weights-stationary token-tile kernel
// (pq2_tile.cu): weights expanded into tensor memory, 16, 32 or 64 token
// rows per tile, split-K partial sums reduced in a fixed order.
constexpr int kTileMaxM = 64;
size_t tile_workspace_bytes(int64_t M, int64_t N, int64_t K);
size_t tile_scratch_bytes(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_tile(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                        const __half* ws, float* y, int32_t* dots, int64_t M, int64_t N, int64_t K,
                        void* workspace, cudaStream_t st, const pq2::DevCtl& ctl,
                        const DeviceInfo& dev);
// The same from the fp16 activations x [M][K]: one kernel quantises x
// straight into the token tiles (see pq2_tokens.cuh); y bit-identical.
cudaError_t launch_tile_x(const __half* x, const uint8_t* codes, const __half* ws, float* y,
                          int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                          const pq2::DevCtl& ctl, const DeviceInfo& dev);

// 1 <= M <= kTileMaxM: the weights-wide token-tile kernel (pq2_wtile.cu):
// 128 expanded weight rows per MMA, the tokens' hi and lo parts as the
// 128-row operand (16, 32 or 64 tokens), split-K partial sums reduced in a
// fixed order.  pq2_gemm_prefill runs it by default for 33-64 tokens when
// the call has few items a CTA (wtile_default: at most 4 (128-row tile,
// 4-group) items per CTA, measured at 6144 -> 5120, 48 and 64 tokens: 30.3
// and 32.6 us against 38.9 and 39.4 for the 128 x 128 tile kernel; at
// 5120 -> 17408, 9 items a CTA, 47.2 and 48.9 against 34.7 and 35.5).
constexpr int kWTileDefaultMinM = 32;
constexpr int kWTileDefaultItemsPerCta = 4;
bool wtile_default(int64_t M, int64_t N, int64_t K, int num_sms);
size_t wtile_workspace_bytes(int64_t M, int64_t N, int64_t K);
size_t wtile_scratch_bytes(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_wtile(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                         const __half* ws, float* y, int32_t* dots, int64_t M, int64_t N,
                         int64_t K, void* workspace, cudaStream_t st, const pq2::DevCtl& ctl,
                         const DeviceInfo& dev);
cudaError_t launch_wtile_x(const __half* x, const uint8_t* codes, const __half* ws, float* y,
                           int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                           const pq2::DevCtl& ctl, const DeviceInfo& dev);

// Back-to-back tcgen05 e4m3 MMAs (M = 128, N = n, K = 32) on every SM:
// cycles[sm] = clock cycles for `iters` of them (pq2_debug_mma_rate).
cudaError_t launch_mma_rate(int n, int iters, unsigned long long* cycles, cudaStream_t st,
                            const pq2::DevCtl& ctl, const DeviceInfo& dev);

// The tensor-core kernel pq2_gemm_small runs for 5 to 16 tokens (and for
// fewer when the DP4A kernel cannot take the shape): the token-tile kernel,
// or small_kernel when forced.  Scratch for this device / for any device.
size_t small_tc_scratch_bytes(int64_t M, int64_t N, int64_t K, int num_sms);
size_t small_tc_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_small_tc(const int8_t* qp, const float* S, const int32_t* T,
                            const uint8_t* codes, const __half* ws, float* y, int32_t* dots,
                            int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                            const pq2::DevCtl& ctl, const DeviceInfo& dev);

// The token-tile kernels (their tiles can be quantised straight from x).
enum class TokenTile { kNone, kSmall, kTile, kWide };
// The token-tile kernel pq2_gemm_prefill runs for this call (its routing):
// kTile (tile_kernel), kWide (wtile_kernel) or kNone (a 128-token kernel).
TokenTile prefill_token_tile_kernel(int64_t M, int64_t N, int64_t K, int num_sms);

// Any M: tcgen05 tensor-core kernel (token planes prepared in the workspace).
size_t prefill_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_prefill(const int8_t* qp, const float* S, const int32_t* T, const uint8_t* codes,
                           const __half* ws, float* y, int32_t* dots, int64_t M, int64_t N,
                           int64_t K, void* workspace, cudaStream_t st, const pq2::DevCtl& ctl,
                           const DeviceInfo& dev);

}  // namespace pq2h
