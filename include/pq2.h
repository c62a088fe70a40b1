/*
 * pq2.h -- C ABI of the GB300 (sm_103a) PQ2_0 ternary-weight matmul library.
 *
 * The operation, as the pages define it:
 *   [P1] "Making a ternary reasoning model fast in vLLM", page "From CUDA to
 *        Triton and Gluon";
 *   [P2] the same series, page "Chasing llama.cpp at batch one".
 *
 *   y[m,n] = sum_g (dot(codes[n,g], q[m,g]) - sum(q[m,g])) * S[m,g] * WS[n,g]
 *
 * Weights are 2-bit codes 0,1,2 standing for -1,0,+1, four to a byte, with
 * one fp16 scale per 128 weights ([P1] "One token at a time": the PQ2_0 code
 * and the per-group scale).  Activations are quantised to int8 per 128 values
 * and stored in plane order, so the activation of weight 4*byte+s sits at
 * position s*32+byte of its group; plane s of a 32-bit code word,
 * (w >> 2s) & 0x03030303, then lines up with four consecutive activation
 * bytes, and the -1 offset is one subtraction of sum(q) per group (same
 * section).
 *
 * Notation and layouts (all row-major, all buffers owned by the caller):
 *   M tokens, K inputs (K % 128 == 0), N outputs, G = K / 128.
 *   x      fp16  [M, K]      activations
 *   qp     int8  [M, K]      quantised activations, plane order: the value of
 *                            natural index k is at g*128 + (k&3)*32 + ((k&127)>>2)
 *   S      fp32  [M, G]      activation scale per group
 *   T      int32 [M, G]      sum of the group's int8 values
 *   codes  uint8 [N, K/4]    weight k of row n in byte n*K/4 + (k>>2), bits 2*(k&3)
 *   WS     fp16  [N, G]      weight scale per group
 *   y      fp32  [M, N]      output (fully overwritten, never accumulated into)
 *
 * Conventions shared by every entry point:
 *   - Pointers are device pointers unless stated, 16-byte aligned
 *     (PQ2_ERR_MISALIGNED otherwise); sizes are element counts.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it; nothing here
 *     synchronises, except pq2_last_device_error.
 *   - The library allocates and frees no memory.  Scratch space, where an
 *     operation needs it, is passed in as `workspace` / `workspace_bytes`
 *     (size from pq2_workspace_bytes).
 *   - Arguments are checked on the host before any launch; on error nothing
 *     is enqueued and the status says why.  A failed launch returns
 *     PQ2_ERR_CUDA.  Device faults surface at the caller's next
 *     synchronisation, as for any CUDA call.
 *   - Results are deterministic: the same inputs give bit-identical outputs
 *     (fixed-order reductions, no atomics on data).
 *   - NaN or Inf in x is not checked; the result is then undefined.
 *   - Kernels wait on on-chip barriers with a bounded spin; a wait that runs
 *     out sets a device error word that pq2_last_device_error reports as
 *     PQ2_ERR_TIMEOUT.
 */
#ifndef PQ2_H
#define PQ2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pq2_status {
    PQ2_OK = 0,
    PQ2_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad op  */
    PQ2_ERR_UNSUPPORTED_SHAPE = 2, /* K % 128 != 0, M out of range, ...    */
    PQ2_ERR_MISALIGNED = 3,        /* a pointer is not 16-byte aligned      */
    PQ2_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed  */
    PQ2_ERR_TIMEOUT = 5,           /* a kernel's bounded wait ran out       */
    PQ2_ERR_WORKSPACE = 6,         /* workspace missing or too small        */
    PQ2_ERR_BOUNDS = 7             /* bounds-checked build: a kernel skipped
                                      a store outside its buffer            */
} pq2_status;

/* Operation selectors for pq2_workspace_bytes and pq2_group_dots. */
enum {
    PQ2_OP_GEMV = 0,     /* pq2_gemv            (M == 1)            */
    PQ2_OP_SMALL = 1,    /* pq2_gemm_small      (2 <= M <= 16)      */
    PQ2_OP_PREFILL = 2,  /* pq2_gemm_prefill    (M >= 1)            */
    PQ2_OP_MATMUL = 3,   /* pq2_matmul          (M >= 1, from fp16) */
    PQ2_OP_SWIGLU_DOWN = 4 /* pq2_mlp_down_swiglu (M >= 1; K = I)     */
};

/* Largest K any entry point accepts (G <= 2048 groups). */
#define PQ2_MAX_K 262144

/* Static text for a status code; never NULL. */
const char* pq2_status_string(int status);

/* Library version string, e.g. "pq2-gb300 0.1 sm_103a". */
const char* pq2_version(void);

/*
 * pq2_quantize_act -- fused activation quantisation and plane reorder.
 *   [P1] "Prompt processing": the quantize kernel writes q [m,k] int8,
 *   s [m,G] fp32 and t [m,G] int32 per 128-value group; [P1] "One token at
 *   a time": q is stored in plane order.
 * Per (m, g): amax = max |x|; d = amax / 127 (fp32, round to nearest even);
 * q = round-half-even(x / d) clamped to [-127, 127]; S = d; T = sum q.  A
 * group of zeros gives d = 0, q = 0, T = 0.  (The pages fix the outputs but
 * not the scale formula; this is the plain symmetric reading.)
 *   x_f16  in   fp16 [M, K]
 *   qp     out  int8 [M, K] plane order
 *   S, T   out  fp32 / int32 [M, G]
 * M >= 0 (M == 0 enqueues nothing), 1 <= K <= PQ2_MAX_K, K % 128 == 0.
 */
pq2_status pq2_quantize_act(const void* x_f16, int64_t M, int64_t K,
                            int8_t* qp, float* S, int32_t* T, void* stream);

/*
 * pq2_quantize_swiglu -- the activation between the two projections of a
 * decode MLP, fused with the quantisation of pq2_quantize_act.  The pages
 * link the MLP's gate/up and down projections ([P1] "Choose the
 * configuration with the proxy": replayed gate -> down pairs) but do not
 * define the activation; this is the plain SwiGLU reading:
 *   gate = gu[m, 0..I), up = gu[m, I..2I);  h = silu(gate) * up,
 *   silu(g) = g / (1 + exp(-g)),
 * every step one fp32 operation with round-to-nearest, exp computed by Cody
 * and Waite's argument reduction and a degree-7 Taylor polynomial (a fixed
 * sequence of fused multiply-adds, so a CPU restatement gets the same bits);
 * h is rounded to fp16, saturating at +-65504, then quantised exactly as
 * pq2_quantize_act quantises x.
 *   gu     in   fp32 [M, 2I]  (typically the y of the gate/up projection)
 *   qp     out  int8 [M, I] plane order
 *   S, T   out  fp32 / int32 [M, I/128]
 * M >= 0 (M == 0 enqueues nothing), 1 <= I <= PQ2_MAX_K, I % 128 == 0.
 * NaN or Inf in gu: the result is undefined.
 */
pq2_status pq2_quantize_swiglu(const float* gu, int64_t M, int64_t I,
                               int8_t* qp, float* S, int32_t* T, void* stream);

/*
 * pq2_pack_weights -- the "prepared" weight planes: ternary values to codes.
 *   [P1] "One token at a time": codes 0,1,2 for -1,0,+1, four to a byte,
 *   weight 4*byte+s in bits 2s; [P1] "A power proxy for the rest of the
 *   model": prepared weights carry the scales as a separate plane.
 *   tern    in   int8 [N, K], every value in {-1, 0, +1}
 *   ws_f16  in   fp16 [N, G]  (may be NULL together with ws_out)
 *   codes   out  uint8 [N, K/4]
 *   ws_out  out  fp16 [N, G]  copy of ws_f16 (may alias ws_f16)
 * A value outside {-1,0,1} is stored as code 3 (read as +2 by the matmul
 * kernels) and sets the device error word; the host cannot see it without a
 * synchronisation, so validate ternary inputs before packing.
 */
pq2_status pq2_pack_weights(const int8_t* tern, const void* ws_f16, int64_t N, int64_t K,
                            uint8_t* codes, void* ws_out, void* stream);

/*
 * pq2_gemv -- the M = 1 decode matmul y[n] for all n.
 *   [P1] "One token at a time: plain Triton is enough" (plane extraction
 *   with (w >> 2s) & 0x03030303 feeding DP4A, the per-group sum(q)
 *   subtraction, fp32 accumulation of dot * s * ws); [P2] "The win: a program
 *   just for one token" (no token dimension, separate scale plane).
 *   qp [1,K], S [1,G], T [1,G], codes [N,K/4], ws_f16 [N,G] in; y [1,N] out.
 * N >= 1, 128 <= K <= PQ2_MAX_K, K % 128 == 0.
 */
pq2_status pq2_gemv(const int8_t* qp, const float* S, const int32_t* T,
                    const uint8_t* codes, const void* ws_f16, float* y,
                    int64_t N, int64_t K, void* stream);

/*
 * pq2_gemm_small -- small batches, 2 <= M <= 16 token rows.
 *   [P1] "Small batches: make the register layout explicit", "Use a ring
 *   buffer for longer rows", "Extend the kernels to sixteen token rows";
 *   split-K partial sums, where used, are reduced in the fixed order
 *   0,1,2,... ([P1] "Choose the configuration with the proxy").
 *   Same operands as pq2_gemv with M rows; y [M,N].
 *   workspace: device scratch of pq2_workspace_bytes(PQ2_OP_SMALL, M, N, K)
 *   bytes (may be NULL when that is 0).
 *   2 to 4 token rows run on DP4A, each code word shared by the rows, where
 *   a CTA's group terms fit its shared memory (the workspace is then not
 *   touched; each row's y equals pq2_gemv on that row, bit for bit); larger
 *   M on the tensor cores.
 */
pq2_status pq2_gemm_small(const int8_t* qp, const float* S, const int32_t* T,
                          const uint8_t* codes, const void* ws_f16, float* y,
                          int64_t M, int64_t N, int64_t K,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * pq2_gemm_small_ex -- pq2_gemm_small with a flags word: 0, or
 *   PQ2_WEIGHTS_STATIC (defined below, as for pq2_matmul_ex): the caller
 *   promises that codes and ws_f16 are not written by any operation enqueued
 *   on `stream` before this call that may still be running when it starts.
 *   The DP4A kernel for 2 to 4 token rows then requests its weights (an L2
 *   prefetch of its slice and its first rows) before the preceding kernel
 *   has finished; qp, S and T are still read only after it.  y is
 *   bit-identical to pq2_gemm_small.  Other bits give PQ2_ERR_INVALID_ARG;
 *   the tensor-core path ignores the flag.
 */
pq2_status pq2_gemm_small_ex(const int8_t* qp, const float* S, const int32_t* T,
                             const uint8_t* codes, const void* ws_f16, float* y, int64_t M,
                             int64_t N, int64_t K, uint32_t flags, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * pq2_gemm_prefill -- prompt processing, any M >= 1 (built for M > 16).
 *   [P1] "Prompt processing: check configuration and launch costs" (2-D
 *   output tiles, per-group integer products and the same per-group
 *   dequantise-accumulate order as the M = 1 path).
 *   Same operands as pq2_gemm_small; y [M,N].
 *   workspace: pq2_workspace_bytes(PQ2_OP_PREFILL, M, N, K) bytes; for
 *   shapes the 128 x 256 tile kernel may take (at least 8 tiles of 128
 *   tokens, M > 896, and at least 128 tiles of 128 x 256) it includes the
 *   weights expanded to one byte per weight (N*K bytes), written once per
 *   call.
 */
pq2_status pq2_gemm_prefill(const int8_t* qp, const float* S, const int32_t* T,
                            const uint8_t* codes, const void* ws_f16, float* y,
                            int64_t M, int64_t N, int64_t K,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * pq2_matmul -- the whole path from fp16 activations: pq2_quantize_act, then
 * pq2_gemv (M == 1), pq2_gemm_small (M <= 16) or pq2_gemm_prefill.  The
 * pages' routing by token count ([P1] "Defaults and switches").
 *   x_f16 [M,K] fp16, codes, ws_f16 in; y [M,N] fp32 out.
 *   workspace: pq2_workspace_bytes(PQ2_OP_MATMUL, M, N, K) bytes (holds the
 *   quantised activations plus the chosen kernel's own scratch).  For M == 1
 *   and K <= 32768 the GEMV kernel quantises x itself (one launch) and no
 *   workspace is needed (size 0, workspace may be NULL).
 */
pq2_status pq2_matmul(const void* x_f16, const uint8_t* codes, const void* ws_f16, float* y,
                      int64_t M, int64_t N, int64_t K,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Flags of pq2_matmul_ex. */
#define PQ2_WEIGHTS_STATIC 1u

/*
 * pq2_matmul_ex -- pq2_matmul with flags.  (The pages have no counterpart to
 * the flag; it lets a decode loop overlap one call's weight stream with the
 * preceding call's arithmetic.)
 *   flags: 0 or PQ2_WEIGHTS_STATIC; other bits give PQ2_ERR_INVALID_ARG.
 *   PQ2_WEIGHTS_STATIC: the caller promises that codes and ws_f16 are not
 *     written by any operation enqueued on `stream` before this call that may
 *     still be running when it starts (typically: weights packed or copied
 *     once, then many calls).  The M == 1 fused kernel and the DP4A kernel
 *     for a few tokens (2 <= M <= 4 where the shape allows) may then read
 *     them before the preceding kernel on the stream has finished
 *     (programmatic dependent launch).  x_f16 is still read only after that
 *     kernel is done.  If the promise is broken, y is undefined.  Results
 *     are bit-identical to pq2_matmul.  The other paths ignore the flag.
 *   Other arguments, workspace and errors as pq2_matmul.
 */
pq2_status pq2_matmul_ex(const void* x_f16, const uint8_t* codes, const void* ws_f16, float* y,
                         int64_t M, int64_t N, int64_t K, uint32_t flags,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * pq2_mlp_down_swiglu -- the down projection of a decode MLP from its gate/up
 * output: pq2_quantize_swiglu, then pq2_gemv (M == 1), pq2_gemm_small
 * (M <= 16) or pq2_gemm_prefill, as pq2_matmul routes.
 *   gu [M, 2I] fp32 in; codes [N, I/4], ws_f16 [N, I/128] in; y [M, N] fp32 out.
 *   workspace: pq2_workspace_bytes(PQ2_OP_SWIGLU_DOWN, M, N, I) bytes (the
 *   quantised h plus the matmul's own scratch); never 0.
 * Errors as pq2_matmul.
 */
pq2_status pq2_mlp_down_swiglu(const float* gu, const uint8_t* codes, const void* ws_f16, float* y,
                               int64_t M, int64_t N, int64_t I,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * pq2_gemm_bf16_splitk -- the small unquantised projection of a decode step
 * ([P1] "Speed up a small unquantised projection": in_proj_ba, N = 96,
 * K = 5120, a few tokens at a time): y = bf16(x . w^T), computed as a
 * split-K GEMM whose fp32 partial sums are added in a fixed order, so the
 * same inputs give the same bits on every call.
 *   x [M, K] bf16 in, w [N, K] bf16 in, y [M, N] bf16 out; bf16 values are
 *   passed as their 16-bit patterns, rows contiguous.  Products and sums in
 *   fp32, one rounding of each output to bf16 (nearest, ties to even).
 *   M >= 0 and N >= 0 (either 0 enqueues nothing), 0 <= K <= PQ2_MAX_K
 *   (K == 0 writes zeros; x and w may then be null), K % 8 == 0, M <= PQ2_MAX_M_BF16,
 *   N <= PQ2_MAX_N_BF16: PQ2_ERR_UNSUPPORTED_SHAPE otherwise.  x and w
 *   16-byte aligned, y 2-byte aligned: PQ2_ERR_MISALIGNED otherwise.
 *   flags: 0 or PQ2_WEIGHTS_STATIC (w may be read before the preceding
 *   kernel on the stream has finished); other bits: PQ2_ERR_INVALID_ARG.
 *   One launch, no workspace.  Built for M <= 16; a larger M runs as
 *   independent 16-token tiles that each read w again.
 */
#define PQ2_MAX_M_BF16 1048560
#define PQ2_MAX_N_BF16 1073741824
pq2_status pq2_gemm_bf16_splitk(const uint16_t* x, const uint16_t* w, uint16_t* y, int64_t M,
                                int64_t N, int64_t K, uint32_t flags, void* stream);

/*
 * pq2_workspace_bytes -- scratch bytes `op` needs for this shape (0 if none,
 * SIZE_MAX if the shape is not supported).
 */
size_t pq2_workspace_bytes(int op, int64_t M, int64_t N, int64_t K);

/*
 * pq2_group_dots -- debug view of the integer part of a kernel: the same
 * kernel as `op` (PQ2_OP_GEMV, PQ2_OP_SMALL or PQ2_OP_PREFILL), writing the
 * per-group ternary dots dot(codes,q) - sum(q) instead of y
 * ([P1] "One token at a time": the -1 offset as one subtraction per group).
 *   dots out int32 [M, N, G].  Other operands as for `op`; workspace as for
 *   `op`.  For PQ2_OP_GEMV, M must be 1.
 */
pq2_status pq2_group_dots(int op, const int8_t* qp, const int32_t* T, const uint8_t* codes,
                          int64_t M, int64_t N, int64_t K, int32_t* dots,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * pq2_last_device_error -- synchronises `stream`, then reads and clears the
 * current device's error word: PQ2_ERR_TIMEOUT if a kernel's bounded wait ran
 * out, PQ2_ERR_BOUNDS (bounds-checked build only) if a kernel skipped a store
 * outside its buffer, PQ2_ERR_INVALID_ARG if pq2_pack_weights met a
 * non-ternary value,
 * PQ2_OK otherwise (PQ2_ERR_CUDA if the synchronisation itself failed).
 */
pq2_status pq2_last_device_error(void* stream);

/*
 * pq2_gemm_small_noalloc -- pq2_gemm_small for callers that cannot allocate
 * device memory (no allocator of their own, or allocation not allowed where
 * they run): the same kernel, with its split-K scratch in a fixed 4 MiB
 * device array that the library holds on every device it is loaded on until
 * the process exits.  (The pages have no counterpart to this entry point;
 * it exists for callers of this library.)
 *   Same operands as pq2_gemm_small, no workspace.  Returns
 *   PQ2_ERR_WORKSPACE if the shape needs more than
 *   pq2_gemm_small_noalloc_max_scratch() bytes of scratch on this device.
 *   For the tensor-core kernel (5 or more tokens) the scratch is about
 *   (min(SMs, 256) + ceil(N/128)) * M * 512 bytes of partial sums plus
 *   ceil(K/512) * 16 KB of token tiles: on a 152-SM GPU, 16 tokens fit up
 *   to about N = 40,000 at K = 5120, and an lm_head-scale N = 248,320 gets
 *   PQ2_ERR_WORKSPACE.  2 to 4 tokens, where the DP4A kernel takes them,
 *   need no scratch.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) and should come before any stream capture.
 *   All calls share the array: calls that may run at the same time on the
 *   GPU (unordered streams) race on it.  No cudaMalloc, cudaFree or other
 *   allocating call is made.
 */
pq2_status pq2_gemm_small_noalloc(const int8_t* qp, const float* S, const int32_t* T,
                                  const uint8_t* codes, const void* ws_f16, float* y,
                                  int64_t M, int64_t N, int64_t K, void* stream);

/* Size in bytes of the fixed scratch array behind pq2_gemm_small_noalloc. */
size_t pq2_gemm_small_noalloc_max_scratch(void);

/* Kernel variants for pq2_debug_force_kernel. */
#define PQ2_VARIANT_DEFAULT 0        /* the library's own routing                  */
#define PQ2_VARIANT_GEMV_DIRECT 1    /* M = 1: look-ahead loads into registers      */
#define PQ2_VARIANT_GEMV_RING 2      /* M = 1: bulk-copy ring in shared memory      */
#define PQ2_VARIANT_GEMV_STAGED 3    /* M = 1 fused: whole slice staged before wait */
#define PQ2_VARIANT_SMALL_DP4A 1     /* 2..8 tokens: DP4A, code words shared        */
#define PQ2_VARIANT_SMALL_TC 2       /* tcgen05, weights in tensor memory, 16-token
                                        tile (5..16 tokens by default)              */
#define PQ2_VARIANT_SMALL_TILE 3     /* tcgen05 token-tile kernel (16 tokens)       */
#define PQ2_VARIANT_SMALL_WTILE 4    /* tcgen05, 128 weight rows per MMA, tokens as
                                        the 128-row operand (16 tokens)             */
#define PQ2_VARIANT_PREFILL_128 1    /* tcgen05 128 x 128 tiles, in-kernel expansion */
#define PQ2_VARIANT_PREFILL_WIDE 2   /* tcgen05 128 x 256 tiles, pre-expanded weights */
#define PQ2_VARIANT_PREFILL_TILE 3   /* tcgen05 token-tile kernel, M <= 64 (by
                                        default 17-32 tokens)                       */
#define PQ2_VARIANT_PREFILL_WTILE 4  /* tcgen05, 128 weight rows per MMA, tokens as
                                        the 128-row operand, M <= 64 (by default
                                        33-64 tokens when a CTA gets at most 4
                                        items of 128 rows x 4 groups)               */

/*
 * pq2_debug_force_kernel -- test hook: from now on, calls of `op`
 * (PQ2_OP_GEMV, PQ2_OP_SMALL or PQ2_OP_PREFILL; pq2_matmul, pq2_group_dots
 * and pq2_mlp_down_swiglu route through them) run kernel `variant` of that op
 * (PQ2_VARIANT_*), or follow the library's own routing again with
 * PQ2_VARIANT_DEFAULT.  Every variant computes the same integer group dots
 * and the same y, bit for bit; the hook exists so that tests can check each
 * kernel on shapes the routing would give to another.  A call whose shape
 * the forced variant cannot take returns PQ2_ERR_UNSUPPORTED_SHAPE.
 * pq2_workspace_bytes accounts for the forced variant, so set it before
 * sizing a workspace.  Process-wide; not for use while other threads call
 * the library.  PQ2_ERR_INVALID_ARG for an unknown op or variant.
 */
pq2_status pq2_debug_force_kernel(int op, int variant);

/*
 * pq2_debug_gemv_floor -- measurement hook: enqueues one launch of an empty
 * kernel (it waits for the preceding kernel on the stream and lets the next
 * one start launching, nothing else) with the grid, block and shared memory
 * that pq2_matmul_ex(M = 1, N, K, flags) gets.  A chain of these times the
 * launch and dependency latency a chain of real calls pays before any byte
 * moves: the floor of a dependent sequence of M = 1 calls.  No pointer is
 * passed and nothing is written.  Errors as pq2_matmul_ex (shape, flags).
 */
pq2_status pq2_debug_gemv_floor(int64_t N, int64_t K, uint32_t flags, void* stream);

/*
 * pq2_debug_mma_rate -- measurement hook: the rate at which one thread per SM
 * can issue tcgen05 MMAs of the kind the tensor-core kernels use
 * (kind::f8f6f4, e4m3 operands, M = 128, N = n, K = 32; A in tensor memory,
 * B in shared memory), back to back into one accumulator.  Enqueues one
 * launch of one CTA per SM; on completion cycles[sm] holds the SM clock
 * cycles from the first issue to the completion of `iters` MMAs (0 if the
 * bounded wait ran out).  n in {32, 64, 128, 256}, 1 <= iters <= 2^24.
 *   cycles  device uint64 array of at least (number of SMs) entries.
 * Multiply-adds per cycle per SM: 128 * n * 32 * iters / cycles.
 */
pq2_status pq2_debug_mma_rate(int n, int iters, uint64_t* cycles, void* stream);

/*
 * pq2_debug_set_wait_limit_ns -- bound on every on-chip barrier wait, in
 * nanoseconds (default 2e9).  For tests of the timeout path only.
 */
pq2_status pq2_debug_set_wait_limit_ns(uint64_t ns);

/*
 * pq2_debug_skip_stage -- test hook: from now on, the producer of every
 * bulk-copy pipeline withholds its stage number `stage` (never issues it), so
 * the consumers' bounded wait runs out and the call reports PQ2_ERR_TIMEOUT
 * through pq2_last_device_error.  -1 turns it off (the default).
 */
pq2_status pq2_debug_skip_stage(int stage);

/*
 * pq2_bounds_checked -- 1 in the bounds-checked build of the library
 * (libpq2_debug.so, compiled with PQ2_DEBUG=1), 0 in the normal one.  In the
 * bounds-checked build every kernel store to y, to the integer-dot output and
 * to the split-K scratch first checks that it lies inside its buffer; a store
 * that does not is skipped and pq2_last_device_error reports PQ2_ERR_BOUNDS.
 * Results are otherwise bit-identical to the normal build's.  It stands in
 * for a memory checker on GPUs where none can be run.
 */
int pq2_bounds_checked(void);

/*
 * pq2_debug_shrink_bounds -- test hook of the bounds-checked build: from now
 * on the checks treat the last `elements` elements of every checked buffer as
 * outside it, so that the stores a call makes there are reported
 * (PQ2_ERR_BOUNDS) and skipped (no memory outside the buffers is touched).
 * 0 turns it off (the default); no effect in the normal build.
 * PQ2_ERR_INVALID_ARG for a negative count.
 */
pq2_status pq2_debug_shrink_bounds(int elements);

#ifdef __cplusplus
}
#endif

#endif /* PQ2_H */
