/*
 * PQ2_0 ternary matmul -- CPU ORACLE.
 *
 * This file is test infrastructure.  It is the plain, slow, obviously
 * correct statement of what the ternary matmul computes, used only by the
 * test-suite, by the package smoke check and by the benchmark's CPU-baseline
 * leg.  The CUDA library never links, loads or calls it, and it shares no
 * code, header or table with the CUDA library.
 *
 * Sources (web pages; section names as printed on them):
 *   [P1] "Making a ternary reasoning model fast in vLLM" -- the page
 *        "From CUDA to Triton and Gluon".
 *   [P2] "Making a ternary reasoning model fast in vLLM" -- the page
 *        "Chasing llama.cpp at batch one".
 *
 * Notation: M tokens, K inputs, N outputs, G = K/128 groups of 128 weights.
 *
 * What each function follows:
 *   pq2o_quantize      activation int8 quantisation per 128 values, emitting
 *                      q, the scale s and the sum t per group ([P1]
 *                      "Prompt processing", the quantize kernel's outputs
 *                      q [m,k] int8, s [m,G] fp32, t [m,G] int32).  The
 *                      pages do not print the scale formula or the rounding;
 *                      this oracle takes the plain symmetric reading:
 *                      d = amax/127 (IEEE fp32), q = round-half-even(x/d)
 *                      clamped to [-127,127], d = 0 and q = 0 when amax = 0.
 *   pq2o_plane_order   the plane order of activations: the activation of
 *                      weight 4*byte+s goes to position s*32+byte of its
 *                      group ([P1] "One token at a time").
 *   pq2o_pack          the PQ2_0 weight code: codes 0,1,2 stand for
 *                      -1,0,+1, four to a byte, weight k of a row in byte
 *                      k>>2 at bits 2*(k&3) ([P1] "One token at a time";
 *                      [P2] "Recover four weights with one lookup").
 *   pq2o_unpack        the inverse map code -> code-1.
 *   pq2o_group_dots    dot_g[m,n] = sum over the 128 k of group g of
 *                      (code[n,k]-1) * q[m,k], in natural k order, int64
 *                      arithmetic -- the ternary dot the kernels compute as
 *                      dot(codes,q) - sum(q) ([P1] "One token at a time").
 *   pq2o_codes_dots    sum of code[n,k]*q[m,k] per group (no offset), for the
 *                      identity dot(codes,q) - sum(q) = sum((code-1)*q).
 *   pq2o_swiglu        h = silu(gate) * up of a gate/up output (an assumed
 *                      activation: the pages do not define it), with exp by
 *                      a stated method (pq2o_exp); see the function.
 *   pq2o_matmul        y[m,n] = sum_g dot_g[m,n] * s[m,g] * ws[n,g], every
 *                      product and sum in float64, plus the magnitude
 *                      A[m,n] = sum_g |dot_g * s * ws| used by the
 *                      tolerance of the fp32 kernels ([P1] "One token at a
 *                      time": per-group dequantise and accumulate).
 *
 * Parity pins (tests/test_oracle_pins.py): the worked lookup example of
 * [P2], one-hot plane-layout cases, the identity above, all-minus-one /
 * all-zero / all-plus-one codes, brute force in pure Python on tiny inputs,
 * the integer matmul with unit scales, and exact quantisation cases.
 *
 * Plain C99, no vector intrinsics; OpenMP (if enabled) only splits the
 * independent output rows n across threads.  Compile without fast-math and
 * with -ffp-contract=off so every float operation is a single IEEE op.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PQ2O_OK 0
#define PQ2O_BAD_SHAPE 1
#define PQ2O_BAD_VALUE 2

/* Number of threads the parallel loops below use. */
int pq2o_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets that number (n >= 1); used to time the oracle on one core.  Returns
   the number in effect afterwards. */
int pq2o_set_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
    return pq2o_threads();
}

/* Position of natural index k (within a row) in plane order. */
static int64_t plane_pos(int64_t k) {
    int64_t g = k / 128;        /* group                        */
    int64_t j = k % 128;        /* weight index inside group    */
    int64_t byte = j / 4;       /* byte of the group's 32 bytes */
    int64_t s = j % 4;          /* 2-bit field inside that byte */
    return g * 128 + s * 32 + byte;
}

/*
 * x      float32 [M,K]  (the fp16 activations, widened exactly)
 * q      int8    [M,K]  natural order
 * S      float32 [M,G]
 * T      int32   [M,G]
 */
int pq2o_quantize(const float* x, int64_t M, int64_t K,
                  int8_t* q, float* S, int32_t* T) {
    if (M < 0 || K < 0 || K % 128 != 0) return PQ2O_BAD_SHAPE;
    int64_t G = K / 128;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < G; ++g) {
            const float* xg = x + m * K + g * 128;
            int8_t* qg = q + m * K + g * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float a = fabsf(xg[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            int32_t t = 0;
            for (int i = 0; i < 128; ++i) {
                int32_t v = 0;
                if (amax != 0.0f) {
                    float r = rintf(xg[i] / d);   /* default mode: half-even */
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    v = (int32_t)r;
                }
                qg[i] = (int8_t)v;
                t += v;
            }
            S[m * G + g] = (amax != 0.0f) ? d : 0.0f;
            T[m * G + g] = t;
        }
    }
    return PQ2O_OK;
}

/* q natural [M,K] -> qp plane-ordered [M,K]. */
int pq2o_plane_order(const int8_t* q, int64_t M, int64_t K, int8_t* qp) {
    if (M < 0 || K < 0 || K % 128 != 0) return PQ2O_BAD_SHAPE;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            qp[m * K + plane_pos(k)] = q[m * K + k];
    return PQ2O_OK;
}

/* qp plane-ordered [M,K] -> q natural [M,K]. */
int pq2o_natural_order(const int8_t* qp, int64_t M, int64_t K, int8_t* q) {
    if (M < 0 || K < 0 || K % 128 != 0) return PQ2O_BAD_SHAPE;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            q[m * K + k] = qp[m * K + plane_pos(k)];
    return PQ2O_OK;
}

/* ternary int8 [N,K] in {-1,0,1} -> codes uint8 [N,K/4]. */
int pq2o_pack(const int8_t* tern, int64_t N, int64_t K, uint8_t* codes) {
    if (N < 0 || K < 0 || K % 4 != 0) return PQ2O_BAD_SHAPE;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < K / 4; ++b) {
            unsigned byte = 0;
            for (int s = 0; s < 4; ++s) {
                int t = tern[n * K + 4 * b + s];
                if (t < -1 || t > 1) return PQ2O_BAD_VALUE;
                unsigned code = (unsigned)(t + 1);      /* -1,0,+1 -> 0,1,2 */
                byte |= code << (2 * s);
            }
            codes[n * (K / 4) + b] = (uint8_t)byte;
        }
    }
    return PQ2O_OK;
}

/* codes uint8 [N,K/4] -> code-1 as int8 [N,K] (code 3 reads as +2). */
int pq2o_unpack(const uint8_t* codes, int64_t N, int64_t K, int8_t* tern) {
    if (N < 0 || K < 0 || K % 4 != 0) return PQ2O_BAD_SHAPE;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            unsigned byte = codes[n * (K / 4) + k / 4];
            unsigned code = (byte >> (2 * (k % 4))) & 3u;
            tern[n * K + k] = (int8_t)((int)code - 1);
        }
    return PQ2O_OK;
}

static int code_at(const uint8_t* codes, int64_t K, int64_t n, int64_t k) {
    unsigned byte = codes[n * (K / 4) + k / 4];
    return (int)((byte >> (2 * (k % 4))) & 3u);
}

/* dots int32 [M,N,G]: sum over group g of (code-1)*q, natural order. */
int pq2o_group_dots(const int8_t* qp, const uint8_t* codes,
                    int64_t M, int64_t N, int64_t K, int32_t* dots) {
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0) return PQ2O_BAD_SHAPE;
    int64_t G = K / 128;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t g = 0; g < G; ++g) {
                int64_t acc = 0;
                for (int64_t k = g * 128; k < (g + 1) * 128; ++k) {
                    int64_t q = qp[m * K + plane_pos(k)];
                    int64_t t = code_at(codes, K, n, k) - 1;
                    acc += t * q;
                }
                dots[(m * N + n) * G + g] = (int32_t)acc;
            }
    return PQ2O_OK;
}

/* out int32 [M,N,G]: sum over group g of code*q (no offset), natural order. */
int pq2o_codes_dots(const int8_t* qp, const uint8_t* codes,
                    int64_t M, int64_t N, int64_t K, int32_t* out) {
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0) return PQ2O_BAD_SHAPE;
    int64_t G = K / 128;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t g = 0; g < G; ++g) {
                int64_t acc = 0;
                for (int64_t k = g * 128; k < (g + 1) * 128; ++k)
                    acc += (int64_t)code_at(codes, K, n, k) * qp[m * K + plane_pos(k)];
                out[(m * N + n) * G + g] = (int32_t)acc;
            }
    return PQ2O_OK;
}

/*
 * y  float64 [M,N] = sum_g dot_g * S[m,g] * WS[n,g]
 * A  float64 [M,N] = sum_g |dot_g * S[m,g] * WS[n,g]|   (may be NULL)
 * WS is given as float64 [N,G] (the fp16 group scales, widened exactly).
 * Rows n_begin..n_end-1 only (n_end <= N), so a caller can time a sample.
 */
int pq2o_matmul_rows(const int8_t* qp, const float* S, const uint8_t* codes,
                     const double* WS, int64_t M, int64_t N, int64_t K,
                     int64_t n_begin, int64_t n_end, double* y, double* A) {
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0) return PQ2O_BAD_SHAPE;
    if (n_begin < 0 || n_end > N || n_begin > n_end) return PQ2O_BAD_SHAPE;
    int64_t G = K / 128;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = n_begin; n < n_end; ++n)
        for (int64_t m = 0; m < M; ++m) {
            double sum = 0.0, mag = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                int64_t dot = 0;
                for (int64_t k = g * 128; k < (g + 1) * 128; ++k) {
                    int64_t q = qp[m * K + plane_pos(k)];
                    int64_t t = code_at(codes, K, n, k) - 1;
                    dot += t * q;
                }
                double term = (double)dot * (double)S[m * G + g] * WS[n * G + g];
                sum += term;
                mag += fabs(term);
            }
            y[m * N + n] = sum;
            if (A) A[m * N + n] = mag;
        }
    return PQ2O_OK;
}

int pq2o_matmul(const int8_t* qp, const float* S, const uint8_t* codes,
                const double* WS, int64_t M, int64_t N, int64_t K,
                double* y, double* A) {
    return pq2o_matmul_rows(qp, S, codes, WS, M, N, K, 0, N, y, A);
}

/*
 * Selected entries only: y[i] and A[i] for the pairs (ms[i], ns[i]),
 * i < count -- the same definition as pq2o_matmul_rows, evaluated one output
 * at a time, for checking full-size problems on a sample of outputs.
 */
int pq2o_matmul_entries(const int8_t* qp, const float* S, const uint8_t* codes,
                        const double* WS, int64_t M, int64_t N, int64_t K,
                        int64_t count, const int64_t* ms, const int64_t* ns,
                        double* y, double* A) {
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0 || count < 0) return PQ2O_BAD_SHAPE;
    int64_t G = K / 128;
    for (int64_t i = 0; i < count; ++i)
        if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return PQ2O_BAD_SHAPE;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = ms[i], n = ns[i];
        double sum = 0.0, mag = 0.0;
        for (int64_t g = 0; g < G; ++g) {
            int64_t dot = 0;
            for (int64_t k = g * 128; k < (g + 1) * 128; ++k) {
                int64_t q = qp[m * K + plane_pos(k)];
                int64_t t = code_at(codes, K, n, k) - 1;
                dot += t * q;
            }
            double term = (double)dot * (double)S[m * G + g] * WS[n * G + g];
            sum += term;
            mag += fabs(term);
        }
        y[i] = sum;
        if (A) A[i] = mag;
    }
    return PQ2O_OK;
}

/*
 * SwiGLU of the MLP's gate/up output, the activation between the two
 * projections of a decode MLP.  The pages do not define it, so it is an
 * assumed activation.  This oracle takes the plain reading:
 *   gate = gu[m, 0..I), up = gu[m, I..2I);  h = silu(gate) * up,
 *   silu(g) = g / (1 + exp(-g)),
 * every step one IEEE fp32 operation in this order (the caller rounds h to
 * fp16, saturating at +-65504, before quantising it).
 * exp is computed by a stated method rather than libm's expf, so that a
 * kernel that follows the same steps gets the same bits: Cody and Waite's
 * argument reduction (W. J. Cody, W. Waite, "Software Manual for the
 * Elementary Functions", 1980): n = rint(x log2 e), r = x - n ln2 with ln2
 * split in two fp32 parts (each subtraction one fused multiply-add), then the
 * degree-7 Taylor polynomial of e^r (coefficients 1/i!, Horner with fused
 * multiply-adds), then the exact scaling by 2^n.  x is clamped to [-87, 88]
 * first (e^x stays a normal fp32 number).
 */
static float pq2o_exp_cw(float x) {
    if (x < -87.0f) x = -87.0f;
    if (x > 88.0f) x = 88.0f;
    const float log2e = 0x1.715476p+0f;
    const float ln2_hi = 0x1.62e430p-1f;
    const float ln2_lo = -0x1.05c610p-29f;
    const float n = rintf(x * log2e);
    float r = fmaf(-n, ln2_hi, x);
    r = fmaf(-n, ln2_lo, r);
    float p = 0x1.a01a02p-13f;         /* 1/7! */
    p = fmaf(p, r, 0x1.6c16c2p-10f);   /* 1/6! */
    p = fmaf(p, r, 0x1.111112p-7f);    /* 1/5! */
    p = fmaf(p, r, 0x1.555556p-5f);    /* 1/4! */
    p = fmaf(p, r, 0x1.555556p-3f);    /* 1/3! */
    p = fmaf(p, r, 0x1.0p-1f);         /* 1/2! */
    p = fmaf(p, r, 1.0f);              /* 1/1! */
    p = fmaf(p, r, 1.0f);              /* 1/0! */
    return ldexpf(p, (int)n);          /* exact: the result is a normal number */
}

/* y[i] = the exp above, for the pin tests. */
int pq2o_exp(const float* x, int64_t count, float* y) {
    if (count < 0) return PQ2O_BAD_SHAPE;
    for (int64_t i = 0; i < count; ++i) y[i] = pq2o_exp_cw(x[i]);
    return PQ2O_OK;
}

/*
 * gu  float32 [M, 2I]  (gate | up)
 * h   float32 [M, I]   silu(gate) * up in fp32
 */
int pq2o_swiglu(const float* gu, int64_t M, int64_t I, float* h) {
    if (M < 0 || I < 0) return PQ2O_BAD_SHAPE;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < I; ++k) {
            const float g = gu[m * 2 * I + k];
            const float u = gu[m * 2 * I + I + k];
            const float e = pq2o_exp_cw(-g);
            const float s = g / (1.0f + e);
            h[m * I + k] = s * u;
        }
    return PQ2O_OK;
}
