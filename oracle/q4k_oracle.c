/*
 * q4k_oracle.c -- plain, slow, obviously-correct CPU oracle for the Q4_K
 * decode hot path.  TEST INFRASTRUCTURE ONLY: nothing in the product library
 * links, includes or calls this file; only the tests, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code with the CUDA path.
 *
 * What it computes (all sources are web pages on GGUF Q4_K_M inference):
 *   - "fused scale x int dot-product kernels operating directly on quantized
 *     blocks" (dotLLM README, Key Features / Performance).  Such a kernel is
 *     only a re-association of the plain product y = W_deq . x, so the oracle
 *     is that plain product: dequantize every weight, multiply, sum in fp64 in
 *     increasing k order.
 *   - the batched verification pass that streams the weights once for K+1
 *     tokens (Glacier.Inference article, section 4 "Beating Hardware Bandwidth
 *     Ceilings with Speculative Decoding"): the oracle simply evaluates every
 *     batch row independently.
 *   - the greedy argmax that emits one int32 token id per row (Glacier.Inference
 *     article, section 2 "Eliminating PCIe Starvation: In-VRAM Warp-Shuffle
 *     Argmax"): a scalar scan with a strict '>' so the lowest index wins ties.
 *   - the prefill product with bf16 activations ("cuBLAS HGEMM for prefill",
 *     dotLLM README, News 2026-03 "CUDA GPU backend"): same fp64 sum with the
 *     bf16 activations decoded exactly.
 *   - the Q6_K GEMV (dotLLM README, News 2026-03 "CUDA GPU backend": "custom
 *     quantized GEMV for decode (Q8_0, Q4_K, Q6_K)"): the same plain fp64
 *     product over the Q6_K weights, layout at oracle_q6k_dequant_block.
 *   - Q8_K activation quantization and the Q4_K x Q8_K product (dotLLM README,
 *     News 2026-03 "Mixed quantization + Q8_K"): the int8 codes and block
 *     scales by the rule written at oracle_q8k_quantize, then the same fp64
 *     sum over the dequantized activations.
 *
 * The Q4_K super-block (the pages name the format -- Q4_K / Q4_K_M -- but never
 * print its bytes; the reading used here is the GGUF packing):
 *   144 bytes hold 256 weights in 8 sub-blocks of 32.
 *   bytes 0-1   d     (IEEE binary16, little-endian)
 *   bytes 2-3   dmin  (IEEE binary16, little-endian)
 *   bytes 4-15  s[12] eight 6-bit scales sc_j and eight 6-bit mins m_j:
 *                 j < 4 : sc_j = s[j] & 63,  m_j = s[j+4] & 63
 *                 j >= 4: sc_j = (s[j+4] & 15) | ((s[j-4] >> 6) << 4)
 *                         m_j  = (s[j+4] >> 4) | ((s[j]   >> 6) << 4)
 *   bytes 16-143 qs[128]: for sub-block pair p = 0..3 and i = 0..31,
 *                 q[64p + i]      = qs[32p + i] & 15   (sub-block 2p)
 *                 q[64p + 32 + i] = qs[32p + i] >> 4   (sub-block 2p+1)
 *   weight 32j + i of the block:  w = d * sc_j * q - dmin * m_j
 *
 * Every value the oracle forms from a block (d*sc*q, dmin*m, their difference)
 * is exact in fp64 (at most 11+6+4 significant bits each), so the only
 * rounding in y is the fp64 accumulation.
 *
 * Threads: an optional OpenMP loop over independent rows; each row's sum is
 * still formed by one thread in k order, so the result does not depend on the
 * thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 256
#define QBYTES 144

/* IEEE binary16 -> double, from the bit fields (exact for every pattern). */
double oracle_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 (upper half of an IEEE binary32) -> double, exact. */
double oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 255;
    int f = b & 127;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);                /* f * 2^-7 * 2^-126 */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 134);     /* (1 + f/128) * 2^(e-127) */
    }
    return sign ? -v : v;
}

/* Round a double to the nearest bfloat16 value, ties to even, returned as a
 * double (finite inputs of normal bf16 range; used only by the diagnostic
 * prefill variant that shows how much error weight rounding contributes). */
double oracle_round_bf16(double v)
{
    if (v == 0.0 || !isfinite(v)) return v;
    int e;
    double f = frexp(v, &e);               /* v = f * 2^e, 0.5 <= |f| < 1 */
    double r = nearbyint(ldexp(f, 8));     /* 8 significant bits, ties-to-even */
    return ldexp(r, e - 8);
}

/* The 6-bit scale/min unpack of bytes 4..15 of a block. */
void oracle_unpack_scales(const uint8_t s[12], int sc[8], int m[8])
{
    for (int j = 0; j < 8; ++j) {
        if (j < 4) {
            sc[j] = s[j] & 63;
            m[j] = s[j + 4] & 63;
        } else {
            sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
            m[j] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
        }
    }
}

/* The 256 4-bit quants of a block, in weight order. */
void oracle_unpack_quants(const uint8_t qs[128], int q[256])
{
    for (int p = 0; p < 4; ++p) {
        for (int i = 0; i < 32; ++i) {
            q[64 * p + i] = qs[32 * p + i] & 15;
            q[64 * p + 32 + i] = qs[32 * p + i] >> 4;
        }
    }
}

/* w[32j+i] = d * sc_j * q[32j+i] - dmin * m_j  (exact in fp64). */
void oracle_dequant_block(const uint8_t blk[QBYTES], double w[QK])
{
    uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    uint16_t mbits = (uint16_t)(blk[2] | (blk[3] << 8));
    double d = oracle_fp16_to_double(dbits);
    double dmin = oracle_fp16_to_double(mbits);
    int sc[8], m[8], q[256];
    oracle_unpack_scales(blk + 4, sc, m);
    oracle_unpack_quants(blk + 16, q);
    for (int j = 0; j < 8; ++j)
        for (int i = 0; i < 32; ++i)
            w[32 * j + i] = d * (double)sc[j] * (double)q[32 * j + i] - dmin * (double)m[j];
}

/* Inverse of the unpack functions, for building hand-made test blocks. */
void oracle_pack_block(uint16_t d, uint16_t dmin, const int sc[8], const int m[8],
                       const int q[256], uint8_t out[QBYTES])
{
    memset(out, 0, QBYTES);
    out[0] = (uint8_t)(d & 255);
    out[1] = (uint8_t)(d >> 8);
    out[2] = (uint8_t)(dmin & 255);
    out[3] = (uint8_t)(dmin >> 8);
    uint8_t *s = out + 4;
    for (int j = 0; j < 4; ++j) {
        s[j] = (uint8_t)((sc[j] & 63) | (((sc[j + 4] >> 4) & 3) << 6));
        s[j + 4] = (uint8_t)((m[j] & 63) | (((m[j + 4] >> 4) & 3) << 6));
        s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
    uint8_t *qs = out + 16;
    for (int p = 0; p < 4; ++p)
        for (int i = 0; i < 32; ++i)
            qs[32 * p + i] = (uint8_t)((q[64 * p + i] & 15) | ((q[64 * p + 32 + i] & 15) << 4));
}

/* Dequantize row n of W (K weights) into buf. */
static void dequant_row(const uint8_t *W, int64_t n, int64_t K, double *buf)
{
    int64_t nb = K / QK;
    const uint8_t *row = W + n * nb * QBYTES;
    for (int64_t b = 0; b < nb; ++b) oracle_dequant_block(row + b * QBYTES, buf + b * QK);
}

static void set_threads(int threads)
{
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
}

/* Dense fp64 copy of the dequantized matrix, [N][K] row-major. */
void oracle_dequant_matrix(const uint8_t *W, int64_t N, int64_t K, double *out, int threads)
{
    set_threads(threads);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) dequant_row(W, n, K, out + n * K);
}

/* y[b][n] = sum_k w[n][k] * x[b][k]; x is fp32 [B][K], y fp64 [B][N]. */
void oracle_gemv(const uint8_t *W, const float *x, double *y, int64_t N, int64_t K, int B, int threads)
{
    set_threads(threads);
#pragma omp parallel
    {
        double *buf = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            dequant_row(W, n, K, buf);
            for (int b = 0; b < B; ++b) {
                const float *xb = x + (int64_t)b * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += buf[k] * (double)xb[k];
                y[(int64_t)b * N + n] = acc;
            }
        }
        free(buf);
    }
}

/* Same product for an explicit row subset (rows[r] -> y[b][r]), used to check
 * sampled outputs of very large matrices.  y is [B][R]. */
void oracle_gemv_rows(const uint8_t *W, const float *x, double *y, int64_t N, int64_t K, int B,
                      const int64_t *rows, int64_t R, int threads)
{
    (void)N;
    set_threads(threads);
#pragma omp parallel
    {
        double *buf = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            dequant_row(W, rows[r], K, buf);
            for (int b = 0; b < B; ++b) {
                const float *xb = x + (int64_t)b * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += buf[k] * (double)xb[k];
                y[(int64_t)b * R + r] = acc;
            }
        }
        free(buf);
    }
}

/*
 * Q8_K-style activation quantization.  The dotLLM README (News 2026-03, "Mixed
 * quantization + Q8_K") describes x quantized in 256-element blocks with a
 * float32 scale, int8 codes and precomputed block sums, feeding a fused
 * Q4_K x Q8_K GEMV.  It fixes the block size, the float32 scale and the int8
 * codes but no rounding rule; this oracle takes the plainest one, in fp32:
 *   a = max |x| over the block,  d = a / 127,
 *   q = rint(x * (127 / a))   (round half to even; |q| <= 127),
 * an all-zero block giving d = 0, q = 0.  When a < 2^-64 the same fp32 values
 * are formed as (x * 2^64) * (127 / (a * 2^64)), so that the reciprocal stays
 * finite for every finite x (scaling by 2^64 is exact).  Finite x only.
 */
void oracle_q8k_quantize(const float *x, int64_t K, int8_t *q, float *d)
{
    for (int64_t b = 0; b < K / QK; ++b) {
        const float *xb = x + b * QK;
        float a = 0.0f;
        for (int i = 0; i < QK; ++i) {
            const float v = fabsf(xb[i]);
            if (v > a) a = v;
        }
        d[b] = a / 127.0f;
        const float pre = (a < 0x1p-64f) ? 0x1p64f : 1.0f;
        const float inv = (a > 0.0f) ? 127.0f / (a * pre) : 0.0f;
        for (int i = 0; i < QK; ++i) {
            const float t = (xb[i] * pre) * inv;
            q[b * QK + i] = (int8_t)rintf(t);
        }
    }
}

/* y[n] = sum_k w[n][k] * (d_{k/256} * q[k]) in fp64, k order: the product of
 * the dequantized weights with the dequantized Q8_K activations (batch 1). */
void oracle_gemv_q8k(const uint8_t *W, const int8_t *q, const float *d, double *y, int64_t N, int64_t K,
                     int threads)
{
    set_threads(threads);
#pragma omp parallel
    {
        double *buf = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            dequant_row(W, n, K, buf);
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += buf[k] * ((double)d[k / QK] * (double)q[k]);
            y[n] = acc;
        }
        free(buf);
    }
}

/*
 * Q6_K, the other block format of Q4_K_M files ("custom quantized GEMV for
 * decode (Q8_0, Q4_K, Q6_K)", dotLLM README, News 2026-03 "CUDA GPU
 * backend"; the pages print no bytes, the reading used here is the GGUF Q6_K
 * packing):  210 bytes hold 256 weights in 16 sub-blocks of 16.
 *   bytes   0..127  ql[128]  low 4 bits of the 6-bit codes
 *   bytes 128..191  qh[64]   high 2 bits of the codes
 *   bytes 192..207  sc[16]   int8 scale of each 16 weights
 *   bytes 208..209  d        IEEE binary16, little-endian
 * For weight k = 128 h + 32 c + l  (h < 2, c < 4, l < 32):
 *   low  = ql[64 h + 32 (c & 1) + l]: its low nibble when c < 2, else its high
 *   high = (qh[32 h + l] >> (2 c)) & 3
 *   q = low + 16 high  (0..63),   w = d * sc[k / 16] * (q - 32)
 * (d * sc * (q - 32) has at most 11 + 8 + 6 significant bits: exact in fp64.)
 */
#define Q6BYTES 210

void oracle_q6k_dequant_block(const uint8_t blk[Q6BYTES], double w[QK])
{
    const uint8_t *ql = blk, *qh = blk + 128;
    const int8_t *sc = (const int8_t *)(blk + 192);
    const double d = oracle_fp16_to_double((uint16_t)(blk[208] | (blk[209] << 8)));
    for (int k = 0; k < QK; ++k) {
        const int h = k / 128, c = (k % 128) / 32, l = k % 32;
        const int byte = ql[64 * h + 32 * (c & 1) + l];
        const int low = (c < 2) ? (byte & 15) : (byte >> 4);
        const int high = (qh[32 * h + l] >> (2 * c)) & 3;
        const int q = low + 16 * high;
        w[k] = d * (double)sc[k / 16] * (double)(q - 32);
    }
}

static void q6k_dequant_row(const uint8_t *W, int64_t n, int64_t K, double *buf)
{
    const int64_t nb = K / QK;
    for (int64_t b = 0; b < nb; ++b) oracle_q6k_dequant_block(W + (n * nb + b) * Q6BYTES, buf + b * QK);
}

/* y[b][n] = sum_k w[n][k] * x[b][k] for a Q6_K matrix; x fp32 [B][K], y fp64 [B][N]. */
void oracle_q6k_gemv(const uint8_t *W, const float *x, double *y, int64_t N, int64_t K, int B, int threads)
{
    set_threads(threads);
#pragma omp parallel
    {
        double *buf = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            q6k_dequant_row(W, n, K, buf);
            for (int b = 0; b < B; ++b) {
                const float *xb = x + (int64_t)b * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += buf[k] * (double)xb[k];
                y[(int64_t)b * N + n] = acc;
            }
        }
        free(buf);
    }
}

/* The same for an explicit row subset (rows[r] -> y[b][r]); y is [B][R]. */
void oracle_q6k_gemv_rows(const uint8_t *W, const float *x, double *y, int64_t K, int B, const int64_t *rows,
                          int64_t R, int threads)
{
    set_threads(threads);
#pragma omp parallel
    {
        double *buf = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            q6k_dequant_row(W, rows[r], K, buf);
            for (int b = 0; b < B; ++b) {
                const float *xb = x + (int64_t)b * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += buf[k] * (double)xb[k];
                y[(int64_t)b * R + r] = acc;
            }
        }
        free(buf);
    }
}

/* Greedy argmax: the first index holding the largest value (strict '>' scan).
 * NaN never wins; an all-NaN (or empty) row gives 0.  -0.0 and +0.0 compare
 * equal, so the lower index wins between them. */
int64_t oracle_argmax_f64(const double *v, int64_t n)
{
    int64_t best = -1;
    for (int64_t i = 0; i < n; ++i) {
        if (isnan(v[i])) continue;
        if (best < 0 || v[i] > v[best]) best = i;
    }
    return best < 0 ? 0 : best;
}

int64_t oracle_argmax_f32(const float *v, int64_t n)
{
    int64_t best = -1;
    for (int64_t i = 0; i < n; ++i) {
        if (isnan(v[i])) continue;
        if (best < 0 || v[i] > v[best]) best = i;
    }
    return best < 0 ? 0 : best;
}

/* Prefill: Y[t][n] = sum_k w[n][k] * X[t][k], X given as bf16 bit patterns
 * [T][K], Y fp64 [T][N].  round_w != 0 rounds every weight to bf16 first (a
 * diagnostic of the weight-rounding share of the error, not the reference). */
void oracle_prefill(const uint8_t *W, const uint16_t *X, double *Y, int64_t N, int64_t K, int64_t T,
                    int round_w, int threads)
{
    set_threads(threads);
    double *Xd = (double *)malloc((size_t)(T * K) * sizeof(double));
    for (int64_t i = 0; i < T * K; ++i) Xd[i] = oracle_bf16_to_double(X[i]);
#pragma omp parallel
    {
        double *buf = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            dequant_row(W, n, K, buf);
            if (round_w)
                for (int64_t k = 0; k < K; ++k) buf[k] = oracle_round_bf16(buf[k]);
            for (int64_t t = 0; t < T; ++t) {
                const double *xt = Xd + t * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += buf[k] * xt[k];
                Y[t * N + n] = acc;
            }
        }
        free(buf);
    }
    free(Xd);
}

/* Processors available to this process (not the current OpenMP thread
 * count, which a call with threads > 0 changes). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_num_procs();
#else
    return 1;
#endif
}
