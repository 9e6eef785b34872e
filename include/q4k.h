/*
 * q4k.h -- C ABI of the GB300 (sm_103a) Q4_K decode library.
 *
 * The library computes the memory-bound decode products of a GGUF Q4_K_M
 * engine directly on 4-bit block-quantized weights:
 *   - q4k_gemv         y = W x for one token or a small batch of tokens
 *                      ("custom quantized GEMV for decode (Q8_0, Q4_K, Q6_K)"
 *                      with "on-the-fly weight dequantization", dotLLM README,
 *                      News 2026-03 "CUDA GPU backend"; the batch form is the
 *                      VerifyBatch pass of the Glacier.Inference article,
 *                      section 4 "Beating Hardware Bandwidth Ceilings with
 *                      Speculative Decoding": one weight read for K+1 tokens)
 *   - q4k_gemv_argmax  the LM-head product fused with a greedy argmax that
 *                      writes one int32 token id per batch row (Glacier.Inference
 *                      article, section 2 "Eliminating PCIe Starvation: In-VRAM
 *                      Warp-Shuffle Argmax")
 *   - q4k_gemm_prefill the prefill product with bf16 activations ("cuBLAS HGEMM
 *                      for prefill", dotLLM README, News 2026-03), here on the
 *                      tcgen05 tensor cores after a dequantize-to-fp16 step
 *                      (q4k_gemm_prefill_exact: the same with exact integer
 *                      weight tiles).
 *   - q6k_gemv         y = W x for a Q6_K matrix, the other block format of
 *                      Q4_K_M files ("custom quantized GEMV for decode (Q8_0,
 *                      Q4_K, Q6_K)", same page and item); q6k_repack_planar
 *                      and q6k_gemv_planar: the same product on a copy of
 *                      the matrix split into aligned planes once, at load
 *                      time (the dotLLM README repacks its weights at model
 *                      load time too: News 2026-03, the R4 row interleave).
 *
 * ---------------------------------------------------------------------------
 * Q4_K super-block (144 bytes, 256 weights, 4.5 bits per weight)
 * ---------------------------------------------------------------------------
 * The pages name the format (Q4_K, Q4_K_M) but print no byte layout; this
 * library fixes the GGUF Q4_K packing:
 *   bytes   0..1   d     IEEE binary16, little-endian (super-block scale)
 *   bytes   2..3   dmin  IEEE binary16, little-endian (super-block min scale)
 *   bytes   4..15  s[12] eight 6-bit scales sc_j and eight 6-bit mins m_j:
 *                    j < 4 : sc_j = s[j] & 63,  m_j = s[j+4] & 63
 *                    j >= 4: sc_j = (s[j+4] & 15) | ((s[j-4] >> 6) << 4)
 *                            m_j  = (s[j+4] >> 4) | ((s[j]   >> 6) << 4)
 *   bytes  16..143 qs[128] 4-bit quants; for p = 0..3 and i = 0..31:
 *                    q[64p + i]      = qs[32p + i] & 15   (sub-block 2p)
 *                    q[64p + 32 + i] = qs[32p + i] >> 4   (sub-block 2p+1)
 *   weight 32j + i of the block:   w = d * sc_j * q[32j+i] - dmin * m_j
 *
 * A matrix W of N rows and K columns (K a positive multiple of 256) is stored
 * row-major as N rows of K/256 consecutive super-blocks: row n starts at byte
 * n * (K/256) * 144.  Every row therefore starts on a 16-byte boundary when W
 * does.
 *
 * ---------------------------------------------------------------------------
 * Conventions for every entry point
 * ---------------------------------------------------------------------------
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     never frees or retains them.  Calls are asynchronous on `stream` (a
 *     cudaStream_t passed as void*; NULL is the legacy default stream) and
 *     never synchronize the host.
 *   - Outputs are overwritten, never accumulated.  Inputs and outputs must not
 *     overlap.
 *   - Argument errors are detected on the host before anything is launched and
 *     returned as a status; Q4K_ERR_CUDA reports a launch failure (the CUDA
 *     error is left for cudaGetLastError to clear).
 *   - x and X are read only inside the kernels; they may be produced by the
 *     kernel that ran just before on the same stream.
 */
#ifndef Q4K_H
#define Q4K_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q4K_BLOCK_WEIGHTS 256
#define Q4K_BLOCK_BYTES 144
#define Q4K_MAX_BATCH 16
#define Q4K_ABI_VERSION 1

typedef enum {
    Q4K_OK = 0,
    Q4K_ERR_INVALID_ARG = 1,        /* null pointer, bad size or batch */
    Q4K_ERR_MISALIGNED = 2,         /* a pointer is not 16-byte aligned */
    Q4K_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
    Q4K_ERR_CUDA = 4                /* a CUDA call or a launch failed */
} q4k_status;

/* Human-readable text of a status (static storage, never NULL). */
const char *q4k_status_string(q4k_status s);

/* Q4K_ABI_VERSION of the loaded library. */
int q4k_abi_version(void);

/*
 * y[b][n] = sum_k w[n][k] * x[b][k]   for b < batch, n < N.
 *   W     uint8  [N][K/256*144]  Q4_K rows (layout above), 16-byte aligned
 *   x     fp32   [batch][K]      row-major, 16-byte aligned
 *   y     fp32   [batch][N]      row-major
 *   N >= 0 (N == 0 is a no-op and W, y may then be NULL), K a positive multiple
 *   of 256, K/256 < 2^24, 1 <= batch <= 16.
 * Accumulation is fp32.  Each weight super-block is read from memory once for
 * all batch rows.  x may hold any finite fp32 values.  Inside, each
 * super-block of x is carried in one of two forms:
 *   - batch 1: two int8 parts, x ~= (a/32258)(254 xh + xl) with a = max|x| of
 *     the super-block (error <= a (1/64516 + 2^-16)); the weight nibbles are
 *     multiplied with them by integer dot products (dp4a), exact in int32,
 *     and the scales applied per super-block in fp32;
 *   - batch >= 2 (and batch 1 with Q4K_FLAG_TENSOR_CORE): two fp16 parts after
 *     a power-of-two scale (error <= 2^-22 |x|), multiplied with the weights as
 *     exact fp16 integers on the tensor cores (mma.sync), fp32 accumulation.
 * Errors: INVALID_ARG (null pointer, N < 0, K <= 0 or K % 256 != 0, batch out
 * of range), MISALIGNED (W or x), UNSUPPORTED_DEVICE, CUDA.
 */
q4k_status q4k_gemv(const void *W, const float *x, float *y, int64_t N, int64_t K, int batch,
                    void *stream);

/*
 * idx[b] = the smallest n with y[b][n] == max_n' y[b][n'], where y = W x is the
 * product q4k_gemv computes (the very same fp32 values).  NaN never wins; a row
 * whose values are all NaN gives 0; -0.0 and +0.0 compare equal.  No logits
 * leave the device: the only output is batch int32 values.
 *   idx   int32 [batch]
 *   1 <= N <= 2^31 - 1; other arguments as for q4k_gemv.
 * Scratch: 144 bytes taken from the stream-ordered allocator (cudaMallocAsync,
 * cleared with cudaMemsetAsync, released with cudaFreeAsync, all on `stream`),
 * so concurrent calls on different streams are independent.
 */
q4k_status q4k_gemv_argmax(const void *W, const float *x, int32_t *idx, int64_t N, int64_t K,
                           int batch, void *stream);

/*
 * Same as q4k_gemv_argmax, and also writes the logits it reduced to
 * `logits` (fp32 [batch][N]); meant for tests that check the argmax bit for bit
 * against a scan of the very values the kernel compared.
 */
q4k_status q4k_gemv_argmax_debug(const void *W, const float *x, int32_t *idx, float *logits,
                                 int64_t N, int64_t K, int batch, void *stream);

/*
 * Allocation-free q4k_gemv_argmax.  (No counterpart on the pages: this is an
 * interface choice of this library.)  Same arguments, same result bit for bit.
 * Meant for callers that must not allocate device memory while they run --
 * code working from a fixed, pre-sized memory budget, real-time loops that
 * forbid allocator calls, or processes whose stream-ordered allocator is
 * unavailable or replaced.  Instead of cudaMallocAsync it uses a static device
 * array of 16 keys + a ticket (144 bytes) that every GPU loading the library
 * keeps until the process exits.
 *   - batch must be <= 16 (the array's capacity); larger batches return
 *     Q4K_ERR_INVALID_ARG.
 *   - The array's device address is looked up (cudaGetSymbolAddress) on the
 *     first call on a device and on every call made outside stream capture;
 *     a call made during capture reuses the last address looked up, so make a
 *     first call on each device before any stream capture (and again after a
 *     cudaDeviceReset, which may move the array).
 *   - Each call clears the array with cudaMemsetAsync on `stream` before its
 *     kernel.  All calls share the array: calls that overlap on the GPU
 *     (different streams, concurrently running graphs) race and may return
 *     wrong indices.  Serialize them.
 *   - Allocates nothing: no cudaMalloc, cudaMallocAsync or cudaFree.
 */
q4k_status q4k_gemv_argmax_noalloc(const void *W, const float *x, int32_t *idx, int64_t N, int64_t K,
                                   int batch, void *stream);

/*
 * ---------------------------------------------------------------------------
 * Q6_K super-block (210 bytes, 256 weights, 6.5625 bits per weight), the other
 * block format of Q4_K_M files ("custom quantized GEMV for decode (Q8_0, Q4_K,
 * Q6_K)", dotLLM README, News 2026-03 "CUDA GPU backend").  The pages print no
 * bytes; this library fixes the GGUF Q6_K packing:
 *   bytes   0..127  ql[128] low 4 bits of the 6-bit codes
 *   bytes 128..191  qh[64]  high 2 bits of the codes
 *   bytes 192..207  sc[16]  int8 scale of each 16 weights
 *   bytes 208..209  d       IEEE binary16, little-endian
 *   weight k = 128h + 32c + l (h < 2, c < 4, l < 32):
 *     low  = ql[64h + 32(c & 1) + l], its low nibble for c < 2, high for c >= 2
 *     high = (qh[32h + l] >> 2c) & 3,   q = low + 16 high (0..63)
 *     w = d * sc[k / 16] * (q - 32)
 * Rows hold K/256 consecutive blocks (row n at byte n * (K/256) * 210); blocks
 * are therefore only 2-byte aligned.
 * ---------------------------------------------------------------------------
 * y[b][n] = sum_k w[n][k] * x[b][k] for a Q6_K matrix W, b < batch, n < N.
 *   W uint8 [N][K/256*210] (16-byte aligned), x fp32 [batch][K] (16-byte
 *   aligned), y fp32 [batch][N]; N >= 0 (0: no-op), K a positive multiple of
 *   256, 1 <= batch <= 16.  Each block is read once for all batch rows;
 *   deterministic.  For batch <= 4 and K <= 4096, whole 8-row tiles take an
 *   integer inner product: x enters per 256-block as two int8 parts
 *   (x ~ (a/32258)(254 xh + xl), a = the block's max |x|, error <=
 *   a (1/64516 + 2^-16) per element), the weight codes meet them in exact
 *   int32 dot products and the scales in fp32; the other rows and shapes
 *   multiply in fp32.  Both stay far inside the stated tolerance.
 * Errors: INVALID_ARG, MISALIGNED (W or x), UNSUPPORTED_DEVICE, CUDA.
 */
q4k_status q6k_gemv(const void *W, const float *x, float *y, int64_t N, int64_t K, int batch, void *stream);

/*
 * Planar Q6_K: the bytes of a Q6_K matrix regrouped so that every block's
 * codes and scales start on a 16-byte boundary (GGUF blocks are only 2-byte
 * aligned), for the GEMV below.  For N rows and nb = K/256 blocks per row,
 * with DP = 2*nb rounded up to a multiple of 16, the planar buffer holds
 *   QS  [N][nb][208]  bytes 0..207 of each block (ql, qh, sc), unchanged
 *   D   [N][DP]       d of block j at bytes 2j, 2j+1 of the row; the rest 0
 * QS at byte 0 and D at byte N*nb*208, q6k_planar_bytes(N, K) =
 * N * (nb*208 + DP) bytes in all (2940 + 4 bytes per row for K = 3584).  The
 * weights it encodes are exactly those of the GGUF matrix.  Returns -1 for
 * N < 0 or K not a positive multiple of 256.
 */
int64_t q6k_planar_bytes(int64_t N, int64_t K);

/*
 * Wp = the planar form of the Q6_K matrix W (above).  W uint8 [N][K/256*210]
 * (16-byte aligned); Wp device memory of q6k_planar_bytes(N, K) bytes
 * (16-byte aligned), not overlapping W; asynchronous on stream.  N >= 0 (0:
 * no-op), K a positive multiple of 256.  Errors: INVALID_ARG, MISALIGNED,
 * UNSUPPORTED_DEVICE, CUDA.
 */
q4k_status q6k_repack_planar(const void *W, void *Wp, int64_t N, int64_t K, void *stream);

/*
 * y = W x as q6k_gemv computes it, from the planar form Wp of W: the same
 * arguments, with Wp (q6k_planar_bytes(N, K) bytes, 16-byte aligned) in place
 * of W.  Every block is read once for all batch rows.  The planes stream into
 * shared memory as 2-D TMA boxes of 128 rows (one block per stage), so each
 * thread reads its codes, scales and d with 16-byte loads; x enters per
 * 256-block as the two int8 parts of q6k_gemv's integer path and the codes
 * meet them in exact int32 dot products (batch rows 1..8 per launch; larger
 * batches take one launch per eight rows).  Deterministic; K splits over the
 * CTAs of a cluster add their partial rows in rank order.
 * Errors: INVALID_ARG, MISALIGNED (Wp or x), UNSUPPORTED_DEVICE, CUDA.
 */
q4k_status q6k_gemv_planar(const void *Wp, const float *x, float *y, int64_t N, int64_t K, int batch,
                           void *stream);

/*
 * Y[t][n] = sum_k w[n][k] * X[t][k]   for t < T, n < N (prefill).
 *   W  Q4_K rows as above (16-byte aligned)
 *   X  bf16 [T][K] row-major (16-byte aligned)
 *   Y  fp32 [T][N] row-major
 * Up to 32 tokens this is q4k_gemm_prefill_exact (below: no weight is
 * rounded).  Above that each weight is dequantized in fp32 (one fma),
 * multiplied by a power of two chosen per row from the row's largest possible
 * |w|, and rounded to fp16 (nearest even) in shared memory; each token's
 * activations are converted to fp16
 * under a power of two chosen per token from its largest |x| (exact for every
 * value of at least 2^-31 times that largest).  The tcgen05 tensor cores
 * multiply them with fp32 accumulation in tensor memory and the epilogue
 * removes both scales.  Result: |Y - exact| <= ~2^-11 sum_k |w||x| for any
 * finite inputs, no overflow from large d, dmin or x.
 * Scratch: the converted X (2*T*K bytes), T scale exponents and, up to 32
 * tokens, T*K/2 bytes of sub-block sums come from cudaMallocAsync on `stream`
 * and are freed on it after the product.
 * Any T >= 0 is accepted (T == 0 or N == 0 is a no-op, and the pointers may
 * then be NULL); tokens go in tiles of 32 (T <= 32), 64 (T <= 64), 128, 256
 * or 512.
 * Errors: INVALID_ARG, MISALIGNED (W or X), UNSUPPORTED_DEVICE, CUDA
 * (including a failed scratch allocation).
 */
q4k_status q4k_gemm_prefill(const void *W, const void *X_bf16, float *Y, int64_t N, int64_t K,
                            int64_t T, void *stream);

/*
 * The same product with no weight rounding at all (arguments, layouts, errors
 * and scratch as q4k_gemm_prefill, plus T*K/2 bytes of scratch for the
 * sub-block sums of X).  The weight tiles hold q * sc_j, an integer of at most
 * 945 that fp16 represents exactly; the tensor cores accumulate
 * D = sum (q sc) x per super-block in tensor memory, one more MMA forms
 * M = sum_j m_j S_j from the sub-block sums S_j of the fp16 X (split into fp16
 * hi + lo), and y += d D - dmin M in fp32.  The only roundings are the fp32
 * accumulations and the hi + lo split of S_j.  Tiles of 32 (T <= 32) or 64
 * tokens; any T >= 0.  q4k_gemm_prefill takes this path up to 32 tokens;
 * from 33 tokens on the fp16 path is faster (14336 x 4096 at 64 tokens: 35.2
 * against 44.2 us), so this entry point is for callers that want the weights
 * exact there too.
 */
q4k_status q4k_gemm_prefill_exact(const void *W, const void *X_bf16, float *Y, int64_t N, int64_t K,
                                  int64_t T, void *stream);

/*
 * Extended launch control (tests and benchmarks).  Zero-initialised options
 * reproduce the plain entry points exactly.
 *   split_k  0 = automatic (up to 16 CTAs per tile for batch <= 8, when all
 *            clusters fit on the GPU at once); 1 <= s <= 8 forces the K range
 *            of every row tile to be split over s cooperating CTAs of a
 *            thread-block cluster (clamped to K/256).
 *   flags    Q4K_FLAG_PDL: launch with programmatic dependent launch, so the
 *            kernel may start streaming W while the previous kernel on the
 *            stream is still running.  W must then not be written by that
 *            previous kernel (weights are constant during decode); x is still
 *            read only after the previous kernel has completed.
 *            Q4K_FLAG_TENSOR_CORE: batch 1 uses the tensor-core inner product
 *            of the larger batches instead of the integer one.
 *            Q4K_FLAG_Q8K_X: batch 1 with x quantized Q8_K style (dotLLM README,
 *            News 2026-03 "Mixed quantization + Q8_K": 256-element blocks, a
 *            float32 scale, int8 codes, precomputed block sums): per block
 *            a = max|x|, d = a/127, q = rint(x * (127/a)) in fp32 (round half
 *            to even); the result is the product of W with d*q (exact integer
 *            dot products, fp32 per block), so it differs from W x by at most
 *            sum_k |w_k| d/2 per row -- its own tolerance, not the one stated
 *            for q4k_gemv.  Returns Q4K_ERR_INVALID_ARG with batch > 1 or
 *            together with Q4K_FLAG_TENSOR_CORE.
 *            Q4K_FLAG_TEST_STALL (failure-path tests only): the first weight
 *            copy of every CTA is awaited for 16 bytes more than it brings, so
 *            that every wait on it runs out.  The kernel then does what it does
 *            after any timed-out wait: sets bit 0 of q4k_device_error_flags(),
 *            stops waiting, writes no outputs, waits (bounded) for its own
 *            copies in flight and returns; the context stays usable.
 *            Q4K_FLAG_ROWS16: batch 1 on the 16-row-tile kernel (a CTA owns 16
 *            rows over the whole K; its warps split K and add their partial
 *            rows in shared memory, in warp order).  Without the flag the
 *            library takes it by itself for batch 1 when 128-row tiles would
 *            need a K split over CTAs and K <= 8192 (the q/k/v and o
 *            projections of a 7B-class layer); a forced split_k keeps the
 *            128-row kernel.  INVALID_ARG with batch > 1, with
 *            Q4K_FLAG_TENSOR_CORE or with K > 8192.
 *   wait_limit_us  bound of each wait inside the kernel in microseconds;
 *            0 = the default of 2 s.
 */
#define Q4K_FLAG_PDL 1u
#define Q4K_FLAG_TENSOR_CORE 2u
#define Q4K_FLAG_Q8K_X 4u
#define Q4K_FLAG_TEST_STALL 8u
#define Q4K_FLAG_ROWS16 16u
typedef struct {
    int split_k;
    unsigned flags;
    unsigned wait_limit_us;
    int reserved[5];
} q4k_launch_opts;

q4k_status q4k_gemv_ex(const void *W, const float *x, float *y, int64_t N, int64_t K, int batch,
                       void *stream, const q4k_launch_opts *opts);

/*
 * Fused dispatch: up to 4 matrices that multiply the same x (the q/k/v
 * projections of a layer, or its gate/up pair) in one launch, each with its
 * own output.  Same numbers as calling q4k_gemv per matrix with the same
 * split (the row tiles of all matrices share one grid, so the automatic split
 * may differ from the per-matrix one).  The dotLLM README lists this fusion
 * for its CPU decode (News 2026-03 "Fused decode dispatch": Q/K/V 3->1,
 * Gate/Up 2->1).
 *   groups[g].W  Q4_K [N_g][K/256*144] (16-byte aligned), groups[g].y fp32
 *   [batch][N_g]; every matrix has the same K; 1 <= ngroups <= 4; opts may be
 *   NULL.  A matrix with N_g == 0 is skipped.
 */
typedef struct {
    const void *W;
    float *y;
    int64_t N;
} q4k_gemv_group;

q4k_status q4k_gemv_grouped(const q4k_gemv_group *groups, int ngroups, const float *x, int64_t K,
                            int batch, void *stream, const q4k_launch_opts *opts);

/*
 * Read-only streaming probe (a measurement aid; no counterpart on the pages):
 * streams the first *bytes_read bytes of buf from device memory into shared
 * memory the way the GEMV kernels stream their weights -- one CTA per SM,
 * each reading a contiguous slice with 32 KB bulk asynchronous copies through
 * a 4-deep ring -- and discards them.  Timing it gives the read-only HBM rate
 * that bounds the GEMVs (a copy's read+write rate is lower).  *bytes_read is
 * bytes rounded down to a whole number of 32 KB chunks per SM (0 when bytes
 * is smaller).  buf: device pointer, 16-byte aligned; asynchronous on stream.
 * Errors: INVALID_ARG (bytes < 0, null buf or bytes_read), MISALIGNED,
 * UNSUPPORTED_DEVICE, CUDA.
 */
q4k_status q4k_stream_read(const void *buf, int64_t bytes, int64_t *bytes_read, void *stream);

/* Launch plan the automatic heuristics pick for a shape (for tests and
 * reports): out[0] = split_k, out[1] = number of CTAs, out[2] = rows per CTA
 * tile, out[3] = K blocks per x chunk held in shared memory. */
q4k_status q4k_gemv_plan(int64_t N, int64_t K, int batch, int out[4]);

/* Sticky device-side error bits of the library's kernels, read synchronously
 * from the current device: bit 0 = a bounded wait inside a GEMV/argmax
 * kernel (Q4_K or Q6_K) or the streaming probe timed out, bit 1 = the same in the prefill
 * kernel; the kernel then wound down early and its outputs are invalid.
 * 0 = no error.  The bits stay set until q4k_device_error_clear(). */
unsigned int q4k_device_error_flags(void);

/* Reset the sticky error bits on the current device (synchronous; call it
 * when no kernel of the library is running).  Q4K_ERR_CUDA if a copy to the
 * device failed. */
q4k_status q4k_device_error_clear(void);

#ifdef __cplusplus
}
#endif

#endif /* Q4K_H */
