// q6k_planar.cu -- Q6_K decode GEMV on the planar form of the weights
// (q6k_repack_planar, q6k_gemv_planar).
//
// What is computed: y[b] = W x[b] for a Q6_K matrix W (GGUF packing, written
// out in include/q4k.h), the other block format of Q4_K_M files ("custom
// quantized GEMV for decode (Q8_0, Q4_K, Q6_K)", dotLLM README, News 2026-03
// "CUDA GPU backend").  The weights are those of the GGUF matrix; only their
// bytes are regrouped once, at load time, so that each block's 208 bytes of
// codes and scales start on a 16-byte boundary and its d sits in a plane of
// its own (the dotLLM README repacks weights at model load time as well: News
// 2026-03, the R4 row interleave).
//
// Design (GB300):
//   * The QS plane ([N][nb][208]) streams HBM -> shared memory as 2-D TMA
//     boxes of one block of 128 rows (26 KB), with the rows' d values of the
//     block's group of eight (a 16-byte box of the D plane) in the same stage,
//     through a 3-stage ring guarded by mbarriers.  As in the Q4_K kernel
//     there is no producer warp: the last warp to leave a slot refills it.
//   * The 208-byte row stride in shared memory spreads the eight rows that a
//     quarter-warp reads over all 32 banks (16-byte chunk 13 g + c of row g),
//     so every code, qh and scale load is one 16-byte (or 8-byte) access.
//   * Thread (g, t) of warp w: rows 16w + g and 16w + g + 8, part t of each
//     block = the 64 weights 128h + 32c + l, h = t/2, c = 0..3,
//     l in [16(t%2), 16(t%2) + 16): 16 ql bytes for c = 0 and 2, 16 for c = 1
//     and 3, 16 qh bytes, and the four int8 scales of those sub-blocks.  Four
//     6-bit codes per 32-bit word are assembled with a few LOP3/shifts.
//   * x enters per block as two int8 parts per element against the block's
//     max |x| (x ~ (a/32258)(254 xh + xl), as in the Q4_K integer path); the
//     codes meet them in exact int32 dot products (dp4a), the -32 offset
//     through per-16 sums of the parts, the scales and d in fp32.
//   * Few row tiles: the K range splits over the CTAs of a cluster (up to 8)
//     and the partial rows are added in rank order through distributed shared
//     memory (deterministic).  Otherwise CTAs loop over row tiles.
//   * Batch rows 1..8 per launch (the dp4a work grows with each row).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "ptx.cuh"
#include "q4k_internal.h"

namespace q4k {
namespace q6p {

constexpr int kQsBytes = 208;                 // ql, qh, sc of a block
constexpr int kRows = 128;                    // rows per tile
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 3;
constexpr int kQsStage = kRows * kQsBytes;    // 26,624
constexpr int kDStage = kRows * 16;           // 2,048: d of 8 blocks per row
constexpr int kStageBytes = kQsStage + kDStage;   // 28,672 (a multiple of 1024)
constexpr int kPreWait = 1;                   // stages issued before the dependency wait
constexpr int kXItem = 576;                   // x of one (batch row, block): xh[256], xl[256], sums[16]
constexpr int kMaxItems = 40;                 // x items held at once (per chunk); two CTAs per SM
constexpr int kRedRows = kRows + 16;          // split-K receive rows (one slot per source rank)
constexpr int kMaxSplit = 8;
constexpr int kMaxB = 8;                      // batch rows per launch
constexpr size_t kSmemBytes = static_cast<size_t>(kStages) * kStageBytes + static_cast<size_t>(kMaxItems) * kXItem +
                              static_cast<size_t>(kRedRows) * kMaxB * 4;
// two CTAs per SM: (dynamic + 1 KB static + 1 KB reserved) x 2 <= 228 KB
static_assert(2 * (kSmemBytes + 2048) <= 228 * 1024, "two CTAs per SM");
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

__device__ unsigned int g_q6p_error = 0;   // bit 0: a bounded wait timed out

// ---------------------------------------------------------------------------
// One (batch row, block) of x -> its two int8 parts and per-16 sums at base,
// by one warp.  v0, v1 = float4 number lane and lane + 32 of the block (k =
// 4 lane .. + 3 and 128 + 4 lane .. + 3).  With a = max |x| of the block and
// q = x (127/a) in fp32: xh = rint(q), xl = rint((q - xh) 254) (ties to even,
// by adding and removing 1.5 * 2^23), so x ~ (a/32258)(254 xh + xl).  Layout:
//   [0, 256)    xh in k order
//   [256, 512)  xl in k order
//   [512, 576)  int32 sums 254 sum(xh) + sum(xl) over the 16 k of sub-block
//               j = 8h + 2c + p, stored at index 4(2h + p) + c (the four
//               sums a thread of part t = 2h + p reads with one load)
// Returns {unscale, pre} with unscale * pre = a / 32258 (a and x first scaled
// by 2^64 when a < 2^-64, pre = 2^-64 then); unscale = 0 for an all-zero
// block and the non-finite max itself when x holds an inf or NaN.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 x_item(float4 v0, float4 v1, int lane, uint8_t *base)
{
    uint32_t m = 0u;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const float4 w = h2 ? v1 : v0;
        m = max(m, max(max(__float_as_uint(fabsf(w.x)), __float_as_uint(fabsf(w.y))),
                       max(__float_as_uint(fabsf(w.z)), __float_as_uint(fabsf(w.w)))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float amax = __uint_as_float(m);
    const bool ok = m != 0u && m < 0x7F800000u;
    const float pre = (m < 0x1F800000u) ? 0x1p64f : 1.0f;
    const float inv = ok ? 127.0f / (amax * pre) : 0.0f;
    constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23
    constexpr uint32_t kMagicBits = 0x4B400000u;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const float4 w = h2 ? v1 : v0;
        const float e[4] = {w.x * pre, w.y * pre, w.z * pre, w.w * pre};
        uint32_t th[4], tl[4];
        uint32_t sum = 0u;   // mod 2^32: the magic offsets cancel below
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float q = e[j] * inv;
            const float t1 = __fadd_rn(q, kMagic);
            const float hq = __fsub_rn(t1, kMagic);
            const float r = __fmul_rn(__fsub_rn(q, hq), 254.0f);
            th[j] = __float_as_uint(t1);
            tl[j] = __float_as_uint(__fadd_rn(r, kMagic));
            sum += 254u * th[j] + tl[j];
        }
        uint32_t hw = __byte_perm(__byte_perm(th[0], th[1], 0x0040), __byte_perm(th[2], th[3], 0x0040), 0x5410);
        uint32_t lw = __byte_perm(__byte_perm(tl[0], tl[1], 0x0040), __byte_perm(tl[2], tl[3], 0x0040), 0x5410);
        sum -= 4u * 255u * kMagicBits;
        if (!ok) hw = lw = sum = 0u;
        const int k = 128 * h2 + 4 * lane;
        *reinterpret_cast<uint32_t *>(base + k) = hw;
        *reinterpret_cast<uint32_t *>(base + 256 + k) = lw;
        int s = static_cast<int>(sum);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if ((lane & 3) == 0) {
            const int j = k >> 4;                               // sub-block 8h + 2c + p
            const int idx = 4 * (2 * (j >> 3) + (j & 1)) + ((j & 7) >> 1);
            reinterpret_cast<int *>(base + 512)[idx] = s;
        }
    }
    const float unscale = ok ? (amax * pre) / 127.0f / 254.0f : (m == 0u ? 0.0f : amax);
    return make_float2(unscale, 1.0f / pre);
}

// ---------------------------------------------------------------------------
// GGUF Q6_K rows -> planar form.  Thread i writes one 16-byte chunk: chunk c
// < 13 of block (n, j) of the QS plane (16 bytes of the 2-byte aligned GGUF
// block, read as eight 16-bit words), or one 16-byte chunk of the D plane
// (the d of eight blocks of a row, zero past the last block).
// ---------------------------------------------------------------------------
__global__ void repack_kernel(const uint8_t *__restrict__ W, uint8_t *__restrict__ Wp, long long N, int nb, int dp)
{
    const long long qs_chunks = N * nb * 13;
    const long long d_chunks = N * (dp / 16);
    const size_t rb = static_cast<size_t>(nb) * 210;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < qs_chunks + d_chunks;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        uint32_t w[4];
        uint8_t *dst;
        if (i < qs_chunks) {
            const long long blk = i / 13;          // n * nb + j
            const int c = static_cast<int>(i - blk * 13);
            const long long n = blk / nb;
            const int j = static_cast<int>(blk - n * nb);
            const unsigned short *src = reinterpret_cast<const unsigned short *>(W + n * rb + static_cast<size_t>(j) * 210 + 16 * c);
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = static_cast<uint32_t>(src[2 * q]) | (static_cast<uint32_t>(src[2 * q + 1]) << 16);
            dst = Wp + static_cast<size_t>(blk) * kQsBytes + 16 * c;
        } else {
            const long long e = i - qs_chunks;
            const int per = dp / 16;
            const long long n = e / per;
            const int c = static_cast<int>(e - n * per);
            unsigned short d[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int j = 8 * c + q;
                d[q] = (j < nb) ? *reinterpret_cast<const unsigned short *>(W + n * rb + static_cast<size_t>(j) * 210 + 208)
                                : static_cast<unsigned short>(0);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = static_cast<uint32_t>(d[2 * q]) | (static_cast<uint32_t>(d[2 * q + 1]) << 16);
            dst = Wp + static_cast<size_t>(N) * nb * kQsBytes + static_cast<size_t>(n) * dp + 16 * c;
        }
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ---------------------------------------------------------------------------
// The GEMV.  grid = (row-tile CTAs, split), cluster (1, split, 1) when
// split > 1.  Tensor maps: QS as [N rows] x [nb * 26] 8-byte words with a box
// of one block (26 words) x 128 rows; D as [N] x [DP / 8] words with a box of
// 2 words x 128 rows.
// ---------------------------------------------------------------------------
struct Maps {
    CUtensorMap qs;
    CUtensorMap d;
};

struct Args {
    const float *x;
    float *y;
    int N, nb, B, tiles, kc;
    uint64_t wait_ns;
};

// The four 6-bit codes (0..63) of word i of this thread's part, one per byte:
// A = ql bytes of c = 0 (low nibbles) and c = 2 (high), Bq = ql bytes of c = 1
// and 3, H = qh bytes (two bits per c).
struct Codes {
    uint32_t c0, c1, c2, c3;
};
__device__ __forceinline__ Codes codes(uint32_t A, uint32_t Bq, uint32_t H)
{
    Codes q;
    q.c0 = and_or(A, 0x0F0F0F0Fu, (H << 4) & 0x30303030u);
    q.c1 = and_or(Bq, 0x0F0F0F0Fu, (H << 2) & 0x30303030u);
    q.c2 = and_or(A >> 4, 0x0F0F0F0Fu, H & 0x30303030u);
    q.c3 = and_or(Bq >> 4, 0x0F0F0F0Fu, (H >> 2) & 0x30303030u);
    return q;
}

// signed byte S of w as an int (S = 0..3, compile-time)
template <int S>
__device__ __forceinline__ int sbyte(uint32_t w)
{
    return static_cast<int>(w << (24 - 8 * S)) >> 24;
}

template <int BMAX>
__global__ void __launch_bounds__(kThreads, 2) q6k_planar_kernel(const __grid_constant__ Maps maps, const Args args)
{
    static_assert(BMAX <= kMaxB, "the split-K receive buffer holds kMaxB batch rows");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *ring = smem_raw;
    uint8_t *xa = smem_raw + static_cast<size_t>(kStages) * kStageBytes;
    float *s_red = reinterpret_cast<float *>(xa + static_cast<size_t>(kMaxItems) * kXItem);
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ int s_slot_done[kStages];
    __shared__ int s_abort;
    __shared__ int s_issued;
    __shared__ float2 s_up[kMaxItems];   // per x item: (unscale, pre)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane & 7, t = lane >> 3;
    const int B = args.B, nb = args.nb;
    const int split = gridDim.y, rank = blockIdx.y;
    const int kb_begin = static_cast<int>((static_cast<long long>(rank) * nb) / split);
    const int ks = static_cast<int>((static_cast<long long>(rank + 1) * nb) / split) - kb_begin;
    const int my_tiles = (args.tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                         static_cast<int>(gridDim.x);
    const int total = my_tiles * ks;
    uint64_t policy = 0, policy_d = 0;   // codes: evict first; d (read once per block of its group of 8): evict last

    auto issue = [&](int i) {   // stage i of this CTA's schedule -> slot i % kStages
        const int tile = static_cast<int>(blockIdx.x) + (i / ks) * static_cast<int>(gridDim.x);
        const int kb = kb_begin + i % ks;
        const int slot = i % kStages;
        uint8_t *st = ring + static_cast<size_t>(slot) * kStageBytes;
        mbar_arrive_expect_tx(smem_u32(&full[slot]), kStageBytes);
        tma_load_2d_hint(smem_u32(st), &maps.qs, kb * (kQsBytes / 8), tile * kRows, smem_u32(&full[slot]), policy);
        tma_load_2d_hint(smem_u32(st + kQsStage), &maps.d, (kb >> 3) * 2, tile * kRows, smem_u32(&full[slot]), policy_d);
    };

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            s_slot_done[i] = 0;
        }
        s_abort = 0;
        fence_barrier_init();
        prefetch_tensormap(&maps.qs);
        prefetch_tensormap(&maps.d);
        policy = l2_policy_evict_first();
        policy_d = l2_policy_evict_last();
        const int first = min(kPreWait, total);
        for (int i = 0; i < first; ++i) issue(i);
        s_issued = first;
    }
    __syncthreads();
    policy = l2_policy_evict_first();
    policy_d = l2_policy_evict_last();
    if (split > 1) cluster_arrive_relaxed();
    pdl_launch_dependents();
    pdl_wait();   // x may come from the previous kernel

    // this thread's part of a block: h, the first l, the byte offsets of its
    // ql (c = 0/2 and 1/3), qh and sc data
    const int h = t >> 1, p = t & 1;
    const int offA = 64 * h + 16 * p, offB = offA + 32, offH = 128 + 32 * h + 16 * p, offS = 192 + 8 * h;
    // x chunk: items (batch row, block) of kc blocks of this CTA's K slice,
    // item (bl, b) at (bl * B + b) * kXItem
    auto convert = [&](int kb0, int cn, bool first_chunk) {
        const int items = cn * B;
        float4 v[2][2];
        // two rounds of loads in flight, then the conversions
        for (int it0 = warp; it0 < items; it0 += 2 * kWarps) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int it = it0 + r * kWarps;
                if (it < items) {
                    const int bl = it / B, b = it - bl * B;
                    const float4 *src = reinterpret_cast<const float4 *>(
                        args.x + static_cast<size_t>(b) * nb * 256 + static_cast<size_t>(kb0 + bl) * 256);
                    v[r][0] = __ldg(src + lane);
                    v[r][1] = __ldg(src + 32 + lane);
                }
            }
            if (first_chunk && it0 == warp && tid == 0) {
                const int first = min(kStages, total);
                for (int i = s_issued; i < first; ++i) issue(i);
                s_issued = first;
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int it = it0 + r * kWarps;
                if (it < items) {
                    const int bl = it / B, b = it - bl * B;
                    const float2 up = x_item(v[r][0], v[r][1], lane, xa + static_cast<size_t>(bl * B + b) * kXItem);
                    if (lane == 0) s_up[bl * B + b] = up;
                }
            }
        }
        named_bar_sync(1, kThreads);
    };

    int consumed = 0;
    const bool single_chunk = args.kc >= ks;
    if (single_chunk) convert(kb_begin, ks, true);
    for (int ti_idx = 0; ti_idx < my_tiles; ++ti_idx) {
        const int tile = static_cast<int>(blockIdx.x) + ti_idx * static_cast<int>(gridDim.x);
        float acc[2][BMAX];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int b = 0; b < BMAX; ++b) acc[r][b] = 0.f;
        int chunk_end = single_chunk ? ks : -1;
        int blk = -1;
        for (int kbl = 0; kbl < ks; ++kbl) {
            ++blk;
            if (kbl >= chunk_end) {
                const int cn = min(args.kc, ks - kbl);
                named_bar_sync(1, kThreads);   // everyone done with the previous chunk
                convert(kb_begin + kbl, cn, ti_idx == 0 && kbl == 0);
                chunk_end = kbl + cn;
                blk = 0;
            }
            const int slot = consumed % kStages;
            const uint32_t phase = static_cast<uint32_t>((consumed / kStages) & 1);
            if (!*(volatile int *)&s_abort && !mbar_wait_bounded(smem_u32(&full[slot]), phase, args.wait_ns)) {
                atomicOr(&g_q6p_error, 1u);
                s_abort = 1;
            }
            const uint8_t *st = ring + static_cast<size_t>(slot) * kStageBytes;
            const int kbm = (kb_begin + kbl) & 7;   // this block's d in the row's 16-byte d chunk
            // codes, scales and d of the two rows
            uint4 qa[2], qb[2], qh[2];
            uint2 sc[2];
            float d[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int row = 16 * warp + g + 8 * r;
                const uint8_t *rp = st + row * kQsBytes;
                qa[r] = *reinterpret_cast<const uint4 *>(rp + offA);
                qb[r] = *reinterpret_cast<const uint4 *>(rp + offB);
                qh[r] = *reinterpret_cast<const uint4 *>(rp + offH);
                sc[r] = *reinterpret_cast<const uint2 *>(rp + offS);
                d[r] = __half2float(__ushort_as_half(
                    *reinterpret_cast<const unsigned short *>(st + kQsStage + row * 16 + 2 * kbm)));
            }
            // scales of c = 0..3: byte 2c + p of the thread's 8 scale bytes
            int scv[2][4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t lo = p ? (sc[r].x >> 8) : sc[r].x;   // bytes p, p + 2
                const uint32_t hi = p ? (sc[r].y >> 8) : sc[r].y;   // bytes 4 + p, 6 + p
                scv[r][0] = sbyte<0>(lo);
                scv[r][1] = sbyte<2>(lo);
                scv[r][2] = sbyte<0>(hi);
                scv[r][3] = sbyte<2>(hi);
            }
#pragma unroll
            for (int b = 0; b < BMAX; ++b) {
                if (b >= B) break;
                const uint8_t *xi = xa + static_cast<size_t>(blk * B + b) * kXItem;
                // x parts of the thread's weights: 16 bytes per c, xh then xl
                uint4 xh[4], xl[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    xh[c] = *reinterpret_cast<const uint4 *>(xi + 128 * h + 32 * c + 16 * p);
                    xl[c] = *reinterpret_cast<const uint4 *>(xi + 256 + 128 * h + 32 * c + 16 * p);
                }
                const int4 sums = *reinterpret_cast<const int4 *>(xi + 512 + 16 * t);
                const float2 up = s_up[blk * B + b];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t A[4] = {qa[r].x, qa[r].y, qa[r].z, qa[r].w};
                    const uint32_t Bq[4] = {qb[r].x, qb[r].y, qb[r].z, qb[r].w};
                    const uint32_t H[4] = {qh[r].x, qh[r].y, qh[r].z, qh[r].w};
                    int eh[4] = {0, 0, 0, 0}, el[4] = {0, 0, 0, 0};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const Codes q = codes(A[i], Bq[i], H[i]);
                        const uint32_t h0 = (&xh[0].x)[i], h1 = (&xh[1].x)[i], h2 = (&xh[2].x)[i], h3 = (&xh[3].x)[i];
                        const uint32_t l0 = (&xl[0].x)[i], l1 = (&xl[1].x)[i], l2 = (&xl[2].x)[i], l3 = (&xl[3].x)[i];
                        eh[0] = dp4a_us(q.c0, h0, eh[0]);
                        eh[1] = dp4a_us(q.c1, h1, eh[1]);
                        eh[2] = dp4a_us(q.c2, h2, eh[2]);
                        eh[3] = dp4a_us(q.c3, h3, eh[3]);
                        el[0] = dp4a_us(q.c0, l0, el[0]);
                        el[1] = dp4a_us(q.c1, l1, el[1]);
                        el[2] = dp4a_us(q.c2, l2, el[2]);
                        el[3] = dp4a_us(q.c3, l3, el[3]);
                    }
                    // sum_c sc_c (sum q (254 xh + xl) - 32 S_c), exact pieces in int32
                    const int Th = scv[r][0] * eh[0] + scv[r][1] * eh[1] + scv[r][2] * eh[2] + scv[r][3] * eh[3];
                    const int Tl = scv[r][0] * el[0] + scv[r][1] * el[1] + scv[r][2] * el[2] + scv[r][3] * el[3];
                    const int M = scv[r][0] * sums.x + scv[r][1] * sums.y + scv[r][2] * sums.z + scv[r][3] * sums.w;
                    const float v = fmaf(254.0f, static_cast<float>(Th), static_cast<float>(Tl)) - 32.0f * static_cast<float>(M);
                    acc[r][b] = fmaf((v * d[r]) * up.x, up.y, acc[r][b]);
                }
            }
            // the slot's bytes have all been used: the last warp to leave refills it
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                const int prev = atomicAdd(&s_slot_done[slot], 1);
                if (prev % kWarps == kWarps - 1) {
                    const int next = consumed + kStages;
                    if (next < total && !*(volatile int *)&s_abort) {
                        issue(next);
                        atomicAdd(&s_issued, 1);
                    }
                }
            }
            ++consumed;
        }
        // tile epilogue: the four parts of each row (lanes g, g + 8, g + 16, g + 24)
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int b = 0; b < BMAX; ++b) {
                acc[r][b] += __shfl_xor_sync(0xffffffffu, acc[r][b], 8);
                acc[r][b] += __shfl_xor_sync(0xffffffffu, acc[r][b], 16);
            }
        if (split == 1) {
            if (t == 0 && !*(volatile int *)&s_abort) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int row = tile * kRows + 16 * warp + g + 8 * r;
#pragma unroll
                    for (int b = 0; b < BMAX; ++b)
                        if (b < B && row < args.N) args.y[static_cast<size_t>(b) * args.N + row] = acc[r][b];
                }
            }
        } else {
            // push the partial rows into the owner rank's receive buffer: rank
            // q owns tile rows [q*128/split, (q+1)*128/split), one slot per
            // source rank
            cluster_wait_acquire();
            if (t == 0 && !*(volatile int *)&s_abort) {
                const uint32_t red_base = smem_u32(s_red);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int row = 16 * warp + g + 8 * r;
                    const int owner = (row * split + split - 1) / kRows;
                    const int o0 = (owner * kRows) / split, o1 = ((owner + 1) * kRows) / split;
#pragma unroll
                    for (int b = 0; b < BMAX; ++b)
                        if (b < B) {
                            const uint32_t off = static_cast<uint32_t>(((rank * (o1 - o0) + (row - o0)) * B + b) * 4);
                            st_shared_cluster_f32(map_shared_rank(red_base + off, owner), acc[r][b]);
                        }
                }
            }
        }
    }

    // after a timed-out wait: wait (bounded) for the copies still in flight
    __syncthreads();
    if (*(volatile int *)&s_abort && tid == 0) {
        for (int i = max(0, s_issued - kStages); i < s_issued; ++i)
            (void)mbar_wait_bounded(smem_u32(&full[i % kStages]), static_cast<uint32_t>((i / kStages) & 1), args.wait_ns);
    }
    if (split > 1) {
        cluster_arrive_release();
        cluster_wait_acquire();
        if (!*(volatile int *)&s_abort) {
            const int lr0 = (rank * kRows) / split;
            const int rows = ((rank + 1) * kRows) / split - lr0;
            for (int it = tid; it < rows * B; it += kThreads) {
                const int lr = it / B, b = it - lr * B;
                float sum = s_red[lr * B + b];
                for (int q = 1; q < split; ++q) sum += s_red[(q * rows + lr) * B + b];
                const int row = static_cast<int>(blockIdx.x) * kRows + lr0 + lr;
                if (row < args.N) args.y[static_cast<size_t>(b) * args.N + row] = sum;
            }
        }
    }
}

}  // namespace q6p

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

int64_t d_pitch(int64_t nb) { return ((2 * nb + 15) / 16) * 16; }

bool encode(CUtensorMap *map, const void *base, uint64_t words_per_row, uint64_t rows, uint32_t box_words)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(words_per_row), static_cast<cuuint64_t>(rows)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(words_per_row * 8)};
    cuuint32_t box[2] = {box_words, static_cast<cuuint32_t>(q6p::kRows)};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(base), gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of `size` CTAs of the kernel resident at once (per device, cached).
int max_clusters(int size)
{
    static int table[64][q6p::kMaxSplit + 1];
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::call_once(once[dev], [dev]() {
        void (*kern)(const q6p::Maps, const q6p::Args) = q6p::q6k_planar_kernel<1>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(q6p::kSmemBytes));
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        for (int c = 1; c <= q6p::kMaxSplit; ++c) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(1, c, 1);
            cfg.blockDim = dim3(q6p::kThreads, 1, 1);
            cfg.dynamicSmemBytes = q6p::kSmemBytes;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 1;
            attr[0].val.clusterDim.y = c;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
            table[dev][c] = n;
        }
        (void)cudaGetLastError();
    });
    return table[dev][size];
}

// K split: the smallest that gives every SM two CTAs' worth of row tiles, and
// only while all clusters of that size are resident at once.
int choose_split(int tiles, int nb, int sms)
{
    int best = 1;
    for (int s = 1; s <= std::min(nb, q6p::kMaxSplit); ++s) {
        if (s > 1 && max_clusters(s) < tiles) break;
        best = s;
        if (static_cast<long long>(tiles) * s >= 2ll * sms) break;
    }
    return best;
}

template <int BMAX>
cudaError_t launch(const q6p::Maps &maps, const q6p::Args &a, int split, int grid_x, cudaStream_t stream)
{
    void (*kern)(const q6p::Maps, const q6p::Args) = q6p::q6k_planar_kernel<BMAX>;
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!done[dev & 63]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(q6p::kSmemBytes));
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
            if (e != cudaSuccess) return e;
            done[dev & 63] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, split, 1);
    cfg.blockDim = dim3(q6p::kThreads, 1, 1);
    cfg.dynamicSmemBytes = q6p::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (split > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = split;
        attr[0].val.clusterDim.z = 1;
        na = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, maps, a);
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e;
}

bool valid_shape(int64_t N, int64_t K)
{
    return N >= 0 && N <= 0x7FFFFFFFll && K > 0 && K % 256 == 0 && K / 256 < (1ll << 20);
}

}  // namespace

int64_t q6k_planar_bytes_impl(int64_t N, int64_t K)
{
    if (!valid_shape(N, K)) return -1;
    const int64_t nb = K / 256;
    return N * (nb * q6p::kQsBytes + d_pitch(nb));
}

q4k_status q6k_repack_planar_impl(const void *W, void *Wp, int64_t N, int64_t K, void *stream)
{
    if (!valid_shape(N, K)) return Q4K_ERR_INVALID_ARG;
    if (N > 0 && (!W || !Wp)) return Q4K_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(Wp)) & 15u) return Q4K_ERR_MISALIGNED;
    int sms = 0;
    q4k_status st = check_device(&sms);
    if (st != Q4K_OK) return st;
    if (N == 0) return Q4K_OK;
    const int64_t nb = K / 256;
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(W), p0 = reinterpret_cast<uintptr_t>(Wp);
    const uintptr_t wl = static_cast<uintptr_t>(N * nb * 210), pl = static_cast<uintptr_t>(q6k_planar_bytes_impl(N, K));
    if (w0 < p0 + pl && p0 < w0 + wl) return Q4K_ERR_INVALID_ARG;   // overlapping buffers
    q6p::repack_kernel<<<sms * 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(W), static_cast<uint8_t *>(Wp), N, static_cast<int>(nb),
        static_cast<int>(d_pitch(nb)));
    return cudaGetLastError() == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
}

q4k_status q6k_gemv_planar_impl(const void *Wp, const float *x, float *y, int64_t N, int64_t K, int batch,
                                void *stream)
{
    if (!valid_shape(N, K) || !x || batch < 1 || batch > Q4K_MAX_BATCH) return Q4K_ERR_INVALID_ARG;
    if (N > 0 && (!Wp || !y)) return Q4K_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(Wp) | reinterpret_cast<uintptr_t>(x)) & 15u) return Q4K_ERR_MISALIGNED;
    int sms = 0;
    q4k_status st = check_device(&sms);
    if (st != Q4K_OK) return st;
    if (N == 0) return Q4K_OK;
    const int64_t nb = K / 256;
    q6p::Maps maps;
    memset(&maps, 0, sizeof(maps));
    const uint8_t *base = static_cast<const uint8_t *>(Wp);
    if (!encode(&maps.qs, base, static_cast<uint64_t>(nb) * (q6p::kQsBytes / 8), static_cast<uint64_t>(N),
                q6p::kQsBytes / 8) ||
        !encode(&maps.d, base + static_cast<size_t>(N) * nb * q6p::kQsBytes, static_cast<uint64_t>(d_pitch(nb) / 8),
                static_cast<uint64_t>(N), 2))
        return Q4K_ERR_CUDA;
    const int tiles = static_cast<int>((N + q6p::kRows - 1) / q6p::kRows);
    const int split = choose_split(tiles, static_cast<int>(nb), sms);
    const int grid_x = (split > 1) ? tiles : std::min(tiles, 2 * sms);
    for (int b0 = 0; b0 < batch; b0 += q6p::kMaxB) {
        const int B = std::min(q6p::kMaxB, batch - b0);
        q6p::Args a{};
        a.x = x + static_cast<size_t>(b0) * K;
        a.y = y + static_cast<size_t>(b0) * N;
        a.N = static_cast<int>(N);
        a.nb = static_cast<int>(nb);
        a.B = B;
        a.tiles = tiles;
        const int ks_max = static_cast<int>((nb + split - 1) / split);
        a.kc = std::min(ks_max, q6p::kMaxItems / B);
        a.wait_ns = q6p::kWaitLimitNs;
        const cudaStream_t cs = static_cast<cudaStream_t>(stream);
        cudaError_t e = (B == 1)   ? launch<1>(maps, a, split, grid_x, cs)
                        : (B <= 4) ? launch<4>(maps, a, split, grid_x, cs)
                                   : launch<8>(maps, a, split, grid_x, cs);
        if (e != cudaSuccess) return Q4K_ERR_CUDA;
    }
    return Q4K_OK;
}

unsigned int read_q6p_error()
{
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, q6p::g_q6p_error, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    return v;
}

bool clear_q6p_error()
{
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(q6p::g_q6p_error, &z, sizeof(z)) == cudaSuccess;
}

}  // namespace q4k
