// q4k_gemv.cu -- Q4_K decode GEMV / VerifyBatch GEMV / fused LM-head argmax
// for GB300 (sm_103a).
//
// What is computed: y[b][n] = sum_k w[n][k] x[b][k] with w the Q4_K weight
// w = d*sc_j*q - dmin*m_j, directly on the quantized blocks ("fused scale x
// int dot-product kernels operating directly on quantized blocks", dotLLM
// README, Key Features / Performance), reading every super-block once for all
// batch rows (Glacier.Inference article, section 4: VerifyBatch pulls the
// weights through the memory bus once for K+1 tokens), optionally followed by
// the greedy argmax of each batch row (same article, section 2: one int32 per
// row, logits stay on the device).
//
// Design (GB300-first; the pages' own kernels were HLSL Wave32 shaders and
// sm_75..sm_90 cubins):
//   * Weights are streamed HBM -> shared memory with 2-D TMA tensor copies (one
//     super-block of all 128 rows of a tile per stage) into a 4-stage ring
//     guarded by mbarriers.  There is no producer warp: thread 0 issues the
//     first stages before the dependency wait, and the last warp to finish a
//     stage issues the one four ahead into it; the consumers never issue
//     global loads for W.
//   * Batch 1 (default): an integer inner product.  Each super-block of x is
//     carried as two int8 parts per element against its own max|x|, the
//     weight nibbles multiply them with dp4a, the sub-block sums are exact in
//     int32, and the scales are applied once per super-block in fp32.
//   * Batch >= 2 (and batch 1 on request): the tensor cores with mma.sync
//     m16n8k16.  A = the weights' q*sc_j as exact fp16 integers (<= 945),
//     built in registers from the nibbles with one LOP3 (magic-exponent trick)
//     and one HFMA2 per two weights; B = the activations split into fp16 hi +
//     lo parts (x = hi + lo to ~2^-22 relative after a power-of-two scale per
//     super-block and batch row), one column each; column pairs hold batch
//     rows (up to 4 per n8 tile).  The dmin*m_j term is one extra k16 step per
//     super-block whose A holds m_j and whose B holds the per sub-block sums
//     of x; per super-block the two fp32 tiles are combined as d*C - dmin*Cmin.
//   * Row tiles of 128 rows (8 warps x 16 rows), two CTAs per SM.  When there
//     are too few row tiles to fill the GPU the K range of a tile is split
//     over the CTAs of a thread-block cluster (up to 16), and the partial sums
//     are added in rank order through distributed shared memory
//     (deterministic, no atomics, no global scratch).  With a single K slice
//     the grid is persistent and CTAs loop over row tiles, so the weight
//     stream never drains between tiles.
//   * The argmax variant keeps per-CTA (max, lowest index) keys in shared
//     memory and combines CTAs with one 64-bit atomicMax per batch row plus a
//     last-CTA ticket (no spin-waits).

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/q4k.h"
#include "ptx.cuh"
#include "q4k_internal.h"

namespace q4k {

constexpr int kBlockBytes = 144;
constexpr int kWarps = 8;                 // warps per CTA, 16 weight rows each
constexpr int kRows = 16 * kWarps;        // rows per tile (128)
constexpr int kThreads = 32 * kWarps;
constexpr int kKsteps = 17;               // 16 k16 steps + 1 min-term step per super-block
constexpr int kStages = 4;                // W ring depth
constexpr int kStageBytes = kRows * kBlockBytes;   // one super-block of every tile row (18 KB)
constexpr size_t kSmemPerCta2 = 110 * 1024;        // two CTAs per SM (batch <= 8)
constexpr size_t kSmemPerCta1 = 200 * 1024;        // one CTA per SM (batch > 8)
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

__device__ unsigned int g_device_error = 0;   // bit 0: an mbarrier wait timed out

constexpr int kMaxGroups = 4;             // matrices sharing x in one launch

struct GemvArgs {
    const float *x;
    float *y[kMaxGroups];           // outputs per matrix (null in the argmax variant without logits)
    int N[kMaxGroups];              // rows per matrix
    int tile_start[kMaxGroups + 1]; // first row tile of each matrix in the concatenated tile space
    int ngroups;
    int nb;              // super-blocks per row
    int B;               // batch
    int tiles;           // total row tiles over all matrices
    int kc;              // super-blocks per x chunk in shared memory
    unsigned long long *keys;  // argmax: [B] 64-bit keys (zeroed), null otherwise
    unsigned int *ticket;      // argmax: CTA ticket (zeroed)
    int32_t *idx;              // argmax: output [B]
};

__host__ __device__ inline int frag_lanes(int NT, int B) { return NT == 1 ? 8 * B : 32; }

// B fragments are stored lane-major: the 17*NT entries (uint2) of one lane for
// one super-block are contiguous, so a consumer lane reads them at constant
// offsets from one base.  The per-lane stride is odd in 8-byte units for even
// NT so that the 16 lanes of a wavefront hit distinct bank pairs.
__host__ __device__ constexpr int lane_stride(int NT)
{
    // even (16-byte aligned lanes: a k-step's even and odd fragments load as one
    // 16-byte access; lane L starts at bank 4L mod 32 for NT = 1, 2, 4, so the
    // eight lanes of a 16-byte wavefront hit distinct banks); NT = 3 loads
    // 8-byte fragments and keeps an odd stride
    return NT == 3 ? kKsteps * NT : kKsteps * NT + ((kKsteps * NT) & 1);
}

__host__ __device__ inline size_t xfrag_bytes_per_block(int NT, int B)
{
    return static_cast<size_t>(lane_stride(NT)) * frag_lanes(NT, B) * 8;
}

// Dynamic shared memory: [ring | x fragments | split-K receive buffer (split
// slots of at most ceil(128/split) rows x B, only with a split)].
__host__ __device__ inline size_t xfrag_offset() { return static_cast<size_t>(kStages) * kStageBytes; }
__host__ __device__ inline size_t red_offset(int NT, int B, int kc)
{
    return xfrag_offset() + ((xfrag_bytes_per_block(NT, B) * kc + 127) & ~size_t(127));
}
// Split-K receive buffer: the owner of ceil(128 / split) rows keeps one slot
// per source rank, split * ceil(128 / split) <= 128 + 15 rows for split <= 16.
constexpr int kRedRows = kRows + 16;
__host__ inline size_t gemv_smem_bytes(int NT, int B, int kc, int split)
{
    return red_offset(NT, B, kc) + ((split > 1) ? static_cast<size_t>(kRedRows) * B * 4 : 0);
}

// ---------------------------------------------------------------------------
// x chunk -> fp16 hi/lo B fragments in shared memory.
// Entry (bl, s, nt, L) is a uint2 {b01, b23} for lane L = 4*col8 + t of n-tile
// nt at k-step s of local super-block bl.  Thread t of an A fragment handles
// sub-block pair t of each super-block (sub-blocks 2t and 2t+1), so for k-step
// s < 16 (word u = s/2, sub-block 2t + (s&1)) the four B values are the x
// entries 4u..4u+3 of that sub-block ordered {4u, 4u+2 | 4u+1, 4u+3}.  Step 16
// holds the sub-block sums of x for sub-blocks 2t, 2t+1 (the dmin*m term).
// ---------------------------------------------------------------------------
// Power-of-two scale 2^s with max|x| * 2^s in [2^9, 2^10) (s = 0 for an all
// zero or non-finite chunk), clamped to the normal range.
__device__ __forceinline__ int chunk_scale_exp(uint32_t amax_bits)
{
    const int E = static_cast<int>((amax_bits >> 23) & 255u);
    int s = (amax_bits != 0u && E != 255) ? 136 - E : 0;
    return max(-126, min(126, s));
}

// A chunk of x (B rows x nblk super-blocks, B * nblk <= 32) -> B fragments in
// shared memory.  One warp converts one (batch row, super-block) item per
// round; lane l holds float4 l and l + 32 of the super-block (elements
// 4i..4i+3, sub-block i/8, word i%8).  All loads of all rounds are issued
// first.  Each item gets its own power-of-two scale from a warp-level max
// (no shared-memory max, no barrier in between), stored as s_unscale[bl*B + b];
// then the fp16 hi/lo fragments and the sub-block sums (8-lane shuffles).
// Float4 i is sub-block j = i/8 (pair t = j/2, half h = j%2), word u = i%8 ->
// k-step s = 2u + h of pair t.  Ends with a barrier over all nthr threads; the
// caller must have finished reading the previous chunk's fragments and scales.
template <int NT, bool L2ONLY = false>
__device__ void convert_x_blocks(const float *__restrict__ x, int K, int B, int kb0, int nblk, uint2 *xf,
                                 float *s_unscale, int tid, int nthr)
{
    const int LW = frag_lanes(NT, B);
    constexpr int LS = lane_stride(NT);
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int items = B * nblk;   // <= 32: at most 4 rounds of 8 warps
    float4 v[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int it = warp + r * nwarps;
        if (it < items) {   // warp-uniform
            const int b = it / nblk;
            const float4 *src = reinterpret_cast<const float4 *>(
                x + static_cast<size_t>(b) * K + static_cast<size_t>(kb0 + (it - b * nblk)) * 256);
            v[r][0] = L2ONLY ? __ldcg(src + lane) : __ldg(src + lane);
            v[r][1] = L2ONLY ? __ldcg(src + 32 + lane) : __ldg(src + 32 + lane);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int it = warp + r * nwarps;
        if (it >= items) continue;   // warp-uniform
        const int b = it / nblk;
        const int bl = it - b * nblk;
        uint32_t m = 0u;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const float4 w = v[r][h2];
            m = max(m, max(max(__float_as_uint(fabsf(w.x)), __float_as_uint(fabsf(w.y))),
                           max(__float_as_uint(fabsf(w.z)), __float_as_uint(fabsf(w.w)))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int e = chunk_scale_exp(m);
        const float sc = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
        if (lane == 0) s_unscale[bl * B + b] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
        const int chi = 2 * b, clo = 2 * b + 1;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int i = lane + 32 * h2;
            float4 w = v[r][h2];
            w.x *= sc; w.y *= sc; w.z *= sc; w.w *= sc;
            const int sb = i >> 3, u = i & 7;
            const int t = sb >> 1, s = 2 * u + (sb & 1);
            const uint32_t h01 = pack_half2(w.x, w.z);
            const uint32_t h23 = pack_half2(w.y, w.w);
            const uint32_t l01 = pack_half2(w.x - half_lo_f32(h01), w.z - half_hi_f32(h01));
            const uint32_t l23 = pack_half2(w.y - half_lo_f32(h23), w.w - half_hi_f32(h23));
            xf[(bl * LW + 4 * (chi % 8) + t) * LS + s * NT + chi / 8] = make_uint2(h01, h23);
            xf[(bl * LW + 4 * (clo % 8) + t) * LS + s * NT + clo / 8] = make_uint2(l01, l23);
            // sub-block sum over the 8 lanes holding it, then pair it with the
            // odd sub-block held by the next 8 lanes
            float sum = (w.x + w.y) + (w.z + w.w);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            const float sum_odd = __shfl_down_sync(0xffffffffu, sum, 8);
            if ((i & 15) == 0) {
                const uint32_t hs = pack_half2(sum, sum_odd);
                const uint32_t ls = pack_half2(sum - half_lo_f32(hs), sum_odd - half_hi_f32(hs));
                xf[(bl * LW + 4 * (chi % 8) + t) * LS + 16 * NT + chi / 8] = make_uint2(hs, 0u);
                xf[(bl * LW + 4 * (clo % 8) + t) * LS + 16 * NT + clo / 8] = make_uint2(ls, 0u);
            }
        }
    }
    named_bar_sync(1, nthr);
}

// ---------------------------------------------------------------------------
// Batch 1, integer inner product: x of one super-block as two int8 parts per
// element,  x ~= (dx / 254) * (254 * xh + xl)  with dx = max|x| / 127,
// q = x * (127 / max|x|), xh = rint(q) and xl = rint((q - xh) * 254), all in
// fp32 (x and max|x| first scaled by 2^64 when max|x| < 2^-64), so that
// |x - (dx / 254)(254 xh + xl)| <= dx (1/508 + 2^-16).  Per local
// super-block bl, at byte offset bl * blk_bytes of the fragment area:
//   [0, 320)    xh: the 64 values of sub-block pair t at 80 t, in k order
//   [320, 640)  xl: the same at 320 + 80 t
//   [640, 672)  int32 per sub-block j: 254 * sum(xh) + sum(xl) over its 32 k
// (the 16-byte pad per pair puts the four pairs' 16-byte loads of one
// quarter-warp on distinct banks)
// and s_unscale[bl] * s_pre[bl] = dx / 254, with s_unscale[bl] kept in the
// normal range (s_pre = 2^-64 for the scaled blocks, else 1); s_unscale is 0
// for an all-zero super-block and the non-finite max itself when x holds an
// inf or NaN, so that the result is not finite.
// One warp per super-block; lane l holds float4 l and l + 32 (k = 4l..4l+3 and
// 128 + 4l..).  Ends with a barrier over all nthr threads.
// ---------------------------------------------------------------------------
constexpr int kI8Bytes = 672;
constexpr int kI8Pair = 80;        // bytes per sub-block pair in each part
static_assert(kI8Bytes <= lane_stride(1) * 8 * 8, "batch-1 fragment area holds the int8 parts");

template <bool Q8, bool L2ONLY = false>
__device__ void convert_x_i8_blocks(const float *__restrict__ x, int kb0, int nblk, uint8_t *xb, int blk_bytes,
                                    float *s_unscale, float *s_pre, int tid, int nthr)
{
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    float4 v[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int it = warp + r * nwarps;
        if (it < nblk) {   // warp-uniform
            const float4 *src = reinterpret_cast<const float4 *>(x + static_cast<size_t>(kb0 + it) * 256);
            v[r][0] = L2ONLY ? __ldcg(src + lane) : __ldg(src + lane);
            v[r][1] = L2ONLY ? __ldcg(src + 32 + lane) : __ldg(src + 32 + lane);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int it = warp + r * nwarps;
        if (it >= nblk) continue;   // warp-uniform
        uint32_t m = 0u;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const float4 w = v[r][h2];
            m = max(m, max(max(__float_as_uint(fabsf(w.x)), __float_as_uint(fabsf(w.y))),
                           max(__float_as_uint(fabsf(w.z)), __float_as_uint(fabsf(w.w)))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float amax = __uint_as_float(m);
        const bool ok = m != 0u && m < 0x7F800000u;   // finite and not all zero
        // below 2^-64 the reciprocal is taken of the max scaled by 2^64 (exact)
        // and x is scaled alike, so that it stays finite
        const float pre = (m < 0x1F800000u) ? 0x1p64f : 1.0f;
        const float inv = ok ? 127.0f / (amax * pre) : 0.0f;
        uint8_t *base = xb + static_cast<size_t>(it) * blk_bytes;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const float4 w = v[r][h2];
            const float e[4] = {w.x, w.y, w.z, w.w};
            uint32_t hw = 0u, lw = 0u;
            int sum = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float q = (e[j] * pre) * inv;
                const float hq = rintf(q);
                const int hi = static_cast<int>(hq);
                hw |= (static_cast<uint32_t>(hi) & 0xFFu) << (8 * j);
                if constexpr (Q8) {
                    sum += hi;
                } else {
                    const int lo = static_cast<int>(rintf((q - hq) * 254.0f));
                    lw |= (static_cast<uint32_t>(lo) & 0xFFu) << (8 * j);
                    sum += 254 * hi + lo;
                }
            }
            const int i = lane + 32 * h2;   // float4 index: k = 4i..4i+3, sub-block i/8, pair i/16
            const int off = kI8Pair * (i >> 4) + 4 * (i & 15);
            *reinterpret_cast<uint32_t *>(base + off) = hw;
            if constexpr (!Q8) *reinterpret_cast<uint32_t *>(base + 4 * kI8Pair + off) = lw;
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            if ((i & 7) == 0) reinterpret_cast<int *>(base + 8 * kI8Pair)[i >> 3] = sum;
        }
        if (lane == 0) {
            s_unscale[it] = ok ? (Q8 ? (amax * pre) / 127.0f : (amax * pre) / 127.0f / 254.0f)
                               : (m == 0u ? 0.0f : amax);
            s_pre[it] = 1.0f / pre;
        }
    }
    named_bar_sync(1, nthr);
}

// Warm L2 with x[b][kb0*256, kb1*256) for every batch row (one 128-byte line
// per thread and round).  Safe before a dependency wait: L2 is where the
// earlier writes land, so the loads after the wait still see them.
__device__ __forceinline__ void prefetch_x_l2(const float *x, int K, int B, int kb0, int kb1, int tid, int nthr)
{
    const int lines = (kb1 - kb0) * 8;   // 1 KB of floats per super-block
    for (int i = tid; i < B * lines; i += nthr) {
        const int b = i / lines;
        prefetch_l2(x + static_cast<size_t>(b) * K + static_cast<size_t>(kb0) * 256 + (i - b * lines) * 32);
    }
}

// Scale/min constants of one row of a super-block for thread t (pair t).
struct RowConsts {
    uint32_t mulE, addE, mulO, addO;  // f16x2 (sc_2t), (-1024 sc_2t), (sc_2t+1 / 16), (-64 sc_2t+1)
    uint32_t mpair;                   // f16x2 {m_2t, m_2t+1}
    float d, dmin;
};

__device__ __forceinline__ RowConsts decode_header(uint4 h, int t)
{
    RowConsts rc;
    rc.d = half_lo_f32(h.x);
    rc.dmin = half_hi_f32(h.x);
    const uint32_t sh = (t & 1) ? 16u : 0u;
    const uint32_t a0 = (h.y >> sh) & 0xFFFFu;   // s[2(t&1)], s[2(t&1)+1]
    const uint32_t a1 = (h.z >> sh) & 0xFFFFu;   // s[4+...]
    const uint32_t a2 = (h.w >> sh) & 0xFFFFu;   // s[8+...]
    uint32_t scp, mp;
    if (t < 2) {
        scp = a0 & 0x3F3Fu;
        mp = a1 & 0x3F3Fu;
    } else {
        scp = (a2 & 0x0F0Fu) | ((a0 >> 2) & 0x3030u);
        mp = ((a2 >> 4) & 0x0F0Fu) | ((a1 >> 2) & 0x3030u);
    }
    const uint32_t k1024 = 0x64006400u;          // f16x2 {1024, 1024}
    uint32_t sch = hsub2_u32(__byte_perm(scp, 0u, 0x4140u) | k1024, k1024);   // {sc_2t, sc_2t+1}
    rc.mpair = hsub2_u32(__byte_perm(mp, 0u, 0x4140u) | k1024, k1024);       // {m_2t, m_2t+1}
    const uint32_t lo2 = __byte_perm(sch, 0u, 0x1010u);   // {sc_2t, sc_2t}
    const uint32_t hi2 = __byte_perm(sch, 0u, 0x3232u);   // {sc_2t+1, sc_2t+1}
    rc.mulE = lo2;
    rc.addE = hmul2_u32(lo2, 0xE400E400u);        // * -1024
    rc.mulO = hmul2_u32(hi2, 0x2C002C00u);        // * 1/16
    rc.addO = hmul2_u32(hi2, 0xD400D400u);        // * -64
    return rc;
}

// Integer scale/min constants of one row for thread t (sub-blocks 2t, 2t+1).
struct RowConstsI {
    int scE, scO, mE, mO;
    float d, dmin;
};
__device__ __forceinline__ RowConstsI decode_header_i(uint4 h, int t)
{
    RowConstsI rc;
    rc.d = half_lo_f32(h.x);
    rc.dmin = half_hi_f32(h.x);
    const uint32_t sh = (t & 1) ? 16u : 0u;
    const uint32_t a0 = (h.y >> sh) & 0xFFFFu;   // s[2(t&1)], s[2(t&1)+1]
    const uint32_t a1 = (h.z >> sh) & 0xFFFFu;   // s[4+...]
    const uint32_t a2 = (h.w >> sh) & 0xFFFFu;   // s[8+...]
    uint32_t scp, mp;
    if (t < 2) {
        scp = a0 & 0x3F3Fu;
        mp = a1 & 0x3F3Fu;
    } else {
        scp = (a2 & 0x0F0Fu) | ((a0 >> 2) & 0x3030u);
        mp = ((a2 >> 4) & 0x0F0Fu) | ((a1 >> 2) & 0x3030u);
    }
    rc.scE = static_cast<int>(scp & 0xFFu);
    rc.scO = static_cast<int>(scp >> 8);
    rc.mE = static_cast<int>(mp & 0xFFu);
    rc.mO = static_cast<int>(mp >> 8);
    return rc;
}

// Batch 1, integer inner product of one super-block for thread (g, t): rows g
// (ra) and g + 8 (rb), sub-block pair t.  Byte i of the pair's 32 quant bytes
// holds q of weight i of sub-block 2t (low nibble) and of 2t+1 (high nibble);
// dp4a multiplies four of them with four int8 parts of x at a time.  Low
// nibbles go in as q, high nibbles in place as 16 q (one exact shift per sum
// afterwards).  Per row the sums are exact in int32:
//   T = 254 (scE SEh + scO SOh) + (scE SEl + scO SOl)    (|T| < 1.96e9)
//   M = mE BS_2t + mO BS_2t+1                            (|M| < 1.4e8)
// and y += ((d T - dmin M) u) pre with u pre = dx / 254 for this super-block
// (every intermediate in the normal range, whatever the size of x).
template <bool Q8, typename Release>
__device__ __forceinline__ void stage_compute_i8(const uint8_t *ra, const uint8_t *rb, const uint8_t *xb, int t,
                                                 float u, float pre, float (&acc)[1][2], Release &&release)
{
    const RowConstsI r0 = decode_header_i(*reinterpret_cast<const uint4 *>(ra), t);
    const RowConstsI r1 = decode_header_i(*reinterpret_cast<const uint4 *>(rb), t);
    int eh0 = 0, el0 = 0, oh0 = 0, ol0 = 0, eh1 = 0, el1 = 0, oh1 = 0, ol1 = 0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const uint4 qa = *reinterpret_cast<const uint4 *>(ra + 16 + 32 * t + 16 * half);
        const uint4 qb = *reinterpret_cast<const uint4 *>(rb + 16 + 32 * t + 16 * half);
        // x parts of k = 64t + 16 half + 0..15 (sub-block 2t) and + 32 (2t+1)
        const uint8_t *xh = xb + kI8Pair * t + 16 * half;
        const uint4 xhE = *reinterpret_cast<const uint4 *>(xh);
        const uint4 xhO = *reinterpret_cast<const uint4 *>(xh + 32);
        const uint4 xlE = Q8 ? make_uint4(0, 0, 0, 0) : *reinterpret_cast<const uint4 *>(xh + 4 * kI8Pair);
        const uint4 xlO = Q8 ? make_uint4(0, 0, 0, 0) : *reinterpret_cast<const uint4 *>(xh + 4 * kI8Pair + 32);
        const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
        const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
        const uint32_t he[4] = {xhE.x, xhE.y, xhE.z, xhE.w};
        const uint32_t ho[4] = {xhO.x, xhO.y, xhO.z, xhO.w};
        const uint32_t le[4] = {xlE.x, xlE.y, xlE.z, xlE.w};
        const uint32_t lo[4] = {xlO.x, xlO.y, xlO.z, xlO.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t aE = wa[j] & 0x0F0F0F0Fu, aO = wa[j] & 0xF0F0F0F0u;
            const uint32_t bE = wb[j] & 0x0F0F0F0Fu, bO = wb[j] & 0xF0F0F0F0u;
            eh0 = dp4a_us(aE, he[j], eh0);
            oh0 = dp4a_us(aO, ho[j], oh0);
            eh1 = dp4a_us(bE, he[j], eh1);
            oh1 = dp4a_us(bO, ho[j], oh1);
            if constexpr (!Q8) {
                el0 = dp4a_us(aE, le[j], el0);
                ol0 = dp4a_us(aO, lo[j], ol0);
                el1 = dp4a_us(bE, le[j], el1);
                ol1 = dp4a_us(bO, lo[j], ol1);
            }
        }
    }
    release();
    const int2 bs = *reinterpret_cast<const int2 *>(xb + 8 * kI8Pair + 8 * t);
    // the high-nibble sums are multiples of 16: exact shifts
    oh0 >>= 4; ol0 >>= 4; oh1 >>= 4; ol1 >>= 4;
    const int T0 = Q8 ? r0.scE * eh0 + r0.scO * oh0 : 254 * (r0.scE * eh0 + r0.scO * oh0) + (r0.scE * el0 + r0.scO * ol0);
    const int T1 = Q8 ? r1.scE * eh1 + r1.scO * oh1 : 254 * (r1.scE * eh1 + r1.scO * oh1) + (r1.scE * el1 + r1.scO * ol1);
    const int M0 = r0.mE * bs.x + r0.mO * bs.y;
    const int M1 = r1.mE * bs.x + r1.mO * bs.y;
    const float v0 = fmaf(r0.d, static_cast<float>(T0), -r0.dmin * static_cast<float>(M0));
    const float v1 = fmaf(r1.d, static_cast<float>(T1), -r1.dmin * static_cast<float>(M1));
    acc[0][0] = fmaf(v0 * u, pre, acc[0][0]);
    acc[0][1] = fmaf(v1 * u, pre, acc[0][1]);
}

// One super-block of this warp's 16 rows (rows g and g + 8 for thread (g, t)):
// dequantize into A fragments, run the k16 steps against the x fragments at
// xl, call release() once the slot's bytes have been read, then fold the
// super-block into acc as d*C - dmin*Cmin.  NC accumulator chains per
// sub-block parity (2: shorter dependency chains; 1: fewer registers).
template <int NT, int NC, typename Release>
__device__ __forceinline__ void stage_compute(const uint8_t *ra, const uint8_t *rb, const uint2 *xl, int t,
                                              const float (&unscale)[NT], float (&acc)[NT][2], Release &&release)
{
    const RowConsts r0 = decode_header(*reinterpret_cast<const uint4 *>(ra), t);
    const RowConsts r1 = decode_header(*reinterpret_cast<const uint4 *>(rb), t);
    float cE[NC][NT][4], cO[NC][NT][4], cM[NT][4];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const uint4 qa = *reinterpret_cast<const uint4 *>(ra + 16 + 32 * t + 16 * half);
        const uint4 qb = *reinterpret_cast<const uint4 *>(rb + 16 + 32 * t + 16 * half);
        const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
        const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
            const int u = 4 * half + uu;
            const uint32_t a = wa[uu], a8 = a >> 8;
            const uint32_t c = wb[uu], c8 = c >> 8;
            const uint32_t mlo = 0x000F000Fu, mhi = 0x00F000F0u, magic = 0x64006400u;
            const uint32_t e0 = hfma2_u32(and_or(a, mlo, magic), r0.mulE, r0.addE);
            const uint32_t e1 = hfma2_u32(and_or(a8, mlo, magic), r0.mulE, r0.addE);
            const uint32_t o0 = hfma2_u32(and_or(a, mhi, magic), r0.mulO, r0.addO);
            const uint32_t o1 = hfma2_u32(and_or(a8, mhi, magic), r0.mulO, r0.addO);
            const uint32_t f0 = hfma2_u32(and_or(c, mlo, magic), r1.mulE, r1.addE);
            const uint32_t f1 = hfma2_u32(and_or(c8, mlo, magic), r1.mulE, r1.addE);
            const uint32_t p0 = hfma2_u32(and_or(c, mhi, magic), r1.mulO, r1.addO);
            const uint32_t p1 = hfma2_u32(and_or(c8, mhi, magic), r1.mulO, r1.addO);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                uint2 be, bo;
                if constexpr (NT == 1) {   // even and odd fragment of k-step pair u: one 16-byte load
                    const uint4 q = *reinterpret_cast<const uint4 *>(&xl[2 * u]);
                    be = make_uint2(q.x, q.y);
                    bo = make_uint2(q.z, q.w);
                } else if constexpr ((NT & 1) == 0) {   // two n-tiles per 16-byte load
                    const uint4 qe = *reinterpret_cast<const uint4 *>(&xl[2 * u * NT + (nt & ~1)]);
                    const uint4 qo = *reinterpret_cast<const uint4 *>(&xl[(2 * u + 1) * NT + (nt & ~1)]);
                    be = (nt & 1) ? make_uint2(qe.z, qe.w) : make_uint2(qe.x, qe.y);
                    bo = (nt & 1) ? make_uint2(qo.z, qo.w) : make_uint2(qo.x, qo.y);
                } else {
                    be = xl[2 * u * NT + nt];
                    bo = xl[(2 * u + 1) * NT + nt];
                }
                if (u < NC) {   // first k-step of each accumulator chain
                    mma_16816_z(cE[uu % NC][nt], e0, f0, e1, f1, be.x, be.y);
                    mma_16816_z(cO[uu % NC][nt], o0, p0, o1, p1, bo.x, bo.y);
                } else {
                    mma_16816(cE[uu % NC][nt], e0, f0, e1, f1, be.x, be.y);
                    mma_16816(cO[uu % NC][nt], o0, p0, o1, p1, bo.x, bo.y);
                }
            }
        }
    }
    release();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const uint2 bm = xl[16 * NT + nt];
        mma_16816_z(cM[nt], r0.mpair, r1.mpair, 0u, 0u, bm.x, bm.y);
        float s0, s1;
        if constexpr (NC == 2) {
            s0 = ((cE[0][nt][0] + cE[1][nt][0]) + (cO[0][nt][0] + cO[1][nt][0])) +
                 ((cE[0][nt][1] + cE[1][nt][1]) + (cO[0][nt][1] + cO[1][nt][1]));
            s1 = ((cE[0][nt][2] + cE[1][nt][2]) + (cO[0][nt][2] + cO[1][nt][2])) +
                 ((cE[0][nt][3] + cE[1][nt][3]) + (cO[0][nt][3] + cO[1][nt][3]));
        } else {
            s0 = (cE[0][nt][0] + cO[0][nt][0]) + (cE[0][nt][1] + cO[0][nt][1]);
            s1 = (cE[0][nt][2] + cO[0][nt][2]) + (cE[0][nt][3] + cO[0][nt][3]);
        }
        const float m0 = cM[nt][0] + cM[nt][1];
        const float m1 = cM[nt][2] + cM[nt][3];
        acc[nt][0] = fmaf(r0.d * unscale[nt], s0, acc[nt][0]);
        acc[nt][0] = fmaf(-r0.dmin * unscale[nt], m0, acc[nt][0]);
        acc[nt][1] = fmaf(r1.d * unscale[nt], s1, acc[nt][1]);
        acc[nt][1] = fmaf(-r1.dmin * unscale[nt], m1, acc[nt][1]);
    }
}

// ---------------------------------------------------------------------------
// The kernel body.  All 8 warps consume (16 rows each); there is no producer
// warp.  Thread 0 issues the first kStages weight stages right after
// initialising the barriers; afterwards the last warp to finish reading a
// stage (a shared-memory counter per ring slot) refills that slot with the
// stage kStages ahead, so no thread ever waits for a slot to drain.
// grid = (row-tile CTAs, split) with cluster dims (1, split, 1) when split > 1.
// W is read through a 2-D TMA tensor map: [N rows] x [K/256 * 18] 8-byte
// words; one stage = one super-block of all 128 tile rows (rows beyond N are
// zero-filled by the TMA unit).
// ---------------------------------------------------------------------------
// One tensor map per matrix of the launch.
struct WMaps {
    CUtensorMap m[kMaxGroups];
};

// Matrix of a row tile and its per-matrix data, selected with compile-time
// indices only (no dynamically indexed parameter arrays, hence no local copy).
struct TileInfo {
    int grp;
    int row0;     // first row of the tile within its matrix
    int N;
    float *y;
};

template <typename Desc>
__device__ __forceinline__ TileInfo tile_info(const Desc &a, int tile)
{
    TileInfo ti{0, tile * kRows, a.N[0], a.y[0]};
#pragma unroll
    for (int i = 1; i < kMaxGroups; ++i) {
        if (i < a.ngroups && tile >= a.tile_start[i]) {
            ti.grp = i;
            ti.row0 = (tile - a.tile_start[i]) * kRows;
            ti.N = a.N[i];
            ti.y = a.y[i];
        }
    }
    return ti;
}

struct StageIssuer {
    const WMaps *maps;
    const GemvArgs *args;
    int kb_begin, ks, total;    // this CTA's schedule: total = tiles_of_cta * ks stages
    uint8_t *ring;
    uint64_t *full;
    uint64_t policy;

    // Issue global stage i of this CTA's schedule into ring slot i % kStages.
    __device__ __forceinline__ void issue(int i) const
    {
        const int tile = blockIdx.x + (i / ks) * gridDim.x;
        const int kb = kb_begin + i % ks;
        const TileInfo ti = tile_info(*args, tile);
        const CUtensorMap *map = &maps->m[0];
#pragma unroll
        for (int g = 1; g < kMaxGroups; ++g)
            if (g == ti.grp) map = &maps->m[g];
        const int slot = i % kStages;
        mbar_arrive_expect_tx(smem_u32(&full[slot]), kStageBytes);
        tma_load_2d_hint(smem_u32(ring + slot * kStageBytes), map, kb * (kBlockBytes / 8), ti.row0,
                         smem_u32(&full[slot]), policy);
    }
};

// XM: how x enters the inner product.  0: fp16 hi/lo parts on the tensor cores
// (any batch); 1: two int8 parts per element and dp4a (batch 1); 2: one int8
// code per element, Q8_K style, and dp4a (batch 1, on request).
template <int NT, bool ARGMAX, int XM>
__device__ __forceinline__ void gemv_body(const WMaps &maps, const GemvArgs &args)
{
    constexpr bool I8 = XM != 0;
    constexpr bool Q8 = XM == 2;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *ring = smem_raw;
    const int B = args.B;
    const int LW = frag_lanes(NT, B);
    uint2 *xf = reinterpret_cast<uint2 *>(smem_raw + xfrag_offset());
    float *s_red = reinterpret_cast<float *>(smem_raw + red_offset(NT, B, args.kc));
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ float s_unscale[32];   // per (super-block of the chunk, batch row)
    __shared__ float s_pre[32];       // integer path: power-of-two factor per super-block
    __shared__ unsigned long long s_best[16];
    __shared__ int s_abort;
    __shared__ int s_issued;                 // stages issued so far (for the abort drain)
    __shared__ int s_slot_done[kStages];     // warp arrivals per ring slot (monotonic)
    __shared__ int s_cons[kWarps];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int split = gridDim.y;
    const int rank = blockIdx.y;
    const int nb = args.nb;
    const int kb_begin = static_cast<int>((static_cast<long long>(rank) * nb) / split);
    const int kb_end = static_cast<int>((static_cast<long long>(rank + 1) * nb) / split);
    const int ks = kb_end - kb_begin;
    const int my_tiles = (args.tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                         static_cast<int>(gridDim.x);
    StageIssuer iss{&maps, &args, kb_begin, ks, my_tiles * ks, ring, full, 0ull};

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            s_slot_done[i] = 0;
        }
        s_abort = 0;
        fence_barrier_init();
#pragma unroll
        for (int g = 0; g < kMaxGroups; ++g)
            if (g < args.ngroups) prefetch_tensormap(&maps.m[g]);
        // The first stages stream in while the CTA sets up and, under PDL,
        // while the previous kernel finishes (weights never depend on it).
        iss.policy = l2_policy_evict_first();
        const int first = min(kStages, iss.total);
        for (int i = 0; i < first; ++i) iss.issue(i);
        s_issued = first;
    }
    if (ARGMAX && tid < 16) s_best[tid] = 0ull;
    if (tid < kWarps) s_cons[tid] = 0;
    __syncthreads();
    iss.policy = l2_policy_evict_first();
    // every CTA of a cluster has started once this phase completes; it is
    // waited for only before the first remote store, at the very end
    if (split > 1) cluster_arrive_relaxed();

    pdl_launch_dependents();
    pdl_wait();                             // x may come from the previous kernel

    const int g = lane >> 2;
    const int t = lane & 3;
    const int nchunks = (ks + args.kc - 1) / args.kc;
    const bool single_chunk = (nchunks == 1);
    // batch 1 on the integer path: int8 x parts, one block of the fragment area per super-block
    static_assert(!I8 || NT == 1, "the integer path is batch 1 only");
    uint8_t *xb = reinterpret_cast<uint8_t *>(xf);
    const int blk_bytes = static_cast<int>(xfrag_bytes_per_block(1, 1));
    if (single_chunk) {
        if constexpr (I8)
            convert_x_i8_blocks<Q8>(args.x, kb_begin, ks, xb, blk_bytes, s_unscale, s_pre, tid, kThreads);
        else
            convert_x_blocks<NT>(args.x, nb * 256, B, kb_begin, ks, xf, s_unscale, tid, kThreads);
    }
    // B-fragment lane.  Lanes whose column holds no batch row read some other
    // valid entry: MMA columns are independent, and those output columns are
    // never used.
    const int blane = (g < 2 * B) ? lane : (lane % LW);   // NT > 1: LW == 32, every lane is a valid slot
    int consumed = 0;
    const int row_off = (warp * 16 + g) * kBlockBytes;
    for (int ti_idx = 0; ti_idx < my_tiles; ++ti_idx) {
        const int tile = blockIdx.x + ti_idx * gridDim.x;
        const TileInfo ti = tile_info(args, tile);
        const int row0 = ti.row0;   // within matrix ti.grp
        const int Ng = ti.N;
        float *yg = ti.y;
        float acc[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = 0.f;
        float unscale[NT];
        int chunk_end = -1;
        for (int kbl = 0; kbl < ks; ++kbl) {
            if (!single_chunk && kbl > chunk_end) {
                const int cn = min(args.kc, ks - kbl);
                named_bar_sync(1, kThreads);     // everyone done with the previous chunk
                if constexpr (I8)
                    convert_x_i8_blocks<Q8>(args.x, kb_begin + kbl, cn, xb, blk_bytes, s_unscale, s_pre, tid, kThreads);
                else
                    convert_x_blocks<NT>(args.x, nb * 256, B, kb_begin + kbl, cn, xf, s_unscale, tid, kThreads);
                chunk_end = kbl + cn - 1;
            }
            // this super-block's x scale per batch row
            const int blk = single_chunk ? kbl : (kbl % args.kc);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int b = t + 4 * nt;
                // integer path: all four pair lanes of a row work on batch row 0
                unscale[nt] = I8 ? s_unscale[blk] : ((b < B) ? s_unscale[blk * B + b] : 0.f);
            }
            const int slot = consumed % kStages;
            const uint32_t phase = static_cast<uint32_t>((consumed / kStages) & 1);
            // After an abort the warps keep walking the same schedule (every
            // named barrier is still reached) but stop waiting.
            if (!*(volatile int *)&s_abort && !mbar_wait_bounded(smem_u32(&full[slot]), phase, kWaitLimitNs)) {
                atomicOr(&g_device_error, 1u);
                s_abort = 1;
            }
            const uint8_t *ra = ring + slot * kStageBytes + row_off;   // row g of this warp
            const uint8_t *rb = ra + 8 * kBlockBytes;                   // row g + 8
            // this lane's B fragments of this super-block (lane-major layout)
            const uint2 *xl = xf + static_cast<size_t>((single_chunk ? kbl : (kbl % args.kc)) * LW + blane) *
                                       lane_stride(NT);
            // two accumulator chains per parity at batch <= 4 (shorter chains), one above (fewer registers)
            auto release = [&]() {
                // This warp is done with the slot: the last warp to finish refills it.
                __syncwarp();
                if (lane == 0) {
                    __threadfence_block();
                    // monotonic per-slot count: the kWarps-th arrival of each round is last
                    const int prev = atomicAdd(&s_slot_done[slot], 1);
                    if (prev % kWarps == kWarps - 1) {
                        const int next = consumed + kStages;
                        if (next < iss.total && !*(volatile int *)&s_abort) {
                            iss.issue(next);
                            atomicAdd(&s_issued, 1);
                        }
                    }
                }
                ++consumed;
            };
            if constexpr (I8)
                stage_compute_i8<Q8>(ra, rb, xb + blk * blk_bytes, t, unscale[0], s_pre[blk], acc, release);
            else
                stage_compute<NT, NT == 1 ? 2 : 1>(ra, rb, xl, t, unscale, acc, release);
        }
        // ---------------- tile epilogue
        if constexpr (I8) {   // sum the four sub-block-pair lanes of each row
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                acc[0][h] += __shfl_xor_sync(0xffffffffu, acc[0][h], 1);
                acc[0][h] += __shfl_xor_sync(0xffffffffu, acc[0][h], 2);
            }
        }
        if (split == 1 && !*(volatile int *)&s_abort) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int b = t + 4 * nt;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = row0 + warp * 16 + g + 8 * h;
                    if (b < B && row < Ng) {
                        const float v = acc[nt][h];
                        if (yg) yg[static_cast<size_t>(b) * Ng + row] = v;
                        if (ARGMAX && !isnan(v)) atomicMax(&s_best[b], argmax_key(v, static_cast<uint32_t>(row)));
                    }
                }
            }
        } else if (split > 1) {
            // Push this CTA's partial rows into the shared memory of the rank
            // that owns them: rank r owns tile rows [r*128/split, (r+1)*128/split)
            // and keeps one slot per source rank in its receive buffer.  The
            // wait completes the start-of-kernel phase (all CTAs running); the
            // barrier after the tile loop orders the stores before the sums.
            cluster_wait_acquire();
            const uint32_t red_base = smem_u32(s_red);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int b = t + 4 * nt;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = warp * 16 + g + 8 * h;
                    const int owner = (row * split + split - 1) / kRows;
                    const int o0 = (owner * kRows) / split, o1 = ((owner + 1) * kRows) / split;
                    if (b < B && !*(volatile int *)&s_abort) {
                        const uint32_t off = static_cast<uint32_t>(((rank * (o1 - o0) + (row - o0)) * B + b) * 4);
                        st_shared_cluster_f32(map_shared_rank(red_base + off, owner), acc[nt][h]);
                    }
                }
            }
        }
    }
    if (lane == 0) s_cons[warp] = consumed;

    // After a timed-out wait, wait (bounded) for the copies this CTA issued but
    // did not consume, so that none of them lands after the CTA has exited.
    __syncthreads();
    if (*(volatile int *)&s_abort && tid == 0) {
        int lo = s_cons[0];
        for (int w = 1; w < kWarps; ++w) lo = min(lo, s_cons[w]);
        for (int i = lo; i < s_issued; ++i)
            if (!mbar_wait_bounded(smem_u32(&full[i % kStages]), static_cast<uint32_t>((i / kStages) & 1), kWaitLimitNs))
                break;
    }

    if (split > 1) {
        // Deterministic cross-CTA reduction: after this cluster barrier every
        // rank holds the partials of its own rows from all ranks and adds them
        // in rank order.
        cluster_arrive_release();
        cluster_wait_acquire();
        if (!*(volatile int *)&s_abort) {
            const TileInfo ti = tile_info(args, blockIdx.x);
            const int lr0 = (rank * kRows) / split;
            const int rows = ((rank + 1) * kRows) / split - lr0;
            for (int it = tid; it < rows * B; it += kThreads) {
                const int lr = it / B;
                const int b = it - lr * B;
                float sum = s_red[lr * B + b];
                for (int q = 1; q < split; ++q) sum += s_red[(q * rows + lr) * B + b];
                const int row = ti.row0 + lr0 + lr;
                if (row < ti.N) {
                    if (ti.y) ti.y[static_cast<size_t>(b) * ti.N + row] = sum;
                    if (ARGMAX && !isnan(sum)) atomicMax(&s_best[b], argmax_key(sum, static_cast<uint32_t>(row)));
                }
            }
        }
    }

    if (ARGMAX) {
        __syncthreads();
        if (tid == 0 && !*(volatile int *)&s_abort) {
            for (int b = 0; b < B; ++b)
                if (s_best[b]) atomicMax(&args.keys[b], s_best[b]);
            __threadfence();
            const unsigned total = gridDim.x * gridDim.y;
            const unsigned prev = atomicAdd(args.ticket, 1u);
            if (prev == total - 1) {
                __threadfence();
                for (int b = 0; b < B; ++b) {
                    const unsigned long long k = atomicAdd(&args.keys[b], 0ull);
                    args.idx[b] = k ? static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull)) : 0;
                }
            }
        }
    }
}

// Batch <= 8 (one or two n8 tiles): at most 128 registers, so that two CTAs of
// 8 warps (4 warps per SM sub-partition) fit in the register file.
template <int NT, bool ARGMAX, int XM = 0>
__global__ void __maxnreg__(128) q4k_gemv_kernel(const __grid_constant__ WMaps maps, const GemvArgs args)
{
    gemv_body<NT, ARGMAX, XM>(maps, args);
}

// Batch 9..16 (three or four n8 tiles): one CTA per SM, registers as needed.
template <int NT, bool ARGMAX>
__global__ void __launch_bounds__(kThreads, 1) q4k_gemv_kernel_wide(const __grid_constant__ WMaps maps,
                                                                   const GemvArgs args)
{
    gemv_body<NT, ARGMAX, 0>(maps, args);
}

// ---------------------------------------------------------------------------
// Chain: a sequence of GEMV steps (each one grouped GEMV: up to four matrices
// sharing one x) in ONE persistent launch.
//
// The CTAs of a cooperative grid stay resident across steps.  Each CTA works
// through a fixed share of every step (work unit = row tile x K slice; with
// G CTAs, unit u goes to CTA u mod G) and streams its weight stages through
// one ring for the whole chain, so the stages of step s+1 are already in
// flight while step s finishes: the same last-arriver refill as above, with
// the stage -> (step, unit, super-block) map looked up in a per-CTA table.
// Step s+1 reads x only after every CTA has finished step s (a counter in
// global memory, bounded spin), so a step may consume the output of an
// earlier one.  A K split over CTAs (a power of two dividing G, so that a
// CTA's K slice is the same for all its units of a step) is reduced without
// clusters: each slice writes its partial rows to a scratch area and the last
// slice of the tile (global ticket) adds them in slice order.
// ---------------------------------------------------------------------------
// One step as the kernel reads it from device memory (the tensor maps make it
// 128-byte aligned).
struct ChainStep {
    CUtensorMap maps[kMaxGroups];
    const float *x;
    float *y[kMaxGroups];
    int N[kMaxGroups];
    int tile_start[kMaxGroups + 1];
    int ngroups;
    int nb;      // super-blocks per row
    int tiles;   // row tiles of all matrices
    int split;   // K slices per tile (power of two dividing the grid)
    int kc;      // super-blocks per x chunk
};

// The copy each CTA keeps in shared memory, with its own K slice and unit count.
struct ChainStepS {
    float *y[kMaxGroups];
    const float *x;
    int N[kMaxGroups];
    int tile_start[kMaxGroups + 1];
    int ngroups, nb, split, kc;
    int kb0, ks, mine;   // this CTA: first super-block and length of its K slice, units
};

struct ChainArgs {
    const ChainStep *steps;
    int nsteps;
    int B;
    int kc_max;                 // x chunk capacity of the shared-memory layout
    float *partials;            // split-K partial rows [tile][slice][B][128]
    unsigned int *tickets;      // per row tile, zero between uses
    unsigned int *bar;          // arrivals of all CTAs, zeroed before the launch
};

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait until *bar >= target (bounded; gives up early once any kernel of the
// library has flagged an error).
__device__ __forceinline__ bool grid_wait(const unsigned int *bar, unsigned int target)
{
    if (ld_acquire_u32(bar) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(64);
        if (ld_acquire_u32(bar) >= target) return true;
        if (*(volatile unsigned int *)&g_device_error) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

__host__ __device__ inline size_t chain_xf_bytes(int NT, int B, int kc_max)
{
    return (xfrag_bytes_per_block(NT, B) * kc_max + 127) & ~size_t(127);
}

// Issue global stage i of this CTA's chain schedule into ring slot i % kStages.
// The slot's next stage is always kStages further on, so its step is found by
// walking forward from the step of the slot's previous stage (cursor[slot]).
__device__ __forceinline__ void chain_issue(const ChainArgs &args, const ChainStepS *s_steps, const int *s_start,
                                            int *cursor, uint8_t *ring, uint64_t *full, int i)
{
    const int slot = i % kStages;
    int si = cursor[slot];
    while (s_start[si + 1] <= i) ++si;
    cursor[slot] = si;
    const ChainStepS &st = s_steps[si];
    const int local = i - s_start[si];
    const int ul = local / st.ks;
    const int kb = st.kb0 + (local - ul * st.ks);
    const int tile = (static_cast<int>(blockIdx.x) + ul * static_cast<int>(gridDim.x)) / st.split;
    const TileInfo ti = tile_info(st, tile);
    mbar_arrive_expect_tx(smem_u32(&full[slot]), kStageBytes);
    tma_load_2d_hint(smem_u32(ring + slot * kStageBytes), &args.steps[si].maps[ti.grp], kb * (kBlockBytes / 8),
                     ti.row0, smem_u32(&full[slot]), l2_policy_evict_first());
}

template <int NT>
__device__ __forceinline__ void chain_body(const ChainArgs &args)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *ring = smem_raw;
    const int B = args.B;
    const int LW = frag_lanes(NT, B);
    uint2 *xf = reinterpret_cast<uint2 *>(smem_raw + xfrag_offset());
    ChainStepS *s_steps = reinterpret_cast<ChainStepS *>(smem_raw + xfrag_offset() + chain_xf_bytes(NT, B, args.kc_max));
    int *s_start = reinterpret_cast<int *>(s_steps + args.nsteps);   // [nsteps + 1]
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ float s_unscale[32];   // per (super-block of the chunk, batch row)
    __shared__ int s_abort;
    __shared__ int s_issued;
    __shared__ int s_last;
    __shared__ int s_slot_done[kStages];
    __shared__ int s_cons[kWarps];
    __shared__ int s_cursor[kStages];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = gridDim.x;
    const int c = blockIdx.x;
    const int nsteps = args.nsteps;

    // this CTA's copy of the steps and its number of stages per step
    for (int si = tid; si < nsteps; si += kThreads) {
        const ChainStep &st = args.steps[si];
        ChainStepS &d = s_steps[si];
#pragma unroll
        for (int g = 0; g < kMaxGroups; ++g) {
            d.y[g] = st.y[g];
            d.N[g] = st.N[g];
            d.tile_start[g] = st.tile_start[g];
        }
        d.tile_start[kMaxGroups] = st.tile_start[kMaxGroups];
        d.x = st.x;
        d.ngroups = st.ngroups;
        d.nb = st.nb;
        d.split = st.split;
        d.kc = st.kc;
        const int units = st.tiles * st.split;
        const int rank = c & (st.split - 1);
        d.mine = (c < units) ? (units - c + G - 1) / G : 0;
        d.kb0 = (rank * st.nb) / st.split;
        d.ks = ((rank + 1) * st.nb) / st.split - d.kb0;
        s_start[si + 1] = d.mine * d.ks;
    }
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            s_slot_done[i] = 0;
            s_cursor[i] = 0;
        }
        s_abort = 0;
        fence_barrier_init();
    }
    if (tid < kWarps) s_cons[tid] = 0;
    __syncthreads();
    if (tid == 0) {
        s_start[0] = 0;
        for (int si = 0; si < nsteps; ++si) s_start[si + 1] += s_start[si];
    }
    __syncthreads();
    const int total = s_start[nsteps];
    auto issue = [&](int i) { chain_issue(args, s_steps, s_start, s_cursor, ring, full, i); };

    if (tid == 0) {
        // the TMA unit reads the tensor maps from global memory: warm its
        // descriptor cache for the first two steps before the first copies
        for (int si = 0; si < min(nsteps, 2); ++si)
            for (int g = 0; g < s_steps[si].ngroups; ++g) prefetch_tensormap(&args.steps[si].maps[g]);
        const int first = min(kStages, total);
        for (int i = 0; i < first; ++i) issue(i);
        s_issued = first;
    }

    const int g = lane >> 2;
    const int t = lane & 3;
    const int blane = (g < 2 * B) ? lane : (lane % LW);
    const int row_off = (warp * 16 + g) * kBlockBytes;
    int consumed = 0;

    for (int si = 0; si < nsteps; ++si) {
        const ChainStepS &st = s_steps[si];
        const int split = st.split;
        const int rank = c & (split - 1);
        const int kb_begin = st.kb0;
        const int ks = st.ks;
        const int mine = st.mine;
        // x of this step may be an output of an earlier step: wait until
        // every CTA has finished step si - 1
        if (tid == 32 && si + 2 < nsteps)   // maps of the step after next (its copies start during step si + 1)
            for (int gi = 0; gi < s_steps[si + 2].ngroups; ++gi) prefetch_tensormap(&args.steps[si + 2].maps[gi]);
        if (mine > 0) prefetch_x_l2(st.x, st.nb * 256, B, kb_begin, kb_begin + ks, tid, kThreads);
        if (si > 0) {
            if (tid == 0 && !*(volatile int *)&s_abort && !grid_wait(args.bar, static_cast<unsigned>(si * G))) {
                atomicOr(&g_device_error, 1u);
                s_abort = 1;
            }
            __syncthreads();
        }
        if (mine > 0 && !*(volatile int *)&s_abort) {
            const int kc = st.kc;
            const bool single_chunk = ks <= kc;
            if (single_chunk) convert_x_blocks<NT, true>(st.x, st.nb * 256, B, kb_begin, ks, xf, s_unscale, tid, kThreads);
            for (int ul = 0; ul < mine; ++ul) {
                float acc[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = 0.f;
                float unscale[NT];
                int chunk_end = -1;
                for (int kbl = 0; kbl < ks; ++kbl) {
                    if (!single_chunk && kbl > chunk_end) {
                        const int cn = min(kc, ks - kbl);
                        named_bar_sync(1, kThreads);   // everyone done with the previous chunk
                        convert_x_blocks<NT, true>(st.x, st.nb * 256, B, kb_begin + kbl, cn, xf, s_unscale, tid,
                                                   kThreads);
                        chunk_end = kbl + cn - 1;
                    }
                    const int blk = single_chunk ? kbl : (kbl % kc);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int b = t + 4 * nt;
                        unscale[nt] = (b < B) ? s_unscale[blk * B + b] : 0.f;
                    }
                    const int slot = consumed % kStages;
                    const uint32_t phase = static_cast<uint32_t>((consumed / kStages) & 1);
                    if (!*(volatile int *)&s_abort && !mbar_wait_bounded(smem_u32(&full[slot]), phase, kWaitLimitNs)) {
                        atomicOr(&g_device_error, 1u);
                        s_abort = 1;
                    }
                    const uint8_t *ra = ring + slot * kStageBytes + row_off;
                    const uint8_t *rb = ra + 8 * kBlockBytes;
                    const uint2 *xl =
                        xf + static_cast<size_t>((single_chunk ? kbl : (kbl % kc)) * LW + blane) * lane_stride(NT);
                    // the refill runs after the stage (fewer live registers than
                    // inside it: the stage-to-step lookup is longer here)
                    stage_compute<NT, 1>(ra, rb, xl, t, unscale, acc, []() {});
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
                // ---------------- unit epilogue
                const int tile = (c + ul * G) / split;
                const TileInfo ti = tile_info(st, tile);
                if (split == 1) {
                    if (!*(volatile int *)&s_abort) {
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const int b = t + 4 * nt;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int row = ti.row0 + warp * 16 + g + 8 * h;
                                if (b < B && row < ti.N) ti.y[static_cast<size_t>(b) * ti.N + row] = acc[nt][h];
                            }
                        }
                    }
                } else {
                    float *part = args.partials + static_cast<size_t>(tile * split + rank) * B * kRows;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int b = t + 4 * nt;
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            if (b < B) part[b * kRows + warp * 16 + g + 8 * h] = acc[nt][h];
                    }
                    __syncthreads();
                    if (tid == 0) {
                        __threadfence();
                        const unsigned prev = atomicAdd(&args.tickets[tile], 1u);
                        s_last = (prev == static_cast<unsigned>(split - 1));
                    }
                    __syncthreads();
                    if (s_last) {
                        // every slice of the tile is in: add them in slice order
                        __threadfence();
                        const float *p0 = args.partials + static_cast<size_t>(tile * split) * B * kRows;
                        for (int idx = tid; idx < B * kRows; idx += kThreads) {
                            float sum = __ldcg(p0 + idx);
                            for (int q = 1; q < split; ++q) sum += __ldcg(p0 + static_cast<size_t>(q) * B * kRows + idx);
                            const int b = idx / kRows;
                            const int row = ti.row0 + (idx - b * kRows);
                            if (row < ti.N && !*(volatile int *)&s_abort) ti.y[static_cast<size_t>(b) * ti.N + row] = sum;
                        }
                        if (tid == 0) args.tickets[tile] = 0u;
                    }
                }
            }
        }
        // this CTA's share of step si is done: its outputs are written and its x is read
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            atomicAdd(args.bar, 1u);
        }
    }
    if (lane == 0) s_cons[warp] = consumed;

    // After a timed-out wait: wait (bounded) for the copies issued but not consumed.
    __syncthreads();
    if (*(volatile int *)&s_abort && tid == 0) {
        int lo = s_cons[0];
        for (int w = 1; w < kWarps; ++w) lo = min(lo, s_cons[w]);
        for (int i = lo; i < s_issued; ++i)
            if (!mbar_wait_bounded(smem_u32(&full[i % kStages]), static_cast<uint32_t>((i / kStages) & 1), kWaitLimitNs))
                break;
    }
}

template <int NT>
__global__ void __maxnreg__(128) q4k_chain_kernel(const __grid_constant__ ChainArgs args)
{
    chain_body<NT>(args);
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) q4k_chain_kernel_wide(const __grid_constant__ ChainArgs args)
{
    chain_body<NT>(args);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct DeviceInfo {
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    size_t smem_optin = 0;
    bool ok = false;
};

static DeviceInfo g_dev[64];
static std::once_flag g_dev_once[64];

static const DeviceInfo &device_info(int dev)
{
    std::call_once(g_dev_once[dev & 63], [dev]() {
        DeviceInfo &d = g_dev[dev & 63];
        cudaDeviceProp p;
        if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) return;
        d.sms = p.multiProcessorCount;
        d.cc_major = p.major;
        d.cc_minor = p.minor;
        d.smem_optin = p.sharedMemPerBlockOptin;
        d.ok = true;
    });
    return g_dev[dev & 63];
}

q4k_status check_device(int *sms_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4K_ERR_CUDA;
    const DeviceInfo &d = device_info(dev);
    if (!d.ok) return Q4K_ERR_CUDA;
    if (d.cc_major != 10 || d.cc_minor != 3) return Q4K_ERR_UNSUPPORTED_DEVICE;
    if (sms_out) *sms_out = d.sms;
    return Q4K_OK;
}

struct GemvPlan {
    int NT;
    int xm;         // x mode of the batch-1 kernel: 0 tensor cores, 1 two int8 parts, 2 Q8_K codes
    int split;
    int grid_x;
    int tiles;
    int kc;
    size_t smem;
};

static int batch_ntiles(int B) { return (2 * B + 7) / 8; }

// Pick the K split: minimise (max row-tile units per SM) x (blocks per unit
// + per-CTA overhead), preferring fewer CTAs on ties.
// How many thread-block clusters of `size` CTAs (1..16; above 8 only with the
// non-portable opt-in) the batch <= 8 GEMV kernels can keep resident at once
// on the current device, at their largest shared-memory footprint (two CTAs
// per SM).  The planner uses it to keep a K split within one wave.
static int max_resident_clusters(int size)
{
    static int table[64][17];
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::call_once(once[dev], [dev]() {
        void (*kern)(const WMaps, const GemvArgs) = q4k_gemv_kernel<1, false>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemPerCta2));
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        for (int c = 1; c <= 16; ++c) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(1, c, 1);
            cfg.blockDim = dim3(kThreads, 1, 1);
            cfg.dynamicSmemBytes = kSmemPerCta2;
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

static GemvPlan make_plan(int tiles, int64_t K, int B, int sms, int forced_split)
{
    GemvPlan p{};
    const int nb = static_cast<int>(K / 256);
    p.NT = batch_ntiles(B);
    p.xm = (B == 1) ? 1 : 0;
    p.tiles = tiles;
    int best_s = 1;
    if (forced_split > 0) {
        best_s = std::min(std::min(forced_split, nb), 8);
    } else {
        // Cost = (units on the busiest SM) x (blocks per unit + per-CTA
        // overhead) / (units that run concurrently on it, at most the CTAs per
        // SM): a lone CTA is latency-bound and cannot use the whole SM.
        // Splits above 8 (non-portable cluster sizes, batch <= 8 kernels) only
        // when all of the tile's clusters stay resident in one wave.
        const int cps = (p.NT <= 2) ? 2 : 1;
        double best = 1e30;
        const int smax = std::min(nb, p.NT <= 2 ? 16 : 8);
        for (int s = 1; s <= smax; ++s) {
            if (s > 8 && max_resident_clusters(s) < p.tiles) continue;
            const long long units = static_cast<long long>(p.tiles) * s;
            const long long per_sm = (units + sms - 1) / sms;
            const int per_unit = (nb + s - 1) / s;
            const double conc = static_cast<double>(std::min<long long>(per_sm, cps));
            const double cost = static_cast<double>(per_sm) * (per_unit + 0.75) / conc;
            if (cost < best - 1e-9) { best = cost; best_s = s; }
        }
    }
    p.split = best_s;
    const int ks_max = (nb + p.split - 1) / p.split;
    const size_t per_blk = xfrag_bytes_per_block(p.NT, B);
    const size_t fixed = gemv_smem_bytes(p.NT, B, 0, p.split) + 128;
    const size_t budget = (p.NT <= 2) ? kSmemPerCta2 : kSmemPerCta1;
    int kc = static_cast<int>(std::max<size_t>(1, (budget - fixed) / per_blk));
    // the conversion holds at most 8 float4 of x per thread: B * kc * 64 <= 8 * 256
    kc = std::min(kc, std::max(1, 32 / B));
    p.kc = std::min(kc, ks_max);
    p.smem = gemv_smem_bytes(p.NT, B, p.kc, p.split);
    if (p.split == 1) {
        const int ctas_per_sm = (p.NT <= 2) ? 2 : 1;
        p.grid_x = std::min(p.tiles, sms * ctas_per_sm);
    } else {
        p.grid_x = p.tiles;
    }
    return p;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// W as a 2-D tensor of 8-byte words: [N rows] x [K/256 * 18 words], box =
// one super-block (18 words) of kRows rows.
static bool encode_w_map(CUtensorMap *map, const void *W, int64_t N, int64_t K)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const int64_t nb = K / 256;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(nb * (kBlockBytes / 8)), static_cast<cuuint64_t>(N)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(nb * kBlockBytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockBytes / 8), static_cast<cuuint32_t>(kRows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(W), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int NT, bool ARGMAX, int XM = 0>
static cudaError_t launch_one(const GemvPlan &p, const WMaps &maps, const GemvArgs &a, cudaStream_t stream,
                              bool pdl)
{
    void (*kern)(const WMaps, const GemvArgs);
    if constexpr (NT <= 2)
        kern = q4k_gemv_kernel<NT, ARGMAX, XM>;
    else
        kern = q4k_gemv_kernel_wide<NT, ARGMAX>;
    static std::mutex mu;
    static int smem_set[64] = {0};   // per device: largest dynamic smem size already allowed
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (smem_set[dev & 63] < static_cast<int>(p.smem)) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(p.smem));
            if (e != cudaSuccess) return e;
            // all of the unified L1 / shared array as shared memory, so that two
            // CTAs fit on an SM
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
            if (e != cudaSuccess) return e;
            // K splits over up to 16 CTAs (clusters above 8 are non-portable)
            if (NT <= 2) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e != cudaSuccess) return e;
            }
            smem_set[dev & 63] = static_cast<int>(p.smem);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid_x, p.split, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.split > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = p.split;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    // Batch-1 launches with clusters above 8 CTAs go without PDL: placed early
    // beside the previous kernel's CTAs, not all of their clusters found room
    // at once (measured: the down projection after gate/up, 15.9 us with PDL,
    // 13.8 us without; the tensor-core kernels gain from PDL there).
    if (pdl && !(XM != 0 && p.split > 8)) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, maps, a);
    if (e != cudaSuccess) (void)cudaGetLastError();   // a failed launch leaves no sticky error behind
    return e;
}

template <bool ARGMAX>
static cudaError_t launch_gemv(const GemvPlan &p, const void *const *Ws, int64_t K, const GemvArgs &a,
                               cudaStream_t s, bool pdl)
{
    WMaps maps;
    memset(&maps, 0, sizeof(maps));
    for (int g = 0; g < a.ngroups; ++g)
        if (!encode_w_map(&maps.m[g], Ws[g], a.N[g], K)) return cudaErrorInvalidValue;
    switch (p.NT) {
        case 1:
            if (p.xm == 1) return launch_one<1, ARGMAX, 1>(p, maps, a, s, pdl);
            if (p.xm == 2) return launch_one<1, ARGMAX, 2>(p, maps, a, s, pdl);
            return launch_one<1, ARGMAX, 0>(p, maps, a, s, pdl);
        case 2: return launch_one<2, ARGMAX>(p, maps, a, s, pdl);
        case 3: return launch_one<3, ARGMAX>(p, maps, a, s, pdl);
        default: return launch_one<4, ARGMAX>(p, maps, a, s, pdl);
    }
}

static int row_tiles(int64_t N) { return static_cast<int>((N + kRows - 1) / kRows); }

static q4k_status validate(const void *W, const void *x, const void *out, int64_t N, int64_t K, int batch,
                           bool argmax)
{
    if (!x) return Q4K_ERR_INVALID_ARG;
    if ((!W || !out) && !(N == 0 && !argmax)) return Q4K_ERR_INVALID_ARG;   // N == 0: W, y are never touched
    if (N < 0 || K <= 0 || (K % 256) != 0 || K / 256 >= (1ll << 24)) return Q4K_ERR_INVALID_ARG;
    if (batch < 1 || batch > Q4K_MAX_BATCH) return Q4K_ERR_INVALID_ARG;
    if (argmax && (N < 1 || N > 0x7FFFFFFFll)) return Q4K_ERR_INVALID_ARG;
    if (N > 0x7FFFFFFFll) return Q4K_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15u) || (reinterpret_cast<uintptr_t>(x) & 15u)) return Q4K_ERR_MISALIGNED;
    return Q4K_OK;
}

q4k_status gemv_impl(const void *W, const float *x, float *y, int64_t N, int64_t K, int batch, void *stream,
                     const q4k_launch_opts *opts)
{
    q4k_status st = validate(W, x, y, N, K, batch, false);
    if (st != Q4K_OK) return st;
    int sms = 0;
    st = check_device(&sms);
    if (st != Q4K_OK) return st;
    if (N == 0) return Q4K_OK;
    const int forced = opts ? opts->split_k : 0;
    if (forced < 0 || forced > 8) return Q4K_ERR_INVALID_ARG;
    GemvPlan p = make_plan(row_tiles(N), K, batch, sms, forced);
    GemvArgs a{};
    a.x = x;
    a.y[0] = y;
    a.N[0] = static_cast<int>(N);
    a.ngroups = 1;
    a.tile_start[0] = 0;
    a.tile_start[1] = p.tiles;
    a.nb = static_cast<int>(K / 256);
    a.B = batch;
    a.tiles = p.tiles;
    a.kc = p.kc;
    const bool pdl = opts && (opts->flags & Q4K_FLAG_PDL);
    if (opts && (opts->flags & Q4K_FLAG_TENSOR_CORE)) p.xm = 0;
    if (opts && (opts->flags & Q4K_FLAG_Q8K_X)) {
        if (batch != 1 || (opts->flags & Q4K_FLAG_TENSOR_CORE)) return Q4K_ERR_INVALID_ARG;
        p.xm = 2;
    }
    cudaError_t e = launch_gemv<false>(p, &W, K, a, static_cast<cudaStream_t>(stream), pdl);
    return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
}

q4k_status gemv_grouped_impl(const q4k_gemv_group *groups, int ngroups, const float *x, int64_t K, int batch,
                             void *stream, const q4k_launch_opts *opts)
{
    if (!groups || ngroups < 1 || ngroups > kMaxGroups) return Q4K_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int g = 0; g < ngroups; ++g) {
        q4k_status st = validate(groups[g].W, x, groups[g].y, groups[g].N, K, batch, false);
        if (st != Q4K_OK) return st;
        total += groups[g].N;
    }
    int sms = 0;
    q4k_status st = check_device(&sms);
    if (st != Q4K_OK) return st;
    const int forced = opts ? opts->split_k : 0;
    if (forced < 0 || forced > 8) return Q4K_ERR_INVALID_ARG;
    GemvArgs a{};
    const void *Ws[kMaxGroups] = {nullptr, nullptr, nullptr, nullptr};
    int tiles = 0;
    for (int g = 0; g < ngroups; ++g) {
        if (groups[g].N == 0) continue;          // empty matrices take no tiles
        const int i = a.ngroups++;
        Ws[i] = groups[g].W;
        a.y[i] = groups[g].y;
        a.N[i] = static_cast<int>(groups[g].N);
        a.tile_start[i] = tiles;
        tiles += row_tiles(groups[g].N);
    }
    if (a.ngroups == 0) return Q4K_OK;
    a.tile_start[a.ngroups] = tiles;
    (void)total;
    GemvPlan p = make_plan(tiles, K, batch, sms, forced);
    a.x = x;
    a.nb = static_cast<int>(K / 256);
    a.B = batch;
    a.tiles = p.tiles;
    a.kc = p.kc;
    const bool pdl = opts && (opts->flags & Q4K_FLAG_PDL);
    if (opts && (opts->flags & Q4K_FLAG_TENSOR_CORE)) p.xm = 0;
    if (opts && (opts->flags & Q4K_FLAG_Q8K_X)) {
        if (batch != 1 || (opts->flags & Q4K_FLAG_TENSOR_CORE)) return Q4K_ERR_INVALID_ARG;
        p.xm = 2;
    }
    cudaError_t e = launch_gemv<false>(p, Ws, K, a, static_cast<cudaStream_t>(stream), pdl);
    return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
}

q4k_status gemv_argmax_impl(const void *W, const float *x, int32_t *idx, float *logits, int64_t N, int64_t K,
                            int batch, void *stream, unsigned long long *scratch_keys, unsigned int *scratch_ticket,
                            const q4k_launch_opts *opts)
{
    q4k_status st = validate(W, x, idx, N, K, batch, true);
    if (st != Q4K_OK) return st;
    int sms = 0;
    st = check_device(&sms);
    if (st != Q4K_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int forced = opts ? opts->split_k : 0;
    if (forced < 0 || forced > 8) return Q4K_ERR_INVALID_ARG;
    GemvPlan p = make_plan(row_tiles(N), K, batch, sms, forced);
    GemvArgs a{};
    a.x = x;
    a.y[0] = logits;
    a.N[0] = static_cast<int>(N);
    a.ngroups = 1;
    a.tile_start[0] = 0;
    a.tile_start[1] = p.tiles;
    a.nb = static_cast<int>(K / 256);
    a.B = batch;
    a.tiles = p.tiles;
    a.kc = p.kc;
    a.idx = idx;
    const bool pdl = opts && (opts->flags & Q4K_FLAG_PDL);
    if (opts && (opts->flags & Q4K_FLAG_TENSOR_CORE)) p.xm = 0;
    if (opts && (opts->flags & Q4K_FLAG_Q8K_X)) {
        if (batch != 1 || (opts->flags & Q4K_FLAG_TENSOR_CORE)) return Q4K_ERR_INVALID_ARG;
        p.xm = 2;
    }
    void *buf = nullptr;
    const size_t bytes = 8 * 16 + 16;
    if (scratch_keys == nullptr) {
        if (cudaMallocAsync(&buf, bytes, s) != cudaSuccess) return Q4K_ERR_CUDA;
        if (cudaMemsetAsync(buf, 0, bytes, s) != cudaSuccess) {
            cudaFreeAsync(buf, s);
            return Q4K_ERR_CUDA;
        }
        a.keys = static_cast<unsigned long long *>(buf);
        a.ticket = reinterpret_cast<unsigned int *>(static_cast<uint8_t *>(buf) + 8 * 16);
    } else {
        a.keys = scratch_keys;
        a.ticket = scratch_ticket;
    }
    cudaError_t e = launch_gemv<true>(p, &W, K, a, s, pdl);
    if (buf) {
        cudaError_t e2 = cudaFreeAsync(buf, s);
        if (e == cudaSuccess) e = e2;
    }
    return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the fused argmax.
//
// For callers that cannot allocate device memory while they run -- code that
// works from a fixed, pre-sized memory budget, real-time loops that forbid any
// allocator call, or processes whose stream-ordered allocator is unavailable
// or replaced -- the argmax's small scratch (one 64-bit key per batch row plus
// a CTA ticket) lives in this file-scope device array instead of coming from
// cudaMallocAsync.  Every GPU that loads the library holds these bytes until
// the process exits.  Host code cannot use the array's name as a device
// address, so the address is looked up with cudaGetSymbolAddress once per
// device (with that device current) on the first call there; make that first
// call before any stream capture.  All calls share the array: it is cleared
// with cudaMemsetAsync on the caller's stream before every launch, and calls
// whose executions overlap on the GPU (different streams, concurrent graphs)
// race on it.
// ---------------------------------------------------------------------------
constexpr int kNoAllocMaxBatch = 16;   // keys held by the static scratch
__device__ __align__(256) static unsigned long long g_argmax_scratch[kNoAllocMaxBatch + 2];

static unsigned long long *g_scratch_addr[64];
static std::once_flag g_scratch_once[64];
static cudaError_t g_scratch_err[64];

q4k_status gemv_argmax_noalloc_impl(const void *W, const float *x, int32_t *idx, int64_t N, int64_t K, int batch,
                                    void *stream)
{
    if (batch > kNoAllocMaxBatch) return Q4K_ERR_INVALID_ARG;   // beyond the static scratch
    q4k_status st = validate(W, x, idx, N, K, batch, true);
    if (st != Q4K_OK) return st;
    st = check_device(nullptr);
    if (st != Q4K_OK) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q4K_ERR_CUDA;
    std::call_once(g_scratch_once[dev], [dev]() {
        void *p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_argmax_scratch);
        g_scratch_addr[dev] = static_cast<unsigned long long *>(p);
    });
    if (g_scratch_err[dev] != cudaSuccess || g_scratch_addr[dev] == nullptr) return Q4K_ERR_CUDA;
    unsigned long long *keys = g_scratch_addr[dev];
    unsigned int *ticket = reinterpret_cast<unsigned int *>(keys + kNoAllocMaxBatch);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(keys, 0, sizeof(g_argmax_scratch), s) != cudaSuccess) return Q4K_ERR_CUDA;
    return gemv_argmax_impl(W, x, idx, nullptr, N, K, batch, stream, keys, ticket, nullptr);
}

q4k_status gemv_plan_impl(int64_t N, int64_t K, int batch, int out[4])
{
    if (!out || N < 0 || K <= 0 || K % 256 || batch < 1 || batch > Q4K_MAX_BATCH) return Q4K_ERR_INVALID_ARG;
    int sms = 0;
    q4k_status st = check_device(&sms);
    if (st != Q4K_OK) return st;
    GemvPlan p = make_plan(row_tiles(N), K, batch, sms, 0);
    out[0] = p.split;
    out[1] = p.grid_x * p.split;
    out[2] = kRows;
    out[3] = p.kc;
    return Q4K_OK;
}

// ---------------------------------------------------------------------------
// Chains (host side)
// ---------------------------------------------------------------------------
// K split of one chain step: a power of two dividing the grid (so that a CTA's
// K slice is the same for all its units), chosen to minimise (units on the
// busiest CTA) x (super-blocks per unit + per-unit overhead), with a small
// charge for the partial-sum fix-up.
static int chain_split(int tiles, int nb, int G)
{
    int best = 1;
    double best_cost = 1e30;
    for (int s = 1; s <= 16 && s <= nb; s *= 2) {
        if (G % s) break;
        const long long units = static_cast<long long>(tiles) * s;
        const long long per_cta = (units + G - 1) / G;
        const int per_unit = (nb + s - 1) / s;
        const double cost = static_cast<double>(per_cta) * (per_unit + 0.75) + (s > 1 ? 0.25 : 0.0);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

template <int NT>
static void (*chain_kernel())(const ChainArgs)
{
    if constexpr (NT <= 2)
        return q4k_chain_kernel<NT>;
    else
        return q4k_chain_kernel_wide<NT>;
}

static void (*chain_kernel_for(int NT))(const ChainArgs)
{
    switch (NT) {
        case 1: return chain_kernel<1>();
        case 2: return chain_kernel<2>();
        case 3: return chain_kernel<3>();
        default: return chain_kernel<4>();
    }
}

}  // namespace q4k

struct q4k_chain {
    int dev;
    int NT;
    int grid;
    size_t smem;
    size_t counter_bytes;   // tickets + barrier counter, cleared before every run
    void *dmem;
    q4k::ChainArgs args;
};

namespace q4k {

q4k_status chain_create_impl(const q4k_chain_step *steps, int nsteps, int batch, q4k_chain **chain)
{
    if (!chain) return Q4K_ERR_INVALID_ARG;
    *chain = nullptr;
    if (!steps || nsteps < 1 || nsteps > Q4K_CHAIN_MAX_STEPS || batch < 1 || batch > Q4K_MAX_BATCH)
        return Q4K_ERR_INVALID_ARG;
    for (int si = 0; si < nsteps; ++si) {
        const q4k_chain_step &st = steps[si];
        if (!st.x || st.ngroups < 1 || st.ngroups > kMaxGroups) return Q4K_ERR_INVALID_ARG;
        if (st.K <= 0 || (st.K % 256) != 0 || st.K / 256 >= (1ll << 24)) return Q4K_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(st.x) & 15u) return Q4K_ERR_MISALIGNED;
        for (int g = 0; g < st.ngroups; ++g) {
            const q4k_gemv_group &gr = st.groups[g];
            if (gr.N < 0 || gr.N > 0x7FFFFFFFll) return Q4K_ERR_INVALID_ARG;
            if (gr.N == 0) continue;
            if (!gr.W || !gr.y) return Q4K_ERR_INVALID_ARG;
            if (reinterpret_cast<uintptr_t>(gr.W) & 15u) return Q4K_ERR_MISALIGNED;
        }
    }
    int sms = 0;
    q4k_status st = check_device(&sms);
    if (st != Q4K_OK) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4K_ERR_CUDA;

    const int NT = batch_ntiles(batch);
    const int cps = (NT <= 2) ? 2 : 1;
    // shared memory: W ring | x chunk | step table
    const size_t table = static_cast<size_t>(nsteps) * sizeof(ChainStepS) + static_cast<size_t>(nsteps + 1) * 4;
    const size_t budget = (NT <= 2) ? kSmemPerCta2 : kSmemPerCta1;
    const size_t per_blk = xfrag_bytes_per_block(NT, batch);
    if (xfrag_offset() + table + chain_xf_bytes(NT, batch, 1) > budget) return Q4K_ERR_INVALID_ARG;
    int kc_need = 1;
    for (int si = 0; si < nsteps; ++si) kc_need = std::max(kc_need, static_cast<int>(steps[si].K / 256));
    int kc_max = static_cast<int>((budget - xfrag_offset() - table) / per_blk);
    while (kc_max > 1 && xfrag_offset() + table + chain_xf_bytes(NT, batch, kc_max) > budget) --kc_max;
    kc_max = std::max(1, std::min(std::min(kc_max, 32 / batch), kc_need));
    const size_t smem = xfrag_offset() + chain_xf_bytes(NT, batch, kc_max) + table;

    void (*kern)(const ChainArgs) = chain_kernel_for(NT);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess) {
        (void)cudaGetLastError();
        return Q4K_ERR_CUDA;
    }
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem) != cudaSuccess || occ < 1) {
        (void)cudaGetLastError();
        return Q4K_ERR_CUDA;
    }
    const int G = sms * std::min(occ, cps);

    // the device-side step table
    std::vector<ChainStep> hs(nsteps);
    size_t partial_floats = 0;
    int max_tiles = 1;
    for (int si = 0; si < nsteps; ++si) {
        const q4k_chain_step &in = steps[si];
        ChainStep &d = hs[si];
        memset(&d, 0, sizeof(d));
        d.x = in.x;
        d.nb = static_cast<int>(in.K / 256);
        int tiles = 0;
        for (int g = 0; g < in.ngroups; ++g) {
            const q4k_gemv_group &gr = in.groups[g];
            if (gr.N == 0) continue;
            const int i = d.ngroups++;
            d.y[i] = gr.y;
            d.N[i] = static_cast<int>(gr.N);
            d.tile_start[i] = tiles;
            tiles += row_tiles(gr.N);
            if (!encode_w_map(&d.maps[i], gr.W, gr.N, in.K)) return Q4K_ERR_CUDA;
        }
        for (int g = d.ngroups; g <= kMaxGroups; ++g) d.tile_start[g] = tiles;
        d.tiles = tiles;
        d.split = tiles > 0 ? chain_split(tiles, d.nb, G) : 1;
        const int ks_max = (d.nb + d.split - 1) / d.split;
        d.kc = std::min(kc_max, ks_max);
        if (d.split > 1) {
            partial_floats = std::max(partial_floats, static_cast<size_t>(tiles) * d.split * batch * kRows);
            max_tiles = std::max(max_tiles, tiles);
        }
    }
    // one allocation: steps | partial rows | tickets | barrier counter
    const size_t steps_bytes = (static_cast<size_t>(nsteps) * sizeof(ChainStep) + 255) & ~size_t(255);
    const size_t part_bytes = (partial_floats * 4 + 255) & ~size_t(255);
    const size_t counter_bytes = static_cast<size_t>(max_tiles + 1) * 4;
    void *dmem = nullptr;
    if (cudaMalloc(&dmem, steps_bytes + part_bytes + counter_bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return Q4K_ERR_CUDA;
    }
    uint8_t *base = static_cast<uint8_t *>(dmem);
    if (cudaMemcpy(base, hs.data(), static_cast<size_t>(nsteps) * sizeof(ChainStep), cudaMemcpyHostToDevice) !=
        cudaSuccess) {
        cudaFree(dmem);
        return Q4K_ERR_CUDA;
    }
    q4k_chain *ch = new (std::nothrow) q4k_chain;
    if (!ch) {
        cudaFree(dmem);
        return Q4K_ERR_CUDA;
    }
    ch->dev = dev;
    ch->NT = NT;
    ch->grid = G;
    ch->smem = smem;
    ch->counter_bytes = counter_bytes;
    ch->dmem = dmem;
    ch->args.steps = reinterpret_cast<const ChainStep *>(base);
    ch->args.nsteps = nsteps;
    ch->args.B = batch;
    ch->args.kc_max = kc_max;
    ch->args.partials = reinterpret_cast<float *>(base + steps_bytes);
    ch->args.tickets = reinterpret_cast<unsigned int *>(base + steps_bytes + part_bytes);
    ch->args.bar = ch->args.tickets + max_tiles;
    *chain = ch;
    return Q4K_OK;
}

q4k_status chain_run_impl(const q4k_chain *ch, void *stream)
{
    if (!ch) return Q4K_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4K_ERR_CUDA;
    if (dev != ch->dev) return Q4K_ERR_INVALID_ARG;   // the chain's memory lives on another device
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ch->args.tickets, 0, ch->counter_bytes, s) != cudaSuccess) return Q4K_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ch->grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = ch->smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: they wait for one another between steps
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, chain_kernel_for(ch->NT), ch->args);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return Q4K_ERR_CUDA;
    }
    return Q4K_OK;
}

q4k_status chain_destroy_impl(q4k_chain *ch)
{
    if (!ch) return Q4K_OK;
    const cudaError_t e = cudaFree(ch->dmem);
    delete ch;
    return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
}

unsigned int read_device_error()
{
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    return v;
}

}  // namespace q4k
