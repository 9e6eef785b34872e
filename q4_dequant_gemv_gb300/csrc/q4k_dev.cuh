// q4k_dev.cuh -- device code shared by the Q4_K GEMV kernels (q4k_gemv.cu) and
// the persistent decode-step kernel (q4k_chain.cu): the super-block header
// decode, the two inner products (integer dp4a for batch 1, mma.sync for any
// batch) and the conversion of x into the forms they consume.
//
// What is computed per super-block and weight row: the contribution
//   d * sum_j sc_j * sum_i q[32j+i] x[32j+i]  -  dmin * sum_j m_j * sum_i x[32j+i]
// of w = d*sc_j*q - dmin*m_j to y = W x ("fused scale x int dot-product kernels
// operating directly on quantized blocks", dotLLM README, Key Features /
// Performance): the 4-bit quants are multiplied with x as integers, the
// sub-block sums of x carry the min term, and the two scales are applied once
// per sub-block and super-block.
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace q4k {

constexpr int kBlockBytes = 144;
constexpr int kKsteps = 17;               // 16 k16 steps + 1 min-term step per super-block

__host__ __device__ inline int frag_lanes(int NT, int B) { return NT == 1 ? 8 * B : 32; }

// B fragments are stored lane-major: the 17*NT entries (uint2) of one lane for
// one super-block are contiguous, so a consumer lane reads them at constant
// offsets from one base.
__host__ __device__ constexpr int lane_stride(int NT)
{
    // even for NT = 1, 2, 4 (16-byte aligned lanes: a k-step's even and odd
    // fragments load as one 16-byte access; lane L starts at bank 4L mod 32, so
    // the eight lanes of a 16-byte wavefront hit distinct banks); NT = 3 loads
    // 8-byte fragments and keeps an odd stride
    return NT == 3 ? kKsteps * NT : kKsteps * NT + ((kKsteps * NT) & 1);
}

__host__ __device__ inline size_t xfrag_bytes_per_block(int NT, int B)
{
    return static_cast<size_t>(lane_stride(NT)) * frag_lanes(NT, B) * 8;
}

// x -> fp16 hi/lo B fragments in shared memory, per super-block.
// Entry (bl, s, nt, L) is a uint2 {b01, b23} for lane L = 4*col8 + t of n-tile
// nt at k-step s of local super-block bl.  Thread t of an A fragment handles
// sub-block pair t of each super-block (sub-blocks 2t and 2t+1), so for k-step
// s < 16 (word u = s/2, sub-block 2t + (s&1)) the four B values are the x
// entries 4u..4u+3 of that sub-block ordered {4u, 4u+2 | 4u+1, 4u+3}.  Step 16
// holds the sub-block sums of x for sub-blocks 2t, 2t+1 (the dmin*m term).
// Power-of-two scale 2^s with max|x| * 2^s in [2^9, 2^10) (s = 0 for an all
// zero or non-finite super-block), clamped to the normal range.
__device__ __forceinline__ int chunk_scale_exp(uint32_t amax_bits)
{
    const int E = static_cast<int>((amax_bits >> 23) & 255u);
    int s = (amax_bits != 0u && E != 255) ? 136 - E : 0;
    return max(-126, min(126, s));
}

// One (batch row b, super-block) item of x -> its fp16 hi/lo B fragments and
// the hi/lo sub-block sums, written into the super-block's fragment block xfb
// (lane-major, LW lanes of lane_stride(NT) uint2 each), by one warp.  v0, v1 =
// float4 number lane and lane + 32 of the super-block (elements 4i..4i+3, i =
// lane or lane + 32: sub-block i/8, word i%8).  The item gets its own
// power-of-two scale 2^e (warp max); returns 2^-e, the factor that undoes it.
// Float4 i is sub-block j = i/8 (pair t = j/2, half h = j%2), word u = i%8 ->
// k-step s = 2u + h of pair t.
template <int NT>
__device__ __forceinline__ float x_item_tc(float4 v0, float4 v1, int lane, int b, int LW, uint2 *xfb)
{
    (void)LW;
    constexpr int LS = lane_stride(NT);
    uint32_t m = 0u;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const float4 w = h2 ? v1 : v0;
        m = max(m, max(max(__float_as_uint(fabsf(w.x)), __float_as_uint(fabsf(w.y))),
                       max(__float_as_uint(fabsf(w.z)), __float_as_uint(fabsf(w.w)))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int e = chunk_scale_exp(m);
    const float sc = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    const int chi = 2 * b, clo = 2 * b + 1;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const int i = lane + 32 * h2;
        float4 w = h2 ? v1 : v0;
        w.x *= sc; w.y *= sc; w.z *= sc; w.w *= sc;
        const int sb = i >> 3, u = i & 7;
        const int t = sb >> 1, s = 2 * u + (sb & 1);
        const uint32_t h01 = pack_half2(w.x, w.z);
        const uint32_t h23 = pack_half2(w.y, w.w);
        const uint32_t l01 = pack_half2(w.x - half_lo_f32(h01), w.z - half_hi_f32(h01));
        const uint32_t l23 = pack_half2(w.y - half_lo_f32(h23), w.w - half_hi_f32(h23));
        xfb[(4 * (chi % 8) + t) * LS + s * NT + chi / 8] = make_uint2(h01, h23);
        xfb[(4 * (clo % 8) + t) * LS + s * NT + clo / 8] = make_uint2(l01, l23);
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
            xfb[(4 * (chi % 8) + t) * LS + 16 * NT + chi / 8] = make_uint2(hs, 0u);
            xfb[(4 * (clo % 8) + t) * LS + 16 * NT + clo / 8] = make_uint2(ls, 0u);
        }
    }
    return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
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
// and unscale * pre = dx / 254, with unscale kept in the normal range (pre =
// 2^-64 for the scaled blocks, else 1); unscale is 0 for an all-zero
// super-block and the non-finite max itself when x holds an inf or NaN, so
// that the result is not finite.  With Q8 (one code per element, Q8_K style)
// only xh is written, unscale * pre = dx and the sums are sum(xh).
// ---------------------------------------------------------------------------
constexpr int kI8Bytes = 672;
constexpr int kI8Pair = 80;        // bytes per sub-block pair in each part
static_assert(kI8Bytes <= lane_stride(1) * 8 * 8, "batch-1 fragment area holds the int8 parts");

// One super-block of x (batch 1) -> the layout above at `base`, by one warp.
// v0, v1 = float4 number lane and lane + 32 of the super-block (k = 4l..4l+3
// and 128 + 4l..).  Rounding to the nearest integer (ties to even) is done by
// adding and removing 1.5 * 2^23 in fp32 (|q| <= 127 here), which leaves the
// integer in the low bits of the sum: its low byte is the int8 code.  Returns
// {unscale, pre} of the super-block (see above).
template <bool Q8>
__device__ __forceinline__ float2 x_item_i8(float4 v0, float4 v1, int lane, uint8_t *base)
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
    const bool ok = m != 0u && m < 0x7F800000u;   // finite and not all zero
    // below 2^-64 the reciprocal is taken of the max scaled by 2^64 (exact)
    // and x is scaled alike, so that it stays finite
    const float pre = (m < 0x1F800000u) ? 0x1p64f : 1.0f;
    const float inv = ok ? 127.0f / (amax * pre) : 0.0f;
    if (pre != 1.0f) {   // warp-uniform; exact scaling by a power of two
        v0.x *= pre; v0.y *= pre; v0.z *= pre; v0.w *= pre;
        v1.x *= pre; v1.y *= pre; v1.z *= pre; v1.w *= pre;
    }
    constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23
    constexpr uint32_t kMagicBits = 0x4B400000u;   // its bit pattern
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const float4 w = h2 ? v1 : v0;
        const float e[4] = {w.x, w.y, w.z, w.w};
        uint32_t th[4], tl[4];
        uint32_t sum = 0u;   // mod 2^32: the constant offsets cancel below
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float q = e[j] * inv;
            const float t1 = __fadd_rn(q, kMagic);     // kMagic + rint(q)
            const float hq = __fsub_rn(t1, kMagic);    // rint(q), exact
            th[j] = __float_as_uint(t1);
            if constexpr (Q8) {
                tl[j] = 0u;
                sum += th[j];
            } else {
                const float r = __fmul_rn(__fsub_rn(q, hq), 254.0f);
                tl[j] = __float_as_uint(__fadd_rn(r, kMagic));
                sum += 254u * th[j] + tl[j];
            }
        }
        uint32_t hw = __byte_perm(__byte_perm(th[0], th[1], 0x0040), __byte_perm(th[2], th[3], 0x0040), 0x5410);
        uint32_t lw = __byte_perm(__byte_perm(tl[0], tl[1], 0x0040), __byte_perm(tl[2], tl[3], 0x0040), 0x5410);
        sum -= (Q8 ? 4u : 4u * 255u) * kMagicBits;
        if (!ok) hw = lw = sum = 0u;
        const int i = lane + 32 * h2;   // float4 index: k = 4i..4i+3, sub-block i/8, pair i/16
        const int off = kI8Pair * (i >> 4) + 4 * (i & 15);
        *reinterpret_cast<uint32_t *>(base + off) = hw;
        if constexpr (!Q8) *reinterpret_cast<uint32_t *>(base + 4 * kI8Pair + off) = lw;
        int s = static_cast<int>(sum);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        if ((i & 7) == 0) reinterpret_cast<int *>(base + 8 * kI8Pair)[i >> 3] = s;
    }
    const float unscale = ok ? (Q8 ? (amax * pre) / 127.0f : (amax * pre) / 127.0f / 254.0f) : (m == 0u ? 0.0f : amax);
    return make_float2(unscale, 1.0f / pre);
}

// Scale/min constants of one row of a super-block for thread t (pair t).
struct RowConsts {
    uint32_t mulE, addE, mulO, addO;  // f16x2 (sc_2t), (-1024 sc_2t), (sc_2t+1 / 16), (-64 sc_2t+1)
    uint32_t mpair;                   // f16x2 {m_2t, m_2t+1}
    float d, dmin;
};

// Scale/min bytes of pair t: scp = {sc_2t, sc_2t+1}, mp = {m_2t, m_2t+1} as
// two bytes each, branch-free for a lane with fixed t (see PairSel).
struct PairSel {
    uint32_t sh;    // 16 for odd t
    uint32_t hi;    // t >= 2: sub-blocks 4..7
    uint32_t mA;    // 0x3F3F (t < 2) or 0x0F0F
    uint32_t mB;    // 0 (t < 2) or 0x3030
};
__device__ __forceinline__ PairSel pair_sel(int t)
{
    PairSel p;
    p.sh = (t & 1) ? 16u : 0u;
    p.hi = (t >= 2) ? 1u : 0u;
    p.mA = p.hi ? 0x0F0Fu : 0x3F3Fu;
    p.mB = p.hi ? 0x3030u : 0u;
    return p;
}

__device__ __forceinline__ void pair_scales(uint4 h, const PairSel &p, uint32_t &scp, uint32_t &mp)
{
    const uint32_t a0 = h.y >> p.sh;   // s[2(t&1)], s[2(t&1)+1] in the low 16 bits
    const uint32_t a1 = h.z >> p.sh;   // s[4+...]
    const uint32_t a2 = h.w >> p.sh;   // s[8+...]
    // t < 2:  sc = a0 & 63,                       m = a1 & 63
    // t >= 2: sc = (a2 & 15) | (a0 >> 6) << 4,     m = (a2 >> 4 & 15) | (a1 >> 6) << 4
    const uint32_t lsc = p.hi ? a2 : a0;
    const uint32_t lm = p.hi ? (a2 >> 4) : a1;
    scp = (lsc & p.mA) | ((a0 >> 2) & p.mB);
    mp = (lm & p.mA) | ((a1 >> 2) & p.mB);
}

__device__ __forceinline__ RowConsts decode_header(uint4 h, const PairSel &ps)
{
    RowConsts rc;
    rc.d = half_lo_f32(h.x);
    rc.dmin = half_hi_f32(h.x);
    uint32_t scp, mp;
    pair_scales(h, ps, scp, mp);
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
__device__ __forceinline__ RowConstsI decode_header_i(uint4 h, const PairSel &p)
{
    RowConstsI rc;
    rc.d = half_lo_f32(h.x);
    rc.dmin = half_hi_f32(h.x);
    uint32_t scp, mp;
    pair_scales(h, p, scp, mp);
    rc.scE = static_cast<int>(scp & 0xFFu);
    rc.scO = static_cast<int>((scp >> 8) & 0xFFu);
    rc.mE = static_cast<int>(mp & 0xFFu);
    rc.mO = static_cast<int>((mp >> 8) & 0xFFu);
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
                                                 const PairSel &ps, float u, float pre, float (&acc)[1][2],
                                                 Release &&release)
{
    const RowConstsI r0 = decode_header_i(*reinterpret_cast<const uint4 *>(ra), ps);
    const RowConstsI r1 = decode_header_i(*reinterpret_cast<const uint4 *>(rb), ps);
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
                                              const PairSel &ps, const float (&unscale)[NT], float (&acc)[NT][2],
                                              Release &&release)
{
    const RowConsts r0 = decode_header(*reinterpret_cast<const uint4 *>(ra), ps);
    const RowConsts r1 = decode_header(*reinterpret_cast<const uint4 *>(rb), ps);
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

}  // namespace q4k
