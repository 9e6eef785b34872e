// q4k_prefill.cu -- Q4_K prefill GEMM on the GB300 tcgen05 tensor cores.
//
// Y[t][n] = sum_k w[n][k] X[t][k] for a block of T prompt tokens: the dense
// contraction that the dotLLM README's CUDA backend sends to "cuBLAS HGEMM for
// prefill" after "on-the-fly weight dequantization" (News 2026-03).  Here the
// weights are dequantized straight into shared memory as 16-bit floats and
// multiplied by hand-issued tcgen05.mma instructions, fp32 accumulation in
// tensor memory.
//
// Precision: kind::f16 takes A and B of one type, and X arrives as bf16.  Both
// sides go to fp16 (11 significant bits, 3 more than bf16: one fp16 rounding
// of w keeps the product well inside the decode path's error budget, one bf16
// rounding does not), each under a power-of-two scale that keeps it in fp16's
// range whatever the data: a small kernel first converts X per token (max|x|
// brought to [2^14, 2^15), so every bf16 value of at least 2^-31 times the
// token's max converts exactly), and each dequantizing thread scales its weight
// row by 2^r chosen from the row's largest possible |w| (|d|*945 + |dmin|*63
// over its super-blocks).  The epilogue multiplies by 2^-r and the token's
// inverse scale.
//
// CTA tile: 128 weight rows (the MMA M side) x TN*NTT tokens (the N side),
// full K.  Per 64-wide K chunk (a quarter of a super-block):
//   * warps 0-7 (two threads per weight row, one per nibble half) read the
//     row's sub-block pair from the raw weight ring, compute
//     w = d*sc*q - dmin*m in fp32, scale it by 2^r and round it to fp16 into
//     a 128-byte-swizzled K-major tile (with one thread per row the dequant
//     took ~900 cycles a chunk against 512 for the MMAs at 256 tokens);
//   * warp 8 loads the X tile [TN x 64] (fp16) with a TMA tensor copy (128B
//     swizzle), warp 9 the raw weight super-blocks;
//   * warps 10 and 11 (one elected thread each) issue the tcgen05.mma (K = 16
//     each) into TMEM and commit to the stage's "empty" barriers: with two
//     token tiles (NTT = 2) warp 10 + j takes tile j, otherwise warp 10 takes
//     the even chunks and warp 11 the odd ones, into an accumulator of its own
//     that the epilogue adds (one issuing warp spent ~500 cycles a chunk on
//     its barrier waits, fences and commits on top of ~100 per MMA issued).
// A ring of NS stages overlaps the three.  The epilogue reads TMEM with
// tcgen05.ld (warps w and w + 4 own TMEM lanes 32w..32w+31 = weight rows) and
// writes Y with coalesced stores.  Every mbarrier wait is bounded in time.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "ptx.cuh"
#include "q4k_dev.cuh"
#include "q4k_internal.h"

namespace q4k {

__device__ unsigned int g_prefill_error = 0;   // bit 1: a bounded wait in the prefill kernel timed out

unsigned int read_prefill_error()
{
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    return v;
}

bool clear_prefill_error()
{
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(g_prefill_error, &z, sizeof(z)) == cudaSuccess;
}

namespace pf {

constexpr int kRowsM = 128;          // MMA M
constexpr int kChunk = 64;           // K elements per stage (one 128-byte swizzle row)
constexpr int kThreads = 192;        // 4 dequant/epilogue warps + TMA warp + MMA warp
// fp16 kernel: 8 dequant/epilogue warps (two threads per weight row, one per
// nibble half), an X-tile TMA warp, a weight TMA warp and two MMA warps
// Thread layout of the fp16 kernel for token tiles of TN: P dequant threads
// per weight row (P = 4 for the small tiles, where the dequant bounds the
// kernel: each thread one nibble half of half of every chunk), then the X
// warp, the weight warp and the two MMA warps.
template <int TN>
struct FLay {
    static constexpr int P = (TN <= 64) ? 4 : 2;
    static constexpr int kProd = 128 * P;
    static constexpr int kThreads = kProd + 128;
    static constexpr int kTmaWarp = kProd / 32;      // X tiles; the next warp: raw weights
    static constexpr int kMmaWarp = kTmaWarp + 2;    // and the one after it
};
constexpr int kATileBytes = kRowsM * kChunk * 2;    // 16 KB: one fp16 weight tile
constexpr int kAStageBytes = kATileBytes;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// tcgen05.mma and tcgen05.commit issued by one elected lane of a warp that
// runs the issue loop as a whole: the loop's descriptor arithmetic then stays
// warp-uniform.  (Measured on this GPU: an M128 K16 MMA every ~40 cycles at
// N <= 32 this way, against ~108 cycles from a loop that only lane 0 runs.)
// The caller keeps the warp converged at every call.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms of
// 1024 bytes (stride byte offset 1024), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1) << 16;                 // leading byte offset (unused for this layout)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;         // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                 // version
    d |= static_cast<uint64_t>(2) << 61;                 // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (format 0), fp32 D, both
// K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N)
{
    return (1u << 4)                                   // D format f32
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Power-of-two exponent e with v * 2^e in [2^14, 2^15) for a positive finite
// v (0 for 0, inf or NaN), clamped so that 2^e and 2^-e stay normal.
__device__ __forceinline__ int f16_range_exp(float v)
{
    const uint32_t b = __float_as_uint(v);
    const int E = static_cast<int>((b >> 23) & 255u);
    if (b == 0u || E == 255) return 0;
    return max(-126, min(126, 141 - E));
}

// X (bf16 [T][K]) -> fp16 [T][K] times 2^e_t per token, and xexp[t] = e_t.
// One CTA per token: the max |x|, then the exact conversion.  A token of up
// to kXv * 8 * 256 elements is read once and held in registers; longer rows
// are read twice.  The prefill kernel that follows is launched as its
// programmatic dependent: it starts streaming and dequantizing W while this
// runs.
//
// EXACT (the small-T kernel's layout): within every aligned group of four k
// the middle two are swapped (k order 0, 2, 1, 3), the order in which that
// kernel's weight tiles come out of its nibble arithmetic, and XS[t][sb][0..15]
// receives the sums of the scaled x over the eight 32-wide sub-blocks of
// super-block sb, times 2^-6, as fp16 hi (0..7) and lo (8..15) parts; entries
// 16..63 of each super-block are zero.
constexpr int kXv = 8;
template <bool EXACT>
__global__ void __launch_bounds__(256) x_to_f16_kernel(const uint16_t *__restrict__ X, uint16_t *__restrict__ Xh,
                                                       int *__restrict__ xexp, uint16_t *__restrict__ XS, int K)
{
    __shared__ uint32_t s_max[8];
    pdl_launch_dependents();
    const size_t t = blockIdx.x;
    const uint4 *src = reinterpret_cast<const uint4 *>(X + t * K);
    uint4 *dst = reinterpret_cast<uint4 *>(Xh + t * K);
    const int nv = K / 8;
    const bool in_regs = nv <= kXv * static_cast<int>(blockDim.x);
    uint4 v[kXv];
    uint32_t m = 0u;   // max |x| as fp32 bits
    auto absmax = [](uint32_t m, const uint4 &q) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) m = max(m, max((w[j] << 16) & 0x7FFFFFFFu, w[j] & 0x7FFF0000u));
        return m;
    };
    if (in_regs) {
#pragma unroll
        for (int r = 0; r < kXv; ++r) {
            const int i = threadIdx.x + r * blockDim.x;
            v[r] = (i < nv) ? src[i] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int r = 0; r < kXv; ++r) m = absmax(m, v[r]);
    } else {
        for (int i = threadIdx.x; i < nv; i += blockDim.x) m = absmax(m, src[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
    __syncthreads();
    m = s_max[0];
    for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) m = max(m, s_max[i]);
    const int e = f16_range_exp(__uint_as_float(m));
    const float sc = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    if (threadIdx.x == 0) xexp[t] = e;
    // converts one 8-element group; i = its index in the row
    auto convert = [&](const uint4 &q, int i) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        float f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = __uint_as_float(w[j] << 16) * sc;
            f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u) * sc;
        }
        if (EXACT) {
            dst[i] = make_uint4(pack_half2(f[0], f[2]), pack_half2(f[1], f[3]), pack_half2(f[4], f[6]),
                                pack_half2(f[5], f[7]));
            // sub-block j = i / 4 is held by the four lanes 4(i/4) .. +3 of
            // this warp (the row stride of the loop is a multiple of 4)
            float sum = ((f[0] + f[1]) + (f[2] + f[3])) + ((f[4] + f[5]) + (f[6] + f[7]));
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if ((i & 3) == 0) {
                const int j = i >> 2;
                uint16_t *xs = XS + (t * (K / 256) + (j >> 3)) * 64;
                const float s6 = sum * 0.015625f;
                const __half hi = __float2half_rn(s6);
                const __half lo = __float2half_rn(s6 - __half2float(hi));
                xs[j & 7] = __half_as_ushort(hi);
                xs[8 + (j & 7)] = __half_as_ushort(lo);
                if ((j & 7) == 0) {
                    uint4 *z = reinterpret_cast<uint4 *>(xs + 16);
#pragma unroll
                    for (int u = 0; u < 6; ++u) z[u] = make_uint4(0, 0, 0, 0);
                }
            }
        } else {
            dst[i] = make_uint4(pack_half2(f[0], f[1]), pack_half2(f[2], f[3]), pack_half2(f[4], f[5]),
                                pack_half2(f[6], f[7]));
        }
    };
    if (in_regs) {
#pragma unroll
        for (int r = 0; r < kXv; ++r) {
            const int i = threadIdx.x + r * blockDim.x;
            // (whole warps take the same branch: nv is a multiple of 32)
            if (i < nv) convert(v[r], i);
        }
    } else {
        for (int i = threadIdx.x; i < nv; i += blockDim.x) convert(src[i], i);
    }
}


// The raw weight super-blocks of the tile (128 rows x 144 bytes) come by TMA
// into a ring of their own, kWSlots super-blocks ahead of the dequant: loaded
// by each producer thread from global memory one super-block ahead, they kept
// the producers waiting on memory (long-scoreboard stalls on top in ncu).
constexpr int kWSlots = 3;
constexpr int kWSlotBytes = kRowsM * 144;
template <int TN, int NTT>
struct Cfg {
    static constexpr int kBBytes = TN * kChunk * 2;                       // one token subtile
    static constexpr int kStageBytes = kAStageBytes + NTT * kBBytes;
    static constexpr int kRoom = 224 * 1024 - kWSlots * kWSlotBytes;      // for the stage ring
    static constexpr int kStages = (kRoom / kStageBytes) < 4 ? (kRoom / kStageBytes) : 4;
    static constexpr int kTmemCols = TN * 2;   // NTT = 2: one accumulator per tile; NTT = 1: one per MMA warp
    static constexpr size_t kWOffset = static_cast<size_t>(kStages) * kStageBytes;
    static constexpr size_t kSmem = kWOffset + static_cast<size_t>(kWSlots) * kWSlotBytes;
    static_assert(kStages >= 2, "at least two stages");
};

// Named barrier 1 over the first `count` threads (the epilogue warps),
// returning the AND of p over them.
__device__ __forceinline__ bool bar_and_n(bool p, uint32_t count)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred a, b;\n\t"
        "setp.ne.u32 a, %1, 0;\n\t"
        "bar.red.and.pred b, 1, %2, a;\n\t"
        "selp.u32 %0, 1, 0, b;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(p)), "r"(count)
        : "memory");
    return r != 0;
}

// Packed pairs of fp32 (one 64-bit register pair; low word = first value)
// and the paired fp32 add and fma of sm_100+.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f2_pack_bits(uint32_t lo, uint32_t hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
// fp16 pair {round(lo), round(hi)} of an fp32 pair
__device__ __forceinline__ uint32_t f2_to_half2(uint64_t v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return pack_half2(lo, hi);
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// K-split reduction over a cluster of S CTAs.  Every rank holds its scaled
// partial tile as fp32 [col][128 rows] at part_addr; rank kz sums rows
// [kz*128/S, (kz+1)*128/S) over the ranks in rank order (0 + p_0 + p_1 + ...,
// the same order for every element) and stores them to Y [T][N].  An item is
// four consecutive rows of one column (16-byte loads); 8/S items per round put
// eight remote loads in flight per thread (one at a time left a 128 x 256
// tile's reduction at tens of microseconds).
template <int S>
__device__ __forceinline__ void reduce_split_tile(uint32_t part_addr, int kz, int cols, int row0, int t0, float *Y,
                                                  int N, int T, int tid, int nthreads)
{
    constexpr int kU = 8 / S;
    constexpr int kQuads = kRowsM / S / 4;
    static_assert(S >= 2 && S <= 8 && kRowsM % (4 * S) == 0, "split of 2, 4 or 8");
    const int r0 = kz * (kRowsM / S);
    const int items = kQuads * cols;
    const bool vec = (N % 4) == 0 && (reinterpret_cast<uintptr_t>(Y) & 15u) == 0;
    for (int base = tid; base < items; base += kU * nthreads) {
        float4 v[kU][S];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int it = min(base + u * nthreads, items - 1);
            const int c = it / kQuads, r = r0 + 4 * (it % kQuads);
            const uint32_t off = static_cast<uint32_t>((c * kRowsM + r) * 4);
#pragma unroll
            for (int q = 0; q < S; ++q) v[u][q] = ld_cluster_v4(map_shared_rank(part_addr + off, q));
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int it = base + u * nthreads;
            if (it < items) {
                const int c = it / kQuads, r = r0 + 4 * (it % kQuads);
                float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int q = 0; q < S; ++q) {
                    s.x += v[u][q].x;
                    s.y += v[u][q].y;
                    s.z += v[u][q].z;
                    s.w += v[u][q].w;
                }
                const int n = row0 + r, t = t0 + c;
                if (t < T) {
                    float *yp = Y + static_cast<size_t>(t) * N + n;
                    if (vec && n + 3 < N) {
                        *reinterpret_cast<float4 *>(yp) = s;
                    } else {
                        const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (n + i < N) yp[i] = sv[i];
                    }
                }
            }
        }
    }
}

// Rank-order sum of any split (the host launches 2, 4 or 8).
__device__ __forceinline__ void reduce_split(uint32_t part_addr, int split, int kz, int cols, int row0, int t0,
                                             float *Y, int N, int T, int tid, int nthreads)
{
    switch (split) {
    case 2: reduce_split_tile<2>(part_addr, kz, cols, row0, t0, Y, N, T, tid, nthreads); break;
    case 4: reduce_split_tile<4>(part_addr, kz, cols, row0, t0, Y, N, T, tid, nthreads); break;
    case 8: reduce_split_tile<8>(part_addr, kz, cols, row0, t0, Y, N, T, tid, nthreads); break;
    default: {
        const int r0 = (kz * kRowsM) / split, rows = ((kz + 1) * kRowsM) / split - r0;
        for (int it = tid; it < rows * cols; it += nthreads) {
            const int c = it / rows, r = r0 + it % rows;
            const uint32_t off = static_cast<uint32_t>((c * kRowsM + r) * 4);
            float sum = 0.f;
            for (int q = 0; q < split; ++q) sum += ld_shared_cluster_f32(map_shared_rank(part_addr + off, q));
            const int n = row0 + r, t = t0 + c;
            if (n < N && t < T) Y[static_cast<size_t>(t) * N + n] = sum;
        }
    }
    }
}

template <int TN, int NTT>
__global__ void __launch_bounds__(FLay<TN>::kThreads, 1)
    q4k_prefill_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                       const uint8_t *__restrict__ W, const int *__restrict__ xexp, float *__restrict__ Y, int N,
                       int K, int T)
{
    using C = Cfg<TN, NTT>;
    using L = FLay<TN>;
    constexpr int P = L::P;
    constexpr int kProdF16 = L::kProd;
    constexpr int kThreadsF16 = L::kThreads;
    constexpr int kTmaWarpF16 = L::kTmaWarp;
    constexpr int kMmaWarpF16 = L::kMmaWarp;
    static_assert(P == 2 || NTT == 1, "four dequant threads per row only with one token tile");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;   // 1024-byte aligned: the 128B-swizzle atoms need it
    // full_a/empty: the stage's weight tile; full_x/empty_x: each token
    // tile's X tile of the stage (freed as soon as its own MMAs finish)
    __shared__ __align__(8) uint64_t full_a[C::kStages], empty[C::kStages], done_bar;
    __shared__ __align__(8) uint64_t full_x[C::kStages * NTT], empty_x[C::kStages * NTT];
    __shared__ __align__(8) uint64_t wfull[kWSlots], wempty[kWSlots];
    __shared__ uint32_t tmem_base_s;
    __shared__ int s_abort;
    __shared__ __align__(16) int s_xexp[TN * NTT];   // token scale exponents of this CTA's tokens
    __shared__ __align__(16) float s_xinv[TN * NTT]; // 2^-e_t
    __shared__ int s_rexp[kRowsM];                   // row scale exponents (from the prescan)

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int row0 = blockIdx.x * kRowsM;
    const int t0 = blockIdx.y * TN * NTT;
    int rexp = 0;   // dequant/epilogue threads: r of the tile row they own (w scaled by 2^r)
    const int nsub = min(NTT, (T - t0 + TN - 1) / TN);
    // K split over the CTAs of a cluster along z (split == 1: whole K)
    const int split = gridDim.z;
    const int kz = blockIdx.z;
    // (whole super-blocks per CTA: four chunks each)
    const int c_begin = 4 * static_cast<int>((static_cast<long long>(kz) * (K / 256)) / split);
    const int c_end = 4 * static_cast<int>((static_cast<long long>(kz + 1) * (K / 256)) / split);
    const size_t row_bytes = static_cast<size_t>(K / 256) * 144;
    // Super-blocks of this CTA's K range in a per-row-tile rotated order (so
    // that the CTAs' X tile requests spread over L2).
    const int sb_begin = c_begin >> 2, sb_end = c_end >> 2, nloc = sb_end - sb_begin;
    const int rot = static_cast<int>(blockIdx.x % static_cast<unsigned>(nloc));
    auto sb_of = [&](int i) {
        const int j = i + rot;
        return sb_begin + (j >= nloc ? j - nloc : j);
    };

    // Row-scale prescan, first round of header loads issued before the setup
    // barrier by the low-nibble thread of each row (the other thread of the
    // row reads the result from shared memory): the prescan is pure load
    // latency at the start of the launch.
    const bool pre_thread = tid < kRowsM;
    const bool pre_live = pre_thread && row0 + tid < N;
    uint32_t hb0[16];
    {
        const uint8_t *wr = W + static_cast<size_t>(pre_live ? row0 + tid : 0) * row_bytes;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            hb0[i] = (pre_live && sb_begin + i < sb_end)
                         ? __ldg(reinterpret_cast<const uint32_t *>(wr + static_cast<size_t>(sb_begin + i) * 144))
                         : 0u;
    }

    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&full_a[s]), kProdF16);
            mbar_init(smem_u32(&empty[s]), NTT == 2 ? 2 : 1);   // both tiles' warps read the weight tile
        }
        for (int s = 0; s < C::kStages * NTT; ++s) {
            mbar_init(smem_u32(&full_x[s]), 1);
            mbar_init(smem_u32(&empty_x[s]), 1);
        }
        mbar_init(smem_u32(&done_bar), 2);   // a final commit from each MMA warp
        s_abort = 0;
        fence_barrier_init();
    }
    // The weight warp sets up its own ring and issues the first super-blocks
    // before the setup barrier (the weight stream is the first thing the
    // dequant needs, with the prescan).
    const int w_first = min(kWSlots, nloc);
    if (warp == kTmaWarpF16 + 1 && lane == 0) {
        for (int s = 0; s < kWSlots; ++s) {
            mbar_init(smem_u32(&wfull[s]), 1);
            mbar_init(smem_u32(&wempty[s]), kProdF16);
        }
        fence_barrier_init();
        const uint64_t pol = l2_policy_evict_first();
        for (int i = 0; i < w_first; ++i) {
            mbar_arrive_expect_tx(smem_u32(&wfull[i]), kWSlotBytes);
            tma_load_2d_hint(smem_u32(smem + C::kWOffset + i * kWSlotBytes), &tmW, sb_of(i) * 18, row0,
                             smem_u32(&wfull[i]), pol);
        }
    }
    if (warp == kMmaWarpF16) {
        tmem_alloc(smem_u32(&tmem_base_s), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kTmaWarpF16 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp < kTmaWarpF16) {
        // ------------------------------------------------ dequant producers
        const int r = tid & (kRowsM - 1);     // tile row 0..127
        const int hsel = (tid >> 7) & 1;      // 0: low nibbles (k 0..31 of a chunk), 1: high nibbles (k 32..63)
        // P = 4: which half of the chunk's four 16-byte output chunks (and of
        // its 32 quant bytes) this thread takes
        const int quarter = (P == 4) ? (tid >> 8) : 0;
        constexpr int NQ = (P == 4) ? 5 : 9;  // 16-byte words of a super-block a thread reads
        constexpr int NC8 = 8 / P;            // 16-byte output chunks per chunk and thread
        const int n = row0 + r;
        const bool live = n < N;
        const uint8_t *wrow = W + static_cast<size_t>(live ? n : 0) * row_bytes;
        int stage = 0;
        uint32_t phase = 0;
        // Row scale 2^rs: the largest |w| this CTA's super-blocks of the row
        // can hold, |d|*945 + |dmin|*63, brought to [2^14, 2^15).
        if (tid < kRowsM) {   // one thread per row
            float wmax = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                wmax = fmaxf(wmax, fmaf(fabsf(half_lo_f32(hb0[i])), 945.0f, fabsf(half_hi_f32(hb0[i])) * 63.0f));
            if (live) {   // sixteen headers in flight per further round
                for (int b = sb_begin + 16; b < sb_end; b += 16) {
                    uint32_t hb[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        hb[i] = (b + i < sb_end) ? __ldg(reinterpret_cast<const uint32_t *>(wrow + static_cast<size_t>(b + i) * 144)) : 0u;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        wmax = fmaxf(wmax, fmaf(fabsf(half_lo_f32(hb[i])), 945.0f, fabsf(half_hi_f32(hb[i])) * 63.0f));
                }
            }
            s_rexp[r] = f16_range_exp(wmax);
        }
        named_bar_sync(2, kProdF16);
        rexp = s_rexp[r];
        const float rscale = __uint_as_float(static_cast<uint32_t>(rexp + 127) << 23);
        // A super-block of the row as nine 16-byte words (header, then the
        // 128 quant bytes), read from the weight ring one super-block ahead of
        // its dequant.  Rows past N arrive as zeros from the TMA unit (d =
        // dmin = 0 makes every weight of them zero); super-blocks past the
        // CTA's range read as zeros.
        const uint8_t *wring = smem + C::kWOffset;
        auto load_sb = [&](int i, uint4 (&q)[NQ]) {
            if (i < nloc) {
                const int slot = i % kWSlots;
                if (!*(volatile int *)&s_abort &&
                    !mbar_wait_bounded(smem_u32(&wfull[slot]), static_cast<uint32_t>((i / kWSlots) & 1), kWaitLimitNs)) {
                    atomicOr(&g_prefill_error, 2u);
                    s_abort = 1;
                }
                const uint4 *bp = reinterpret_cast<const uint4 *>(wring + slot * kWSlotBytes + r * 144);
                if constexpr (P == 4) {   // the header and this thread's half of each part's quant bytes
                    q[0] = bp[0];
#pragma unroll
                    for (int p = 0; p < 4; ++p) q[1 + p] = bp[1 + 2 * p + quarter];
                } else {
#pragma unroll
                    for (int u = 0; u < 9; ++u) q[u] = bp[u];
                }
                mbar_arrive(smem_u32(&wempty[slot]));   // (release: orders the reads before the refill)
            } else {
#pragma unroll
                for (int u = 0; u < NQ; ++u) q[u] = make_uint4(0, 0, 0, 0);
            }
        };
        // One super-block = four K chunks; chunk p holds sub-blocks 2p (low
        // nibbles of quant bytes 32p..32p+31) and 2p+1 (their high nibbles):
        // this thread's sub-block is 2p + hsel.
        auto dequant_sb = [&](const uint4 (&q)[NQ]) {
            const float d = half_lo_f32(q[0].x) * rscale, dmin = half_hi_f32(q[0].x) * rscale;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t scp, mp;
                pair_scales(q[0], pair_sel(p), scp, mp);
                // (the high nibbles come out as 16 q: their scale carries 1/16)
                const float ds = hsel ? d * static_cast<float>((scp >> 8) & 0xFFu) * 0.0625f
                                      : d * static_cast<float>(scp & 0xFFu);
                const float dm = dmin * static_cast<float>(hsel ? ((mp >> 8) & 0xFFu) : (mp & 0xFFu));
                if (!*(volatile int *)&s_abort && !mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, kWaitLimitNs)) {
                    atomicOr(&g_prefill_error, 2u);
                    s_abort = 1;
                }
                uint32_t words[2 * NC8];
                if constexpr (P == 4) {
                    words[0] = q[1 + p].x; words[1] = q[1 + p].y; words[2] = q[1 + p].z; words[3] = q[1 + p].w;
                } else {
                    const uint32_t w8[8] = {q[1 + 2 * p].x, q[1 + 2 * p].y, q[1 + 2 * p].z, q[1 + 2 * p].w,
                                            q[2 + 2 * p].x, q[2 + 2 * p].y, q[2 + 2 * p].z, q[2 + 2 * p].w};
#pragma unroll
                    for (int u = 0; u < 2 * NC8; ++u) words[u] = w8[u];
                }
                uint8_t *arow = smem + stage * C::kStageBytes + r * 128;
                // Each nibble goes straight under the fp32 exponent of 2^23 (one
                // LOP3 on the word shifted by 0, 8, 16 or 24 bits: 2^23 + q 2^s,
                // s = 0 for the low nibbles, 4 for the high ones, whose ds
                // carries the 1/16), the paired add takes 2^23 off exactly and
                // the paired fma gives q ds - dm in fp32, rounded once more to
                // fp16: the same two roundings as a scalar fma, in 13
                // instructions per four weights instead of 15.
                const uint32_t m0 = 0x0000000Fu << (4 * hsel);
                const uint32_t kMag = 0x4B000000u;
                const uint64_t nmag2 = f2_pack(-8388608.0f, -8388608.0f);
                const uint64_t ds2 = f2_pack(ds, ds);
                const uint64_t ndm2 = f2_pack(-dm, -dm);
#pragma unroll
                for (int c8 = 0; c8 < NC8; ++c8) {               // 16-byte chunk: k = 32*hsel + 8*(c8 + c8 base) .. +7
                    uint32_t out[4];
#pragma unroll
                    for (int uu = 0; uu < 2; ++uu) {             // word u = 2*c8 + uu -> k offset 4u..4u+3
                        const uint32_t w = words[2 * c8 + uu];
                        // {2^23 + q(4u) 2^s, 2^23 + q(4u+1) 2^s}, {.. q(4u+2) .., .. q(4u+3) ..}
                        const uint64_t A = f2_pack_bits(and_or(w, m0, kMag), and_or(w >> 8, m0, kMag));
                        const uint64_t B = f2_pack_bits(and_or(w >> 16, m0, kMag), and_or(w >> 24, m0, kMag));
                        out[2 * uu] = f2_to_half2(f2_fma(f2_add(A, nmag2), ds2, ndm2));
                        out[2 * uu + 1] = f2_to_half2(f2_fma(f2_add(B, nmag2), ds2, ndm2));
                    }
                    const int chunk = 4 * hsel + 2 * quarter + c8;
                    *reinterpret_cast<uint4 *>(arow + ((chunk ^ (r & 7)) << 4)) =
                        make_uint4(out[0], out[1], out[2], out[3]);
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&full_a[stage]));
                if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
            }
        };
        // Two register sets alternate so that no loaded word is ever moved.
        uint4 qa[NQ], qb[NQ];
        load_sb(0, qa);
        for (int i = 0; i < nloc; i += 2) {
            load_sb(i + 1, qb);
            dequant_sb(qa);
            if (i + 1 < nloc) {
                load_sb(i + 2, qa);
                dequant_sb(qb);
            }
        }
    } else if (warp == kTmaWarpF16 + 1) {
        // ------------------------------------------------ weight super-blocks by TMA (lane 0)
        // (a warp of its own: as a second lane of the X warp, its bounded
        // waits held up the X copies of the diverged lane)
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int issued = w_first;   // (the first ones went out before the setup barrier)
            for (int i = w_first; i < nloc; ++i) {
                const int slot = i % kWSlots;
                if (i >= kWSlots && !*(volatile int *)&s_abort &&
                    !mbar_wait_bounded(smem_u32(&wempty[slot]), static_cast<uint32_t>(((i / kWSlots) - 1) & 1),
                                       kWaitLimitNs)) {
                    atomicOr(&g_prefill_error, 2u);
                    s_abort = 1;
                }
                if (*(volatile int *)&s_abort) break;
                mbar_arrive_expect_tx(smem_u32(&wfull[slot]), kWSlotBytes);
                tma_load_2d_hint(smem_u32(smem + C::kWOffset + slot * kWSlotBytes), &tmW, sb_of(i) * 18, row0,
                                 smem_u32(&wfull[slot]), pol);
                ++issued;
            }
            if (*(volatile int *)&s_abort) {   // let the copies in flight land before the CTA exits
                for (int j = max(0, issued - kWSlots); j < issued; ++j)
                    if (!mbar_wait_bounded(smem_u32(&wfull[j % kWSlots]), static_cast<uint32_t>((j / kWSlots) & 1),
                                           kWaitLimitNs))
                        break;
            }
        }
    } else if (warp == kTmaWarpF16) {
        // ------------------------------------------------ X tiles by TMA (lane 0)
        if (lane == 0) {
            pdl_wait();   // X (fp16) is written by the conversion kernel launched just before
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;   // X tiles issued (nsub per stage use)
            for (int c = c_begin; c < c_end; ++c) {
                uint8_t *bbase = smem + stage * C::kStageBytes + kAStageBytes;
                const int kc = 4 * sb_of((c - c_begin) >> 2) + (c & 3);
                for (int j = 0; j < nsub; ++j) {
                    const uint32_t bx = smem_u32(&empty_x[stage * NTT + j]);
                    if (!*(volatile int *)&s_abort && !mbar_wait_bounded(bx, phase ^ 1u, kWaitLimitNs)) {
                        atomicOr(&g_prefill_error, 2u);
                        s_abort = 1;
                    }
                    if (*(volatile int *)&s_abort) break;
                    mbar_arrive_expect_tx(smem_u32(&full_x[stage * NTT + j]), static_cast<uint32_t>(C::kBBytes));
                    tma_load_2d(smem_u32(bbase + j * C::kBBytes), &tmX, kc * kChunk, t0 + j * TN,
                                smem_u32(&full_x[stage * NTT + j]));
                    ++issued;
                }
                if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
            }
            // After an abort, wait (bounded) for the copies still in flight so
            // none lands after the CTA has exited.
            if (*(volatile int *)&s_abort) {
                for (int i = max(0, issued - C::kStages * nsub); i < issued; ++i) {
                    const int use = i / nsub, j = i % nsub;
                    if (!mbar_wait_bounded(smem_u32(&full_x[(use % C::kStages) * NTT + j]),
                                           static_cast<uint32_t>((use / C::kStages) & 1), kWaitLimitNs))
                        break;
                }
            }
        }
    } else {
        // ------------------------------------------------ MMA issuers (two whole warps, one elected lane issues)
        {
            const int w = warp - kMmaWarpF16;
            constexpr uint32_t idesc = idesc_f16(kRowsM, TN);
            // NTT == 2: every chunk, token tile w.  NTT == 1: chunks c_begin + w,
            // c_begin + w + 2, ...  Either way into accumulator columns w*TN.
            constexpr int kStep = (NTT == 2) ? 1 : 2;
            const int first = (NTT == 2) ? c_begin : c_begin + w;
            const int j = (NTT == 2) ? w : 0;
            const bool active = j < nsub;   // (a second tile past T has no X and no MMAs)
            for (int c = first; c < c_end; c += kStep) {
                const int u = c - c_begin;
                const int stage = u % C::kStages;
                const uint32_t phase = static_cast<uint32_t>((u / C::kStages) & 1);
                bool ok = !*(volatile int *)&s_abort;
                if (ok && !mbar_wait_bounded(smem_u32(&full_a[stage]), phase, kWaitLimitNs)) ok = false;
                if (active && ok && !mbar_wait_bounded(smem_u32(&full_x[stage * NTT + j]), phase, kWaitLimitNs))
                    ok = false;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok && lane == 0 && !*(volatile int *)&s_abort) {
                    atomicOr(&g_prefill_error, 2u);
                    s_abort = 1;
                }
                tc_fence_after();
                if (active) {
                    if (ok) {
                        const uint32_t a_addr = smem_u32(smem + stage * C::kStageBytes);
                        const uint32_t b_addr = a_addr + kAStageBytes + j * C::kBBytes;
#pragma unroll
                        for (int kk = 0; kk < kChunk / 16; ++kk)
                            umma_f16(tmem + w * TN, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32), idesc,
                                     (c > first || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(smem_u32(&empty_x[stage * NTT + j]));   // frees this X tile
                }
                umma_commit(smem_u32(&empty[stage]));   // this warp is done with the weight tile
            }
            umma_commit(smem_u32(&done_bar));
        }
    }

    // ---------------------------------------------------- epilogue (warps 0-7)
    // Warps w and w + 4 read TMEM lanes 32w..32w+31 (= tile rows); thread group
    // g = tid / 128 takes token tile g (NTT == 2) or column half g (NTT == 1).
    // With a K split the partial tile goes to this CTA's shared memory
    // (column-major, so a warp's stores are consecutive); after a cluster
    // barrier CTA rank z sums rows [z*128/split, (z+1)*128/split) over ranks
    // 0..split-1 in order and writes Y.
    float *part = reinterpret_cast<float *>(smem);   // pipeline buffers are idle by now
    if (warp < kTmaWarpF16) {
        pdl_wait();   // the token exponents come from the conversion kernel
        // token factors 2^-e_t; moderate = every |e_t| <= 63 (then, for rows
        // with |r| <= 63 too, 2^-r 2^-e_t is an exact normal float and one
        // multiply scales a value)
        bool mod = true;
        for (int i = tid; i < TN * NTT; i += kProdF16) {
            const int e = (t0 + i < T) ? __ldg(xexp + t0 + i) : 0;
            s_xexp[i] = e;
            s_xinv[i] = __uint_as_float(static_cast<uint32_t>(127 - max(-126, min(126, e))) << 23);
            mod = mod && e >= -63 && e <= 63;
        }
        const bool all_mod = bar_and_n(mod, kProdF16);
        const bool ok = mbar_wait_bounded(smem_u32(&done_bar), 0u, kWaitLimitNs);
        if (!ok) {
            atomicOr(&g_prefill_error, 2u);
            s_abort = 1;
        }
        tc_fence_after();
        const int r = tid & (kRowsM - 1);
        const int n = row0 + r;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const bool fast = all_mod && rexp >= -63 && rexp <= 63;
        const float rinv = __uint_as_float(static_cast<uint32_t>(127 - max(-126, min(126, rexp))) << 23);
        // Four tensor-memory loads in flight per wait (a wait per 16 columns
        // left the 512-token epilogue at ~14 us): 64 columns of a tile per
        // round, or with NTT == 1 32 columns of each MMA warp's accumulator,
        // added (D0 + D1).
        constexpr int kGroupCols = TN / P;   // NTT == 1: columns per thread group
        constexpr int kRound = (NTT == 1) ? (kGroupCols < 32 ? kGroupCols : 32) : 64;
        const int g = tid >> 7;
        const int j_lo = (NTT == 2) ? g : 0, j_hi = (NTT == 2) ? min(g + 1, nsub) : nsub;
        const int c_lo = (NTT == 1) ? g * kGroupCols : 0, c_hi = (NTT == 1) ? c_lo + kGroupCols : TN;
        for (int j = j_lo; j < j_hi; ++j) {
#pragma unroll 1
            for (int c64 = c_lo; c64 < c_hi; c64 += kRound) {
                uint32_t v[4][16];
                if (NTT == 1) {
#pragma unroll
                    for (int q = 0; q < kRound / 16; ++q) {
                        tmem_ld16(lane_addr + c64 + 16 * q, v[q]);
                        tmem_ld16(lane_addr + TN + c64 + 16 * q, v[q + 2]);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) tmem_ld16(lane_addr + j * TN + c64 + 16 * q, v[q]);
                }
                tmem_wait_ld();
                if (NTT == 1) {
#pragma unroll
                    for (int q = 0; q < kRound / 16; ++q)
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            v[q][i] = __float_as_uint(__uint_as_float(v[q][i]) + __uint_as_float(v[q + 2][i]));
                }
#pragma unroll
                for (int q = 0; q < kRound / 16; ++q) {
                    const int c0 = c64 + 16 * q;
                    // undo the row's and the tokens' power-of-two scales: times
                    // 2^-(r + e_t), one correctly rounded multiply by an exact
                    // power of two when both are moderate, else as two factors
                    // that are normal floats (the second is 1 unless
                    // |r + e_t| > 126)
                    float o[16];
                    if (fast) {
                        const float4 *gx = reinterpret_cast<const float4 *>(s_xinv + j * TN + c0);
#pragma unroll
                        for (int i4 = 0; i4 < 4; ++i4) {
                            const float4 g = gx[i4];
                            o[4 * i4 + 0] = __uint_as_float(v[q][4 * i4 + 0]) * (rinv * g.x);
                            o[4 * i4 + 1] = __uint_as_float(v[q][4 * i4 + 1]) * (rinv * g.y);
                            o[4 * i4 + 2] = __uint_as_float(v[q][4 * i4 + 2]) * (rinv * g.z);
                            o[4 * i4 + 3] = __uint_as_float(v[q][4 * i4 + 3]) * (rinv * g.w);
                        }
                    } else {
                        const int4 *ex = reinterpret_cast<const int4 *>(s_xexp + j * TN + c0);
#pragma unroll
                        for (int i4 = 0; i4 < 4; ++i4) {
                            const int4 e4 = ex[i4];
                            const int es[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int tot = -rexp - es[u];
                                const int a = max(-126, min(126, tot));
                                const float f1 = __uint_as_float(static_cast<uint32_t>(a + 127) << 23);
                                const float f2 = __uint_as_float(static_cast<uint32_t>(tot - a + 127) << 23);
                                o[4 * i4 + u] = __uint_as_float(v[q][4 * i4 + u]) * f1 * f2;
                            }
                        }
                    }
                    const int tb = t0 + j * TN + c0;
                    if (split > 1) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) part[(j * TN + c0 + i) * kRowsM + r] = o[i];
                    } else if (ok && n < N) {
                        float *yp = Y + static_cast<size_t>(tb) * N + n;
                        if (tb + 16 <= T) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) yp[static_cast<size_t>(i) * N] = o[i];
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (tb + i < T) yp[static_cast<size_t>(i) * N] = o[i];
                        }
                    }
                }
            }
        }
        tc_fence_before();
    }
    if (split > 1) {
        __syncthreads();
        cluster_sync_all();
        if (!*(volatile int *)&s_abort)
            reduce_split(smem_u32(part), split, kz, nsub * TN, row0, t0, Y, N, T, tid, kThreadsF16);
        cluster_sync_all();
    }
    __syncthreads();
    if (warp == kMmaWarpF16) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}


// ---------------------------------------------------------------------------
// Small token counts: exact integer weight tiles, scales applied per super-block.
//
// For T up to a few dozen tokens the fp32 dequant above costs far more than
// the weight stream.  This kernel never forms w: the weight tile holds
// q * sc_j, an integer of at most 945 that fp16 represents exactly (two
// instructions per two weights: the nibbles under the exponent of 1024, one
// f16x2 fma with sc and -1024 sc), the MMAs of one super-block accumulate
// D = sum_k (q sc)_k x_k in tensor memory, one more MMA per super-block forms
// M = sum_j m_j S_j from the sub-block sums S_j of x, and the epilogue warps
// add d * D - dmin * M into fp32 registers before tensor memory is reused.
// D and M are double-buffered so that the next super-block's MMAs run while
// the epilogue reads the last one.  Every product is exact; the only
// roundings are fp32 accumulation and the split of S_j into fp16 hi + lo.
//
// Per super-block five parts go through the stage ring: its four 64-wide K
// chunks (weight tile + X tile) and a "min" part whose weight tile holds
// {m_0..m_7, m_0..m_7} in its first 16 columns and whose X tile holds
// {S_hi 0..7, S_lo 0..7} (one K16 MMA).  PS parts share one stage (one
// barrier hand-off): PS = 5 puts a whole super-block in a stage.  X arrives
// in the converted layout with the middle two of every four k swapped, which
// is the order in which the nibble arithmetic emits the weights.
template <int TN, int PS>
struct ECfg {
    static constexpr int kBBytes = TN * kChunk * 2;                 // X tile of a part
    static constexpr int kStageBytes = PS * (kATileBytes + kBBytes);  // PS weight tiles, then PS X tiles
    static constexpr int kStages = (PS == 1) ? ((TN <= 32) ? 5 : (200 * 1024) / kStageBytes) : (200 * 1024) / kStageBytes;
    static constexpr int kTmemCols = 4 * TN;      // {D, M} x 2 buffers
    static constexpr size_t kSmem = static_cast<size_t>(kStages) * kStageBytes;
    static constexpr bool kTwoPerSm = PS == 1 && TN <= 32;
    static_assert(kStages >= 2, "at least two stages");
    static_assert(static_cast<size_t>(TN) * kRowsM * 4 <= kSmem, "split-K partial tile must fit the ring");
};

template <int TN, int PS>
__global__ void __launch_bounds__(kThreads, (PS == 1 && TN <= 32) ? 2 : 1)
    q4k_prefill_exact_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmS,
                             const uint8_t *__restrict__ W, const int *__restrict__ xexp, float *__restrict__ Y,
                             int N, int K, int T)
{
    using C = ECfg<TN, PS>;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_a[C::kStages], full_b[C::kStages], empty[C::kStages];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ int s_abort;
    __shared__ __align__(16) int s_xexp[TN];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int row0 = blockIdx.x * kRowsM;
    const int t0 = blockIdx.y * TN;
    const int split = gridDim.z;
    const int kz = blockIdx.z;
    const int nsb = K / 256;
    const int sb_begin = static_cast<int>((static_cast<long long>(kz) * nsb) / split);
    const int sb_end = static_cast<int>((static_cast<long long>(kz + 1) * nsb) / split);
    const int nloc = sb_end - sb_begin;    // >= 1 (the planner keeps split <= nsb / 2)
    // Every row tile walks its super-blocks from a different start (wrapping
    // around), so that the CTAs do not all ask L2 for the same X tile at the
    // same moment.
    const int rot = static_cast<int>(blockIdx.x % static_cast<unsigned>(nloc));
    auto sb_of = [&](int i) {
        const int j = i + rot;
        return sb_begin + (j >= nloc ? j - nloc : j);
    };
    const size_t row_bytes = static_cast<size_t>(nsb) * 144;

    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&full_a[s]), 128);
            mbar_init(smem_u32(&full_b[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 128);
        }
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(&tmem_base_s), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    auto fail = [&]() {
        atomicOr(&g_prefill_error, 2u);
        s_abort = 1;
    };
    auto aborted = [&]() { return *(volatile int *)&s_abort != 0; };

    float acc[TN];
#pragma unroll
    for (int i = 0; i < TN; ++i) acc[i] = 0.f;

    if (warp < 4) {
        // ------------------------------------------------ weight tiles + epilogue
        const int r = tid;
        const int n = row0 + r;
        const bool live = n < N;
        const uint8_t *wrow = W + static_cast<size_t>(live ? n : 0) * row_bytes;
        int stage = 0;
        uint32_t phase = 0;
        auto load_sb = [&](int i, uint4 (&q)[9]) {
            const bool ok = live && i < nloc;
            const uint4 *bp = reinterpret_cast<const uint4 *>(wrow + static_cast<size_t>(sb_of(ok ? i : 0)) * 144);
#pragma unroll
            for (int u = 0; u < 9; ++u) q[u] = ok ? __ldg(bp + u) : make_uint4(0, 0, 0, 0);
            // and ask L2 for the super-block after it, so that its loads,
            // issued one super-block from now, find it there
            if (live && i + 1 < nloc) {
                const uint8_t *nb = wrow + static_cast<size_t>(sb_of(i + 1)) * 144;
                prefetch_l2(nb);
                prefetch_l2(nb + 128);
                prefetch_l2(nb + 143);
            }
        };
        auto next_stage = [&]() {
            if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        };
        auto wait_empty = [&]() {
            if (!aborted() && !mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, kWaitLimitNs)) fail();
        };
        // part g of a super-block: the stage it goes to is entered at its
        // first part and handed over after its last
        auto part_begin = [&](int g) {
            if (g % PS == 0) wait_empty();
            return smem + stage * C::kStageBytes + (g % PS) * kATileBytes + r * 128;
        };
        auto part_end = [&](int g) {
            if (g % PS == PS - 1) {
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&full_a[stage]));
                next_stage();
            }
        };
        // the five parts of one super-block; returns its {d, 64 dmin}
        auto produce_sb = [&](const uint4 (&q)[9]) {
            uint32_t mpairs[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const RowConsts rc = decode_header(q[0], pair_sel(p));
                mpairs[p] = rc.mpair;
                uint8_t *arow = part_begin(p);
                const uint32_t words[8] = {q[1 + 2 * p].x, q[1 + 2 * p].y, q[1 + 2 * p].z, q[1 + 2 * p].w,
                                           q[2 + 2 * p].x, q[2 + 2 * p].y, q[2 + 2 * p].z, q[2 + 2 * p].w};
                const uint32_t k1024 = 0x64006400u;
#pragma unroll
                for (int half = 0; half < 2; ++half) {       // 0: sub-block 2p (low nibbles), 1: 2p+1
                    const uint32_t mask = half ? 0x00F000F0u : 0x000F000Fu;
                    const uint32_t mul = half ? rc.mulO : rc.mulE;
                    const uint32_t add = half ? rc.addO : rc.addE;
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        uint32_t out[4];
#pragma unroll
                        for (int uu = 0; uu < 2; ++uu) {
                            const uint32_t w = words[2 * c8 + uu];
                            // {q sc (4u), q sc (4u+2)}, {q sc (4u+1), q sc (4u+3)}
                            out[2 * uu] = hfma2_u32(and_or(w, mask, k1024), mul, add);
                            out[2 * uu + 1] = hfma2_u32(and_or(w >> 8, mask, k1024), mul, add);
                        }
                        const int chunk = 4 * half + c8;
                        *reinterpret_cast<uint4 *>(arow + ((chunk ^ (r & 7)) << 4)) =
                            make_uint4(out[0], out[1], out[2], out[3]);
                    }
                }
                part_end(p);
            }
            // min part: {m_0..m_7} in k 0..7 and again in k 8..15
            {
                uint8_t *arow = part_begin(4);
                const uint4 mv = make_uint4(mpairs[0], mpairs[1], mpairs[2], mpairs[3]);
                *reinterpret_cast<uint4 *>(arow + ((0 ^ (r & 7)) << 4)) = mv;
                *reinterpret_cast<uint4 *>(arow + ((1 ^ (r & 7)) << 4)) = mv;
            }
            part_end(4);
            return make_float2(half_lo_f32(q[0].x), 64.0f * half_hi_f32(q[0].x));
        };
        // acc += d D - 64 dmin M for local super-block i, then free its buffer
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        auto epilogue_sb = [&](int i, float2 dd) {
            const int buf = i & 1;
            if (!aborted() && !mbar_wait_bounded(smem_u32(&acc_full[buf]), static_cast<uint32_t>((i >> 1) & 1), kWaitLimitNs))
                fail();
            tc_fence_after();
            const uint32_t col = lane_addr + static_cast<uint32_t>(buf * 2 * TN);
#pragma unroll
            for (int c0 = 0; c0 < TN; c0 += 16) {
                uint32_t vd[16], vm[16];
                tmem_ld16(col + c0, vd);
                tmem_ld16(col + TN + c0, vm);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    acc[c0 + u] = fmaf(dd.x, __uint_as_float(vd[u]), fmaf(-dd.y, __uint_as_float(vm[u]), acc[c0 + u]));
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&acc_empty[buf]));
        };
        uint4 qa[9], qb[9];
        float2 dprev = make_float2(0.f, 0.f);
        load_sb(0, qa);
        for (int i = 0; i < nloc; i += 2) {
            load_sb(i + 1, qb);
            const float2 da = produce_sb(qa);
            if (i > 0) epilogue_sb(i - 1, dprev);
            dprev = da;
            if (i + 1 < nloc) {
                load_sb(i + 2, qa);
                const float2 db = produce_sb(qb);
                epilogue_sb(i, dprev);
                dprev = db;
            }
        }
        epilogue_sb(nloc - 1, dprev);
    } else if (warp == 4) {
        // ------------------------------------------------ X tiles and sub-block sums by TMA
        if (lane == 0) {
            pdl_wait();   // X and the sums are written by the conversion kernel launched just before
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            for (int i = 0; i < nloc; ++i) {
                const int sb = sb_of(i);
                for (int p = 0; p < 5; ++p) {
                    const uint32_t bar = smem_u32(&full_b[stage]);
                    if (p % PS == 0) {
                        if (!aborted() && !mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, kWaitLimitNs)) fail();
                        if (!aborted()) {
                            mbar_arrive_expect_tx(bar, PS * C::kBBytes);
                            ++issued;
                        }
                    }
                    if (!aborted()) {
                        const uint32_t dst =
                            smem_u32(smem + stage * C::kStageBytes + PS * kATileBytes + (p % PS) * C::kBBytes);
                        if (p < 4) tma_load_2d(dst, &tmX, (4 * sb + p) * kChunk, t0, bar);
                        else tma_load_2d(dst, &tmS, sb * kChunk, t0, bar);
                    }
                    if (p % PS == PS - 1 && ++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (aborted()) {
                for (int j = max(0, issued - C::kStages); j < issued; ++j)
                    if (!mbar_wait_bounded(smem_u32(&full_b[j % C::kStages]), static_cast<uint32_t>((j / C::kStages) & 1),
                                           kWaitLimitNs))
                        break;
            }
        }
    } else {
        // ------------------------------------------------ MMA issuer (whole warp, one elected lane issues)
        {
            int stage = 0;
            uint32_t phase = 0;
            constexpr uint32_t idesc = idesc_f16(kRowsM, TN);
            for (int i = 0; i < nloc; ++i) {
                const int buf = i & 1;
                bool bok = i < 2 || aborted() ||
                           mbar_wait_bounded(smem_u32(&acc_empty[buf]), static_cast<uint32_t>(((i >> 1) - 1) & 1), kWaitLimitNs);
                bok = __all_sync(0xffffffffu, bok);
                if (!bok && lane == 0) fail();
                tc_fence_after();
                const uint32_t dcol = tmem + static_cast<uint32_t>(buf * 2 * TN);
                bool ok = true;
                for (int p = 0; p < 5; ++p) {
                    if (p % PS == 0) {
                        ok = !aborted();
                        if (ok && !mbar_wait_bounded(smem_u32(&full_a[stage]), phase, kWaitLimitNs)) ok = false;
                        if (ok && !mbar_wait_bounded(smem_u32(&full_b[stage]), phase, kWaitLimitNs)) ok = false;
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok && lane == 0 && !aborted()) fail();
                        tc_fence_after();
                    }
                    if (ok) {
                        const uint32_t a_addr = smem_u32(smem + stage * C::kStageBytes + (p % PS) * kATileBytes);
                        const uint32_t b_addr = smem_u32(smem + stage * C::kStageBytes + PS * kATileBytes + (p % PS) * C::kBBytes);
                        if (p < 4) {
#pragma unroll
                            for (int kk = 0; kk < kChunk / 16; ++kk)
                                umma_f16(dcol, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32), idesc,
                                         (p > 0 || kk > 0) ? 1u : 0u);
                        } else {
                            umma_f16(dcol + TN, sw128_desc(a_addr), sw128_desc(b_addr), idesc, 0u);
                        }
                    }
                    if (p % PS == PS - 1) {
                        umma_commit(smem_u32(&empty[stage]));
                        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                    }
                }
                umma_commit(smem_u32(&acc_full[buf]));
            }
        }
    }

    // ---------------------------------------------------- output (warps 0-3)
    // y = acc * 2^-e_t.  With a K split the scaled partial rows go to shared
    // memory and CTA rank z of the cluster sums its share of rows over the
    // ranks in order (as in the kernel above).
    float *part = reinterpret_cast<float *>(smem);
    if (warp < 4) {
        pdl_wait();
        if (tid < TN) s_xexp[tid] = (t0 + tid < T) ? __ldg(xexp + t0 + tid) : 0;
        named_bar_sync(1, 128);
        const int r = tid;
        const int n = row0 + r;
        const bool ok = !aborted();
#pragma unroll
        for (int i = 0; i < TN; ++i) {
            const float o = acc[i] * __uint_as_float(static_cast<uint32_t>(127 - s_xexp[i]) << 23);
            if (split > 1) part[i * kRowsM + r] = o;
            else if (ok && n < N && t0 + i < T) Y[static_cast<size_t>(t0 + i) * N + n] = o;
        }
    }
    if (split > 1) {
        __syncthreads();
        cluster_sync_all();
        if (!aborted()) reduce_split(smem_u32(part), split, kz, TN, row0, t0, Y, N, T, tid, kThreads);
        cluster_sync_all();
    }
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace pf

// ------------------------------------------------------------------ host
// Parts of a super-block per stage of the exact kernel at 32-token tiles (5:
// the whole super-block in one stage, one barrier hand-off per super-block).
constexpr int kExactParts32 = 5;

static q4k_status validate_prefill(const void *W, const void *X, const float *Y, int64_t N, int64_t K, int64_t T)
{
    const bool empty = (N == 0 || T == 0);       // nothing is read or written
    if (!empty && (!W || !X || !Y)) return Q4K_ERR_INVALID_ARG;
    if (N < 0 || N > 0x7FFFFFFFll || T < 0 || T > 0x7FFFFFFFll) return Q4K_ERR_INVALID_ARG;
    if (K <= 0 || (K % 256) != 0 || K / 256 >= (1ll << 24)) return Q4K_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15u) || (reinterpret_cast<uintptr_t>(X) & 15u)) return Q4K_ERR_MISALIGNED;
    return Q4K_OK;
}

template <int TN, int NTT>
static cudaError_t launch_prefill(const uint8_t *W, const void *Xh, const int *xexp, float *Y, int N, int K, int T,
                                  int split, cudaStream_t s)
{
    using C = pf::Cfg<TN, NTT>;
    // the split-K partial tile (128 x TN*NTT fp32) reuses the pipeline buffers
    if (static_cast<size_t>(TN) * NTT * pf::kRowsM * 4 > C::kSmem) split = 1;
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap map;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(T)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(pf::kChunk), static_cast<cuuint32_t>(TN)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(Xh), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // W as a 2-D tensor of 8-byte words: [N rows] x [K/256 * 18 words], box =
    // one super-block of 128 rows (rows past N read as zeros)
    CUtensorMap wmap;
    {
        const int64_t nb = K / 256;
        cuuint64_t wdim[2] = {static_cast<cuuint64_t>(nb * 18), static_cast<cuuint64_t>(N)};
        cuuint64_t wstride[1] = {static_cast<cuuint64_t>(nb * 144)};
        cuuint32_t wbox[2] = {18, static_cast<cuuint32_t>(pf::kRowsM)};
        if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t *>(W), wdim, wstride, wbox, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    auto kern = pf::q4k_prefill_kernel<TN, NTT>;
    // the shared-memory limit is a per-device attribute: set it once per device
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return de;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    std::call_once(once[dev], [&]() {
        attr_err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem));
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + pf::kRowsM - 1) / pf::kRowsM, (T + TN * NTT - 1) / (TN * NTT), split);
    cfg.blockDim = dim3(pf::FLay<TN>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = split;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (split > 1) attrs[na++] = attr[0];
    // W streams and dequantizes while the X conversion before it finishes;
    // the kernel waits for it (griddepcontrol.wait) before reading X
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, map, wmap, W, xexp, Y, N, K, T);
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e;
}

static bool encode_f16_map(CUtensorMap *map, const void *base, int cols, int rows, int box_rows)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(pf::kChunk), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int TN, int PS>
static cudaError_t launch_prefill_exact(const uint8_t *W, const void *Xh, const void *XS, const int *xexp, float *Y,
                                        int N, int K, int T, int split, cudaStream_t s)
{
    using C = pf::ECfg<TN, PS>;
    CUtensorMap mx, ms;
    if (!encode_f16_map(&mx, Xh, K, T, TN) || !encode_f16_map(&ms, XS, (K / 256) * pf::kChunk, T, TN))
        return cudaErrorInvalidValue;
    auto kern = pf::q4k_prefill_exact_kernel<TN, PS>;
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return de;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    std::call_once(once[dev], [&]() {
        attr_err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem));
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + pf::kRowsM - 1) / pf::kRowsM, (T + TN - 1) / TN, split);
    cfg.blockDim = dim3(pf::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (split > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = split;
        ++na;
    }
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mx, ms, W, xexp, Y, N, K, T);
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e;
}

// Clusters of csize CTAs (2, 4 or 8) of kernel `kid` (0: exact 32-token,
// 1: exact 64-token, 2: fp16 128-token, 3: fp16 256-token, 4: fp16 64-token
// tiles) that the GPU
// holds at once, queried once per device; -1 when the query fails (the caller
// then does not limit the split on it).
static int max_active_clusters(int kid, int csize)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return -1;
    }
    const int ci = (csize == 2) ? 0 : (csize == 4) ? 1 : 2;
    static std::mutex mu;
    static int cache[64][5][3];
    static bool have[64][5][3];
    std::lock_guard<std::mutex> lock(mu);
    if (have[dev][kid][ci]) return cache[dev][kid][ci];
    const void *kern = nullptr;
    size_t smem = 0;
    int threads = pf::kThreads;
    switch (kid) {
    case 0: kern = reinterpret_cast<const void *>(pf::q4k_prefill_exact_kernel<32, kExactParts32>);
            smem = pf::ECfg<32, kExactParts32>::kSmem; break;
    case 1: kern = reinterpret_cast<const void *>(pf::q4k_prefill_exact_kernel<64, 1>); smem = pf::ECfg<64, 1>::kSmem; break;
    case 2: kern = reinterpret_cast<const void *>(pf::q4k_prefill_kernel<128, 1>); smem = pf::Cfg<128, 1>::kSmem;
            threads = pf::FLay<128>::kThreads; break;
    case 4: kern = reinterpret_cast<const void *>(pf::q4k_prefill_kernel<64, 1>); smem = pf::Cfg<64, 1>::kSmem;
            threads = pf::FLay<64>::kThreads; break;
    default: kern = reinterpret_cast<const void *>(pf::q4k_prefill_kernel<256, 1>); smem = pf::Cfg<256, 1>::kSmem;
             threads = pf::FLay<256>::kThreads; break;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, csize);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = 1;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = csize;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        n = -1;
    }
    cache[dev][kid][ci] = n;
    have[dev][kid][ci] = true;
    return n;
}

// Up to this many tokens the plain entry point takes the exact kernel too:
// with the weights streamed from HBM it is as fast there or a little faster
// (14336 x 4096 at 32 tokens: 35.3 against 36.2 us), and no weight is rounded.
constexpr int kExactDefaultMaxT = 32;

q4k_status prefill_impl(const void *W, const void *X, float *Y, int64_t N, int64_t K, int64_t T, void *stream,
                        bool exact_requested)
{
    q4k_status st = validate_prefill(W, X, Y, N, K, T);
    if (st != Q4K_OK) return st;
    int sms = 0;
    st = check_device(&sms);
    if (st != Q4K_OK) return st;
    if (N == 0 || T == 0) return Q4K_OK;
    const auto *Wb = static_cast<const uint8_t *>(W);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int n = static_cast<int>(N), k = static_cast<int>(K), t = static_cast<int>(T);
    const int mtiles = (n + pf::kRowsM - 1) / pf::kRowsM;
    // Token tiling: one CTA covers up to 512 tokens (weights dequantized once)
    // unless that leaves too few CTAs, then 256-token tiles.
    int tn, ntt;
    if (t <= 32) { tn = 32; ntt = 1; }
    else if (t <= 64) { tn = 64; ntt = 1; }
    else if (t <= 128) { tn = 128; ntt = 1; }
    else if (t <= 256) { tn = 256; ntt = 1; }
    // 512-token tiles dequantize each weight tile half as often; they pay
    // once they fill at least 70 % of the SMs (14336 rows: 112 tiles on 152
    // SMs take about three quarters of the time of two waves of 256-token
    // tiles)
    else if (static_cast<long long>(mtiles) * ((t + 511) / 512) * 10 >= static_cast<long long>(sms) * 7) { tn = 256; ntt = 2; }
    else { tn = 256; ntt = 1; }
    // The exact kernel (integer weight tiles, no weight rounding) on request or
    // up to kExactDefaultMaxT tokens, in 32- or 64-token tiles; the fp16
    // kernel otherwise, whose 64-token tiles beat the exact kernel from 33 to
    // 64 tokens (14336 x 4096 at 64 tokens: 35.2 against 44.2 us).
    const bool exact = exact_requested || t <= kExactDefaultMaxT;
    if (exact) {
        tn = (t <= 32) ? 32 : 64;
        ntt = 1;
    } else if (tn < 64) {
        tn = 64;   // the fp16 kernel's smallest token tile
    }
    const long long ctas = static_cast<long long>(mtiles) * ((t + tn * ntt - 1) / (tn * ntt));
    // K split over a cluster until the GPU is covered (at most 8, at least
    // two super-blocks per CTA).
    // (one CTA per SM, except the exact kernel's 32-token tiles with one part per stage)
    const long long slots = exact && tn == 32 && pf::ECfg<32, kExactParts32>::kTwoPerSm ? 2LL * sms
                                                                                         : static_cast<long long>(sms);
    // ... and only while every cluster of the split fits on the GPU at once
    // (clusters of eight CTAs that take a whole SM each stop fitting well
    // before 152 CTAs: at 1024 x 4096 and 512 tokens, sixteen of them ran
    // in two waves, 30 us, against 19 us for sixteen clusters of four)
    const int kid = exact ? (tn == 32 ? 0 : 1) : (tn == 64 ? 4 : tn == 128 ? 2 : 3);
    int split = 1;
    while (ntt == 1 && split < 8 && ctas * split * 2 <= slots && (k / 256) / (split * 2) >= 2) {
        const int fit = max_active_clusters(kid, split * 2);
        if (fit > 0 && ctas > fit) break;
        split *= 2;
    }
    // X in fp16 under a power-of-two scale per token: T*K*2 bytes, the
    // exponents, and for the exact kernel the sub-block sums (T*K/2 bytes),
    // from the stream-ordered allocator on the caller's stream
    const size_t xh_bytes = (static_cast<size_t>(T) * static_cast<size_t>(K) * 2 + 255) & ~size_t(255);
    const size_t xe_bytes = (static_cast<size_t>(T) * 4 + 255) & ~size_t(255);
    const size_t xs_bytes = exact ? static_cast<size_t>(T) * static_cast<size_t>(K) / 2 : 0;
    void *scratch = nullptr;
    if (cudaMallocAsync(&scratch, xh_bytes + xe_bytes + xs_bytes, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return Q4K_ERR_CUDA;
    }
    uint16_t *Xh = static_cast<uint16_t *>(scratch);
    int *xexp = reinterpret_cast<int *>(static_cast<uint8_t *>(scratch) + xh_bytes);
    uint16_t *XS = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(scratch) + xh_bytes + xe_bytes);
    if (exact) pf::x_to_f16_kernel<true><<<t, 256, 0, s>>>(static_cast<const uint16_t *>(X), Xh, xexp, XS, k);
    else pf::x_to_f16_kernel<false><<<t, 256, 0, s>>>(static_cast<const uint16_t *>(X), Xh, xexp, nullptr, k);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) {
        if (exact && tn == 32) e = launch_prefill_exact<32, kExactParts32>(Wb, Xh, XS, xexp, Y, n, k, t, split, s);
        else if (exact) e = launch_prefill_exact<64, 1>(Wb, Xh, XS, xexp, Y, n, k, t, split, s);
        else if (tn == 64) e = launch_prefill<64, 1>(Wb, Xh, xexp, Y, n, k, t, split, s);
        else if (tn == 128) e = launch_prefill<128, 1>(Wb, Xh, xexp, Y, n, k, t, split, s);
        else if (ntt == 1) e = launch_prefill<256, 1>(Wb, Xh, xexp, Y, n, k, t, split, s);
        else e = launch_prefill<256, 2>(Wb, Xh, xexp, Y, n, k, t, split, s);
    }
    const cudaError_t ef = cudaFreeAsync(scratch, s);
    if (e == cudaSuccess) e = ef;
    return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
}

}  // namespace q4k
