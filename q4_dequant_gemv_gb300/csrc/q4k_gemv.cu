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
//   * Batch 1 with too few 128-row tiles and K <= 8192 (q/k/v, o): 16-row
//     tiles instead, one CTA per tile over the whole K, the K split between
//     its warps and their partial rows added in shared memory (no cluster).
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

#include "q4k_dev.cuh"

namespace q4k {

constexpr int kWarps = 8;                 // warps per CTA, 16 weight rows each
constexpr int kRows = 16 * kWarps;        // rows per tile (128)
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 4;                // W ring depth
constexpr int kPreWait = 1;               // stages issued before the dependency wait
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
    uint64_t wait_ns;          // bound of every wait (default 2 s)
    int test_stall;            // tests: the first stage expects 16 bytes more than its copy brings
};


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

// ---------------------------------------------------------------------------
// A chunk of x (B rows x nblk super-blocks, B * nblk <= 32) -> B fragments in
// shared memory (x_item_tc per item).  One warp converts one (batch row,
// super-block) item per round; all loads of all rounds are issued first, then
// after_loads() runs (the kernel issues its remaining weight stages there, so
// that they queue behind x, not ahead of it).  The
// item scales go to s_unscale[bl*B + b].  Ends with a barrier over all nthr
// threads; the caller must have finished reading the previous chunk's
// fragments and scales.
template <int NT, typename AfterLoads>
__device__ void convert_x_blocks(const float *__restrict__ x, int K, int B, int kb0, int nblk, uint2 *xf,
                                 float *s_unscale, int tid, int nthr, AfterLoads after_loads)
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
            v[r][0] = __ldg(src + lane);
            v[r][1] = __ldg(src + 32 + lane);
        }
    }
    after_loads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int it = warp + r * nwarps;
        if (it >= items) continue;   // warp-uniform
        const int b = it / nblk;
        const int bl = it - b * nblk;
        const float us = x_item_tc<NT>(v[r][0], v[r][1], lane, b, LW, xf + static_cast<size_t>(bl) * LW * LS);
        if (lane == 0) s_unscale[bl * B + b] = us;
    }
    named_bar_sync(1, nthr);
}

// Batch 1: a chunk of x (nblk <= 32 super-blocks) -> the int8 parts of
// x_item_i8, one super-block per warp and round, at xb + bl * blk_bytes; the
// scales go to s_unscale[bl], s_pre[bl].  Ends with a barrier over all nthr
// threads.
template <bool Q8, typename AfterLoads>
__device__ void convert_x_i8_blocks(const float *__restrict__ x, int kb0, int nblk, uint8_t *xb, int blk_bytes,
                                    float *s_unscale, float *s_pre, int tid, int nthr, AfterLoads after_loads)
{
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    float4 v[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int it = warp + r * nwarps;
        if (it < nblk) {   // warp-uniform
            const float4 *src = reinterpret_cast<const float4 *>(x + static_cast<size_t>(kb0 + it) * 256);
            v[r][0] = __ldg(src + lane);
            v[r][1] = __ldg(src + 32 + lane);
        }
    }
    after_loads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int it = warp + r * nwarps;
        if (it >= nblk) continue;   // warp-uniform
        const float2 sp = x_item_i8<Q8>(v[r][0], v[r][1], lane, xb + static_cast<size_t>(it) * blk_bytes);
        if (lane == 0) {
            s_unscale[it] = sp.x;
            s_pre[it] = sp.y;
        }
    }
    named_bar_sync(1, nthr);
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

template <int R = kRows, typename Desc>
__device__ __forceinline__ TileInfo tile_info(const Desc &a, int tile)
{
    TileInfo ti{0, tile * R, a.N[0], a.y[0]};
#pragma unroll
    for (int i = 1; i < kMaxGroups; ++i) {
        if (i < a.ngroups && tile >= a.tile_start[i]) {
            ti.grp = i;
            ti.row0 = (tile - a.tile_start[i]) * R;
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
        // (test_stall: the first stage waits for 16 bytes that never come, so
        // that a test can make the bounded waits run out)
        mbar_arrive_expect_tx(smem_u32(&full[slot]), kStageBytes + ((args->test_stall && i == 0) ? 16 : 0));
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
        // Only kPreWait of them: the x loads after the wait queue behind every
        // weight byte already requested by this SM, and a CTA that starts only
        // when the previous kernel ends would otherwise wait for its whole
        // ring before it sees x.  The rest follow the x loads.
        iss.policy = l2_policy_evict_first();
        const int first = min(kPreWait, iss.total);
        for (int i = 0; i < first; ++i) iss.issue(i);
        s_issued = first;
    }
    if (ARGMAX && tid < 16) s_best[tid] = 0ull;
    __syncthreads();
    iss.policy = l2_policy_evict_first();
    // every CTA of a cluster has started once this phase completes; it is
    // waited for only before the first remote store, at the very end
    if (split > 1) cluster_arrive_relaxed();

    pdl_launch_dependents();
    pdl_wait();                             // x may come from the previous kernel

    // the rest of the first kStages stages, once this thread's x loads are out
    auto issue_rest = [&]() {
        if (tid == 0) {
            const int first = min(kStages, iss.total);
            for (int i = s_issued; i < first; ++i) iss.issue(i);
            s_issued = first;
        }
    };
    const int g = lane >> 2;
    const int t = lane & 3;
    const PairSel psel = pair_sel(t);
    const int nchunks = (ks + args.kc - 1) / args.kc;
    const bool single_chunk = (nchunks == 1);
    // batch 1 on the integer path: int8 x parts, one block of the fragment area per super-block
    static_assert(!I8 || NT == 1, "the integer path is batch 1 only");
    uint8_t *xb = reinterpret_cast<uint8_t *>(xf);
    const int blk_bytes = static_cast<int>(xfrag_bytes_per_block(1, 1));
    if (single_chunk) {
        if constexpr (I8)
            convert_x_i8_blocks<Q8>(args.x, kb_begin, ks, xb, blk_bytes, s_unscale, s_pre, tid, kThreads, issue_rest);
        else
            convert_x_blocks<NT>(args.x, nb * 256, B, kb_begin, ks, xf, s_unscale, tid, kThreads, issue_rest);
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
        int blk = -1;   // this super-block's place in the x chunk (counted, not divided)
        for (int kbl = 0; kbl < ks; ++kbl) {
            ++blk;
            if (!single_chunk && kbl > chunk_end) {
                const int cn = min(args.kc, ks - kbl);
                named_bar_sync(1, kThreads);     // everyone done with the previous chunk
                const bool first_chunk = ti_idx == 0 && kbl == 0;
                auto maybe_rest = [&]() {
                    if (first_chunk) issue_rest();
                };
                if constexpr (I8)
                    convert_x_i8_blocks<Q8>(args.x, kb_begin + kbl, cn, xb, blk_bytes, s_unscale, s_pre, tid, kThreads,
                                            maybe_rest);
                else
                    convert_x_blocks<NT>(args.x, nb * 256, B, kb_begin + kbl, cn, xf, s_unscale, tid, kThreads, maybe_rest);
                chunk_end = kbl + cn - 1;
                blk = 0;
            }
            // this super-block's x scale per batch row
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
            if (!*(volatile int *)&s_abort && !mbar_wait_bounded(smem_u32(&full[slot]), phase, args.wait_ns)) {
                atomicOr(&g_device_error, 1u);
                s_abort = 1;
            }
            const uint8_t *ra = ring + slot * kStageBytes + row_off;   // row g of this warp
            const uint8_t *rb = ra + 8 * kBlockBytes;                   // row g + 8
            // this lane's B fragments of this super-block (lane-major layout)
            const uint2 *xl = xf + static_cast<size_t>(blk * LW + blane) * lane_stride(NT);
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
                stage_compute_i8<Q8>(ra, rb, xb + blk * blk_bytes, t, psel, unscale[0], s_pre[blk], acc, release);
            else
                stage_compute<NT, NT == 1 ? 2 : 1>(ra, rb, xl, t, psel, unscale, acc, release);
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

    // After a timed-out wait, wait (bounded) for the copies this CTA may still
    // have in flight, so that none of them lands after the CTA has exited.
    // Stage i + kStages is issued only once every warp has waited for stage i,
    // and nothing is issued after the abort, so only the last kStages stages
    // issued can be outstanding.
    __syncthreads();
    if (*(volatile int *)&s_abort && tid == 0) {
        for (int i = max(0, s_issued - kStages); i < s_issued; ++i)
            (void)mbar_wait_bounded(smem_u32(&full[i % kStages]), static_cast<uint32_t>((i / kStages) & 1), args.wait_ns);
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
// Batch 1, 16-row tiles (q4k_gemv_rows16_kernel).  For matrices with too few
// 128-row tiles to fill the GPU (the q/k/v and o projections of a decoder
// layer), the 128-row kernel splits K over the CTAs of a cluster, and its
// epilogue (distributed shared-memory stores, a cluster barrier that waits
// for the slowest CTA, the rank-ordered sum) is most of such a launch.  Here
// a CTA of 8 warps owns 16 rows over the whole K instead: the K split is
// between its warps, and their partial rows meet in shared memory.
//   * Stage = the tile's 16 rows x kT16Sb super-blocks (one 2-D TMA box; the
//     row stride kT16Sb*144 bytes, kT16Sb odd, keeps the fragment loads free
//     of bank conflicts).  Super-block j of the row goes to warp j % 8.
//   * Warp w converts the x of its own super-blocks (w, w + 8, ...) into the
//     integer parts of the 128-row kernel, once per CTA (all tiles of a CTA
//     share x), into shared memory of its own: no barrier comes before the
//     first inner product.
//   * The ring and its refill are those of the 128-row kernel: every warp
//     waits for every stage, and the last warp to leave a slot issues the
//     stage kT16Stages ahead into it.
// ---------------------------------------------------------------------------
constexpr int kT16Rows = 16;
constexpr int kT16Sb = 7;                                          // super-blocks per stage
constexpr int kT16Stages = 4;                                      // ring depth
constexpr int kT16StageBytes = kT16Rows * kT16Sb * kBlockBytes;    // 16,128
constexpr int kT16XPerWarp = 4;                                    // x super-blocks per warp
constexpr int kT16MaxNb = kWarps * kT16XPerWarp;                   // K <= 8192
constexpr int kT16PreWait = 1;                                     // stages issued before the dependency wait
__host__ __device__ constexpr size_t t16_smem_bytes()
{
    return static_cast<size_t>(kT16Stages) * kT16StageBytes + static_cast<size_t>(kWarps) * kT16XPerWarp * kI8Bytes;
}

template <int XM>
__global__ void __launch_bounds__(kThreads, 2) q4k_gemv_rows16_kernel(const __grid_constant__ WMaps maps,
                                                                     const GemvArgs args)
{
    constexpr bool Q8 = XM == 2;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *ring = smem_raw;
    uint8_t *xarea = smem_raw + static_cast<size_t>(kT16Stages) * kT16StageBytes;
    __shared__ __align__(8) uint64_t full[kT16Stages];
    __shared__ int s_slot_done[kT16Stages];
    __shared__ int s_abort;
    __shared__ int s_issued;
    __shared__ float2 s_sc[kT16MaxNb];         // per super-block: (unscale, pre) of its x
    __shared__ float s_red[2][kWarps][kT16Rows];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int nb = args.nb;
    const int spt = (nb + kT16Sb - 1) / kT16Sb;   // stages per tile
    const int my_tiles = (args.tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                         static_cast<int>(gridDim.x);
    const int total = my_tiles * spt;
    uint64_t policy = 0;

    // stage i of this CTA's schedule -> ring slot i % kT16Stages
    auto issue = [&](int i) {
        const int tile = static_cast<int>(blockIdx.x) + (i / spt) * static_cast<int>(gridDim.x);
        const TileInfo ti = tile_info<kT16Rows>(args, tile);
        const CUtensorMap *map = &maps.m[0];
#pragma unroll
        for (int gi = 1; gi < kMaxGroups; ++gi)
            if (gi == ti.grp) map = &maps.m[gi];
        const int slot = i % kT16Stages;
        mbar_arrive_expect_tx(smem_u32(&full[slot]), kT16StageBytes + ((args.test_stall && i == 0) ? 16 : 0));
        tma_load_2d_hint(smem_u32(ring + static_cast<size_t>(slot) * kT16StageBytes), map,
                         (i % spt) * kT16Sb * (kBlockBytes / 8), ti.row0, smem_u32(&full[slot]), policy);
    };

    if (tid == 0) {
        for (int i = 0; i < kT16Stages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            s_slot_done[i] = 0;
        }
        s_abort = 0;
        fence_barrier_init();
#pragma unroll
        for (int gi = 0; gi < kMaxGroups; ++gi)
            if (gi < args.ngroups) prefetch_tensormap(&maps.m[gi]);
        policy = l2_policy_evict_first();
        const int first = min(kT16PreWait, total);
        for (int i = 0; i < first; ++i) issue(i);
        s_issued = first;
    }
    __syncthreads();
    policy = l2_policy_evict_first();

    pdl_launch_dependents();
    pdl_wait();   // x may come from the previous kernel

    // x of this warp's super-blocks, four at a time: loads first (the rest of
    // the ring is issued behind the first four), then the conversion
    uint8_t *xw = xarea + static_cast<size_t>(warp) * kT16XPerWarp * kI8Bytes;
#pragma unroll 1
    for (int r0 = 0; r0 < kT16XPerWarp && warp + kWarps * r0 < nb; r0 += 4) {
        float4 v[4][2];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int j = warp + kWarps * (r0 + r);
            if (r0 + r < kT16XPerWarp && j < nb) {   // warp-uniform
                const float4 *src = reinterpret_cast<const float4 *>(args.x + static_cast<size_t>(j) * 256);
                v[r][0] = __ldg(src + lane);
                v[r][1] = __ldg(src + 32 + lane);
            }
        }
        if (r0 == 0 && tid == 0) {
            const int first = min(kT16Stages, total);
            for (int i = s_issued; i < first; ++i) issue(i);
            s_issued = first;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int j = warp + kWarps * (r0 + r);
            if (r0 + r < kT16XPerWarp && j < nb) {
                const float2 sp = x_item_i8<Q8>(v[r][0], v[r][1], lane, xw + (r0 + r) * kI8Bytes);
                if (lane == 0) s_sc[j] = sp;
            }
        }
    }
    __syncwarp();

    const PairSel psel = pair_sel(t);
    int consumed = 0;
    for (int ti_idx = 0; ti_idx < my_tiles; ++ti_idx) {
        const int tile = static_cast<int>(blockIdx.x) + ti_idx * static_cast<int>(gridDim.x);
        const TileInfo ti = tile_info<kT16Rows>(args, tile);
        float acc[1][2] = {{0.f, 0.f}};
        for (int st = 0; st < spt; ++st) {
            const int slot = consumed % kT16Stages;
            const uint32_t phase = static_cast<uint32_t>((consumed / kT16Stages) & 1);
            if (!*(volatile int *)&s_abort && !mbar_wait_bounded(smem_u32(&full[slot]), phase, args.wait_ns)) {
                atomicOr(&g_device_error, 1u);
                s_abort = 1;
            }
            auto release = [&]() {
                // the last of the 8 warps to leave the slot refills it
                __syncwarp();
                if (lane == 0) {
                    __threadfence_block();
                    const int prev = atomicAdd(&s_slot_done[slot], 1);
                    if (prev % kWarps == kWarps - 1) {
                        const int next = consumed + kT16Stages;
                        if (next < total && !*(volatile int *)&s_abort) {
                            issue(next);
                            atomicAdd(&s_issued, 1);
                        }
                    }
                }
                ++consumed;
            };
            // this warp's super-block of the stage: the first j >= j0 with j % 8 == warp
            const int j0 = st * kT16Sb;
            const int jw = j0 + ((warp - j0 % kWarps) + kWarps) % kWarps;
            if (jw < min(j0 + kT16Sb, nb) && !*(volatile int *)&s_abort) {
                const uint8_t *ra = ring + static_cast<size_t>(slot) * kT16StageBytes +
                                    g * (kT16Sb * kBlockBytes) + (jw - j0) * kBlockBytes;
                const uint8_t *rb = ra + 8 * (kT16Sb * kBlockBytes);
                const float2 sp = s_sc[jw];
                stage_compute_i8<Q8>(ra, rb, xw + (jw / kWarps) * kI8Bytes, t, psel, sp.x, sp.y, acc, release);
            } else {
                release();
            }
        }
        // tile epilogue: the four pair lanes of each row, then the 8 warps in order
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            acc[0][h] += __shfl_xor_sync(0xffffffffu, acc[0][h], 1);
            acc[0][h] += __shfl_xor_sync(0xffffffffu, acc[0][h], 2);
        }
        const int buf = ti_idx & 1;
        if (t == 0) {
            s_red[buf][warp][g] = acc[0][0];
            s_red[buf][warp][g + 8] = acc[0][1];
        }
        named_bar_sync(1, kThreads);
        if (tid < kT16Rows && !*(volatile int *)&s_abort) {
            float sum = s_red[buf][0][tid];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) sum += s_red[buf][w][tid];
            const int row = ti.row0 + tid;
            if (row < ti.N && ti.y) ti.y[row] = sum;
        }
    }

    // after a timed-out wait: wait (bounded) for the copies still in flight
    __syncthreads();
    if (*(volatile int *)&s_abort && tid == 0) {
        for (int i = max(0, s_issued - kT16Stages); i < s_issued; ++i)
            (void)mbar_wait_bounded(smem_u32(&full[i % kT16Stages]), static_cast<uint32_t>((i / kT16Stages) & 1),
                                    args.wait_ns);
    }
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
    if (pdl) {
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
static int row_tiles16(int64_t N) { return static_cast<int>((N + kT16Rows - 1) / kT16Rows); }

// W as [N rows] x [K/256 * 18 words] with a box of kT16Sb super-blocks of 16
// rows (columns past K and rows past N are zero-filled by the TMA unit).
static bool encode_w_map16(CUtensorMap *map, const void *W, int64_t N, int64_t K)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const int64_t nb = K / 256;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(nb * (kBlockBytes / 8)), static_cast<cuuint64_t>(N)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(nb * kBlockBytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kT16Sb * (kBlockBytes / 8)), static_cast<cuuint32_t>(kT16Rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(W), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Batch 1 on the 16-row kernel: automatically when the 128-row plan would
// split K over CTAs (too few row tiles) and x fits the per-warp area, or on
// request (Q4K_FLAG_ROWS16).  A forced split keeps the 128-row kernel.
static bool use_rows16(const GemvPlan &p, int batch, int64_t K, const q4k_launch_opts *opts)
{
    if (batch != 1 || p.xm == 0 || K / 256 > kT16MaxNb) return false;
    if (opts && (opts->flags & Q4K_FLAG_ROWS16)) return true;
    if (opts && opts->split_k > 0) return false;
    return p.split > 1;
}

// a.tile_start and a.tiles in 16-row tiles.
static cudaError_t launch_rows16(int xm, const void *const *Ws, int64_t K, const GemvArgs &a, int sms,
                                 cudaStream_t stream, bool pdl)
{
    WMaps maps;
    memset(&maps, 0, sizeof(maps));
    for (int g = 0; g < a.ngroups; ++g)
        if (!encode_w_map16(&maps.m[g], Ws[g], a.N[g], K)) return cudaErrorInvalidValue;
    void (*kern)(const WMaps, const GemvArgs) = (xm == 2) ? q4k_gemv_rows16_kernel<2> : q4k_gemv_rows16_kernel<1>;
    static std::mutex mu;
    static bool attr_set[64][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(mu);
        bool &done = attr_set[dev & 63][xm == 2 ? 1 : 0];
        if (!done) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(t16_smem_bytes()));
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
            if (e != cudaSuccess) return e;
            done = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(a.tiles, 2 * sms), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = t16_smem_bytes();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, maps, a);
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e;
}

// Wait bound and the test-only stall of the launch options.
static void set_wait_opts(GemvArgs &a, const q4k_launch_opts *opts)
{
    a.wait_ns = (opts && opts->wait_limit_us > 0) ? static_cast<uint64_t>(opts->wait_limit_us) * 1000ull : kWaitLimitNs;
    a.test_stall = (opts && (opts->flags & Q4K_FLAG_TEST_STALL)) ? 1 : 0;
}

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
    set_wait_opts(a, opts);
    if (opts && (opts->flags & Q4K_FLAG_TENSOR_CORE)) p.xm = 0;
    if (opts && (opts->flags & Q4K_FLAG_Q8K_X)) {
        if (batch != 1 || (opts->flags & Q4K_FLAG_TENSOR_CORE)) return Q4K_ERR_INVALID_ARG;
        p.xm = 2;
    }
    if (opts && (opts->flags & Q4K_FLAG_ROWS16) && (batch != 1 || p.xm == 0 || K / 256 > kT16MaxNb))
        return Q4K_ERR_INVALID_ARG;
    if (use_rows16(p, batch, K, opts)) {
        a.tile_start[1] = a.tiles = row_tiles16(N);
        cudaError_t e = launch_rows16(p.xm, &W, K, a, sms, static_cast<cudaStream_t>(stream), pdl);
        return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
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
    set_wait_opts(a, opts);
    if (opts && (opts->flags & Q4K_FLAG_TENSOR_CORE)) p.xm = 0;
    if (opts && (opts->flags & Q4K_FLAG_Q8K_X)) {
        if (batch != 1 || (opts->flags & Q4K_FLAG_TENSOR_CORE)) return Q4K_ERR_INVALID_ARG;
        p.xm = 2;
    }
    if (opts && (opts->flags & Q4K_FLAG_ROWS16) && (batch != 1 || p.xm == 0 || K / 256 > kT16MaxNb))
        return Q4K_ERR_INVALID_ARG;
    if (use_rows16(p, batch, K, opts)) {
        int t16 = 0;
        for (int g = 0; g < a.ngroups; ++g) {
            a.tile_start[g] = t16;
            t16 += row_tiles16(a.N[g]);
        }
        a.tile_start[a.ngroups] = a.tiles = t16;
        cudaError_t e = launch_rows16(p.xm, Ws, K, a, sms, static_cast<cudaStream_t>(stream), pdl);
        return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
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
    set_wait_opts(a, opts);
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
// address, so the address is looked up with cudaGetSymbolAddress with the
// device current: on the first call on each device, and again on every call
// made outside stream capture (a device reset reloads the module and may move
// the array); a call made during capture uses the address of the last call
// made outside it, so make a first call before any stream capture.  All calls
// share the array: it is cleared with cudaMemsetAsync on the caller's stream
// before every launch, and calls whose executions overlap on the GPU
// (different streams, concurrent graphs) race on it.
// ---------------------------------------------------------------------------
constexpr int kNoAllocMaxBatch = 16;   // keys held by the static scratch
__device__ __align__(256) static unsigned long long g_argmax_scratch[kNoAllocMaxBatch + 2];

static unsigned long long *g_scratch_addr[64];   // per device: address from the last lookup
static std::mutex g_scratch_mu;

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
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return Q4K_ERR_CUDA;
    unsigned long long *keys = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        if (cap == cudaStreamCaptureStatusNone || g_scratch_addr[dev] == nullptr) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_argmax_scratch) != cudaSuccess || p == nullptr) {
                (void)cudaGetLastError();
                return Q4K_ERR_CUDA;
            }
            g_scratch_addr[dev] = static_cast<unsigned long long *>(p);
        }
        keys = g_scratch_addr[dev];
    }
    unsigned int *ticket = reinterpret_cast<unsigned int *>(keys + kNoAllocMaxBatch);
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
    if (use_rows16(p, batch, K, nullptr)) {
        out[0] = 1;
        out[1] = std::min(row_tiles16(N), 2 * sms);
        out[2] = kT16Rows;
        out[3] = static_cast<int>(K / 256);
        return Q4K_OK;
    }
    out[0] = p.split;
    out[1] = p.grid_x * p.split;
    out[2] = kRows;
    out[3] = p.kc;
    return Q4K_OK;
}

unsigned int read_device_error()
{
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
    return v;
}

bool clear_device_error()
{
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(g_device_error, &z, sizeof(z)) == cudaSuccess;
}

}  // namespace q4k
