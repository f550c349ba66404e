// Routing-map unpermute on GB300.
//
// "MoeTokenUnpermuteWithRoutingMap 算子全解析", 功能说明与计算公式 (branches
// (1)-(4)) and Kernel 实现 (pad-kernel prob lookup, IsValidInputIndex, the
// prob != 0 skip, fp32 Cast/Muls/Add and the CAST_RINT back-cast).
//
// Launch sequence on the caller's stream (PDL-chained):
//   not padded, probs : maskedSelect: one cooperative kernel (counts per
//                       tile, a grid barrier, the scatter and zero tail) up
//                       to 4096 tiles of 1024 map entries, else column
//                       bitmasks -> csort prefix -> scatter from the
//                       bitmasks; for a small
//                       routing map the gather-reduce selects the weights
//                       itself instead
//   always            : stable sort of sortedIndices -> outIndex,
//                       permuteTokenId: one pass of the counting-sort engine
//                       up to 4096 keys; up to 2^22 keys a coarse pass on
//                       the high bits and fine_sort_kernel; else 2-3 LSD
//                       passes. Padded, the per-token row ranges (CSR) are the
//                       one pass's key starts, the fine sort's, or built from
//                       the sorted keys
//   padded, probs     : permuteProbs[i] = probs[sortedIndices[i], i // capacity],
//                       written by the sort's first scatter
//   not padded        : the sort runs on the caller stream's auxiliary
//                       stream, overlapping the maskedSelect and the
//                       gather-reduce (fork/join events)
//   always            : gather-reduce (reduce.cuh), one warp per (token, run
//                       of hidden chunks), fp32 accumulation in ascending slot
//                       / row order, atomic-free, one RNE cast per output
//                       element; a persistent grid, or, when short and the
//                       sort runs beside it, a plain-order launch of one work
//                       unit per warp.
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include <cooperative_groups.h>

#include "index_sort.cuh"
#include "reduce.cuh"
#include "routing.cuh"

namespace mr {
namespace cg = cooperative_groups;

// maskedSelect beyond the one-kernel form's limit, from the column masks:
// one thread per (32-token block, expert) item; the routed tokens of the
// item's mask land at bucket_start[e] + offs[blk][e] + (set bits below
// them). Threads of consecutive experts read consecutive mask, offset and
// probs words; the routing map itself is not read again.
__global__ void __launch_bounds__(256)
mask_scatter_kernel(const uint32_t* __restrict__ masks, const uint32_t* __restrict__ offs,
                    const uint32_t* __restrict__ bucket_start, int64_t T, int64_t Eu, int64_t n,
                    const uint8_t* __restrict__ probs, int pes, uint8_t* __restrict__ pp) {
    pdl_enter();
    const int64_t items = (T + 31) / 32 * Eu;
    const int64_t nnz = bucket_start[Eu];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t item = tid; item < items; item += stride) {
        uint32_t bits = masks[item];
        if (bits == 0u) continue;
        const int64_t blk = item / Eu;
        const int64_t e = item - blk * Eu;
        int64_t pos = (int64_t)bucket_start[e] + offs[item];
        while (bits) {
            const int j = __ffs(bits) - 1;
            bits &= bits - 1u;
            if (pos < n) copy_prob(pp, pos, probs, (blk * 32 + j) * Eu + e, pes);
            ++pos;
        }
    }
    for (int64_t i = nnz + tid; i < n; i += stride) zero_prob(pp, i, pes);
}

// One-kernel maskedSelect (not padded, with probs) for maps of at most
// kMsMaxTiles tiles: the routed elements of probs.T in expert-major order
// (f = e*T + t, tokens ascending within an expert). Tiles of kMsTile
// consecutive f; each block counts the routed entries of its tiles, a grid
// barrier (cooperative launch: every block resident), then each block sums
// the counts of the lower tiles and scatters its tiles' probs; positions at
// and beyond the routed count are zeroed.
constexpr int kMsThreads = 256;
constexpr int kMsPer = 4;
constexpr int64_t kMsTile = (int64_t)kMsThreads * kMsPer;
constexpr int64_t kMsMaxTiles = 4096;

__device__ __forceinline__ uint32_t ld_prob_bits(const uint8_t* p, int64_t i, int pes) {
    return pes == 4 ? __ldg(reinterpret_cast<const uint32_t*>(p) + i)
                    : (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p) + i);
}
__device__ __forceinline__ void st_prob_bits(uint8_t* p, int64_t i, uint32_t v, int pes) {
    if (pes == 4) reinterpret_cast<uint32_t*>(p)[i] = v;
    else reinterpret_cast<uint16_t*>(p)[i] = (uint16_t)v;
}

__global__ void __launch_bounds__(kMsThreads)
mask_select_kernel(const int8_t* __restrict__ map, int64_t T, int64_t Eu, int64_t n,
                   const uint8_t* __restrict__ probs, int pes, uint32_t* __restrict__ tile_cnt,
                   uint8_t* __restrict__ pp) {
    __shared__ uint32_t wsum[32];
    cg::grid_group grid = cg::this_grid();
    pdl_enter();  // launched in plain stream order (cooperative): returns at once
    const int64_t N = T * Eu;
    const int64_t ntiles = (N + kMsTile - 1) / kMsTile;
    if (ntiles <= (int64_t)gridDim.x) {
        // One tile per block: the map entries, their probs (loaded together
        // with the map, whether routed or not) and the in-tile positions stay
        // in registers across the grid barrier; after it only the tile's base
        // position is added and the probs are stored.
        const int64_t tile = blockIdx.x;
        const bool has = tile < ntiles;
        const int64_t f0 = tile * kMsTile + (int64_t)threadIdx.x * kMsPer;
        int64_t e = f0 / T, t = f0 - e * T;
        int8_t m[kMsPer];
        uint32_t pv[kMsPer];
#pragma unroll
        for (int q = 0; q < kMsPer; ++q) {
            const bool in = has && f0 + q < N;
            m[q] = in ? map[t * Eu + e] : (int8_t)0;
            pv[q] = in ? ld_prob_bits(probs, t * Eu + e, pes) : 0u;
            if (++t == T) {
                t = 0;
                ++e;
            }
        }
        uint32_t c = 0u;
#pragma unroll
        for (int q = 0; q < kMsPer; ++q) c += m[q] != 0 ? 1u : 0u;
        uint32_t tot = 0u;
        const uint32_t excl = block_exclusive_scan(c, wsum, &tot);
        if (has && threadIdx.x == 0) tile_cnt[tile] = tot;
        grid.sync();
        uint32_t s_lo = 0u, s_all = 0u;
        for (int64_t u = threadIdx.x; u < ntiles; u += kMsThreads) {
            const uint32_t v = __ldcg(&tile_cnt[u]);
            s_all += v;
            if (u < tile) s_lo += v;
        }
        uint32_t below = 0u, nnz = 0u;
        block_exclusive_scan(s_lo, wsum, &below);
        block_exclusive_scan(s_all, wsum, &nnz);
        uint32_t pos = below + excl;
#pragma unroll
        for (int q = 0; q < kMsPer; ++q) {
            if (m[q] != 0) {
                if ((int64_t)pos < n) st_prob_bits(pp, pos, pv[q], pes);
                ++pos;
            }
        }
        const int64_t stride = (int64_t)gridDim.x * kMsThreads;
        for (int64_t i = (int64_t)nnz + (int64_t)blockIdx.x * kMsThreads + threadIdx.x; i < n; i += stride)
            zero_prob(pp, i, pes);
        return;
    }
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t f0 = tile * kMsTile + (int64_t)threadIdx.x * kMsPer;
        int64_t e = f0 / T, t = f0 - e * T;
        int8_t m[kMsPer];
#pragma unroll
        for (int q = 0; q < kMsPer; ++q) {
            m[q] = f0 + q < N ? map[t * Eu + e] : (int8_t)0;
            if (++t == T) { t = 0; ++e; }
        }
        uint32_t c = 0u;
#pragma unroll
        for (int q = 0; q < kMsPer; ++q) c += m[q] != 0 ? 1u : 0u;
        uint32_t tot = 0u;
        block_exclusive_scan(c, wsum, &tot);
        if (threadIdx.x == 0) tile_cnt[tile] = tot;
    }
    grid.sync();
    // total routed count, and the blocks' tile prefixes
    uint32_t nnz = 0u;
    {
        uint32_t s = 0u;
        for (int64_t u = threadIdx.x; u < ntiles; u += kMsThreads) s += __ldcg(&tile_cnt[u]);
        block_exclusive_scan(s, wsum, &nnz);
    }
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        uint32_t below = 0u;
        {
            uint32_t s = 0u;
            for (int64_t u = threadIdx.x; u < tile; u += kMsThreads) s += __ldcg(&tile_cnt[u]);
            block_exclusive_scan(s, wsum, &below);
        }
        const int64_t f0 = tile * kMsTile + (int64_t)threadIdx.x * kMsPer;
        int64_t e = f0 / T, t = f0 - e * T;
        int64_t src[kMsPer];
        uint32_t c = 0u;
#pragma unroll
        for (int q = 0; q < kMsPer; ++q) {
            src[q] = -1;
            if (f0 + q < N && map[t * Eu + e] != 0) {
                src[q] = t * Eu + e;
                ++c;
            }
            if (++t == T) { t = 0; ++e; }
        }
        uint32_t tot = 0u;
        uint32_t pos = below + block_exclusive_scan(c, wsum, &tot);
#pragma unroll
        for (int q = 0; q < kMsPer; ++q) {
            if (src[q] >= 0) {
                if ((int64_t)pos < n) copy_prob(pp, pos, probs, src[q], pes);
                ++pos;
            }
        }
    }
    const int64_t stride = (int64_t)gridDim.x * kMsThreads;
    for (int64_t i = (int64_t)nnz + (int64_t)blockIdx.x * kMsThreads + threadIdx.x; i < n; i += stride)
        zero_prob(pp, i, pes);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

constexpr int kRadixDigitBits = 12;
constexpr double kShortReduceBytes = 1e9;  // see the not-padded launch below
constexpr int64_t kSortReserveSMs = 8;    // SMs a short reduce leaves to the concurrent sort

struct UnpermutePlan {
    int64_t rows, H, n, T, Eu, topk, cap;
    int tdt, pdt, pes, es;
    bool probs, padded;
    // sort
    uint32_t key_range;  // number of distinct full keys
    int fine_bits;       // beyond one pass: a coarse pass on the key's high bits
                         // (s = fine_bits), then fine_sort_kernel (0: LSD passes
                         // or one pass)
    int passes;
    int shift[3];
    int bits[3];
    int Bmax;
    // workspace
    uint64_t ms_bytes, sort_bytes, ws_bytes;
};

static int bits_for(uint64_t range) {  // bits to represent values 0..range-1
    int b = 0;
    while (b < 63 && (UINT64_C(1) << b) < range) ++b;
    return b;
}

static mr_status plan_unpermute(int64_t permutedRows, int64_t hidden, int32_t tokenDtype,
                                int64_t n, int32_t hasProbs, int32_t probsDtype, int64_t numTokens,
                                int64_t numExperts, int32_t paddedMode,
                                const int64_t* restoreShape, UnpermutePlan* p) {
    if (tokenDtype != MR_DTYPE_F16 && tokenDtype != MR_DTYPE_BF16 && tokenDtype != MR_DTYPE_F32)
        return MR_ERR_PARAM_INVALID;
    if (hasProbs && probsDtype != tokenDtype && probsDtype != MR_DTYPE_F32)
        return MR_ERR_PARAM_INVALID;
    if (paddedMode != 0 && paddedMode != 1) return MR_ERR_PARAM_INVALID;
    if (hidden <= 0 || permutedRows < 0 || n < 0) return MR_ERR_PARAM_INVALID;
    if (permutedRows >= (INT64_C(1) << 31) || n >= (INT64_C(1) << 31)) return MR_ERR_PARAM_INVALID;
    int64_t T;
    if (hasProbs) {
        if (numTokens <= 0 || numExperts <= 0) return MR_ERR_INNER;
        T = numTokens;
        if (restoreShape && (restoreShape[0] != T || restoreShape[1] != hidden))
            return MR_ERR_PARAM_INVALID;
    } else {
        if (!restoreShape) return MR_ERR_PARAM_NULLPTR;
        T = restoreShape[0];
        if (T <= 0 || restoreShape[1] != hidden) return MR_ERR_PARAM_INVALID;
    }
    if (T >= (INT64_C(1) << 31) - 1) return MR_ERR_PARAM_INVALID;
    const int64_t topk = permutedRows / T;
    if (topk > MR_MAX_TOPK_NUM) return MR_ERR_INNER;
    int64_t cap = 0;
    if (!paddedMode) {
        if (n != T * topk) return MR_ERR_PARAM_INVALID;
    } else {
        if (n != permutedRows) return MR_ERR_PARAM_INVALID;
        if (hasProbs) {
            if (numExperts > n || n % numExperts != 0) return MR_ERR_INNER;
            cap = n / numExperts;
        }
    }
    if (hasProbs && numExperts > MR_MAX_EXPERT_NUM) return MR_ERR_INNER;
    if (hasProbs && T * numExperts >= (INT64_C(1) << 40)) return MR_ERR_INNER;
    if (paddedMode && hasProbs && getenv("MR_VERBOSE")) {
        if (topk > numExperts)
            fprintf(stderr, "moe_unpermute warning: paddedMode with topK_num %lld > experts %lld\n",
                    (long long)topk, (long long)numExperts);
        if (cap > T)
            fprintf(stderr, "moe_unpermute warning: paddedMode with capacity %lld > tokens %lld\n",
                    (long long)cap, (long long)T);
    }
    p->rows = permutedRows;
    p->H = hidden;
    p->n = n;
    p->T = T;
    p->Eu = hasProbs ? numExperts : 0;
    p->topk = topk;
    p->cap = cap;
    p->tdt = tokenDtype;
    p->pdt = hasProbs ? probsDtype : tokenDtype;
    p->pes = p->pdt == MR_DTYPE_F32 ? 4 : 2;
    p->es = tokenDtype == MR_DTYPE_F32 ? 4 : 2;
    p->probs = hasProbs != 0;
    p->padded = paddedMode != 0;

    // sort passes: one pass of the counting sort over every key up to
    // 2^kRadixDigitBits keys, else LSD passes of at most that many bits (a
    // dense histogram of many more keys than a tile's 2048 items costs more
    // than a second pass)
    const uint64_t range = paddedMode ? (uint64_t)T + 1 : (uint64_t)permutedRows + 1;
    p->key_range = (uint32_t)range;
    p->fine_bits = 0;
    if (range > (UINT64_C(1) << kRadixDigitBits) &&
        range <= (UINT64_C(1) << (kRadixDigitBits + kMaxFineBits))) {
        // two levels: a coarse counting sort on the key's high bits (about 2^8
        // buckets padded, 2^9 not padded -- the faster choices measured on
        // GB300 -- and at most 4097), then one block per coarse bucket sorts
        // by the low s bits, s <= kMaxFineBits so that the fine keys fit a
        // block. The span = range - 1 valid keys take ((span - 1) >> s) + 1
        // buckets and the invalid key one more (padded: the last, after the
        // digits key >> s; not padded: bucket 0, before the digits
        // 1 + (key - 1) >> s).
        const uint64_t span = range - 1;
        const int b = bits_for(span);
        const int coarse_bits = paddedMode ? 8 : 9;
        const int sbits = b - coarse_bits < kMaxFineBits ? b - coarse_bits : kMaxFineBits;
        p->fine_bits = sbits;
        p->passes = 1;
        p->shift[0] = sbits;
        p->bits[0] = kRadixDigitBits;
        p->Bmax = (int)(((span - 1) >> sbits) + 2);
    } else if (range <= (UINT64_C(1) << kRadixDigitBits)) {
        p->passes = 1;
        p->shift[0] = 0;
        p->bits[0] = bits_for(range);
        p->Bmax = (int)range;
    } else {
        const int b = bits_for(range);
        const int P = (b + kRadixDigitBits - 1) / kRadixDigitBits;
        p->passes = P;
        int sh = 0;
        for (int q = 0; q < P; ++q) {
            const int d = b / P + (q < b % P ? 1 : 0);
            p->shift[q] = sh;
            p->bits[q] = d;
            sh += d;
        }
        p->Bmax = 1 << p->bits[0];
    }

    // workspace
    uint64_t ms = 0;
    if (hasProbs && !paddedMode) {
        const int64_t nblk = (T + 31) / 32;
        const uint64_t items = (uint64_t)nblk * numExperts;
        ms = align_up(items * 4u, 256) * 2 + align_up((uint64_t)numExperts * 4u, 256) +
             align_up((uint64_t)(numExperts + 1) * 4u, 256) + 256;
    }
    const int Bsort = p->fine_bits ? p->Bmax : p->passes == 1 ? (int)range : p->Bmax;
    uint64_t sb = csort_workspace_bytes(n, Bsort) + 4 * align_up((uint64_t)n * 4u, 256);
    if (paddedMode) sb += align_up((uint64_t)(T + 1) * 4u, 256);
    p->ms_bytes = ms;
    p->sort_bytes = sb;
    p->ws_bytes = ms + sb;
    return MR_OK;
}

static int elementwise_grid(int64_t n) {
    const int64_t want = (n + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

// Whether the gather-reduce takes the 16-byte vector path (row bytes and
// buffers 16-byte aligned); the element-wise kernel serves the rest.
static bool reduce_vec_ok(const UnpermutePlan& p, const void* permuted, const void* out) {
    return (p.H * p.es) % 16 == 0 && reinterpret_cast<uintptr_t>(permuted) % 16 == 0 &&
           reinterpret_cast<uintptr_t>(out) % 16 == 0;
}

// Not padded with probs: whether the gather-reduce derives the weights from a
// small routing map itself (SmallMap), instead of the maskedSelect kernels.
static bool use_small_map(const UnpermutePlan& p, const void* permuted, const void* out) {
    return p.probs && !p.padded && p.T * p.Eu <= kSmallMapEntries &&
           small_map_smem_words(p.T, p.Eu) * 4 <= 32 * 1024 && reduce_vec_ok(p, permuted, out);
}

template <int TDT, int PDT, bool HAS_PROBS, bool PADDED, bool SMALL>
static cudaError_t launch_reduce_vec(const UnpermutePlan& p, const uint8_t* permuted,
                                     const int32_t* si, const void* pp, const int32_t* out_index,
                                     const int32_t* ptr, uint8_t* out, const SmallMap& smap,
                                     cudaStream_t s, bool short_grid) {
    const int64_t row_bytes = p.H * p.es;
    const int64_t nvec = row_bytes / 16;
    const int64_t chunks = (nvec + 32 * kRedVQ - 1) / (32 * kRedVQ);
    const int64_t warps = p.T * chunks;
    const size_t smem = SMALL ? (size_t)small_map_smem_words(p.T, p.Eu) * 4u : 0u;
    static int blocks_per_sm[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int bps = dev < 64 ? blocks_per_sm[dev] : 0;
    if (bps == 0) {
        // registers set the occupancy (the small-map shared memory is at most 32 KB)
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &bps, unpermute_reduce_warp_kernel<TDT, PDT, HAS_PROBS, PADDED, kRedRun, SMALL>, 256, 0) !=
                cudaSuccess || bps <= 0)
            bps = 4;
        if (dev < 64) blocks_per_sm[dev] = bps;
    }
    int64_t grid = (warps + 7) / 8;
    const int64_t cap = (int64_t)device_sm_count() * bps;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    // runs of kRedRun chunks share one slot-list read; when they would
    // leave resident warps idle (a few tokens), one chunk per unit
    // (measured on GB300: decode-sized call 22.8 -> 20.8 us; longer
    // runs keep the padded reduce at 98 us instead of 106 us)
    const int64_t long_units = p.T * ((chunks + kRedRun - 1) / kRedRun);
    auto kern = long_units < cap * 8 ? unpermute_reduce_warp_kernel<TDT, PDT, HAS_PROBS, PADDED, 1, SMALL>
                                     : unpermute_reduce_warp_kernel<TDT, PDT, HAS_PROBS, PADDED, kRedRun, SMALL>;
    if (short_grid) {
        // A short reduce has the index sort running beside it on the
        // (higher-priority) auxiliary stream. Its grid is one work unit per
        // warp (blocks retire as they finish and the sort's blocks take the
        // freed slots), capped at a persistent grid on all SMs but
        // kSortReserveSMs, so that the sort also has SMs of its own
        // (measured on GB300, top-k T=4096, k=8, H=4096: a persistent grid on
        // every SM 55.6 us, one unit per warp 53.5 us, with the cap 51.5 us;
        // a decode step's few units stay below the cap)
        const int64_t run = long_units < cap * 8 ? 1 : kRedRun;
        const int64_t units = p.T * ((chunks + run - 1) / run);
        grid = (units + 7) / 8;
        const int64_t sms = device_sm_count();
        const int64_t pgrid = (sms > 2 * kSortReserveSMs ? sms - kSortReserveSMs : sms) * bps;
        if (grid > pgrid) grid = pgrid;
        if (grid > 0x7fffffff) grid = 0x7fffffff;
        if (grid < 1) grid = 1;
    }
    return launch_pdl(kern, dim3((unsigned)grid), dim3(256), smem, s, permuted, p.rows, row_bytes, nvec, chunks,
                      si, p.topk, pp, out_index, ptr, p.T, out, smap);
}

template <int TDT, int PDT, bool HAS_PROBS, bool PADDED>
static cudaError_t launch_reduce(const UnpermutePlan& p, const uint8_t* permuted,
                                 const int32_t* si, const void* pp, const int32_t* out_index,
                                 const int32_t* ptr, uint8_t* out, const SmallMap& smap,
                                 cudaStream_t s, bool short_grid) {
    if (reduce_vec_ok(p, permuted, out)) {
        if constexpr (HAS_PROBS && !PADDED) {
            if (smap.map)
                return launch_reduce_vec<TDT, PDT, HAS_PROBS, PADDED, true>(p, permuted, si, pp, out_index,
                                                                           ptr, out, smap, s, short_grid);
        }
        return launch_reduce_vec<TDT, PDT, HAS_PROBS, PADDED, false>(p, permuted, si, pp, out_index, ptr,
                                                                    out, smap, s, short_grid);
    }
    int64_t threads = p.H < 256 ? (p.H + 31) / 32 * 32 : 256;
    const int64_t gx = p.T < 0x7fffffff ? p.T : 0x7fffffff;
    return launch_pdl(unpermute_reduce_scalar_kernel<TDT, PDT, HAS_PROBS, PADDED>, dim3((unsigned)gx),
                      dim3((unsigned)threads), 0, s, permuted, p.rows, p.H, si, p.topk, pp, out_index, ptr, p.T,
                      out);
}

template <int TDT, int PDT>
static cudaError_t dispatch_reduce(const UnpermutePlan& p, const uint8_t* permuted,
                                   const int32_t* si, const void* pp, const int32_t* out_index,
                                   const int32_t* ptr, uint8_t* out, const SmallMap& smap,
                                   cudaStream_t s, bool short_grid) {
    if (p.probs) {
        return p.padded ? launch_reduce<TDT, PDT, true, true>(p, permuted, si, pp, out_index, ptr, out, smap, s, short_grid)
                        : launch_reduce<TDT, PDT, true, false>(p, permuted, si, pp, out_index, ptr, out, smap, s, short_grid);
    }
    return p.padded ? launch_reduce<TDT, PDT, false, true>(p, permuted, si, pp, out_index, ptr, out, smap, s, short_grid)
                    : launch_reduce<TDT, PDT, false, false>(p, permuted, si, pp, out_index, ptr, out, smap, s, short_grid);
}

// The one-kernel maskedSelect: a cooperative launch (every block resident for
// its grid barrier) of at most the resident blocks, and no more than the tiles.
static cudaError_t launch_mask_select(const UnpermutePlan& p, const int8_t* map, const uint8_t* probs,
                                      uint32_t* tile_cnt, uint8_t* pp, cudaStream_t s) {
    static int blocks_per_sm[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int bps = dev < 64 ? blocks_per_sm[dev] : 0;
    if (bps == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, mask_select_kernel, kMsThreads, 0) !=
                cudaSuccess || bps <= 0)
            return cudaErrorInvalidConfiguration;
        if (dev < 64) blocks_per_sm[dev] = bps;
    }
    const int64_t tiles = (p.T * p.Eu + kMsTile - 1) / kMsTile;
    int64_t grid = (int64_t)device_sm_count() * bps;
    if (grid > tiles) grid = tiles;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kMsThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mask_select_kernel, map, p.T, p.Eu, p.n, probs, p.pes, tile_cnt, pp);
}

MR_CHECK_ACCESSOR(unpermute)

}  // namespace mr

using namespace mr;

extern "C" mr_status moe_unpermute_get_workspace_size(int64_t permutedRows, int64_t hidden,
                                                       int32_t tokenDtype, int64_t numSortedIndices,
                                                       int32_t hasProbs, int32_t probsDtype,
                                                       int64_t numTokens, int64_t numExperts,
                                                       int32_t paddedMode,
                                                       const int64_t* restoreShape,
                                                       uint64_t* workspaceSize) {
    if (!workspaceSize) return MR_ERR_PARAM_NULLPTR;
    UnpermutePlan p;
    const mr_status st = plan_unpermute(permutedRows, hidden, tokenDtype, numSortedIndices,
                                        hasProbs, probsDtype, numTokens, numExperts, paddedMode,
                                        restoreShape, &p);
    if (st != MR_OK) return st;
    *workspaceSize = p.ws_bytes;
    return MR_OK;
}

extern "C" mr_status moe_unpermute(const void* permutedTokens, const int32_t* sortedIndices,
                                   const int8_t* routingMap, const void* probs,
                                   int64_t permutedRows, int64_t hidden, int32_t tokenDtype,
                                   int64_t numSortedIndices, int32_t probsDtype, int64_t numTokens,
                                   int64_t numExperts, int32_t paddedMode,
                                   const int64_t* restoreShape, void* unpermutedTokens,
                                   int32_t* outIndex, int32_t* permuteTokenId, void* permuteProbs,
                                   void* workspace, uint64_t workspaceSize, void* stream) {
    if ((probs == nullptr) != (routingMap == nullptr)) return MR_ERR_PARAM_INVALID;
    const int32_t hasProbs = probs != nullptr ? 1 : 0;
    UnpermutePlan p;
    mr_status st = plan_unpermute(permutedRows, hidden, tokenDtype, numSortedIndices, hasProbs,
                                  probsDtype, numTokens, numExperts, paddedMode, restoreShape, &p);
    if (st != MR_OK) return st;
    if (!permutedTokens || !sortedIndices || !unpermutedTokens || !outIndex || !permuteTokenId)
        return MR_ERR_PARAM_NULLPTR;
    if (hasProbs && !permuteProbs) return MR_ERR_PARAM_NULLPTR;
    if (!workspace && p.ws_bytes > 0) return MR_ERR_PARAM_NULLPTR;
    if (workspaceSize < p.ws_bytes) return MR_ERR_WORKSPACE;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* wp = reinterpret_cast<uint8_t*>(workspace);
    uint8_t* pp = reinterpret_cast<uint8_t*>(permuteProbs);

    // A small routing map (not padded, with probs): the gather-reduce selects
    // the weights from it itself and writes permuteProbs (SmallMap).
    SmallMap smap{nullptr, nullptr, nullptr, 0};
    if (use_small_map(p, permutedTokens, unpermutedTokens))
        smap = SmallMap{routingMap, reinterpret_cast<const uint8_t*>(probs), pp, p.Eu};

    // ---- stable sort of sortedIndices -> outIndex, permuteTokenId ----------
    uint8_t* q = wp + p.ms_bytes;
    const int Bsort = p.fine_bits ? p.Bmax : p.passes == 1 ? (int)p.key_range : p.Bmax;
    CsortBufs cs = csort_carve(q, p.n, Bsort);
    uint32_t* keys[2];
    int32_t* idx[2];
    keys[0] = reinterpret_cast<uint32_t*>(q);
    q += align_up((uint64_t)p.n * 4u, 256);
    keys[1] = reinterpret_cast<uint32_t*>(q);
    q += align_up((uint64_t)p.n * 4u, 256);
    idx[0] = reinterpret_cast<int32_t*>(q);
    q += align_up((uint64_t)p.n * 4u, 256);
    idx[1] = reinterpret_cast<int32_t*>(q);
    q += align_up((uint64_t)p.n * 4u, 256);
    // padded: per-token row ranges. One pass: the key starts are exactly that
    // (key = token, invalid rows in the last bucket); several passes: built
    // from the sorted keys.
    int32_t* ptr = !p.padded ? nullptr
                   : (p.passes == 1 && !p.fine_bits) ? reinterpret_cast<int32_t*>(cs.bucket_start)
                                                     : reinterpret_cast<int32_t*>(q);

    auto launch_sort = [&](cudaStream_t ss) -> cudaError_t {
        const int64_t limit = p.padded ? p.T : p.rows;
        const uint32_t* kin = nullptr;
        const int32_t* iin = nullptr;
        for (int pass = 0; pass < p.passes; ++pass) {
            const int B = p.fine_bits ? p.Bmax : p.passes == 1 ? (int)p.key_range : (1 << p.bits[pass]);
            const uint32_t mask = (p.passes == 1 || p.fine_bits)
                                      ? 0xffffffffu : (uint32_t)((1u << p.bits[pass]) - 1u);
            RadixKey kf{sortedIndices, kin, limit, p.padded ? 1 : 0, p.shift[pass], mask,
                        p.fine_bits ? 1 : 0, (uint32_t)(p.Bmax - 1)};
            GroupListOut none{nullptr, nullptr, 0};
            const bool last = pass == p.passes - 1 && !p.fine_bits;
            PaddedProbs ppr{reinterpret_cast<const uint8_t*>(probs), nullptr, p.Eu, p.cap, p.pes};
            if (pass == 0 && p.padded && p.probs) ppr.pp = pp;
            const bool apart = p.fine_bits != 0;
            RadixScatter sc{kf, iin, keys[pass & 1], last ? nullptr : idx[pass & 1],
                            last ? outIndex : nullptr, last ? permuteTokenId : nullptr,
                            p.topk > 0 ? p.topk : (int64_t)1, ppr,
                            apart ? outIndex : nullptr, apart ? permuteTokenId : nullptr, p.n};
            cudaError_t e;
            if (p.n <= kSortTile) {
                e = csort_single_tile(kf, p.n, B, cs, none, sc, ss);  // one block
            } else {
                e = csort_run(kf, p.n, B, cs, none, ss);
                if (e != cudaSuccess) return e;
                e = launch_pdl(radix_scatter_kernel, dim3(elementwise_grid(p.n)), dim3(256), 0, ss, kf,
                               p.n, B, cs, sc);
            }
            if (e != cudaSuccess) return e;
            kin = keys[pass & 1];
            iin = idx[pass & 1];
        }
        if (p.fine_bits) {
            const size_t smem = (size_t)(2 + kFineWarps) * ((size_t)1 << p.fine_bits) * 4u;
            auto kern = p.padded ? fine_sort_kernel<true> : fine_sort_kernel<false>;
            if (smem > 48 * 1024) {
                cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
                if (e != cudaSuccess) return e;
            }
            // the invalid entries' bucket is already in place
            const int blocks = p.Bmax - 1;
            return launch_pdl(kern, dim3((unsigned)blocks), dim3(kFineThreads), smem, ss,
                              (const uint32_t*)kin, (const int32_t*)iin, (const uint32_t*)cs.bucket_start,
                              p.fine_bits, p.T, p.topk > 0 ? p.topk : (int64_t)1, sortedIndices, outIndex,
                              permuteTokenId, ptr, p.n);
        }
        if (p.padded && p.passes > 1) {
            return launch_pdl(csr_from_keys_kernel, dim3(elementwise_grid(p.n + 1)), dim3(256), 0,
                              ss, kin, p.n, p.T, ptr);
        }
        return cudaSuccess;
    };

    // ---- permuteProbs (maskedSelect or the padded lookup) --------------------
    auto launch_probs = [&](cudaStream_t ss) -> cudaError_t {
        // padded with probs: the lookup runs in the sort's first scatter; a
        // small map: inside the gather-reduce
        if (!p.probs || p.padded || smap.map) return cudaSuccess;
        if ((p.T * p.Eu + kMsTile - 1) / kMsTile <= kMsMaxTiles)
            return launch_mask_select(p, routingMap, reinterpret_cast<const uint8_t*>(probs),
                                      reinterpret_cast<uint32_t*>(wp), pp, ss);
        // beyond: column bitmasks, the prefix kernel, the scatter
        const int64_t nblk = (p.T + 31) / 32;
        const int64_t items = nblk * p.Eu;
        uint8_t* q = wp;
        uint32_t* masks = reinterpret_cast<uint32_t*>(q);
        q += align_up((uint64_t)items * 4u, 256);
        uint32_t* offs = reinterpret_cast<uint32_t*>(q);
        q += align_up((uint64_t)items * 4u, 256);
        uint32_t* totals = reinterpret_cast<uint32_t*>(q);
        q += align_up((uint64_t)p.Eu * 4u, 256);
        uint32_t* bstart = reinterpret_cast<uint32_t*>(q);
        q += align_up((uint64_t)(p.Eu + 1) * 4u, 256);
        uint32_t* ticket = reinterpret_cast<uint32_t*>(q);
        cudaError_t e = launch_mask_columns(routingMap, p.T, p.Eu, masks, offs, ticket, ss);
        if (e != cudaSuccess) return e;
        GroupListOut none{nullptr, nullptr, 0};
        e = csort_prefix(offs, nblk, (int)p.Eu, totals, bstart, ticket, none, ss);
        if (e != cudaSuccess) return e;
        const int64_t work = items > p.n ? items : p.n;
        return launch_pdl(mask_scatter_kernel, dim3(elementwise_grid(work)), dim3(256), 0, ss,
                          (const uint32_t*)masks, (const uint32_t*)offs, (const uint32_t*)bstart, p.T, p.Eu,
                          p.n, reinterpret_cast<const uint8_t*>(probs), p.pes, pp);
    };

    // ---- gather-reduce --------------------------------------------------------
    const uint8_t* permuted = reinterpret_cast<const uint8_t*>(permutedTokens);
    uint8_t* out = reinterpret_cast<uint8_t*>(unpermutedTokens);
    auto launch_reduce_any = [&](cudaStream_t ss, bool short_grid) -> cudaError_t {
        switch (p.tdt * 4 + p.pdt) {
            case MR_DTYPE_F16 * 4 + MR_DTYPE_F16:
                return dispatch_reduce<MR_DTYPE_F16, MR_DTYPE_F16>(p, permuted, sortedIndices, pp, outIndex, ptr, out, smap, ss, short_grid);
            case MR_DTYPE_F16 * 4 + MR_DTYPE_F32:
                return dispatch_reduce<MR_DTYPE_F16, MR_DTYPE_F32>(p, permuted, sortedIndices, pp, outIndex, ptr, out, smap, ss, short_grid);
            case MR_DTYPE_BF16 * 4 + MR_DTYPE_BF16:
                return dispatch_reduce<MR_DTYPE_BF16, MR_DTYPE_BF16>(p, permuted, sortedIndices, pp, outIndex, ptr, out, smap, ss, short_grid);
            case MR_DTYPE_BF16 * 4 + MR_DTYPE_F32:
                return dispatch_reduce<MR_DTYPE_BF16, MR_DTYPE_F32>(p, permuted, sortedIndices, pp, outIndex, ptr, out, smap, ss, short_grid);
            case MR_DTYPE_F32 * 4 + MR_DTYPE_F32:
                return dispatch_reduce<MR_DTYPE_F32, MR_DTYPE_F32>(p, permuted, sortedIndices, pp, outIndex, ptr, out, smap, ss, short_grid);
        }
        return cudaErrorInvalidValue;
    };

    cudaError_t e = cudaSuccess;
    cudaError_t ea = cudaSuccess;
    AuxStream* ax = p.padded ? nullptr : aux_stream(s, &ea);
    if (ea != cudaSuccess) return MR_ERR_CUDA;
    if (ax) {
        // Not padded, the sort's outputs are not read by the gather-reduce: it
        // runs on the auxiliary stream of the caller's stream, forked from and
        // joined back into it, so it overlaps the reduce.
        std::lock_guard<std::mutex> lock(ax->mu);
        MR_TRY_CUDA(cudaEventRecord(ax->fork, s));
        MR_TRY_CUDA(cudaStreamWaitEvent(ax->stream, ax->fork, 0));
        profile_mark(ax->stream, 8);
        e = launch_sort(ax->stream);
        profile_mark(ax->stream, 9);
        const cudaError_t ej = cudaEventRecord(ax->join, ax->stream);
        if (e == cudaSuccess) {
            profile_mark(s, 4);
            e = launch_probs(s);
            profile_mark(s, 5);
        }
        if (e == cudaSuccess) {
            profile_mark(s, 6);
            // A persistent reduce, launched early under PDL, takes the SMs
            // while it waits for the probs, and the concurrent sort then runs
            // on what is left; a short reduce would end up waiting for the
            // sort at the join. So a short one (up to 1 GB of rows, ~150 us)
            // gets a grid of one work unit per warp, whose blocks retire as
            // they finish (see launch_reduce_vec); a long one hides the sort
            // either way and keeps the persistent grid (measured on GB300:
            // top-k T=4096, k=8, H=4096: persistent grid 75.7 us; one unit per
            // warp launched in plain order 49.4 us, under PDL 47.4 us)
            const double reduce_bytes = (double)p.T * (double)p.topk * (double)p.H * p.es;
            e = launch_reduce_any(s, reduce_bytes <= kShortReduceBytes);
            profile_mark(s, 7);
        }
        const cudaError_t ew = ej == cudaSuccess ? cudaStreamWaitEvent(s, ax->join, 0) : ej;
        MR_TRY_CUDA(e);
        MR_TRY_CUDA(ew);
    } else {
        profile_mark(s, 4);
        MR_TRY_CUDA(launch_probs(s));
        MR_TRY_CUDA(launch_sort(s));
        profile_mark(s, 5);
        profile_mark(s, 6);
        e = launch_reduce_any(s, false);
        MR_TRY_CUDA(e);
        profile_mark(s, 7);
    }
    MR_TRY_CUDA(cudaGetLastError());
    return MR_OK;
}
