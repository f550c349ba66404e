// Stable counting sort engine: the shared index machinery of both operations.
//
// Items i in [0, N) carry a key in [0, B) (B <= kMaxBuckets); a key < 0 means
// "not counted" (only used for the padding lanes past N). The engine computes,
// for every item, its position in the stable ascending order of the keys:
//
//   dest(i) = bucket_start[key] + tile_off[tile(i)][key] + tile_rank[i]
//
//   rank   kernel: per tile of kSortTile items, the stable rank of each item
//                  among the items of the tile with the same key, and the
//                  tile's histogram (tile-major matrix [tiles][B]).
//   prefix kernel: per bucket (one warp each), the exclusive prefix of the
//                  histogram over the tiles (in place), the bucket totals,
//                  and -- in the block that finishes last -- the exclusive
//                  scan of the totals
//                  (bucket_start) plus an optional compacted
//                  [key, count] list of the non-empty buckets below a limit.
//   consumers:     elementwise kernels of each operation call csort_dest().
//   single tile:   an input of at most one tile sorts in one block
//                  (csort_single_tile_kernel), scatter included.
//
// The stable in-tile rank: each of the kSortWarps warps owns kSortChunks
// consecutive 32-item chunks of the tile and walks them in order. Within a
// chunk, __match_any_sync groups the lanes with equal keys; the lowest lane of
// each group advances the warp's private counter of that key in shared memory
// by the group size, and each lane's rank is the counter before the update
// plus the number of lower lanes in its group. The cross-warp part is the sum
// of the lower warps' counters for the key. Ties therefore keep item order,
// which is what makes the sort stable. No atomics touch global memory and no
// kernel waits on another block: the only inter-block step is the last-block
// ticket of the prefix kernel.
#pragma once

#include "common.cuh"

namespace mr {

constexpr int kSortWarps = 8;
constexpr int kSortThreads = kSortWarps * 32;
constexpr int kSortChunks = 8;  // 32-item chunks per warp
constexpr int kSortTile = kSortWarps * 32 * kSortChunks;  // 2048 items per tile
constexpr int kMaxBuckets = 8194;  // expertNum <= 8192, the sentinel and a no-slot key
constexpr int kPrefixWarps = 8;                            // keys per prefix block (one per warp)
constexpr int kPrefixThreads = kPrefixWarps * 32;
constexpr int kPrefixPrefetch = 4;                         // 32-tile steps loaded together
constexpr int kLastChunk = 8;                              // key totals per load batch (last block)

// At least one tile, so an empty input still produces zero totals.
inline int64_t csort_tiles(int64_t N) { return N > 0 ? (N + kSortTile - 1) / kSortTile : 1; }
inline size_t csort_rank_smem(int B) { return align_up((uint64_t)kSortWarps * B * 2u, 16); }

// Workspace of one sort pass.
struct CsortBufs {
    uint32_t* tile_off;      // [tiles][B]: counts, then exclusive prefixes over tiles
    uint32_t* totals;        // [B]
    uint32_t* bucket_start;  // [B + 1]
    uint16_t* tile_rank;     // [N]
    uint32_t* ticket;        // [1]
    uint32_t* coop_counts;   // key-major counts of the one-launch form (csort_coop.cuh), or null
};

inline uint64_t csort_workspace_bytes(int64_t N, int B) {
    const uint64_t tiles = (uint64_t)csort_tiles(N);
    return align_up(tiles * B * 4u, 256) + align_up((uint64_t)B * 4u, 256) +
           align_up((uint64_t)(B + 1) * 4u, 256) + align_up((uint64_t)N * 2u, 256) + 256;
}

inline CsortBufs csort_carve(uint8_t*& p, int64_t N, int B) {
    CsortBufs b;
    const uint64_t tiles = (uint64_t)csort_tiles(N);
    b.tile_off = reinterpret_cast<uint32_t*>(p);
    p += align_up(tiles * B * 4u, 256);
    b.totals = reinterpret_cast<uint32_t*>(p);
    p += align_up((uint64_t)B * 4u, 256);
    b.bucket_start = reinterpret_cast<uint32_t*>(p);
    p += align_up((uint64_t)(B + 1) * 4u, 256);
    b.tile_rank = reinterpret_cast<uint16_t*>(p);
    p += align_up((uint64_t)N * 2u, 256);
    b.ticket = reinterpret_cast<uint32_t*>(p);
    p += 256;
    b.coop_counts = nullptr;
    return b;
}

template <class KeyFn>
__global__ void __launch_bounds__(kSortThreads)
csort_rank_kernel(KeyFn kf, int64_t N, int B, uint16_t* __restrict__ tile_rank,
                  uint32_t* __restrict__ tile_counts, uint32_t* __restrict__ ticket) {
    extern __shared__ __align__(16) uint16_t tab[];  // [kSortWarps][B] per-warp key counters
    pdl_enter();
    if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0u;

    const int tab_words = (kSortWarps * B + 1) / 2;
    uint32_t* tab32 = reinterpret_cast<uint32_t*>(tab);
    for (int i = threadIdx.x; i < tab_words; i += kSortThreads) tab32[i] = 0u;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t base = (int64_t)blockIdx.x * kSortTile + (int64_t)warp * (32 * kSortChunks);
    int key[kSortChunks];
#pragma unroll
    for (int c = 0; c < kSortChunks; ++c) {
        const int64_t i = base + c * 32 + lane;
        key[c] = i < N ? kf(i) : -1;
        if (key[c] >= 0 && !MR_IN_RANGE(key[c], B, 201)) key[c] = -1;
    }
    __syncthreads();

    uint16_t* mytab = tab + warp * B;
    uint32_t local[kSortChunks];
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int c = 0; c < kSortChunks; ++c) {
        const int k = key[c];
        const uint32_t peers = __match_any_sync(0xffffffffu, k);
        const uint32_t below = __popc(peers & lt);
        uint32_t before = 0u;
        if (k >= 0) before = mytab[k];
        __syncwarp();
        if (k >= 0 && below == 0u) mytab[k] = (uint16_t)(before + __popc(peers));
        __syncwarp();
        local[c] = before + below;
    }
    __syncthreads();

#pragma unroll
    for (int c = 0; c < kSortChunks; ++c) {
        const int k = key[c];
        if (k >= 0) {
            uint32_t r = local[c];
            for (int w = 0; w < warp; ++w) r += tab[w * B + k];
            tile_rank[base + c * 32 + lane] = (uint16_t)r;
        }
    }
    uint32_t* out = tile_counts + (int64_t)blockIdx.x * B;
    for (int b = threadIdx.x; b < B; b += kSortThreads) {
        uint32_t s = 0u;
#pragma unroll
        for (int w = 0; w < kSortWarps; ++w) s += tab[w * B + b];
        out[b] = s;
    }
}

// Optional epilogue of the prefix kernel: a compacted list of the non-empty
// buckets b < limit as int64 rows [b, count], rows past the last one [0, 0],
// and the number of items in those buckets.
struct GroupListOut {
    int64_t* rows;       // [limit][2] or nullptr
    int64_t* count_out;  // [1] or nullptr
    int limit;
};

static __global__ void __launch_bounds__(kPrefixThreads)
csort_prefix_kernel(uint32_t* __restrict__ tile_off, int64_t tiles, int B,
                    uint32_t* __restrict__ totals, uint32_t* __restrict__ bucket_start,
                    uint32_t* __restrict__ ticket, GroupListOut gl) {
    __shared__ uint32_t warp_sums[32];
    __shared__ int is_last;
    pdl_enter();

    // One warp per key: an exclusive scan of the key's tile counts, 32 tiles
    // per step (lane = tile), kPrefixPrefetch steps of loads issued together.
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kPrefixWarps + (threadIdx.x >> 5);
    if (b < B) {
        uint32_t carry = 0u;
        for (int64_t t0 = 0; t0 < tiles; t0 += 32 * kPrefixPrefetch) {
            uint32_t v[kPrefixPrefetch];
#pragma unroll
            for (int u = 0; u < kPrefixPrefetch; ++u) {
                const int64_t t = t0 + 32 * u + lane;
                v[u] = t < tiles ? tile_off[t * B + b] : 0u;
            }
#pragma unroll
            for (int u = 0; u < kPrefixPrefetch; ++u) {
                uint32_t incl = v[u];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const int64_t t = t0 + 32 * u + lane;
                if (t < tiles) tile_off[t * B + b] = carry + incl - v[u];
                carry += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        if (lane == 0) totals[b] = carry;
    }

    // The block that finishes last scans the key totals.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(ticket, 1u) == gridDim.x - 1 ? 1 : 0;
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    // Each thread owns a run of per_t consecutive keys, read kLastChunk at a
    // time with the loads of a chunk issued together.
    const int per_t = (B + kPrefixThreads - 1) / kPrefixThreads;
    const int c0 = threadIdx.x * per_t;
    const int c1 = c0 + per_t < B ? c0 + per_t : B;
    uint32_t s = 0u, ng = 0u;
    for (int i0 = c0; i0 < c1; i0 += kLastChunk) {
        uint32_t v[kLastChunk];
#pragma unroll
        for (int q = 0; q < kLastChunk; ++q) v[q] = i0 + q < c1 ? __ldcg(&totals[i0 + q]) : 0u;
#pragma unroll
        for (int q = 0; q < kLastChunk; ++q) {
            s += v[q];
            if (i0 + q < c1 && i0 + q < gl.limit && v[q] != 0u) ++ng;
        }
    }
    uint32_t total_all = 0u, groups = 0u;
    const uint32_t excl = block_exclusive_scan(s, warp_sums, &total_all);
    const uint32_t gexcl = block_exclusive_scan(ng, warp_sums, &groups);
    uint32_t run = excl, r = gexcl;
    for (int i0 = c0; i0 < c1; i0 += kLastChunk) {
        uint32_t v[kLastChunk];
#pragma unroll
        for (int q = 0; q < kLastChunk; ++q) v[q] = i0 + q < c1 ? __ldcg(&totals[i0 + q]) : 0u;
#pragma unroll
        for (int q = 0; q < kLastChunk; ++q) {
            const int i = i0 + q;
            if (i < c1) {
                bucket_start[i] = run;
                if (gl.rows && i < gl.limit && v[q] != 0u && MR_IN_RANGE(r, gl.limit, 202)) {
                    gl.rows[2 * (int64_t)r] = i;
                    gl.rows[2 * (int64_t)r + 1] = v[q];
                    ++r;
                }
                run += v[q];
            }
        }
    }
    if (threadIdx.x == 0) {
        bucket_start[B] = total_all;
        *ticket = 0u;
    }
    if (gl.rows) {
        for (int64_t q = (int64_t)groups + threadIdx.x; q < gl.limit; q += kPrefixThreads) {
            gl.rows[2 * q] = 0;
            gl.rows[2 * q + 1] = 0;
        }
    }
    __syncthreads();
    if (gl.count_out && threadIdx.x == 0) *gl.count_out = (int64_t)bucket_start[gl.limit];
}

// Launch of the prefix kernel over a [tiles][B] count matrix.
inline cudaError_t csort_prefix(uint32_t* tile_off, int64_t tiles, int B, uint32_t* totals,
                                uint32_t* bucket_start, uint32_t* ticket, GroupListOut gl,
                                cudaStream_t st) {
    const int blocks = (B + kPrefixWarps - 1) / kPrefixWarps;
    return launch_pdl(csort_prefix_kernel, dim3(blocks), dim3(kPrefixThreads), 0, st, tile_off,
                      tiles, B, totals, bucket_start, ticket, gl);
}

// Position of item i (key k) in the stable order.
__device__ __forceinline__ uint32_t csort_dest(int k, int64_t i, const CsortBufs& b, int B) {
    const int64_t t = i / kSortTile;
    return b.bucket_start[k] + b.tile_off[t * B + k] + (uint32_t)b.tile_rank[i];
}

// Host: rank + prefix for one pass. The caller launches its consumer next.
template <class KeyFn>
inline cudaError_t csort_run(KeyFn kf, int64_t N, int B, const CsortBufs& b, GroupListOut gl,
                             cudaStream_t st) {
    const int64_t tiles = csort_tiles(N);
    const size_t smem = csort_rank_smem(B);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(csort_rank_kernel<KeyFn>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_pdl(csort_rank_kernel<KeyFn>, dim3((unsigned)tiles),
                               dim3(kSortThreads), smem, st, kf, N, B, b.tile_rank, b.tile_off,
                               b.ticket);
    if (e != cudaSuccess) return e;
    return csort_prefix(b.tile_off, tiles, B, b.totals, b.bucket_start, b.ticket, gl, st);
}

// The whole sort of an input of one tile (at most kSortTile items) in one
// block: the stable in-tile ranks as in csort_rank_kernel, the tile's
// histogram scanned into key starts in shared memory (the key starts and the
// optional compacted group list written out), then the consumer's scatter
// step for every item, at start[key] + rank. One launch instead of rank,
// prefix and scatter; no block waits on another.
template <class KeyFn, class Consumer>
static __global__ void __launch_bounds__(kSortThreads)
csort_single_tile_kernel(KeyFn kf, int64_t Y, int B, uint32_t* __restrict__ bucket_start,
                         GroupListOut gl, Consumer sc) {
    extern __shared__ __align__(16) uint16_t tab[];  // [kSortWarps][B] u16, then [B + 1] u32
    __shared__ uint32_t warp_sums[32];
    pdl_enter();
    uint32_t* bs = reinterpret_cast<uint32_t*>(tab + (kSortWarps * B + 7) / 8 * 8);  // 16-byte aligned
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int tab_words = (kSortWarps * B + 1) / 2;
    uint32_t* tab32 = reinterpret_cast<uint32_t*>(tab);
    for (int i = threadIdx.x; i < tab_words; i += kSortThreads) tab32[i] = 0u;
    const int64_t base = (int64_t)warp * (32 * kSortChunks);
    int key[kSortChunks];
#pragma unroll
    for (int c = 0; c < kSortChunks; ++c) {
        const int64_t i = base + c * 32 + lane;
        key[c] = i < Y ? kf(i) : -1;
        if (key[c] >= 0 && !MR_IN_RANGE(key[c], B, 203)) key[c] = -1;
    }
    __syncthreads();
    uint16_t* mytab = tab + warp * B;
    uint32_t rnk[kSortChunks];
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int c = 0; c < kSortChunks; ++c) {
        const int k = key[c];
        const uint32_t peers = __match_any_sync(0xffffffffu, k);
        const uint32_t below = __popc(peers & lt);
        uint32_t before = 0u;
        if (k >= 0) before = mytab[k];
        __syncwarp();
        if (k >= 0 && below == 0u) mytab[k] = (uint16_t)(before + __popc(peers));
        __syncwarp();
        rnk[c] = before + below;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < kSortChunks; ++c) {
        const int k = key[c];
        if (k >= 0)
            for (int w = 0; w < warp; ++w) rnk[c] += tab[w * B + k];
    }
    for (int k = threadIdx.x; k < B; k += kSortThreads) {
        uint32_t s = 0u;
#pragma unroll
        for (int w = 0; w < kSortWarps; ++w) s += tab[w * B + k];
        bs[k] = s;
    }
    __syncthreads();
    // key starts: each thread scans a run of consecutive keys
    const int per_t = (B + kSortThreads - 1) / kSortThreads;
    const int c0 = threadIdx.x * per_t < B ? threadIdx.x * per_t : B;
    const int c1 = c0 + per_t < B ? c0 + per_t : B;
    uint32_t s = 0u, ng = 0u;
    for (int k = c0; k < c1; ++k) {
        s += bs[k];
        if (k < gl.limit && bs[k] != 0u) ++ng;
    }
    uint32_t total = 0u, groups = 0u;
    const uint32_t excl = block_exclusive_scan(s, warp_sums, &total);
    const uint32_t gexcl = block_exclusive_scan(ng, warp_sums, &groups);
    uint32_t run = excl, r = gexcl;
    for (int k = c0; k < c1; ++k) {
        const uint32_t v = bs[k];
        bs[k] = run;
        bucket_start[k] = run;
        if (gl.rows && k < gl.limit && v != 0u && MR_IN_RANGE(r, gl.limit, 204)) {
            gl.rows[2 * (int64_t)r] = k;
            gl.rows[2 * (int64_t)r + 1] = v;
            ++r;
        }
        run += v;
    }
    if (threadIdx.x == 0) {
        bs[B] = total;
        bucket_start[B] = total;
    }
    if (gl.rows)
        for (int64_t q = (int64_t)groups + threadIdx.x; q < gl.limit; q += kSortThreads) {
            gl.rows[2 * q] = 0;
            gl.rows[2 * q + 1] = 0;
        }
    __syncthreads();
    if (gl.count_out && threadIdx.x == 0) *gl.count_out = (int64_t)bs[gl.limit];
#pragma unroll
    for (int c = 0; c < kSortChunks; ++c) {
        const int k = key[c];
        if (k >= 0) sc(base + c * 32 + lane, k, bs[k] + rnk[c], bs[k]);
    }
}

// Launch of csort_single_tile_kernel for N <= kSortTile items.
template <class KeyFn, class Consumer>
inline cudaError_t csort_single_tile(KeyFn kf, int64_t N, int B, const CsortBufs& b, GroupListOut gl,
                                     const Consumer& cons, cudaStream_t st) {
    const size_t smem = align_up((uint64_t)kSortWarps * B * 2u, 16) + align_up((uint64_t)(B + 1) * 4u, 16);
    auto kernel = csort_single_tile_kernel<KeyFn, Consumer>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kernel, dim3(1), dim3(kSortThreads), smem, st, kf, N, B, b.bucket_start, gl, cons);
}

}  // namespace mr
