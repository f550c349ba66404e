// One-launch form of the stable counting sort for inputs of a few tens of
// tiles (the batching of a decode step: "aclnnFfnWorkerBatching", 功能说明
// steps 2-4, the sort that yields gather_idx, expertOffsets and group_list).
//
// The multi-kernel engine (csort.cuh) spends most of a mid-sized sort on the
// dependent memory round trips of its three kernels. Here one cooperative
// launch does everything, one block per tile of kCoopTile items:
//
//   1. load the tile's keys and, through the consumer's load(), every value
//      its scatter will need (ids of the slot) -- one DRAM round trip;
//   2. stable in-tile ranks (__match_any_sync, per-warp u16 counters, as in
//      csort_rank_kernel) and the tile's histogram, stored key-major:
//      counts_t[key * TP + tile] (TP = tiles rounded up to 4);
//   3. one grid barrier;
//   4. per key, 16-byte loads of the key's row of counts give the items of
//      that key in lower tiles (the tile offset) and in all tiles (the key
//      total); all of a thread's loads are issued together;
//   5. a block scan of the key totals gives the key starts; block 0 writes
//      them to bucket_start, plus the compacted [key, count] list and the
//      item count below a limit (group_list, actual_token_num);
//   6. each item's position start[key] + offset[key] + rank goes to the
//      consumer's store(), with the values loaded in step 1.
//
// Ties keep item order, so the sort is stable, and the positions are the
// ones the multi-kernel engine gives. The launch is cooperative, so every
// block is resident at the grid barrier; csort_coop() checks that the tiles
// fit the device before launching.
//
// A decoupled look-back form (tile ids from a ticket, per-(tile, key) status
// words holding an aggregate or an inclusive prefix, each tile looking back
// over its predecessors) was measured on GB300 and is not used: the batching
// needs every key's total before any item can be placed, so each tile also
// waits for the last tile's prefix, and the status words need an
// initialising kernel before the look-back kernel (21-23 us for the index
// step of 18432 slots, against 16.9 us for the three-kernel chain and
// 12-14 us for this form).
#pragma once

#include <cooperative_groups.h>

#include "csort.cuh"

namespace mr {

constexpr int kCoopChunks = 2;                              // 32-item chunks per warp
constexpr int kCoopTile = kSortThreads * kCoopChunks;       // 512 items per block
constexpr int kCoopMaxTiles = 64;                           // up to 32768 items
constexpr int kCoopVecs = kCoopMaxTiles / 4;                // 16-byte count loads per key
constexpr int kCoopMaxKeys = 4098;                          // shared memory: 24 bytes per key

inline int64_t csort_coop_tiles(int64_t N) { return (N + kCoopTile - 1) / kCoopTile; }
// Inputs served by the one-launch form: more than one multi-kernel tile (one
// tile takes csort_single_tile_kernel) and at most kCoopMaxTiles of its own.
inline bool csort_coop_eligible(int64_t N, int B) {
    return N > kSortTile && csort_coop_tiles(N) <= kCoopMaxTiles && B <= kCoopMaxKeys;
}
inline int csort_coop_tp(int64_t N) { return (int)((csort_coop_tiles(N) + 3) & ~INT64_C(3)); }
// Workspace of the key-major count matrix (0 when the form does not apply).
inline uint64_t csort_coop_bytes(int64_t N, int B) {
    return csort_coop_eligible(N, B) ? align_up((uint64_t)B * csort_coop_tp(N) * 4u, 256) : 0u;
}
inline size_t csort_coop_smem(int B) {
    return align_up((uint64_t)kSortWarps * B * 2u, 16) + align_up((uint64_t)B * 4u, 16) +
           align_up((uint64_t)(B + 1) * 4u, 16);
}

// Exclusive scan of st[0..B) in place by all 8 warps (warp w owns a run of
// consecutive keys, each lane a run within it), st[B] = the total. With
// `write`, also the starts to bucket_start[0..B] and the compacted list of the
// non-empty keys below gl.limit, rows past it [0, 0], and gl.count_out.
__device__ __forceinline__ void coop_scan_starts(uint32_t* st, int B, bool write, GroupListOut gl,
                                                 uint32_t* bucket_start) {
    __shared__ uint32_t wsum[kSortWarps], wgrp[kSortWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int per_w = (B + kSortWarps - 1) / kSortWarps;
    const int per_l = (per_w + 31) / 32;
    int c0 = warp * per_w + lane * per_l;
    int c1 = c0 + per_l;
    const int w_end = (warp + 1) * per_w < B ? (warp + 1) * per_w : B;
    if (c0 > w_end) c0 = w_end;
    if (c1 > w_end) c1 = w_end;
    uint32_t s = 0u, ng = 0u;
    for (int k = c0; k < c1; ++k) {
        const uint32_t v = st[k];
        s += v;
        ng += (k < gl.limit && v != 0u) ? 1u : 0u;
    }
    uint32_t xs = s, xg = ng;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t a = __shfl_up_sync(0xffffffffu, xs, o);
        const uint32_t b = __shfl_up_sync(0xffffffffu, xg, o);
        if (lane >= o) {
            xs += a;
            xg += b;
        }
    }
    if (lane == 31) {
        wsum[warp] = xs;
        wgrp[warp] = xg;
    }
    __syncthreads();
    uint32_t base = 0u, gbase = 0u, total = 0u, groups = 0u;
#pragma unroll
    for (int w = 0; w < kSortWarps; ++w) {
        const uint32_t a = wsum[w], b = wgrp[w];
        if (w < warp) {
            base += a;
            gbase += b;
        }
        total += a;
        groups += b;
    }
    uint32_t run = base + xs - s, r = gbase + xg - ng;
    for (int k = c0; k < c1; ++k) {
        const uint32_t v = st[k];
        st[k] = run;
        if (write) {
            bucket_start[k] = run;
            if (gl.rows && k < gl.limit && v != 0u && MR_IN_RANGE(r, gl.limit, 206)) {
                gl.rows[2 * (int64_t)r] = k;
                gl.rows[2 * (int64_t)r + 1] = v;
                ++r;
            }
        }
        run += v;
    }
    if (threadIdx.x == 0) {
        st[B] = total;
        if (write) bucket_start[B] = total;
    }
    if (write && gl.rows)
        for (int64_t q = (int64_t)groups + threadIdx.x; q < gl.limit; q += kSortThreads) {
            gl.rows[2 * q] = 0;
            gl.rows[2 * q + 1] = 0;
        }
    __syncthreads();
    if (write && gl.count_out && threadIdx.x == 0) *gl.count_out = (int64_t)st[gl.limit];
}

// The consumer provides `Pre load(int64_t i)` (values item i's scatter reads,
// loaded with its key) and `store(int64_t i, int key, uint32_t pos,
// uint32_t key_start, const Pre&)`.
template <class KeyFn, class Consumer>
static __global__ void __launch_bounds__(kSortThreads)
csort_coop_kernel(KeyFn kf, int64_t N, int B, uint32_t* __restrict__ counts_t,
                  uint32_t* __restrict__ bucket_start, GroupListOut gl, Consumer sc) {
    extern __shared__ __align__(16) uint16_t tab[];  // [8][B] u16, then lo[B], st[B + 1] u32
    cooperative_groups::grid_group grid = cooperative_groups::this_grid();
    pdl_enter();
    uint32_t* lo = reinterpret_cast<uint32_t*>(tab + (kSortWarps * B + 7) / 8 * 8);
    uint32_t* st = lo + (B + 3) / 4 * 4;
    const int tile = (int)blockIdx.x;
    const int tiles = (int)gridDim.x;
    const int TP = (tiles + 3) & ~3;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    {
        const int tab_words = (kSortWarps * B + 1) / 2;
        uint32_t* tab32 = reinterpret_cast<uint32_t*>(tab);
        for (int i = threadIdx.x; i < tab_words; i += kSortThreads) tab32[i] = 0u;
    }
    const int64_t base = (int64_t)tile * kCoopTile + (int64_t)warp * (32 * kCoopChunks);
    int key[kCoopChunks];
    typename Consumer::Pre pre[kCoopChunks];
#pragma unroll
    for (int c = 0; c < kCoopChunks; ++c) {
        const int64_t i = base + c * 32 + lane;
        key[c] = i < N ? kf(i) : -1;
        if (key[c] >= 0 && !MR_IN_RANGE(key[c], B, 205)) key[c] = -1;
        if (i < N) pre[c] = sc.load(i);
    }
    __syncthreads();

    // stable in-tile ranks
    uint16_t* mytab = tab + warp * B;
    const uint32_t lt = lanemask_lt();
    uint32_t rnk[kCoopChunks];
#pragma unroll
    for (int c = 0; c < kCoopChunks; ++c) {
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
    for (int c = 0; c < kCoopChunks; ++c) {
        const int k = key[c];
        if (k >= 0)
            for (int w = 0; w < warp; ++w) rnk[c] += tab[w * B + k];
    }
    for (int k = threadIdx.x; k < B; k += kSortThreads) {
        uint32_t s = 0u;
#pragma unroll
        for (int w = 0; w < kSortWarps; ++w) s += tab[w * B + k];
        counts_t[(int64_t)k * TP + tile] = s;
    }

    grid.sync();

    // per key: items in lower tiles and in all tiles; two keys per step, their
    // loads issued together (the padding columns past `tiles` are skipped)
    const int nv = TP / 4;
    for (int k0 = threadIdx.x; k0 < B; k0 += 2 * kSortThreads) {
        const int k1 = k0 + kSortThreads;
        const bool has1 = k1 < B;
        const uint4* pa = reinterpret_cast<const uint4*>(counts_t + (int64_t)k0 * TP);
        const uint4* pb = reinterpret_cast<const uint4*>(counts_t + (int64_t)(has1 ? k1 : k0) * TP);
        uint4 a[kCoopVecs], b[kCoopVecs];
#pragma unroll
        for (int v = 0; v < kCoopVecs; ++v) {
            if (v < nv) {
                a[v] = __ldcg(pa + v);
                b[v] = has1 ? __ldcg(pb + v) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
        uint32_t la = 0u, ta = 0u, lb = 0u, tb = 0u;
#pragma unroll
        for (int v = 0; v < kCoopVecs; ++v) {
            if (v < nv) {
                const uint32_t xa[4] = {a[v].x, a[v].y, a[v].z, a[v].w};
                const uint32_t xb[4] = {b[v].x, b[v].y, b[v].z, b[v].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int t = v * 4 + q;
                    if (t < tiles) {
                        if (t < tile) {
                            la += xa[q];
                            lb += xb[q];
                        }
                        ta += xa[q];
                        tb += xb[q];
                    }
                }
            }
        }
        lo[k0] = la;
        st[k0] = ta;
        if (has1) {
            lo[k1] = lb;
            st[k1] = tb;
        }
    }
    __syncthreads();
    coop_scan_starts(st, B, tile == 0, gl, bucket_start);

#pragma unroll
    for (int c = 0; c < kCoopChunks; ++c) {
        const int k = key[c];
        if (k >= 0) sc.store(base + c * 32 + lane, k, st[k] + lo[k] + rnk[c], st[k], pre[c]);
    }
}

// Launch of the one-launch sort when the input is eligible, fits the device
// (every block resident) and the workspace holds the count matrix. Returns
// cudaErrorNotSupported, with nothing enqueued, when it does not apply.
template <class KeyFn, class Consumer>
inline cudaError_t csort_coop(KeyFn kf, int64_t N, int B, uint32_t* counts_t, uint32_t* bucket_start,
                              GroupListOut gl, const Consumer& sc, cudaStream_t st) {
    if (!counts_t || !csort_coop_eligible(N, B)) return cudaErrorNotSupported;
    auto kernel = csort_coop_kernel<KeyFn, Consumer>;
    const size_t smem = csort_coop_smem(B);
    // set up once per device for the largest key count, so that the residency
    // check holds for every B
    const size_t smem_max = csort_coop_smem(kCoopMaxKeys);
    static int blocks_per_sm[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int bps = dev < 64 ? blocks_per_sm[dev] : 0;
    if (bps == 0) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kernel, kSortThreads, smem_max);
        if (e != cudaSuccess) return e;
        if (bps <= 0) return cudaErrorNotSupported;
        if (dev < 64) blocks_per_sm[dev] = bps;
    }
    const int64_t tiles = csort_coop_tiles(N);
    if (tiles > (int64_t)device_sm_count() * bps) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles);
    cfg.blockDim = dim3(kSortThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, kf, N, B, counts_t, bucket_start, gl, sc);
}

}  // namespace mr
