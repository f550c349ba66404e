// Routing-map permute on GB300: the producer of the unpermute's inputs.
//
// "MoeTokenUnpermuteWithRoutingMap 算子全解析", 算子定位: the permute step
// rearranges the tokens by routingMap into an expert-grouped compact layout,
// permutedTokens, so that each expert reads its tokens contiguously.
//   not padded: rows = routed (token, expert) pairs in expert-major order;
//               sortedIndices[t*topK + j] = row of t's j-th routed expert, -1
//               for unused slots (and for a pair whose row is past topK*T)
//   padded:     expert e keeps its first `capacity` routed tokens in rows
//               e*capacity + r (sortedIndices = the token); other rows are
//               padding (sortedIndices -1, zero row)
//
// Launch sequence (PDL-chained):
//   1. mask_columns_kernel : 32-token column bitmasks of the routing map
//   2. csort_prefix        : per-expert offsets of the blocks, expert starts
//   3. permute_rows_kernel : one warp per token: ballots over 32 experts at a
//                            time find its routed experts, each pair's row is
//                            start[e] + (block offset) + (routed tokens of the
//                            block below t); the warp writes the slots, then
//                            reads the token row once (up to 256 experts) and
//                            stores it to every destination row; further
//                            warps zero the padding rows
#include <cstdio>
#include <cstdlib>

#include "batching.cuh"
#include "routing.cuh"

namespace mr {

constexpr int kPermuteVPT = 4;     // 16-byte vectors per lane per step
constexpr int kPermuteGroups = 8;  // experts <= 32 * this: destinations held in registers

// Row of the pair (t, e) for lane e of a 32-expert group, or -1 if t is not
// routed to e, the pair is dropped (padded: past the capacity; not padded:
// past topK*T). Writes the pair's slot (not padded) or the row's token
// (padded) and advances j_base by the group's routed count (warp-uniform).
__device__ __forceinline__ int64_t permute_pair_row(const int8_t* __restrict__ map,
                                                    const uint32_t* __restrict__ masks,
                                                    const uint32_t* __restrict__ offs,
                                                    const uint32_t* __restrict__ bstart, int64_t Eu,
                                                    int64_t t, int64_t e, int64_t topk, int padded,
                                                    int64_t cap, int64_t n,
                                                    int32_t* __restrict__ si, int64_t& j_base) {
    const bool routed = e < Eu && map[t * Eu + e] != 0;
    const uint32_t bal = __ballot_sync(0xffffffffu, routed);
    int64_t row = -1;
    if (routed) {
        const int64_t rank = column_rank(masks, offs, Eu, t, e);
        if (!padded) {
            row = (int64_t)bstart[e] + rank;
            const int64_t j = j_base + __popc(bal & lanemask_lt());
            if (row >= n) row = -1;
            if (j < topk) si[t * topk + j] = (int32_t)row;
        } else if (rank < cap) {
            row = e * cap + rank;
            if (MR_IN_RANGE(row, n, 601)) si[row] = (int32_t)t;
            else row = -1;
        }
    }
    j_base += __popc(bal);
    return row;
}

// Copy of one row for the paths off the fast one (rows that are not 16-byte
// vectors, or tokens routed to more than 256 experts), kept out of line so
// its unrolled loops do not raise the kernel's register count.
__device__ __noinline__ void permute_copy_row(const uint8_t* src, uint8_t* dst, int64_t bytes,
                                              int lane) {
    warp_copy_row<4>(src, dst, bytes, lane, false);
}

__device__ __forceinline__ void warp_zero_row(uint8_t* __restrict__ dst, int64_t bytes, int lane) {
    if (((reinterpret_cast<uintptr_t>(dst) | (uintptr_t)bytes) & 15u) == 0u) {
        const int64_t nv = bytes >> 4;
        for (int64_t v = lane; v < nv; v += 32) st_stream_v4(dst + 16 * v, make_uint4(0u, 0u, 0u, 0u));
    } else {
        for (int64_t b = lane; b < bytes; b += 32) dst[b] = 0;
    }
}

static __global__ void __launch_bounds__(256)
permute_rows_kernel(const uint8_t* __restrict__ tokens, int64_t T, int64_t row_bytes,
                    const int8_t* __restrict__ map, int64_t Eu, const uint32_t* __restrict__ masks,
                    const uint32_t* __restrict__ offs, const uint32_t* __restrict__ bstart,
                    const uint32_t* __restrict__ totals, int64_t topk, int padded, int64_t cap,
                    uint8_t* __restrict__ permuted, int32_t* __restrict__ si,
                    int32_t* __restrict__ rows_out) {
    __shared__ uint32_t warp_sums[32];
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int64_t n = padded ? Eu * cap : T * topk;

    if (blockIdx.x == 0 && rows_out) {
        if (!padded) {
            if (threadIdx.x == 0) {
                const int64_t pairs = bstart[Eu];
                *rows_out = (int32_t)(pairs < n ? pairs : n);
            }
        } else {
            uint32_t kept = 0u;
            for (int64_t e = threadIdx.x; e < Eu; e += blockDim.x) {
                const int64_t c = totals[e];
                kept += (uint32_t)(c < cap ? c : cap);
            }
            uint32_t total = 0u;
            block_exclusive_scan(kept, warp_sums, &total);
            if (threadIdx.x == 0) *rows_out = (int32_t)total;
        }
    }

    const bool vec = ((reinterpret_cast<uintptr_t>(tokens) | reinterpret_cast<uintptr_t>(permuted) |
                       (uintptr_t)row_bytes) & 15u) == 0u;
    const int64_t nvec = row_bytes >> 4;
    const int64_t units = T + (padded ? n : 0);
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < units; u += nw) {
        if (u >= T) {
            // a padding row: past the tokens the expert kept
            const int64_t r = u - T;
            const int64_t e = r / cap;
            const int64_t c = totals[e];
            if (r - e * cap >= (c < cap ? c : cap)) {
                if (lane == 0) si[r] = -1;
                warp_zero_row(permuted + r * row_bytes, row_bytes, lane);
            }
            continue;
        }
        const int64_t t = u;
        const uint8_t* src = tokens + t * row_bytes;
        int64_t j_base = 0;
        if (Eu <= 32 * kPermuteGroups) {
            // every destination row of the token first (lane l of group g holds
            // expert 32g + l), then one read of the token row for all of them
            int64_t rowg[kPermuteGroups];
            uint32_t dm[kPermuteGroups];
#pragma unroll
            for (int g = 0; g < kPermuteGroups; ++g) {
                rowg[g] = -1;
                dm[g] = 0u;
                if (32 * g < Eu) {
                    rowg[g] = permute_pair_row(map, masks, offs, bstart, Eu, t, 32 * g + lane, topk,
                                               padded, cap, n, si, j_base);
                    dm[g] = __ballot_sync(0xffffffffu, rowg[g] >= 0);
                }
            }
            if (vec) {
                for (int64_t v0 = 0; v0 < nvec; v0 += 32 * kPermuteVPT) {
                    uint4 x[kPermuteVPT];
#pragma unroll
                    for (int q = 0; q < kPermuteVPT; ++q) {
                        const int64_t v = v0 + 32 * q + lane;
                        if (v < nvec) x[q] = ld_stream_v4(src + 16 * v);
                    }
#pragma unroll
                    for (int g = 0; g < kPermuteGroups; ++g) {
                        uint32_t m = dm[g];
                        while (m) {
                            const int d = __ffs(m) - 1;
                            m &= m - 1u;
                            uint8_t* dst = permuted + __shfl_sync(0xffffffffu, rowg[g], d) * row_bytes;
#pragma unroll
                            for (int q = 0; q < kPermuteVPT; ++q) {
                                const int64_t v = v0 + 32 * q + lane;
                                if (v < nvec) st_stream_v4(dst + 16 * v, x[q]);
                            }
                        }
                    }
                }
            } else {
#pragma unroll
                for (int g = 0; g < kPermuteGroups; ++g) {
                    uint32_t m = dm[g];
                    while (m) {
                        const int d = __ffs(m) - 1;
                        m &= m - 1u;
                        const int64_t drow = __shfl_sync(0xffffffffu, rowg[g], d);
                        permute_copy_row(src, permuted + drow * row_bytes, row_bytes, lane);
                    }
                }
            }
        } else {
            // many experts: 32 at a time, the token row read once per group
            for (int64_t e0 = 0; e0 < Eu; e0 += 32) {
                const int64_t row = permute_pair_row(map, masks, offs, bstart, Eu, t, e0 + lane, topk,
                                                     padded, cap, n, si, j_base);
                uint32_t m = __ballot_sync(0xffffffffu, row >= 0);
                while (m) {
                    const int d = __ffs(m) - 1;
                    m &= m - 1u;
                    const int64_t drow = __shfl_sync(0xffffffffu, row, d);
                    permute_copy_row(src, permuted + drow * row_bytes, row_bytes, lane);
                }
            }
        }
        if (!padded) {
            const int64_t j0 = j_base < topk ? j_base : topk;
            for (int64_t j = j0 + lane; j < topk; j += 32) si[t * topk + j] = -1;
        }
    }
}

struct PermutePlan {
    int64_t T, H, Eu, topk, cap, rows, nblk, row_bytes;
    int padded, dtype;
    uint64_t ws;
};

static mr_status plan_permute(int64_t numTokens, int64_t hidden, int32_t tokenDtype,
                              int64_t numExperts, int64_t topK, int32_t paddedMode,
                              int64_t capacity, PermutePlan* p) {
    if (tokenDtype != MR_DTYPE_F16 && tokenDtype != MR_DTYPE_BF16 && tokenDtype != MR_DTYPE_F32)
        return MR_ERR_PARAM_INVALID;
    if (paddedMode != 0 && paddedMode != 1) return MR_ERR_PARAM_INVALID;
    if (numTokens <= 0 || hidden <= 0 || numExperts <= 0 || numExperts > MR_MAX_EXPERT_NUM)
        return MR_ERR_PARAM_INVALID;
    if (numTokens >= (INT64_C(1) << 31) || hidden > (INT64_C(1) << 40)) return MR_ERR_PARAM_INVALID;
    int64_t rows;
    if (!paddedMode) {
        if (topK <= 0) return MR_ERR_PARAM_INVALID;
        if (topK > MR_MAX_TOPK_NUM) return MR_ERR_INNER;
        rows = numTokens * topK;
    } else {
        if (capacity <= 0) return MR_ERR_PARAM_INVALID;
        rows = numExperts * capacity;
    }
    if (rows >= (INT64_C(1) << 31)) return MR_ERR_PARAM_INVALID;
    p->T = numTokens;
    p->H = hidden;
    p->Eu = numExperts;
    p->topk = paddedMode ? 0 : topK;
    p->cap = paddedMode ? capacity : 0;
    p->rows = rows;
    p->padded = paddedMode;
    p->dtype = tokenDtype;
    p->row_bytes = hidden * (tokenDtype == MR_DTYPE_F32 ? 4 : 2);
    p->nblk = (numTokens + 31) / 32;
    const uint64_t items = (uint64_t)p->nblk * numExperts;
    p->ws = align_up(items * 4u, 256) * 2 + align_up((uint64_t)numExperts * 4u, 256) +
            align_up((uint64_t)(numExperts + 1) * 4u, 256) + 256;
    return MR_OK;
}

static int permute_grid(int64_t units) {
    const int64_t want = (units + 7) / 8;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

MR_CHECK_ACCESSOR(permute)

}  // namespace mr

using namespace mr;

extern "C" mr_status moe_permute_get_workspace_size(int64_t numTokens, int64_t hidden,
                                                     int32_t tokenDtype, int64_t numExperts,
                                                     int64_t topK, int32_t paddedMode,
                                                     int64_t capacity, uint64_t* workspaceSize) {
    if (!workspaceSize) return MR_ERR_PARAM_NULLPTR;
    PermutePlan p;
    const mr_status st = plan_permute(numTokens, hidden, tokenDtype, numExperts, topK, paddedMode,
                                      capacity, &p);
    if (st != MR_OK) return st;
    *workspaceSize = p.ws;
    return MR_OK;
}

extern "C" mr_status moe_permute(const void* tokens, const int8_t* routingMap, int64_t numTokens,
                                 int64_t hidden, int32_t tokenDtype, int64_t numExperts,
                                 int64_t topK, int32_t paddedMode, int64_t capacity,
                                 void* permutedTokens, int32_t* sortedIndices,
                                 int32_t* permutedRowsOut, void* workspace, uint64_t workspaceSize,
                                 void* stream) {
    PermutePlan p;
    const mr_status st = plan_permute(numTokens, hidden, tokenDtype, numExperts, topK, paddedMode,
                                      capacity, &p);
    if (st != MR_OK) return st;
    if (!tokens || !routingMap || !permutedTokens || !sortedIndices || !workspace)
        return MR_ERR_PARAM_NULLPTR;
    if (workspaceSize < p.ws) return MR_ERR_WORKSPACE;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* q = reinterpret_cast<uint8_t*>(workspace);
    const uint64_t items = (uint64_t)p.nblk * p.Eu;
    uint32_t* masks = reinterpret_cast<uint32_t*>(q);
    q += align_up(items * 4u, 256);
    uint32_t* offs = reinterpret_cast<uint32_t*>(q);
    q += align_up(items * 4u, 256);
    uint32_t* totals = reinterpret_cast<uint32_t*>(q);
    q += align_up((uint64_t)p.Eu * 4u, 256);
    uint32_t* bstart = reinterpret_cast<uint32_t*>(q);
    q += align_up((uint64_t)(p.Eu + 1) * 4u, 256);
    uint32_t* ticket = reinterpret_cast<uint32_t*>(q);

    profile_mark(s, 0);
    MR_TRY_CUDA(launch_mask_columns(routingMap, p.T, p.Eu, masks, offs, ticket, s));
    GroupListOut none{nullptr, nullptr, 0};
    MR_TRY_CUDA(csort_prefix(offs, p.nblk, (int)p.Eu, totals, bstart, ticket, none, s));
    profile_mark(s, 1);
    profile_mark(s, 2);
    const int64_t units = p.T + (p.padded ? p.rows : 0);
    MR_TRY_CUDA(launch_pdl(permute_rows_kernel, dim3(permute_grid(units)), dim3(256), 0, s,
                           reinterpret_cast<const uint8_t*>(tokens), p.T, p.row_bytes, routingMap,
                           p.Eu, (const uint32_t*)masks, (const uint32_t*)offs,
                           (const uint32_t*)bstart, (const uint32_t*)totals, p.topk, p.padded, p.cap,
                           reinterpret_cast<uint8_t*>(permutedTokens), sortedIndices,
                           permutedRowsOut));
    profile_mark(s, 3);
    MR_TRY_CUDA(cudaGetLastError());
    return MR_OK;
}
