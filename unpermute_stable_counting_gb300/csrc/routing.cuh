// Routing-map column masks, shared by the unpermute (maskedSelect) and the
// permute: both order the routed (token, expert) pairs expert-major.
#pragma once

#include "csort.cuh"

namespace mr {

// ---------------------------------------------------------------------------
// maskedSelect of probs.T by routingMap.T (not padded, with probs).
// The routing map is cut into blocks of 32 tokens; item (blk, e) holds the
// 32-bit mask of the block's tokens routed to expert e (built by one lane per
// expert, or per four experts, reading 32 routing-map rows). Its popcount is the
// histogram entry of the counting sort whose key is the expert, so the
// engine's prefix kernel turns them into positions: the j-th token of the
// mask lands at bucket_start[e] + tile_off[blk][e] + (set bits below j).
// ---------------------------------------------------------------------------
// EPL experts per lane: 1 (any map), or 4 when the map is 4-byte aligned
// and Eu a multiple of 4 (one 4-byte load per token covers the lane's four
// experts, so a warp reads 128 consecutive map bytes per token).
template <int EPL>
static __global__ void __launch_bounds__(256)
mask_columns_kernel(const int8_t* __restrict__ map, int64_t T, int64_t Eu,
                    uint32_t* __restrict__ masks, uint32_t* __restrict__ counts,
                    uint32_t* __restrict__ ticket) {
    pdl_enter();
    if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0u;
    // one warp per (32-token block, 32 * EPL-expert chunk); 32 coalesced
    // loads of consecutive routing-map bytes, one per token
    const int lane = threadIdx.x & 31;
    const int64_t nblk = (T + 31) / 32;
    const int64_t chunks = (Eu + 32 * EPL - 1) / (32 * EPL);
    const int64_t units = nblk * chunks;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t unit = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; unit < units;
         unit += nwarps) {
        const int64_t blk = unit / chunks;
        const int64_t e = (unit - blk * chunks) * (32 * EPL) + (int64_t)lane * EPL;
        const int64_t t0 = blk * 32;
        if (e >= Eu) continue;  // with EPL = 4, Eu % 4 == 0: all four experts exist
        uint32_t bits[EPL];
#pragma unroll
        for (int k = 0; k < EPL; ++k) bits[k] = 0u;
        if (EPL == 1) {
            int8_t m[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) m[j] = t0 + j < T ? map[(t0 + j) * Eu + e] : (int8_t)0;
#pragma unroll
            for (int j = 0; j < 32; ++j) bits[0] |= (m[j] != 0 ? 1u : 0u) << j;
        } else {
            uint32_t m[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                m[j] = t0 + j < T ? __ldg(reinterpret_cast<const uint32_t*>(map + (t0 + j) * Eu + e)) : 0u;
#pragma unroll
            for (int j = 0; j < 32; ++j)
#pragma unroll
                for (int k = 0; k < EPL; ++k) bits[k] |= (((m[j] >> (8 * k)) & 0xffu) != 0u ? 1u : 0u) << j;
        }
#pragma unroll
        for (int k = 0; k < EPL; ++k) {
            masks[blk * Eu + e + k] = bits[k];
            counts[blk * Eu + e + k] = __popc(bits[k]);
        }
    }
}

// Launch of the column masks over a grid of up to 8 blocks per SM.
inline cudaError_t launch_mask_columns(const int8_t* map, int64_t T, int64_t Eu, uint32_t* masks,
                                       uint32_t* counts, uint32_t* ticket, cudaStream_t s) {
    const bool wide = (Eu % 4) == 0 && (reinterpret_cast<uintptr_t>(map) & 3u) == 0u;
    const int64_t epl = wide ? 4 : 1;
    const int64_t nblk = (T + 31) / 32;
    const int64_t want = (nblk * ((Eu + 32 * epl - 1) / (32 * epl)) * 32 + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    const int grid = (int)(want < cap ? (want > 0 ? want : 1) : cap);
    return wide ? launch_pdl(mask_columns_kernel<4>, dim3(grid), dim3(256), 0, s, map, T, Eu, masks, counts, ticket)
                : launch_pdl(mask_columns_kernel<1>, dim3(grid), dim3(256), 0, s, map, T, Eu, masks, counts, ticket);
}

// Rank of token t among the tokens routed to expert e, from the block masks
// and the per-block offsets the prefix kernel left in `offs`.
__device__ __forceinline__ int64_t column_rank(const uint32_t* __restrict__ masks,
                                               const uint32_t* __restrict__ offs, int64_t Eu,
                                               int64_t t, int64_t e) {
    const int64_t item = (t >> 5) * Eu + e;
    return (int64_t)offs[item] + __popc(masks[item] & ((1u << (t & 31)) - 1u));
}

}  // namespace mr
