// The batching's row gather ("aclnnFfnWorkerBatching", 计算公式 y[i] =
// token_data[gather_idx[i]], and the INT8 dynamic scale of step 3), kept
// apart from the index work so that its source is one file.
#pragma once

#include "common.cuh"

namespace mr {

// 16-byte output vectors from a source that is only 4-byte aligned (INT8 rows
// with their trailing scale have a stride of H + 4 bytes). With o = src % 16
// (4, 8 or 12) and `win` the aligned address src - o, output vector j is the
// tail of window j followed by the head of window j + 1. Lane l loads window
// j = j0 + l and takes window j + 1 from lane l + 1 by a shuffle. Windows up to
// nvec - 1 lie inside [win, src + bytes); the last output vector is read as
// words. The caller uses this only when the buffer base is 16-byte aligned,
// so win never precedes the buffer.
constexpr int kShiftVPT = 8;

__device__ __forceinline__ uint4 shift_combine(const uint4& a, const uint4& b, int o) {
    if (o == 4) return make_uint4(a.y, a.z, a.w, b.x);
    if (o == 8) return make_uint4(a.z, a.w, b.x, b.y);
    return make_uint4(a.w, b.x, b.y, b.z);
}

__device__ __forceinline__ void warp_copy_row_shift(const uint8_t* __restrict__ src,
                                                    uint8_t* __restrict__ dst, int64_t bytes,
                                                    int lane) {
    const int o = (int)(reinterpret_cast<uintptr_t>(src) & 15u);
    const uint4* win = reinterpret_cast<const uint4*>(src - o);
    const int nv1 = (int)(bytes >> 4) - 1;  // vectors built from two windows
    for (int j0 = 0; j0 < nv1; j0 += 32 * kShiftVPT) {
        uint4 a[kShiftVPT];
#pragma unroll
        for (int u = 0; u < kShiftVPT; ++u) {
            const int j = j0 + 32 * u + lane;
            a[u] = j <= nv1 ? ld_stream_v4(win + j) : make_uint4(0u, 0u, 0u, 0u);
        }
        // lane 31's next window: lane 0's window of the next u, or one more load
        const int jl = j0 + 32 * (kShiftVPT - 1) + 31;
        const uint4 extra = (lane == 31 && jl < nv1) ? ld_stream_v4(win + jl + 1)
                                                     : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < kShiftVPT; ++u) {
            const int j = j0 + 32 * u + lane;
            uint4 b;
            b.x = __shfl_down_sync(0xffffffffu, a[u].x, 1);
            b.y = __shfl_down_sync(0xffffffffu, a[u].y, 1);
            b.z = __shfl_down_sync(0xffffffffu, a[u].z, 1);
            b.w = __shfl_down_sync(0xffffffffu, a[u].w, 1);
            if (u + 1 < kShiftVPT) {
                const uint4 nx = make_uint4(__shfl_sync(0xffffffffu, a[u + 1 < kShiftVPT ? u + 1 : u].x, 0),
                                            __shfl_sync(0xffffffffu, a[u + 1 < kShiftVPT ? u + 1 : u].y, 0),
                                            __shfl_sync(0xffffffffu, a[u + 1 < kShiftVPT ? u + 1 : u].z, 0),
                                            __shfl_sync(0xffffffffu, a[u + 1 < kShiftVPT ? u + 1 : u].w, 0));
                if (lane == 31) b = nx;
            } else if (lane == 31) {
                b = extra;
            }
            if (j < nv1) st_stream_v4(dst + 16 * (int64_t)j, shift_combine(a[u], b, o));
        }
    }
    if (lane == 0 && nv1 >= 0) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(src + 16 * (int64_t)nv1);
        st_stream_v4(dst + 16 * (int64_t)nv1, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// Copy `bytes` from src to dst with one warp. Vector width follows the common
// alignment of both addresses and the length: 16-byte vectors (VPT in flight
// per lane), else 4-byte words, else bytes. Addresses are formed from the
// __restrict__ row pointers directly, which leaves the compiler free to start
// the next batch's loads before the current stores (measured on GB300: 616 us
// against 626 us for the round-trip gather with pointer casts).
template <int VPT>
__device__ __forceinline__ void warp_copy_row(const uint8_t* __restrict__ src,
                                              uint8_t* __restrict__ dst, int64_t bytes, int lane,
                                              bool base16) {
    const uintptr_t mis = (reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
                           (uintptr_t)bytes);
    if ((mis & 15u) == 0u) {
        const int64_t nv = bytes >> 4;
        int64_t v = lane;
        for (; v + 32 * (VPT - 1) < nv; v += 32 * VPT) {
            uint4 r[VPT];
#pragma unroll
            for (int u = 0; u < VPT; ++u) r[u] = ld_stream_v4(src + 16 * (v + 32 * u));
#pragma unroll
            for (int u = 0; u < VPT; ++u) st_stream_v4(dst + 16 * (v + 32 * u), r[u]);
        }
        uint4 r[VPT];
#pragma unroll
        for (int u = 0; u < VPT; ++u)
            if (v + 32 * u < nv) r[u] = ld_stream_v4(src + 16 * (v + 32 * u));
#pragma unroll
        for (int u = 0; u < VPT; ++u)
            if (v + 32 * u < nv) st_stream_v4(dst + 16 * (v + 32 * u), r[u]);
    } else if (base16 && ((reinterpret_cast<uintptr_t>(dst) | (uintptr_t)bytes) & 15u) == 0u &&
               (reinterpret_cast<uintptr_t>(src) & 3u) == 0u) {
        warp_copy_row_shift(src, dst, bytes, lane);
    } else if ((mis & 3u) == 0u) {
        constexpr int W = VPT * 4;
        const int64_t nw = bytes >> 2;
        int64_t v = lane;
        for (; v + 32 * (W - 1) < nw; v += 32 * W) {
            uint32_t r[W];
#pragma unroll
            for (int u = 0; u < W; ++u) r[u] = ld_stream_u32(src + 4 * (v + 32 * u));
#pragma unroll
            for (int u = 0; u < W; ++u) st_stream_u32(dst + 4 * (v + 32 * u), r[u]);
        }
        for (; v < nw; v += 32) st_stream_u32(dst + 4 * v, ld_stream_u32(src + 4 * v));
    } else {
        for (int64_t b = lane; b < bytes; b += 32) dst[b] = src[b];
    }
}

template <int VPT>
static __global__ void __launch_bounds__(256)
batching_gather_kernel(const uint8_t* __restrict__ token_data_arg, int64_t row_stride,
                       int64_t row_bytes, int is_int8, const uint8_t* __restrict__ scales,
                       int64_t scale_stride, uint8_t* __restrict__ y, float* __restrict__ dyn,
                       const int32_t* __restrict__ gather_idx,
                       const uint32_t* __restrict__ bucket_start, int row_keys,
                       const uint64_t* __restrict__ token_data_loc, int64_t nrows) {
    pdl_enter();
    // the token rows' address, passed directly or read from device memory
    const uint8_t* __restrict__ token_data =
        token_data_loc ? reinterpret_cast<const uint8_t*>(*token_data_loc) : token_data_arg;
    // rows of the keys below row_keys: the routed rows (row_keys = E), or
    // every row with a token row behind it (the whole-tail option)
    uint32_t U = bucket_start[row_keys];
    if (!MR_IN_RANGE(U, nrows + 1, 301)) U = 0u;
    const int lane = threadIdx.x & 31;
    const bool base16 = (reinterpret_cast<uintptr_t>(token_data) & 15u) == 0u;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    // the next row's source index is loaded while the current row copies
    int64_t gnext = gw < (int64_t)U ? gather_idx[gw] : 0;
    for (int64_t i = gw; i < (int64_t)U; i += nw) {
        const int64_t g = gnext;
        gnext = i + nw < (int64_t)U ? gather_idx[i + nw] : 0;
        if (!MR_IN_RANGE(g, nrows, 302)) continue;
        warp_copy_row<VPT>(token_data + g * row_stride, y + i * row_bytes, row_bytes, lane, base16);
        if (is_int8) {
            const uint8_t* sp = scales ? scales + g * scale_stride : token_data + g * row_stride + row_bytes;
            if ((reinterpret_cast<uintptr_t>(sp) & 3u) == 0u) {
                if (lane == 0) dyn[i] = *reinterpret_cast<const float*>(sp);
            } else if (lane < 4) {
                // an unaligned scale: one byte per lane
                reinterpret_cast<uint8_t*>(dyn + i)[lane] = sp[lane];
            }
        }
    }
}

// The row gather as a flat grid, for rows of 16-byte vectors whose sources
// are 16-byte aligned: each thread copies kGatherVPT vectors of the output
// (vector v of y = vector v % nvec of output row v / nvec) at a stride of the
// block's width, the threads of a block a contiguous stretch of y, and the
// grid covers every vector of the Y possible rows at once (blocks past the
// gathered rows return at their first check). The hardware hands out blocks
// in order, so the blocks running at one time cover a contiguous window of
// y: measured on GB300, the round trip's 140060 rows of 14336 bytes in their
// sorted order move 6.90 TB/s this way, against 6.52 TB/s for the persistent
// grid of warps below (one row per warp) and 6.0-6.3 TB/s for a persistent
// grid of this loop, whose concurrent accesses spread over the whole buffer.
// Rows that are only 4-byte aligned (INT8 rows with their interleaved scale)
// stay with the warp kernel, whose shuffles build the shifted vectors: flat
// forms of that path measured 55-65 us against 38.8 us for the INT8 workload.
// The rows' address is passed directly, or read from device memory (a
// ScheduleContext's token buffer), in which case the host cannot check its
// alignment and a base that is not 16-byte aligned takes a word-by-word form
// of the same loop.
constexpr int kGatherVPT = 4;
constexpr int kGatherThreads = 256;

// One 4-byte word, and one 16-byte vector, from a source of any alignment
// (4-byte words when the address allows, else bytes).
__device__ __forceinline__ uint32_t ld_u32_any(const uint8_t* p) {
    if ((reinterpret_cast<uintptr_t>(p) & 3u) == 0u) return ld_stream_u32(p);
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
__device__ __forceinline__ uint4 ld_stream_v4_any(const uint8_t* p) {
    return make_uint4(ld_u32_any(p), ld_u32_any(p + 4), ld_u32_any(p + 8), ld_u32_any(p + 12));
}

// The flat loop for a source base that turned out not to be 16-byte aligned
// (read from device memory, as from a ScheduleContext): the same vectors, one
// at a time, through ld_stream_v4_any.
static __device__ __noinline__ void gather_flat_unaligned(
    const uint8_t* __restrict__ token_data, int64_t row_stride, int64_t row_bytes, int is_int8,
    const uint8_t* __restrict__ scales, int64_t scale_stride, uint8_t* __restrict__ y, float* __restrict__ dyn,
    const int32_t* __restrict__ gather_idx, int64_t total, int64_t nvec, int64_t nrows) {
    constexpr int64_t per_block = (int64_t)kGatherThreads * kGatherVPT;
    for (int64_t b0 = (int64_t)blockIdx.x * per_block; b0 < total; b0 += (int64_t)gridDim.x * per_block) {
        for (int u = 0; u < kGatherVPT; ++u) {
            const int64_t v = b0 + (int64_t)u * kGatherThreads + threadIdx.x;
            if (v >= total) break;
            const int64_t row = v / nvec;
            const int64_t o = v - row * nvec;
            const int64_t g = gather_idx[row];
            if (!MR_IN_RANGE(g, nrows, 305)) continue;
            st_stream_v4(y + row * row_bytes + 16 * o, ld_stream_v4_any(token_data + g * row_stride + 16 * o));
            if (is_int8 && o == 0) {
                const uint8_t* sp = scales ? scales + g * scale_stride : token_data + g * row_stride + row_bytes;
                dyn[row] = __uint_as_float(ld_u32_any(sp));
            }
        }
    }
}

// SHORT: rows of fewer than kGatherThreads vectors.
template <bool SHORT>
static __global__ void __launch_bounds__(kGatherThreads, 6)
batching_gather_flat_kernel(const uint8_t* __restrict__ token_data_arg, int64_t row_stride, int64_t row_bytes,
                            int is_int8, const uint8_t* __restrict__ scales, int64_t scale_stride,
                            uint8_t* __restrict__ y, float* __restrict__ dyn,
                            const int32_t* __restrict__ gather_idx, const uint32_t* __restrict__ bucket_start,
                            int row_keys, const uint64_t* __restrict__ token_data_loc, int64_t nrows) {
    pdl_enter();
    // the token rows' address, passed directly or read from device memory
    const uint8_t* __restrict__ token_data =
        token_data_loc ? reinterpret_cast<const uint8_t*>(*token_data_loc) : token_data_arg;
    uint32_t U = bucket_start[row_keys];
    if (!MR_IN_RANGE(U, nrows + 1, 303)) U = 0u;
    const int64_t nvec = row_bytes >> 4;
    const int64_t total = (int64_t)U * nvec;
    if ((reinterpret_cast<uintptr_t>(token_data) & 15u) != 0u) {
        gather_flat_unaligned(token_data, row_stride, row_bytes, is_int8, scales, scale_stride, y, dyn,
                              gather_idx, total, nvec, nrows);
        return;
    }
    constexpr int64_t per_block = (int64_t)kGatherThreads * kGatherVPT;
    for (int64_t b0 = (int64_t)blockIdx.x * per_block; b0 < total; b0 += (int64_t)gridDim.x * per_block) {
        const int64_t v0 = b0 + threadIdx.x;
        int64_t row = v0 / nvec;
        int64_t o = v0 - row * nvec;
        uint4 r[kGatherVPT];
        int64_t dst[kGatherVPT];
#pragma unroll
        for (int u = 0; u < kGatherVPT; ++u) {
            dst[u] = -1;
            if (b0 + (int64_t)u * kGatherThreads + threadIdx.x < total) {
                const int64_t g = __ldg(gather_idx + row);
                if (MR_IN_RANGE(g, nrows, 304)) {
                    r[u] = ld_stream_v4(token_data + g * row_stride + 16 * o);
                    dst[u] = row * row_bytes + 16 * o;
                    if (is_int8 && o == 0) {
                        const uint8_t* sp = scales ? scales + g * scale_stride : token_data + g * row_stride + row_bytes;
                        dyn[row] = *reinterpret_cast<const float*>(sp);
                    }
                }
            }
            // the next vector of this thread: kGatherThreads vectors further on
            // (rows of at least kGatherThreads vectors: at most one row
            // boundary per step; SHORT rows: a division, not up to
            // kGatherThreads subtractions)
            o += kGatherThreads;
            if (!SHORT) {
                while (o >= nvec) {
                    o -= nvec;
                    ++row;
                }
            } else if (o >= nvec) {
                const int q = (int)o / (int)nvec;
                row += q;
                o -= (int64_t)q * nvec;
            }
        }
#pragma unroll
        for (int u = 0; u < kGatherVPT; ++u)
            if (dst[u] >= 0) st_stream_v4(y + dst[u], r[u]);
    }
}

// Whether the flat gather serves these rows: 16-byte vectors of the output
// (y and the row length multiples of 16 bytes, at least kGatherFlatMinVectors
// of them over the Y rows: a few small rows go faster through the warp kernel)
// from a 16-byte aligned buffer and row stride; with INT8, a separate scale
// array of aligned floats.
constexpr int64_t kGatherFlatMinVectors = 65536;

inline bool gather_flat_ok(const void* token_data, int64_t row_stride, int64_t row_bytes, const void* y,
                           const void* scales, int64_t scale_stride, int64_t rows) {
    if ((row_bytes & 15) != 0 || (row_stride & 15) != 0) return false;
    if (((reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(token_data)) & 15u) != 0) return false;
    if (scales && (((reinterpret_cast<uintptr_t>(scales) | (uintptr_t)scale_stride) & 3u) != 0)) return false;
    return rows * (row_bytes >> 4) >= kGatherFlatMinVectors;
}

// The same for rows whose address the kernel reads from device memory: the
// host checks the shape and y; the kernel checks the base (see above).
inline bool gather_flat_ok_device_base(int64_t row_stride, int64_t row_bytes, const void* y, int64_t rows) {
    if ((row_bytes & 15) != 0 || (row_stride & 15) != 0) return false;
    if ((reinterpret_cast<uintptr_t>(y) & 15u) != 0) return false;
    return rows * (row_bytes >> 4) >= kGatherFlatMinVectors;
}

// The flat gather's instantiation for rows of row_bytes.
inline auto gather_flat_kernel_for(int64_t row_bytes) {
    return (row_bytes >> 4) < kGatherThreads ? batching_gather_flat_kernel<true>
                                             : batching_gather_flat_kernel<false>;
}

// Blocks of the flat gather for up to `rows` output rows (every vector of
// them in one launch when that fits a grid).
inline unsigned gather_flat_grid(int64_t rows, int64_t row_bytes) {
    const int64_t per_block = (int64_t)kGatherThreads * kGatherVPT;
    const int64_t vecs = rows * (row_bytes >> 4);
    int64_t g = (vecs + per_block - 1) / per_block;
    if (g > 0x7fffffff) g = 0x7fffffff;
    if (g < 1) g = 1;
    return (unsigned)g;
}

static inline int gather_grid(int64_t rows) {
    static int blocks_per_sm[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int bps = dev < 64 ? blocks_per_sm[dev] : 0;
    if (bps == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, batching_gather_kernel<7>, 256, 0) !=
                cudaSuccess || bps <= 0)
            bps = 4;
        if (dev < 64) blocks_per_sm[dev] = bps;
    }
    const int64_t want = (rows + 7) / 8;  // 8 warps per block, one row per warp
    const int64_t cap = (int64_t)device_sm_count() * bps;
    int64_t g = want < cap ? want : cap;
    return (int)(g > 0 ? g : 1);
}

}  // namespace mr
