// The unpermute's gather-reduce kernels ("MoeTokenUnpermuteWithRoutingMap
// 算子全解析", 功能说明与计算公式 branches (1)-(4), and Kernel 实现: the
// IsValidInputIndex and prob != 0 skips, fp32 Cast/Muls/Add, the CAST_RINT
// back-cast), kept apart from the index work so that their source is one file.
#pragma once

#include "common.cuh"

namespace mr {

template <int DT>
__device__ __forceinline__ float ld_f32(const void* base, int64_t i) {
    if constexpr (DT == MR_DTYPE_F32) {
        return __ldg(reinterpret_cast<const float*>(base) + i);
    } else {
        const uint16_t b = __ldg(reinterpret_cast<const unsigned short*>(base) + i);
        return Elem<DT>::to_f32(b);
    }
}

// ---------------------------------------------------------------------------
// Gather-reduce. A token's contributing rows are those with a valid index
// and, with probs, a nonzero prob, taken in ascending slot (not padded) or
// row (padded) order; they are added in fp32, acc = acc + f32(x) * f32(p),
// each operation rounded on its own, then cast once with RNE.
// ---------------------------------------------------------------------------
constexpr int kListCap = 512;   // list entries per pass of the element-wise kernel
constexpr int kRedUnroll = 4;   // rows in flight per warp step
constexpr int kRedVQ = 2;       // 16-byte vectors per lane per hidden chunk
constexpr int kRedRun = 2;      // hidden chunks per work unit (one slot-list read) when the
                                // units of that length still fill the resident warps, else 1

template <bool HAS_PROBS, bool PADDED, int PDT>
__device__ __forceinline__ int build_list(int64_t c0, int64_t c1, const int32_t* __restrict__ si,
                                          int64_t rows, int64_t row_bytes,
                                          const void* __restrict__ pp,
                                          const int32_t* __restrict__ out_index, int64_t* s_row,
                                          float* s_w) {
    const int lane = threadIdx.x & 31;
    int cnt = 0;
    for (int64_t e0 = c0; e0 < c1; e0 += 32) {
        const int64_t e = e0 + lane;
        bool keep = false;
        int64_t r = 0;
        float w = 1.0f;
        if (e < c1) {
            if (PADDED) {
                r = out_index[e];
                keep = MR_IN_RANGE(r, rows, 401);
            } else {
                const int32_t v = si[e];
                keep = v >= 0 && (int64_t)v < rows;
                r = v;
            }
            if (HAS_PROBS && keep) {
                w = ld_f32<PDT>(pp, PADDED ? r : e);
                keep = w != 0.0f;
            }
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, keep);
        if (keep) {
            const int pos = cnt + __popc(bal & lanemask_lt());
            s_row[pos] = r * row_bytes;
            s_w[pos] = w;
        }
        cnt += __popc(bal);
    }
    return cnt;
}

template <int TDT>
struct Vec;
template <>
struct Vec<MR_DTYPE_F32> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void unpack(const uint4& v, float* x) {
        x[0] = __uint_as_float(v.x);
        x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z);
        x[3] = __uint_as_float(v.w);
    }
    static __device__ __forceinline__ uint4 pack(const float* a) {
        return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                          __float_as_uint(a[3]));
    }
};
template <int DT>
struct Vec16 {
    static constexpr int N = 8;
    static __device__ __forceinline__ void unpack(const uint4& v, float* x) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = Elem<DT>::to_f32((uint16_t)(w[k] & 0xffffu));
            x[2 * k + 1] = Elem<DT>::to_f32((uint16_t)(w[k] >> 16));
        }
    }
    static __device__ __forceinline__ uint4 pack(const float* a) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = (uint32_t)Elem<DT>::from_f32(a[2 * k]) |
                   ((uint32_t)Elem<DT>::from_f32(a[2 * k + 1]) << 16);
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <>
struct Vec<MR_DTYPE_F16> : Vec16<MR_DTYPE_F16> {};
template <>
struct Vec<MR_DTYPE_BF16> : Vec16<MR_DTYPE_BF16> {};

// ---------------------------------------------------------------------------
// Not padded, with probs, small routing map (T * Eu <= kSmallMapEntries): the
// weight of slot i is permuteProbs[i], the i-th element of probs.T selected
// by routingMap.T (expert-major, tokens ascending). Instead of a separate
// maskedSelect, every block of the gather-reduce rebuilds that order
// in shared memory -- 32-token column bitmasks and each expert's start -- and
// finds slot i's element by rank: the expert whose range of starts holds i,
// then the (i - start)-th routed token of its column. The warp that owns a
// token's first hidden chunk also writes permuteProbs for the token's slots
// (0 at and beyond the routed count).
// ---------------------------------------------------------------------------
constexpr int64_t kSmallMapEntries = 16384;

struct SmallMap {
    const int8_t* map;     // routingMap [T, Eu] (nullptr: weights come from pp)
    const uint8_t* probs;  // probs [T, Eu], PDT
    uint8_t* pp_out;       // permuteProbs [T * topk], PDT
    int64_t Eu;
};

__host__ __device__ inline int64_t small_map_smem_words(int64_t T, int64_t Eu) {
    return ((T + 31) / 32) * Eu + Eu + 1;  // bitmasks [nb][Eu], starts [Eu + 1]
}

// Every thread of the block takes part (block barriers and a block scan).
__device__ __forceinline__ void small_map_build(const SmallMap& sm, int64_t T, uint32_t* smask,
                                                uint32_t* sstart) {
    __shared__ uint32_t wsum[32];
    const int64_t Eu = sm.Eu;
    const int64_t nb = (T + 31) / 32;
    // one thread per (32-token block, expert) bitmask: 32 independent byte
    // loads, consecutive experts on consecutive threads
    for (int64_t item = threadIdx.x; item < nb * Eu; item += blockDim.x) {
        const int64_t blk = item / Eu;
        const int64_t e = item - blk * Eu;
        const int64_t t0 = blk * 32;
        int8_t m[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) m[j] = t0 + j < T ? sm.map[(t0 + j) * Eu + e] : (int8_t)0;
        uint32_t bits = 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j) bits |= (m[j] != 0 ? 1u : 0u) << j;
        smask[item] = bits;
    }
    __syncthreads();
    uint32_t carry = 0u;
    for (int64_t e0 = 0; e0 < Eu; e0 += blockDim.x) {  // exclusive scan of the column counts
        const int64_t e = e0 + threadIdx.x;
        uint32_t c = 0u;
        if (e < Eu)
            for (int64_t w = 0; w < nb; ++w) c += (uint32_t)__popc(smask[w * Eu + e]);
        uint32_t tot = 0u;
        const uint32_t x = block_exclusive_scan(c, wsum, &tot);
        if (e < Eu) sstart[e] = carry + x;
        carry += tot;
    }
    if (threadIdx.x == 0) sstart[Eu] = carry;
    __syncthreads();
}

// permuteProbs[i]: its element of probs (src, -1 when i >= the routed count)
// and its value.
template <int PDT>
__device__ __forceinline__ float small_map_weight(const SmallMap& sm, const uint32_t* smask,
                                                  const uint32_t* sstart, int64_t i, int64_t T,
                                                  int64_t& src) {
    const int64_t Eu = sm.Eu;
    if (i >= (int64_t)sstart[Eu]) {
        src = -1;
        return 0.0f;
    }
    int64_t lo = 0, hi = Eu;  // sstart[lo] <= i < sstart[hi]
    while (hi - lo > 1) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)sstart[mid] <= i) lo = mid;
        else hi = mid;
    }
    uint32_t r = (uint32_t)(i - (int64_t)sstart[lo]);
    int64_t w = 0;
    uint32_t m = smask[lo];
    uint32_t c = (uint32_t)__popc(m);
    while (r >= c) {  // the column holds more than r routed tokens
        r -= c;
        ++w;
        if (!MR_IN_RANGE(w, (T + 31) / 32, 406)) {
            src = -1;
            return 0.0f;
        }
        m = smask[w * Eu + lo];
        c = (uint32_t)__popc(m);
    }
    for (uint32_t k = 0; k < r; ++k) m &= m - 1u;  // drop the r lower set bits
    src = (w * 32 + (__ffs(m) - 1)) * Eu + lo;
    return ld_f32<PDT>(sm.probs, src);
}

template <int PDT>
__device__ __forceinline__ void small_map_store(const SmallMap& sm, int64_t i, int64_t src) {
    if (PDT == MR_DTYPE_F32) {
        reinterpret_cast<uint32_t*>(sm.pp_out)[i] =
            src < 0 ? 0u : __ldg(reinterpret_cast<const uint32_t*>(sm.probs) + src);
    } else {
        reinterpret_cast<uint16_t*>(sm.pp_out)[i] =
            src < 0 ? (uint16_t)0 : __ldg(reinterpret_cast<const unsigned short*>(sm.probs) + src);
    }
}

// One warp per work unit = (token, run of RUN consecutive chunks of 32*kRedVQ
// 16-byte vectors of the hidden dimension). The warp's lanes load up to 32 of
// the token's slots at a time (index and weight), a ballot keeps the
// contributing ones in ascending order, and the warp adds them kRedUnroll rows
// at a time, each lane owning kRedVQ vectors: no block barrier after the
// start, and shared memory only for the small-map weights (SMALL).
template <int TDT, int PDT, bool HAS_PROBS, bool PADDED, int RUN, bool SMALL>
__global__ void __launch_bounds__(256)
unpermute_reduce_warp_kernel(const uint8_t* __restrict__ permuted, int64_t rows, int64_t row_bytes,
                             int64_t nvec, int64_t chunks, const int32_t* __restrict__ si,
                             int64_t topk, const void* __restrict__ pp,
                             const int32_t* __restrict__ out_index, const int32_t* __restrict__ ptr,
                             int64_t T, uint8_t* __restrict__ out, SmallMap smap) {
    using V = Vec<TDT>;
    static_assert(!SMALL || (HAS_PROBS && !PADDED), "small-map weights are for the not-padded probs branch");
    extern __shared__ __align__(16) uint32_t red_smem[];
    uint32_t* smask = red_smem;
    uint32_t* sstart = red_smem + ((T + 31) / 32) * smap.Eu;
    pdl_enter();
    if constexpr (SMALL) small_map_build(smap, T, smask, sstart);
    const int lane = threadIdx.x & 31;
    // A work unit is a run of consecutive hidden chunks of one token: the
    // token's slot list is read once for the run.
    const int64_t runs = (chunks + RUN - 1) / RUN;
    const int64_t units = T * runs;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t unit = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; unit < units;
         unit += nw) {
        const int64_t t = unit / runs;
        const int64_t c0 = (unit - t * runs) * RUN;
        const int64_t c1 = c0 + RUN < chunks ? c0 + RUN : chunks;
        int64_t L0, L1;
        if (PADDED) {
            L0 = ptr[t];
            L1 = ptr[t + 1];
            // row pointers: 0 <= L0 <= L1 <= rows (padded: one entry per row)
            if (!MR_IN_RANGE(L1, rows + 1, 404) || !MR_IN_RANGE(L1 - L0, L1 + 1, 405)) L0 = L1 = 0;
        } else {
            L0 = t * topk;
            L1 = L0 + topk;
        }
        // this lane's entry of the list's first 32 (kept across the run)
        bool keep0 = false;
        int64_t roff0 = 0;
        float w0 = 1.0f;
        {
            const int64_t e = L0 + lane;
            if (e < L1) {
                int64_t r;
                if (PADDED) {
                    r = out_index[e];
                    keep0 = MR_IN_RANGE(r, rows, 402);
                } else {
                    const int32_t v = si[e];
                    keep0 = v >= 0 && (int64_t)v < rows;
                    r = v;
                }
                if constexpr (SMALL) {
                    int64_t src;
                    const float ws = small_map_weight<PDT>(smap, smask, sstart, e, T, src);
                    if (c0 == 0) small_map_store<PDT>(smap, e, src);
                    if (keep0) {
                        w0 = ws;
                        keep0 = w0 != 0.0f;
                    }
                } else if (HAS_PROBS && keep0) {
                    w0 = ld_f32<PDT>(pp, PADDED ? r : e);
                    keep0 = w0 != 0.0f;
                }
                roff0 = r * row_bytes;
            }
        }
        for (int64_t c = c0; c < c1; ++c) {
        const int64_t v0 = c * (32 * kRedVQ) + lane;
        float acc[kRedVQ][V::N];
#pragma unroll
        for (int q = 0; q < kRedVQ; ++q)
#pragma unroll
            for (int k = 0; k < V::N; ++k) acc[q][k] = 0.0f;

        for (int64_t g0 = L0; g0 < L1; g0 += 32) {
            // this lane's slot of the group: row offset and weight
            const int64_t e = g0 + lane;
            bool keep = keep0;
            int64_t roff = roff0;
            float w = w0;
            if (g0 != L0) {
                keep = false;
                roff = 0;
                w = 1.0f;
                if (e < L1) {
                    int64_t r;
                    if (PADDED) {
                        r = out_index[e];
                        keep = MR_IN_RANGE(r, rows, 403);
                    } else {
                        const int32_t v = si[e];
                        keep = v >= 0 && (int64_t)v < rows;
                        r = v;
                    }
                    if constexpr (SMALL) {
                        int64_t src;
                        const float ws = small_map_weight<PDT>(smap, smask, sstart, e, T, src);
                        if (c == 0) small_map_store<PDT>(smap, e, src);
                        if (keep) {
                            w = ws;
                            keep = w != 0.0f;
                        }
                    } else if (HAS_PROBS && keep) {
                        w = ld_f32<PDT>(pp, PADDED ? r : e);
                        keep = w != 0.0f;
                    }
                    roff = r * row_bytes;
                }
            }
            uint32_t bal = __ballot_sync(0xffffffffu, keep);
            while (bal) {
                int src[kRedUnroll];
                int cnt = 0;
#pragma unroll
                for (int u = 0; u < kRedUnroll; ++u) {
                    src[u] = bal ? __ffs(bal) - 1 : 0;
                    if (bal) {
                        bal &= bal - 1u;
                        ++cnt;
                    }
                }
                uint4 x[kRedUnroll][kRedVQ];
#pragma unroll
                for (int u = 0; u < kRedUnroll; ++u) {
                    const int64_t ro = __shfl_sync(0xffffffffu, roff, src[u]);
                    if (u < cnt) {
#pragma unroll
                        for (int q = 0; q < kRedVQ; ++q) {
                            const int64_t v = v0 + 32 * q;
                            if (v < nvec) x[u][q] = ld_stream_v4(permuted + ro + 16 * v);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kRedUnroll; ++u) {
                    const float wu = __shfl_sync(0xffffffffu, w, src[u]);
                    if (u < cnt) {
#pragma unroll
                        for (int q = 0; q < kRedVQ; ++q) {
                            const int64_t v = v0 + 32 * q;
                            if (v < nvec) {
                                float xs[V::N];
                                V::unpack(x[u][q], xs);
#pragma unroll
                                for (int k = 0; k < V::N; ++k)
                                    acc[q][k] = HAS_PROBS ? __fadd_rn(acc[q][k], __fmul_rn(xs[k], wu))
                                                          : __fadd_rn(acc[q][k], xs[k]);
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kRedVQ; ++q) {
            const int64_t v = v0 + 32 * q;
            if (v < nvec) st_stream_v4(out + t * row_bytes + 16 * v, V::pack(acc[q]));
        }
        }
    }
}

// Element-wise variant for rows that are not 16-byte vectors (odd H or
// buffers not 16-byte aligned; element alignment is required). Same list,
// same order, same arithmetic. One block per token; its list is built once
// (up to kListCap slots) and each thread adds kScalarPer elements at a time
// (their row loads issued together).
constexpr int kScalarPer = 4;
template <int TDT, int PDT, bool HAS_PROBS, bool PADDED>
__global__ void __launch_bounds__(256)
unpermute_reduce_scalar_kernel(const uint8_t* __restrict__ permuted, int64_t rows, int64_t H,
                               const int32_t* __restrict__ si, int64_t topk,
                               const void* __restrict__ pp, const int32_t* __restrict__ out_index,
                               const int32_t* __restrict__ ptr, int64_t T,
                               uint8_t* __restrict__ out) {
    __shared__ int64_t s_row[kListCap];
    __shared__ float s_w[kListCap];
    __shared__ int s_cnt;
    constexpr int es = TDT == MR_DTYPE_F32 ? 4 : 2;
    pdl_enter();
    const int64_t row_bytes = H * es;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        int64_t L0, L1;
        if (PADDED) {
            L0 = ptr[t];
            L1 = ptr[t + 1];
            // row pointers: 0 <= L0 <= L1 <= rows (padded: one entry per row)
            if (!MR_IN_RANGE(L1, rows + 1, 404) || !MR_IN_RANGE(L1 - L0, L1 + 1, 405)) L0 = L1 = 0;
        } else {
            L0 = t * topk;
            L1 = L0 + topk;
        }
        // a list of at most kListCap slots is built once for every hidden
        // step of the token; a longer one a part at a time, in each step
        const bool one_list = L1 - L0 <= kListCap;
        if (one_list && L1 > L0) {
            if (threadIdx.x < 32) {
                const int cnt = build_list<HAS_PROBS, PADDED, PDT>(L0, L1, si, rows, row_bytes, pp,
                                                                   out_index, s_row, s_w);
                if (threadIdx.x == 0) s_cnt = cnt;
            }
            __syncthreads();
        }
        // each thread adds kScalarPer elements, blockDim.x apart, at a time
        for (int64_t h0 = 0; h0 < H; h0 += (int64_t)blockDim.x * kScalarPer) {
            float acc[kScalarPer];
#pragma unroll
            for (int k = 0; k < kScalarPer; ++k) acc[k] = 0.0f;
            for (int64_t c0 = L0; c0 < L1; c0 += kListCap) {
                const int64_t c1 = c0 + kListCap < L1 ? c0 + kListCap : L1;
                if (!one_list) {
                    if (threadIdx.x < 32) {
                        const int cnt = build_list<HAS_PROBS, PADDED, PDT>(c0, c1, si, rows, row_bytes,
                                                                           pp, out_index, s_row, s_w);
                        if (threadIdx.x == 0) s_cnt = cnt;
                    }
                    __syncthreads();
                }
                const int cnt = s_cnt;
                for (int m = 0; m < cnt; ++m) {
                    const uint8_t* rp = permuted + s_row[m];
                    float x[kScalarPer];
#pragma unroll
                    for (int k = 0; k < kScalarPer; ++k) {
                        const int64_t h = h0 + threadIdx.x + (int64_t)k * blockDim.x;
                        x[k] = 0.0f;
                        if (h < H) {
                            if constexpr (TDT == MR_DTYPE_F32) {
                                x[k] = __ldg(reinterpret_cast<const float*>(rp + h * es));
                            } else {
                                x[k] = Elem<TDT>::to_f32(__ldg(reinterpret_cast<const unsigned short*>(rp + h * es)));
                            }
                        }
                    }
#pragma unroll
                    for (int k = 0; k < kScalarPer; ++k)
                        acc[k] = HAS_PROBS ? __fadd_rn(acc[k], __fmul_rn(x[k], s_w[m])) : __fadd_rn(acc[k], x[k]);
                }
                if (!one_list) __syncthreads();  // the next part overwrites the list
            }
#pragma unroll
            for (int k = 0; k < kScalarPer; ++k) {
                const int64_t h = h0 + threadIdx.x + (int64_t)k * blockDim.x;
                if (h < H) {
                    uint8_t* op = out + t * row_bytes + h * es;
                    if constexpr (TDT == MR_DTYPE_F32) {
                        *reinterpret_cast<float*>(op) = acc[k];
                    } else {
                        *reinterpret_cast<uint16_t*>(op) = Elem<TDT>::from_f32(acc[k]);
                    }
                }
            }
        }
        if (one_list && L1 > L0) __syncthreads();  // the next token's list overwrites it
    }
}

}  // namespace mr
