// Index sort of sortedIndices for the unpermute ("MoeTokenUnpermuteWithRoutingMap
// 算子全解析", 功能说明 (1)-(3) and 补充说明: outIndex and permuteTokenId; Kernel
// 实现: the padded prob lookup probs[sortedIndices[i] * num_experts + i /
// capacity]): the key of an entry, the scatter step of a counting-sort pass,
// the per-bucket fine sort of the two-level form and the CSR builder.
#pragma once

#include "csort.cuh"

namespace mr {

// Copy one element of 2 or 4 bytes (the probs dtype) without interpreting it.
__device__ __forceinline__ void copy_prob(uint8_t* dst, int64_t di, const uint8_t* src, int64_t si,
                                          int pes) {
    if (pes == 4) {
        reinterpret_cast<uint32_t*>(dst)[di] = __ldg(reinterpret_cast<const uint32_t*>(src) + si);
    } else {
        reinterpret_cast<uint16_t*>(dst)[di] = __ldg(reinterpret_cast<const unsigned short*>(src) + si);
    }
}
__device__ __forceinline__ void zero_prob(uint8_t* dst, int64_t di, int pes) {
    if (pes == 4) reinterpret_cast<uint32_t*>(dst)[di] = 0u;
    else reinterpret_cast<uint16_t*>(dst)[di] = 0;
}

// ---------------------------------------------------------------------------
// Stable sort of sortedIndices (LSD passes of the counting-sort engine, or a
// coarse pass followed by one block per coarse bucket).
// Full key: not padded (invalid first) v+1 for 0 <= v < rows, else 0;
//           padded (invalid last)      v   for 0 <= v < T,    else T.
// The coarse digit of the two-level sort keeps the invalid entries alone in a
// bucket of their own, so that their final places are known after the coarse
// pass: not padded, bucket 0 (1 + (key - 1) >> shift for the others); padded,
// the last bucket (key >> shift for the others).
// ---------------------------------------------------------------------------
struct RadixKey {
    const int32_t* si;        // pass 0 source
    const uint32_t* keys_in;  // later passes: full keys in the previous order
    int64_t limit;            // rows (not padded) or T (padded)
    int padded;
    int shift;
    uint32_t mask;
    int coarse_invalid_apart;  // two levels: digit as described above
    uint32_t invalid_bucket;   // padded, two levels: the last coarse bucket
    __device__ __forceinline__ uint32_t full(int64_t i) const {
        if (keys_in) return keys_in[i];
        const int32_t v = si[i];
        const bool ok = v >= 0 && (int64_t)v < limit;
        if (padded) return ok ? (uint32_t)v : (uint32_t)limit;
        return ok ? (uint32_t)v + 1u : 0u;
    }
    __device__ __forceinline__ int digit(uint32_t fk) const {
        if (coarse_invalid_apart) {
            if (padded) return fk == (uint32_t)limit ? (int)invalid_bucket : (int)(fk >> shift);
            return fk == 0u ? 0 : (int)(1u + ((fk - 1u) >> shift));
        }
        return (int)((fk >> shift) & mask);
    }
    __device__ __forceinline__ int operator()(int64_t i) const { return digit(full(i)); }
};

// The padded probs lookup of the first pass (pp != nullptr): it reads the same
// sortedIndices element as the key.
struct PaddedProbs {
    const uint8_t* probs;
    uint8_t* pp;
    int64_t Eu, cap;
    int pes;
};

// The scatter step of one sort pass for item i at position d: the full key
// and the item's original index move to d (every pass but the last); the last
// pass writes outIndex and permuteTokenId instead. The first pass of a padded
// sort with probs also writes permuteProbs[i]. In the coarse pass of the
// two-level sort an invalid entry is already in its final place (its bucket,
// first when not padded and last when padded, keeps the original order): it
// writes outIndex and permuteTokenId at once (final_index, final_ptid).
struct RadixScatter {
    RadixKey kf;
    const int32_t* idx_in;
    uint32_t* keys_out;
    int32_t* idx_out;
    int32_t* out_index;
    int32_t* ptid;
    int64_t topk;
    PaddedProbs pprobs;
    int32_t* final_index;
    int32_t* final_ptid;
    int64_t n;  // entries (and positions)
    __device__ __forceinline__ void operator()(int64_t i, int, uint32_t d, uint32_t) const {
        if (!MR_IN_RANGE(d, n, 501)) return;
        if (pprobs.pp) {
            // permuteProbs[i] = probs[sortedIndices[i], i // capacity], 0 if invalid
            const int32_t v = kf.si[i];
            if (v >= 0 && (int64_t)v < kf.limit) {
                copy_prob(pprobs.pp, i, pprobs.probs, (int64_t)v * pprobs.Eu + i / pprobs.cap, pprobs.pes);
            } else {
                zero_prob(pprobs.pp, i, pprobs.pes);
            }
        }
        const uint32_t fk = kf.full(i);
        const int32_t idx = idx_in ? idx_in[i] : (int32_t)i;
        if (final_index && fk == (kf.padded ? (uint32_t)kf.limit : 0u)) {
            final_index[d] = idx;
            final_ptid[d] = kf.padded ? kf.si[idx] : (int32_t)(idx / topk);
            return;
        }
        keys_out[d] = fk;
        if (out_index) {
            out_index[d] = idx;
            ptid[d] = kf.padded ? kf.si[idx] : (int32_t)(idx / topk);
        } else {
            idx_out[d] = idx;
        }
    }
};

__global__ void __launch_bounds__(256)
radix_scatter_kernel(RadixKey kf, int64_t n, int B, CsortBufs cs, RadixScatter sc) {
    pdl_enter();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int digit = kf(i);
        if (!MR_IN_RANGE(digit, B, 502)) continue;
        sc(i, digit, csort_dest(digit, i, cs, B), 0u);
    }
}

// Second level of the two-level sort (one block per coarse bucket). The first
// level is a counting-sort pass on the coarse digit, which leaves each coarse
// bucket [cstart[c], cstart[c+1]) in original order. The block sorts its
// bucket stably by the low s bits of its key (F = 2^s fine keys): a histogram
// and its scan give the fine starts, and 256-item chunks taken in order are
// ranked by key with warp matches, per-warp counters and a running count per
// fine key.
//   padded:     digit key >> s, fine key = key & (F-1); the fine starts are
//               the CSR row pointers ptr[c*F + f] (the last block also writes
//               ptr[T], the start of the invalid bucket that follows it);
//               permuteTokenId = the value.
//   not padded: block b sorts bucket b+1 by (key - 1) & (F-1);
//               permuteTokenId = original index / topK.
// The coarse pass has placed the invalid entries' bucket, which no block takes.
constexpr int kFineThreads = 256;
constexpr int kFineWarps = kFineThreads / 32;
constexpr int kMaxFineBits = 10;

// Fine sort of coarse bucket c, the entries [lo, hi) of keys / idx (in
// original order), by the low `shift` bits of the key; fsm holds
// (2 + kFineWarps) << shift words of shared memory. The last padded bucket
// (`last`) also writes ptr[T]. permuteTokenId of a valid padded entry is its
// full key (its value), so it needs no second read of sortedIndices.
template <bool PADDED>
__device__ __forceinline__ void fine_sort_bucket(int c, uint32_t lo, uint32_t hi, bool last,
                                                 const uint32_t* __restrict__ keys,
                                                 const int32_t* __restrict__ idx, int shift, int64_t T,
                                                 int64_t topk, const int32_t* __restrict__ si,
                                                 int32_t* __restrict__ out_index, int32_t* __restrict__ ptid,
                                                 int32_t* __restrict__ ptr, uint32_t* fsm, int64_t n) {
    const int F = 1 << shift;
    uint32_t* hist = fsm;                     // [F] counts, then fine starts
    uint32_t* running = fsm + F;              // [F] items placed so far
    uint32_t* wcnt = fsm + 2 * F;             // [kFineWarps][F] this chunk's counts
    const int warp = threadIdx.x >> 5;
    const uint32_t fmask = (uint32_t)F - 1u;
    const uint32_t kofs = PADDED ? 0u : 1u;
    for (int i = threadIdx.x; i < (2 + kFineWarps) * F; i += kFineThreads) fsm[i] = 0u;
    __syncthreads();
    for (uint32_t i = lo + threadIdx.x; i < hi; i += kFineThreads)
        atomicAdd(&hist[(__ldcg(keys + i) - kofs) & fmask], 1u);
    __syncthreads();
    if (threadIdx.x == 0) {  // F <= 1024 counts: a serial scan is a few hundred cycles
        uint32_t run = 0u;
        for (int f = 0; f < F; ++f) {
            const uint32_t h = hist[f];
            hist[f] = run;
            run += h;
        }
    }
    __syncthreads();
    if (PADDED) {  // row pointers of the tokens in this coarse bucket
        for (int f = threadIdx.x; f < F; f += kFineThreads) {
            const int64_t t = (int64_t)c * F + f;
            if (t < T) ptr[t] = (int32_t)(lo + hist[f]);
        }
        if (last && threadIdx.x == 0) ptr[T] = (int32_t)hi;
    }
    const uint32_t lt = lanemask_lt();
    for (uint32_t base = lo; base < hi; base += kFineThreads) {
        const uint32_t i = base + threadIdx.x;
        const bool in = i < hi;
        const uint32_t fk = in ? __ldcg(keys + i) : 0u;
        const int f = in ? (int)((fk - kofs) & fmask) : -1;
        const int32_t o = in ? __ldcg(idx + i) : 0;
        const uint32_t peers = __match_any_sync(0xffffffffu, f);
        const uint32_t below = __popc(peers & lt);
        const bool leader = in && below == 0u;
        if (leader) wcnt[warp * F + f] = __popc(peers);
        __syncthreads();
        if (in) {
            uint32_t r = below + running[f] + hist[f];
            for (int w = 0; w < warp; ++w) r += wcnt[w * F + f];
            const uint32_t pos = lo + r;
            if (MR_IN_RANGE(pos, hi, 503) && MR_IN_RANGE(o, n, 504)) {
                out_index[pos] = o;
                // padded, a valid entry's full key is its value sortedIndices[o]
                ptid[pos] = PADDED ? (int32_t)(fk) : (int32_t)(o / topk);
            }
        }
        __syncthreads();
        if (leader) {
            atomicAdd(&running[f], (uint32_t)__popc(peers));
            wcnt[warp * F + f] = 0u;
        }
        __syncthreads();
    }
}

template <bool PADDED>
__global__ void __launch_bounds__(kFineThreads)
fine_sort_kernel(const uint32_t* __restrict__ keys, const int32_t* __restrict__ idx,
                 const uint32_t* __restrict__ cstart, int shift, int64_t T, int64_t topk,
                 const int32_t* __restrict__ si, int32_t* __restrict__ out_index,
                 int32_t* __restrict__ ptid, int32_t* __restrict__ ptr, int64_t n) {
    extern __shared__ __align__(16) uint32_t fsm[];
    pdl_enter();
    const int c = PADDED ? (int)blockIdx.x : (int)blockIdx.x + 1;
    uint32_t lo = cstart[c], hi = cstart[c + 1];
    if (!MR_IN_RANGE(hi, n + 1, 505) || !MR_IN_RANGE(lo, (int64_t)hi + 1, 506)) lo = hi = 0u;
    fine_sort_bucket<PADDED>(c, lo, hi, c == (int)gridDim.x - 1, keys, idx, shift, T, topk, si, out_index,
                             ptid, ptr, fsm, n);
}

// ptr[t] = first position of the sorted keys with key >= t, t in [0, T].
__global__ void __launch_bounds__(256)
csr_from_keys_kernel(const uint32_t* __restrict__ keys, int64_t n, int64_t T,
                     int32_t* __restrict__ ptr) {
    pdl_enter();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p <= n; p += stride) {
        const int64_t prev = p > 0 ? (int64_t)keys[p - 1] : -1;
        const int64_t cur = p < n ? (int64_t)keys[p] : T + 1;
        const int64_t hi = cur < T ? cur : T;
        for (int64_t t = prev + 1; t <= hi; ++t) ptr[t] = (int32_t)p;
    }
}

}  // namespace mr
