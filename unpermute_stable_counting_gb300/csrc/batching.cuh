// Kernels and host planning shared by the batching entry points (flat arrays
// and ScheduleContext). Included by batching.cu and context.cu; the kernels
// have internal linkage in each translation unit.
#pragma once

#include "csort.cuh"
#include "csort_coop.cuh"
#include "gather.cuh"

namespace mr {


// key(s) = layer_id*E_l + id for 0 <= id < E_l, else the sentinel E.
struct BatchKey {
    const int32_t* ids;
    int32_t layer_base;  // layer_id * E_l
    int32_t El;
    int32_t E;
    __device__ __forceinline__ int operator()(int64_t s) const {
        const int32_t id = __ldg(ids + s);
        return (id >= 0 && id < El) ? layer_base + id : E;
    }
};

// Keys already built per slot (the ScheduleContext path); E is the sentinel.
struct KeyArray {
    const int32_t* keys;
    int32_t E;
    __device__ __forceinline__ int operator()(int64_t s) const { return __ldg(keys + s); }
};

// The scatter step for one slot s with key k at output row d (start = the
// first row of key k). Slots with key < kf.E are routed; keys in
// [kf.E, src_keys) are masked slots that still have a token row (their ids are
// looked up when the formula is applied to the whole tail); larger keys have
// no slot behind them.
template <class KeyFn>
struct BatchScatter {
    KeyFn kf;
    int src_keys;
    const int32_t* sess_in;
    const int32_t* micro_in;
    const int32_t* tok_in;
    int32_t* sess_out;
    int32_t* micro_out;
    int32_t* tok_out;
    int32_t* eoff_out;
    int32_t* gather_idx;
    int32_t* slot_row;
    int64_t n;  // slots (and output rows)
    // The slot's ids, loaded apart from the stores (the one-launch sort loads
    // them with the keys).
    struct Pre {
        int32_t sess, micro, tok;
    };
    __device__ __forceinline__ Pre load(int64_t s) const {
        return Pre{sess_in[s], micro_in[s], tok_in ? tok_in[s] : (int32_t)s};
    }
    __device__ __forceinline__ void store(int64_t s, int k, uint32_t d, uint32_t start, const Pre& p) const {
        if (!MR_IN_RANGE(d, n, 101)) return;
        gather_idx[d] = (int32_t)s;
        const bool routed = k < kf.E;
        const bool has_row = k < src_keys;
        sess_out[d] = has_row ? p.sess : -1;
        micro_out[d] = has_row ? p.micro : -1;
        tok_out[d] = has_row ? p.tok : -1;
        eoff_out[d] = routed ? (int32_t)(d - start) : -1;
        if (slot_row && MR_IN_RANGE(s, n, 102)) slot_row[s] = routed ? (int32_t)d : -1;
    }
    __device__ __forceinline__ void operator()(int64_t s, int k, uint32_t d, uint32_t start) const {
        Pre p{-1, -1, -1};
        if (k < src_keys) p = load(s);
        store(s, k, d, start, p);
    }
};

template <class KeyFn>
static __global__ void __launch_bounds__(256)
batching_scatter_kernel(KeyFn kf, int64_t Y, int B, CsortBufs cs, BatchScatter<KeyFn> sc) {
    pdl_enter();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < Y; s += stride) {
        const int k = kf(s);
        if (!MR_IN_RANGE(k, B, 103)) continue;
        sc(s, k, csort_dest(k, s, cs, B), cs.bucket_start[k]);
    }
}

// Index step of the batching: the counting sort of the slots and the scatter
// of the ids. One block for inputs of one tile; the one-launch cooperative
// form for up to kCoopMaxTiles of its tiles (a decode step: measured on
// GB300, 18432 slots index + gather 50.4 -> 47.5 us); otherwise the rank and
// prefix kernels, then the scatter kernel.
template <class KeyFn>
inline cudaError_t batching_index(KeyFn kf, int64_t Y, int B, const CsortBufs& cs, GroupListOut gl,
                                  const BatchScatter<KeyFn>& sc, cudaStream_t s) {
    if (Y <= kSortTile) return csort_single_tile(kf, Y, B, cs, gl, sc, s);  // one block
    cudaError_t e = csort_coop(kf, Y, B, cs.coop_counts, cs.bucket_start, gl, sc, s);
    if (e != cudaErrorNotSupported) return e;
    e = csort_run(kf, Y, B, cs, gl, s);
    if (e != cudaSuccess) return e;
    const int64_t want = (Y + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    const int grid = (int)(want < cap ? (want > 0 ? want : 1) : cap);
    return launch_pdl(batching_scatter_kernel<KeyFn>, dim3(grid), dim3(256), 0, s, kf, Y, B, cs, sc);
}

// ---------------------------------------------------------------------------
// Host planning
// ---------------------------------------------------------------------------


struct BatchPlan {
    int64_t A, BS, K1, H, Y, E, L, El;
    int dtype;
    int B;
    int64_t row_bytes;
    uint64_t ws_bytes;
};

static inline mr_status plan_batching(int64_t expertNum, const int64_t* maxOutShape, int64_t tokenDtype,
                               int64_t needSchedule, int64_t layerNum, BatchPlan* p) {
    if (!maxOutShape) return MR_ERR_PARAM_NULLPTR;
    const int64_t A = maxOutShape[0], BS = maxOutShape[1], K1 = maxOutShape[2], H = maxOutShape[3];
    if (expertNum <= 0 || expertNum > MR_MAX_EXPERT_NUM) return MR_ERR_PARAM_INVALID;
    if (A <= 0 || A > MR_MAX_A || BS <= 0 || K1 <= 0 || K1 > MR_MAX_TOPK1 || H <= 0)
        return MR_ERR_PARAM_INVALID;
    if (tokenDtype != MR_DTYPE_F16 && tokenDtype != MR_DTYPE_BF16 && tokenDtype != MR_DTYPE_INT8)
        return MR_ERR_PARAM_INVALID;
    if (needSchedule != 0 && needSchedule != 1) return MR_ERR_PARAM_INVALID;
    if (layerNum < 0 || layerNum > expertNum) return MR_ERR_PARAM_INVALID;
    const int64_t L = layerNum > 0 ? layerNum : 1;
    if (expertNum % L != 0) return MR_ERR_PARAM_INVALID;
    if (BS > (INT64_C(1) << 31) || A * BS > (INT64_C(1) << 31) || A * BS * K1 >= (INT64_C(1) << 31))
        return MR_ERR_PARAM_INVALID;
    if (H > (INT64_C(1) << 40)) return MR_ERR_PARAM_INVALID;
    if (needSchedule == 1) return MR_ERR_UNSUPPORTED;
    p->A = A;
    p->BS = BS;
    p->K1 = K1;
    p->H = H;
    p->Y = A * BS * K1;
    p->E = expertNum;
    p->L = L;
    p->El = expertNum / L;
    p->dtype = (int)tokenDtype;
    p->B = (int)expertNum + 1;
    p->row_bytes = H * (tokenDtype == MR_DTYPE_INT8 ? 1 : 2);
    p->ws_bytes = csort_workspace_bytes(p->Y, p->B) + align_up((uint64_t)p->Y * 4u, 256) +
                  csort_coop_bytes(p->Y, p->B);
    return MR_OK;
}


}  // namespace mr
