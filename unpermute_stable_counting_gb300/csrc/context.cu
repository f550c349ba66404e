// FFN-worker batching from a ScheduleContext, the page's own input form.
//
// "aclnnFfnWorkerBatching", 功能说明 step 1 and the structs of 调用示例: the
// 1024-byte packed ScheduleContext (CommonArea at byte 0, ControlArea at 128,
// AttentionArea at 256, FfnArea at 384) points, through FfnArea, to
// token_info_buf (one FfnDataDesc per (session, micro-batch) block, sessions
// outer: i32 flag, i32 layer_id, micro_batch_size * selected_expert_num i32
// expert ids) and token_data_buf (one row per slot, same order).
//
// The context lives in device memory and may be written by earlier work on
// the stream, so it is read on the device: the host never synchronises.
//
// Launch sequence (PDL-chained after a memset of the status word):
//   1. context_parse_kernel : one warp per block; with needSchedule = 1 lane 0
//      waits for the block's flag (bounded by a deadline on %globaltimer), then
//      the warp writes the slots' keys (block layer * E_l + id, or the sentinel),
//      session and micro-batch ids into the workspace
//   2-5. the counting-sort rank and prefix, the id scatter and the row gather
//      of the flat-array batching, the gather reading the token rows' address
//      from the context
#include <cstdio>
#include <cstdlib>

#include "batching.cuh"

namespace mr {

constexpr int kCtxCommonOffset = 0;
constexpr int kCtxFfnOffset = 384;
constexpr int kCtxTokenDataField = kCtxFfnOffset + 16;  // FfnArea.token_data_buf
constexpr int64_t kMaxWaitTimeoutUs = 60ll * 1000 * 1000;

__device__ __forceinline__ int32_t ld_acquire_sys(const int32_t* p) {
    int32_t v;
    asm volatile("ld.acquire.sys.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// The context's counts and buffers, and whether they describe slots that fit
// the outputs (every thread derives the same view).
struct CtxView {
    int64_t micro, per_block, blocks, slots, block_bytes;
    const uint8_t* info;
    bool valid;
};

__device__ __forceinline__ CtxView read_context(const uint8_t* ctx, int64_t Y, int32_t El,
                                                int64_t row_stride) {
    const uint32_t* common = reinterpret_cast<const uint32_t*>(ctx + kCtxCommonOffset);
    const uint64_t* ffn = reinterpret_cast<const uint64_t*>(ctx + kCtxFfnOffset);
    const int64_t sessions = common[0], micro = common[1], mbs = common[2], sel = common[3];
    const int64_t expert_num = common[4];
    CtxView v;
    v.micro = micro;
    v.info = reinterpret_cast<const uint8_t*>(ffn[0]);
    bool ok = sessions > 0 && micro > 0 && mbs > 0 && sel > 0 && expert_num == El;
    // slots = sessions * micro * mbs * sel must not exceed Y (each factor >= 1,
    // so checking every partial product keeps the arithmetic in range)
    int64_t p = sessions;
    ok = ok && p <= Y;
    p *= micro;
    ok = ok && p <= Y;
    const int64_t blocks = p;
    p *= mbs;
    ok = ok && p <= Y;
    p *= sel;
    ok = ok && p <= Y;
    v.blocks = ok ? blocks : 0;
    v.per_block = ok ? mbs * sel : 0;
    v.slots = ok ? p : 0;
    v.block_bytes = 8 + 4 * v.per_block;
    ok = ok && ffn[0] != 0 && ffn[2] != 0 && (ffn[0] & 3u) == 0 &&
         (int64_t)ffn[1] >= v.blocks * v.block_bytes && (int64_t)ffn[3] >= v.slots * row_stride;
    v.valid = ok;
    if (!ok) v.blocks = v.slots = v.per_block = 0;
    return v;
}

__global__ void __launch_bounds__(256)
context_parse_kernel(const uint8_t* __restrict__ ctx, int64_t Y, int32_t El, int32_t E,
                     int32_t L, int64_t row_stride, int need_schedule, int64_t timeout_ns,
                     int32_t* __restrict__ keys, int32_t* __restrict__ sess,
                     int32_t* __restrict__ micro_ids, int32_t* __restrict__ status) {
    pdl_enter();
    const CtxView v = read_context(ctx, Y, El, row_stride);
    const uint64_t deadline = global_timer_ns() + (uint64_t)timeout_ns;
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    if (!v.valid && status && blockIdx.x == 0 && threadIdx.x == 0) *status = -1;

    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < v.blocks; b += nw) {
        const int32_t* desc = reinterpret_cast<const int32_t*>(v.info + b * v.block_bytes);
        int ready = 1;
        if (need_schedule && lane == 0) {
            while (ld_acquire_sys(desc) != 1) {
                if (global_timer_ns() > deadline) {
                    ready = 0;
                    break;
                }
                __nanosleep(500);
            }
            if (!ready && status) atomicAdd(status, 1);
        }
        ready = __shfl_sync(0xffffffffu, ready, 0);
        const int32_t layer = desc[1];
        const bool layer_ok = ready && layer >= 0 && layer < L;
        const int32_t s_id = (int32_t)(b / v.micro);
        const int32_t m_id = (int32_t)(b % v.micro);
        for (int64_t j = lane; j < v.per_block; j += 32) {
            const int64_t g = b * v.per_block + j;
            if (!MR_IN_RANGE(g, Y, 801)) continue;
            const int32_t id = desc[2 + j];
            keys[g] = (layer_ok && id >= 0 && id < El) ? layer * El + id : E;
            sess[g] = s_id;
            micro_ids[g] = m_id;
        }
    }
    // output rows past the context's slots belong to the masked tail; their
    // key E + 1 sorts them after the context's masked slots, which (key E)
    // still have a token row
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = v.slots + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < Y; g += stride) {
        keys[g] = E + 1;
        sess[g] = 0;
        micro_ids[g] = 0;
    }
}

static mr_status plan_context(int64_t expertNum, const int64_t* maxOutShape, int64_t tokenDtype,
                              int64_t needSchedule, int64_t layerNum, BatchPlan* p,
                              uint64_t* ws) {
    if (needSchedule != 0 && needSchedule != 1) return MR_ERR_PARAM_INVALID;
    const mr_status st = plan_batching(expertNum, maxOutShape, tokenDtype, 0, layerNum, p);
    if (st != MR_OK) return st;
    p->B = (int)p->E + 2;  // experts, the masked sentinel E, and E + 1 for rows with no slot
    p->ws_bytes = csort_workspace_bytes(p->Y, p->B) + align_up((uint64_t)p->Y * 4u, 256);
    *ws = p->ws_bytes + 3 * align_up((uint64_t)p->Y * 4u, 256) + csort_coop_bytes(p->Y, p->B);
    return MR_OK;
}

MR_CHECK_ACCESSOR(context)

}  // namespace mr

using namespace mr;

extern "C" mr_status ffnwb_batching_context_get_workspace_size(int64_t expertNum,
                                                                const int64_t* maxOutShape,
                                                                int64_t tokenDtype,
                                                                int64_t needSchedule,
                                                                int64_t layerNum,
                                                                uint64_t* workspaceSize) {
    if (!workspaceSize) return MR_ERR_PARAM_NULLPTR;
    BatchPlan p;
    uint64_t ws = 0;
    const mr_status st = plan_context(expertNum, maxOutShape, tokenDtype, needSchedule, layerNum,
                                      &p, &ws);
    if (st != MR_OK) return st;
    *workspaceSize = ws;
    return MR_OK;
}

extern "C" mr_status ffnwb_batching_context_ex(
    const void* scheduleContext, int64_t expertNum, const int64_t* maxOutShape, int64_t tokenDtype,
    int64_t needSchedule, int64_t layerNum, int64_t waitTimeoutUs, void* y, int64_t* groupList,
    int32_t* sessionIds, int32_t* microBatchIds, int32_t* tokenIds, int32_t* expertOffsets,
    float* dynamicScale, int64_t* actualTokenNum, int32_t* scheduleStatus, uint32_t flags,
    void* workspace, uint64_t workspaceSize, void* stream) {
    BatchPlan p;
    uint64_t ws = 0;
    mr_status st = plan_context(expertNum, maxOutShape, tokenDtype, needSchedule, layerNum, &p, &ws);
    if (st != MR_OK) return st;
    if (flags & ~(uint32_t)MR_BATCHING_FULL_TAIL) return MR_ERR_PARAM_INVALID;
    const int row_keys = (int)p.E + ((flags & MR_BATCHING_FULL_TAIL) ? 1 : 0);
    if (!scheduleContext || !y || !groupList || !sessionIds || !microBatchIds || !tokenIds ||
        !expertOffsets || !actualTokenNum)
        return MR_ERR_PARAM_NULLPTR;
    const bool int8 = p.dtype == MR_DTYPE_INT8;
    if (int8 && !dynamicScale) return MR_ERR_PARAM_NULLPTR;
    if (!workspace) return MR_ERR_PARAM_NULLPTR;
    if (waitTimeoutUs < 0 || waitTimeoutUs > kMaxWaitTimeoutUs) return MR_ERR_PARAM_INVALID;
    if ((reinterpret_cast<uintptr_t>(scheduleContext) & 7u) != 0) return MR_ERR_PARAM_INVALID;
    if (workspaceSize < ws) return MR_ERR_WORKSPACE;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* wp = reinterpret_cast<uint8_t*>(workspace);
    CsortBufs cs = csort_carve(wp, p.Y, p.B);
    int32_t* gather_idx = reinterpret_cast<int32_t*>(wp);
    wp += align_up((uint64_t)p.Y * 4u, 256);
    int32_t* keys = reinterpret_cast<int32_t*>(wp);
    wp += align_up((uint64_t)p.Y * 4u, 256);
    int32_t* sess = reinterpret_cast<int32_t*>(wp);
    wp += align_up((uint64_t)p.Y * 4u, 256);
    int32_t* micro = reinterpret_cast<int32_t*>(wp);
    wp += align_up((uint64_t)p.Y * 4u, 256);
    if (csort_coop_bytes(p.Y, p.B) > 0) cs.coop_counts = reinterpret_cast<uint32_t*>(wp);

    const uint8_t* ctx = reinterpret_cast<const uint8_t*>(scheduleContext);
    const int64_t row_stride = p.row_bytes + (int8 ? 4 : 0);
    const int64_t want = (p.Y + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    const int grid = (int)(want < cap ? (want > 0 ? want : 1) : cap);

    profile_mark(s, 0);
    if (scheduleStatus) MR_TRY_CUDA(cudaMemsetAsync(scheduleStatus, 0, sizeof(int32_t), s));
    MR_TRY_CUDA(launch_pdl(context_parse_kernel, dim3(grid), dim3(256), 0, s, ctx, p.Y,
                           (int32_t)p.El, (int32_t)p.E, (int32_t)p.L, row_stride,
                           (int)needSchedule, waitTimeoutUs * 1000, keys, sess, micro,
                           scheduleStatus));
    KeyArray kf{keys, (int32_t)p.E};
    GroupListOut gl{groupList, actualTokenNum, (int)p.E};
    BatchScatter<KeyArray> sc{kf, row_keys, sess, micro, nullptr, sessionIds, microBatchIds, tokenIds,
                              expertOffsets, gather_idx, nullptr, p.Y};
    MR_TRY_CUDA(batching_index(kf, p.Y, p.B, cs, gl, sc, s));
    profile_mark(s, 1);
    profile_mark(s, 2);
    // the token rows' address is the context's token_data_buf, read on the
    // device; 16-byte rows take the flat gather (which checks the address's
    // alignment itself), INT8 rows with their interleaved scale the warp kernel
    const uint64_t* td_loc = reinterpret_cast<const uint64_t*>(ctx + kCtxTokenDataField);
    uint8_t* yb = reinterpret_cast<uint8_t*>(y);
    if (!int8 && gather_flat_ok_device_base(row_stride, p.row_bytes, y, p.Y)) {
        MR_TRY_CUDA(launch_pdl(gather_flat_kernel_for(p.row_bytes), dim3(gather_flat_grid(p.Y, p.row_bytes)),
                               dim3(kGatherThreads), 0, s, (const uint8_t*)nullptr, row_stride, p.row_bytes, 0,
                               (const uint8_t*)nullptr, (int64_t)4, yb, dynamicScale,
                               (const int32_t*)gather_idx, (const uint32_t*)cs.bucket_start, row_keys, td_loc,
                               p.Y));
    } else {
        MR_TRY_CUDA(launch_pdl(batching_gather_kernel<7>, dim3(gather_grid(p.Y)), dim3(256), 0, s,
                               (const uint8_t*)nullptr, row_stride, p.row_bytes, int8 ? 1 : 0,
                               (const uint8_t*)nullptr, (int64_t)4, yb, dynamicScale,
                               (const int32_t*)gather_idx, (const uint32_t*)cs.bucket_start, row_keys,
                               td_loc, p.Y));
    }
    profile_mark(s, 3);
    MR_TRY_CUDA(cudaGetLastError());
    return MR_OK;
}

extern "C" mr_status ffnwb_batching_context(
    const void* scheduleContext, int64_t expertNum, const int64_t* maxOutShape, int64_t tokenDtype,
    int64_t needSchedule, int64_t layerNum, int64_t waitTimeoutUs, void* y, int64_t* groupList,
    int32_t* sessionIds, int32_t* microBatchIds, int32_t* tokenIds, int32_t* expertOffsets,
    float* dynamicScale, int64_t* actualTokenNum, int32_t* scheduleStatus, void* workspace,
    uint64_t workspaceSize, void* stream) {
    return ffnwb_batching_context_ex(scheduleContext, expertNum, maxOutShape, tokenDtype,
                                     needSchedule, layerNum, waitTimeoutUs, y, groupList,
                                     sessionIds, microBatchIds, tokenIds, expertOffsets,
                                     dynamicScale, actualTokenNum, scheduleStatus, 0u, workspace,
                                     workspaceSize, stream);
}
