// FFN-worker batching on GB300.
//
// "aclnnFfnWorkerBatching", 功能说明 steps 2-4 and 计算公式:
//   gather_idx, _ = sort(expert_ids_in)   (masked slots keyed large)
//   y[i] = token_data[gather_idx[i]]      (+ the fp32 dynamic scale in INT8 mode)
//   group_list[e] = [expert_id_e, expert_token_num_e]
//   actual_token_num = sum_e expert_token_num_e
//
// Launch sequence on the caller's stream (all PDL-chained):
//   1. csort rank    : stable in-tile ranks and tile histograms of the keys
//   2. csort prefix  : per-key tile offsets, key starts, group_list and
//                      actual_token_num (replaces the page's single-core
//                      jump-point scan)
//   3. scatter       : every slot's output row; the four int32 id outputs,
//                      gather_idx (workspace) and the optional slot -> row map
//   4. row gather    : y rows (and dynamic scales), one warp per row,
//                      16-byte streaming loads/stores when aligned
// With MR_BATCHING_FULL_TAIL the scatter and the gather also serve the rows of
// the masked slots (keys equal to the sentinel): 计算公式 applied to every i.
#include <cstdio>
#include <cstdlib>

#include "batching.cuh"



namespace mr {
MR_CHECK_ACCESSOR(batching)
}  // namespace mr

using namespace mr;

extern "C" mr_status ffnwb_batching_get_workspace_size(int64_t expertNum, const int64_t* maxOutShape,
                                                        int64_t tokenDtype, int64_t needSchedule,
                                                        int64_t layerNum, uint64_t* workspaceSize) {
    if (!workspaceSize) return MR_ERR_PARAM_NULLPTR;
    BatchPlan p;
    const mr_status st = plan_batching(expertNum, maxOutShape, tokenDtype, needSchedule, layerNum, &p);
    if (st != MR_OK) return st;
    *workspaceSize = p.ws_bytes;
    return MR_OK;
}

extern "C" mr_status ffnwb_batching_ex(const int32_t* expertIds, int32_t layerId,
                                       const void* tokenData, int64_t tokenRowStride,
                                       const void* scales, int64_t scaleStride,
                                       const int32_t* sessionIdsIn, const int32_t* microBatchIdsIn,
                                       const int32_t* tokenIdsIn, int64_t expertNum,
                                       const int64_t* maxOutShape, int64_t tokenDtype,
                                       int64_t needSchedule, int64_t layerNum, void* y,
                                       int64_t* groupList, int32_t* sessionIds,
                                       int32_t* microBatchIds, int32_t* tokenIds,
                                       int32_t* expertOffsets, float* dynamicScale,
                                       int64_t* actualTokenNum, int32_t* sortedIndicesOut,
                                       uint32_t flags, void* workspace, uint64_t workspaceSize,
                                       void* stream) {
    BatchPlan p;
    mr_status st = plan_batching(expertNum, maxOutShape, tokenDtype, needSchedule, layerNum, &p);
    if (st != MR_OK) return st;
    if (flags & ~(uint32_t)MR_BATCHING_FULL_TAIL) return MR_ERR_PARAM_INVALID;
    // keys below this bound have a token row to gather: the experts', and the
    // sentinel's too with the whole-tail option
    const int row_keys = (int)p.E + ((flags & MR_BATCHING_FULL_TAIL) ? 1 : 0);
    if (!expertIds || !tokenData || !sessionIdsIn || !microBatchIdsIn || !y || !groupList ||
        !sessionIds || !microBatchIds || !tokenIds || !expertOffsets || !actualTokenNum)
        return MR_ERR_PARAM_NULLPTR;
    const bool int8 = p.dtype == MR_DTYPE_INT8;
    if (int8 && !dynamicScale) return MR_ERR_PARAM_NULLPTR;
    if (!workspace && p.ws_bytes > 0) return MR_ERR_PARAM_NULLPTR;
    if (layerId < 0 || layerId >= p.L) return MR_ERR_PARAM_INVALID;
    const int64_t need_stride = p.row_bytes + ((int8 && !scales) ? 4 : 0);
    if (tokenRowStride < need_stride) return MR_ERR_PARAM_INVALID;
    if (int8 && scales && scaleStride < 4) return MR_ERR_PARAM_INVALID;
    if (workspaceSize < p.ws_bytes) return MR_ERR_WORKSPACE;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* wp = reinterpret_cast<uint8_t*>(workspace);
    CsortBufs cs = csort_carve(wp, p.Y, p.B);
    int32_t* gather_idx = reinterpret_cast<int32_t*>(wp);
    wp += align_up((uint64_t)p.Y * 4u, 256);
    if (csort_coop_bytes(p.Y, p.B) > 0) cs.coop_counts = reinterpret_cast<uint32_t*>(wp);

    BatchKey kf{expertIds, (int32_t)(layerId * p.El), (int32_t)p.El, (int32_t)p.E};
    GroupListOut gl{groupList, actualTokenNum, (int)p.E};

    profile_mark(s, 0);
    BatchScatter<BatchKey> sc{kf, row_keys, sessionIdsIn, microBatchIdsIn, tokenIdsIn, sessionIds,
                              microBatchIds, tokenIds, expertOffsets, gather_idx, sortedIndicesOut, p.Y};
    MR_TRY_CUDA(batching_index(kf, p.Y, p.B, cs, gl, sc, s));
    profile_mark(s, 1);
    profile_mark(s, 2);
    const uint8_t* td = reinterpret_cast<const uint8_t*>(tokenData);
    const uint8_t* sp = reinterpret_cast<const uint8_t*>(scales);
    uint8_t* yb = reinterpret_cast<uint8_t*>(y);
    if (gather_flat_ok(tokenData, tokenRowStride, p.row_bytes, y, int8 ? scales : nullptr, scaleStride, p.Y)) {
        MR_TRY_CUDA(launch_pdl(gather_flat_kernel_for(p.row_bytes), dim3(gather_flat_grid(p.Y, p.row_bytes)),
                               dim3(kGatherThreads), 0, s, td, tokenRowStride, p.row_bytes, int8 ? 1 : 0, sp,
                               scaleStride, yb, dynamicScale, (const int32_t*)gather_idx,
                               (const uint32_t*)cs.bucket_start, row_keys, (const uint64_t*)nullptr, p.Y));
    } else {
        MR_TRY_CUDA(launch_pdl(batching_gather_kernel<7>, dim3(gather_grid(p.Y)), dim3(256), 0, s, td,
                               tokenRowStride, p.row_bytes, int8 ? 1 : 0, sp, scaleStride, yb, dynamicScale,
                               gather_idx, cs.bucket_start, row_keys, (const uint64_t*)nullptr, p.Y));
    }
    profile_mark(s, 3);
    MR_TRY_CUDA(cudaGetLastError());
    return MR_OK;
}

extern "C" mr_status ffnwb_batching(const int32_t* expertIds, int32_t layerId, const void* tokenData,
                                    int64_t tokenRowStride, const void* scales, int64_t scaleStride,
                                    const int32_t* sessionIdsIn, const int32_t* microBatchIdsIn,
                                    const int32_t* tokenIdsIn, int64_t expertNum,
                                    const int64_t* maxOutShape, int64_t tokenDtype,
                                    int64_t needSchedule, int64_t layerNum, void* y,
                                    int64_t* groupList, int32_t* sessionIds, int32_t* microBatchIds,
                                    int32_t* tokenIds, int32_t* expertOffsets, float* dynamicScale,
                                    int64_t* actualTokenNum, int32_t* sortedIndicesOut,
                                    void* workspace, uint64_t workspaceSize, void* stream) {
    return ffnwb_batching_ex(expertIds, layerId, tokenData, tokenRowStride, scales, scaleStride,
                             sessionIdsIn, microBatchIdsIn, tokenIdsIn, expertNum, maxOutShape,
                             tokenDtype, needSchedule, layerNum, y, groupList, sessionIds,
                             microBatchIds, tokenIds, expertOffsets, dynamicScale, actualTokenNum,
                             sortedIndicesOut, 0u, workspace, workspaceSize, stream);
}
