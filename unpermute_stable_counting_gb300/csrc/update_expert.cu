// MoeUpdateExpert on GB300: logical -> physical expert ids through the EPLB
// table, and pruning of each token's experts by a scale threshold.
//
// "MoeUpdateExpert", 功能说明 and 参数说明:
//   balancedExpertIds[b,k] = eplbTable[e, 1 + c], e = expertIds[b,k],
//     c = localRankId mod count (balanceMode 0, by rank)
//     c = b mod count          (balanceMode 1, by token)
//     count = eplbTable[e, 0]; -1 when e is outside [0, moeExpertNum) or
//     count outside [1, F - 1], so no read leaves the table
//   balancedActiveMask[b,k] = activeMask[b] and not (scale[b,k] < threshold[k])
//
// The op is at most 512 x 16 elements: one element per thread, one launch of
// a few blocks. Each element is a chain of three dependent loads (id, count,
// instance), so the call is bound by launch and memory latency, not by
// bandwidth; every tensor is addressed through element strides, so strided
// (non-contiguous) views need no copy.
#include "common.cuh"

namespace mr {

// Element strides, in the order of the header: expertIds (b, k), eplbTable
// (e, f), scales (b, k), threshold (k), activeMask (b), balancedExpertIds
// (b, k), balancedActiveMask (b, k).
struct UpdateStrides {
    int64_t ids_b, ids_k, tab_e, tab_f, sc_b, sc_k, thr_k, act_b, out_b, out_k, msk_b, msk_k;
};

template <typename Id>
__global__ void __launch_bounds__(256)
    update_expert_kernel(const Id* __restrict__ ids, const int32_t* __restrict__ table,
                         const void* __restrict__ scales, int scales_dt,
                         const float* __restrict__ thr, const uint8_t* __restrict__ active,
                         int64_t BS, int64_t K, int64_t E, int64_t F, int64_t local_rank,
                         int mode, UpdateStrides st, Id* __restrict__ out,
                         uint8_t* __restrict__ mask) {
    pdl_enter();
    const int64_t n = BS * K;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / K;
        const int64_t k = i - b * K;
        const int64_t e = (int64_t)ids[b * st.ids_b + k * st.ids_k];
        int64_t r = -1;
        if (e >= 0 && e < E) {
            const int32_t* row = table + e * st.tab_e;
            const int64_t count = row[0];
            if (count >= 1 && count <= F - 1) {
                const int64_t c = (mode == 0 ? local_rank : b) % count;
                r = row[(1 + c) * st.tab_f];
            }
        }
        out[b * st.out_b + k * st.out_k] = (Id)r;
        if (mask) {
            const bool on = active ? active[b * st.act_b] != 0 : true;
            const float s = load_f32(scales, b * st.sc_b + k * st.sc_k, scales_dt);
            mask[b * st.msk_b + k * st.msk_k] = (on && !(s < thr[k * st.thr_k])) ? 1 : 0;
        }
    }
}

MR_CHECK_ACCESSOR(update_expert)

}  // namespace mr

using namespace mr;

extern "C" mr_status moe_update_expert(const void* expertIds, int32_t idDtype,
                                       const int32_t* eplbTable, const void* expertScales,
                                       int32_t scalesDtype, const float* pruningThreshold,
                                       const uint8_t* activeMask, int64_t BS, int64_t K,
                                       int64_t moeExpertNum, int64_t F, int64_t localRankId,
                                       int64_t worldSize, int64_t balanceMode,
                                       const int64_t* strides, void* balancedExpertIds,
                                       uint8_t* balancedActiveMask, void* stream) {
    if (idDtype != MR_DTYPE_INT32 && idDtype != MR_DTYPE_INT64) return MR_ERR_PARAM_INVALID;
    if (BS <= 0 || BS > MR_MAX_UPDATE_BS || K <= 0 || K > MR_MAX_UPDATE_K) return MR_ERR_PARAM_INVALID;
    if (moeExpertNum <= 0 || moeExpertNum > MR_MAX_UPDATE_EXPERTS || K > moeExpertNum)
        return MR_ERR_PARAM_INVALID;
    if (balanceMode == 0) {
        if (worldSize < 2 || worldSize > 768 || localRankId < 0 || localRankId >= worldSize)
            return MR_ERR_PARAM_INVALID;
    } else if (balanceMode == 1) {
        if (worldSize < 1 || worldSize > MR_MAX_UPDATE_EXPERTS) return MR_ERR_PARAM_INVALID;
    } else {
        return MR_ERR_PARAM_INVALID;
    }
    if (F < 2 || F > worldSize + 1) return MR_ERR_PARAM_INVALID;
    const bool has_scales = expertScales != nullptr;
    if (has_scales != (pruningThreshold != nullptr)) return MR_ERR_PARAM_NULLPTR;
    if (activeMask && !has_scales) return MR_ERR_PARAM_NULLPTR;
    if (has_scales && scalesDtype != MR_DTYPE_F16 && scalesDtype != MR_DTYPE_BF16 &&
        scalesDtype != MR_DTYPE_F32)
        return MR_ERR_PARAM_INVALID;
    if (!expertIds || !eplbTable || !balancedExpertIds) return MR_ERR_PARAM_NULLPTR;
    if (has_scales && !balancedActiveMask) return MR_ERR_PARAM_NULLPTR;

    UpdateStrides st{K, 1, F, 1, K, 1, 1, 1, K, 1, K, 1};
    if (strides) {
        for (int j = 0; j < 12; ++j) {
            // inputs may broadcast (stride 0); outputs advance
            if (strides[j] < (j < 8 ? 0 : 1) || strides[j] > (INT64_C(1) << 40))
                return MR_ERR_PARAM_INVALID;
        }
        st = UpdateStrides{strides[0], strides[1], strides[2], strides[3], strides[4], strides[5],
                           strides[6], strides[7], strides[8], strides[9], strides[10], strides[11]};
    }

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t n = BS * K;
    const int grid = (int)((n + 255) / 256);
    uint8_t* mask = has_scales ? balancedActiveMask : nullptr;
    profile_mark(s, 0);
    if (idDtype == MR_DTYPE_INT32) {
        MR_TRY_CUDA(launch_pdl(update_expert_kernel<int32_t>, dim3(grid), dim3(256), 0, s,
                               reinterpret_cast<const int32_t*>(expertIds), eplbTable,
                               expertScales, (int)scalesDtype, pruningThreshold, activeMask, BS, K,
                               moeExpertNum, F, localRankId, (int)balanceMode, st,
                               reinterpret_cast<int32_t*>(balancedExpertIds), mask));
    } else {
        MR_TRY_CUDA(launch_pdl(update_expert_kernel<int64_t>, dim3(grid), dim3(256), 0, s,
                               reinterpret_cast<const int64_t*>(expertIds), eplbTable,
                               expertScales, (int)scalesDtype, pruningThreshold, activeMask, BS, K,
                               moeExpertNum, F, localRankId, (int)balanceMode, st,
                               reinterpret_cast<int64_t*>(balancedExpertIds), mask));
    }
    profile_mark(s, 1);
    MR_TRY_CUDA(cudaGetLastError());
    return MR_OK;
}
