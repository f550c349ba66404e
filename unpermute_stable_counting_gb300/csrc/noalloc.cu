// Batching for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory at call time: a plugin
// inside an inference engine that reserved all device memory when it started
// and forbids later allocations, or a latency-critical loop where the implicit
// device synchronisation of cudaMalloc/cudaFree is not acceptable. The regular
// ffnwb_batching needs a caller-provided workspace; this entry point instead
// uses a fixed scratch array compiled into the library. It allocates nothing:
// no cudaMalloc, no cudaFree, no allocating library routine.
//
// Costs and rules:
//  * The array (MR_NOALLOC_SCRATCH_BYTES) occupies device memory on a GPU from
//    the moment the library's code is loaded there until the process exits.
//    Under CUDA's default lazy module loading that happens at the first call
//    on the device (the address lookup below loads it), so the first call on
//    each device may allocate: a caller that must not allocate after its
//    start-up makes one call per device during start-up (before it reserves
//    the device's memory), or sets CUDA_MODULE_LOADING=EAGER so that loading
//    the library loads the array. Later calls allocate nothing.
//  * Every call on a device shares the one array. Calls whose work overlaps on
//    the GPU (for example on two streams at once) race on it; callers must
//    order such calls (one stream, or events between streams).
//  * The array keeps the last call's contents. The batching kernels write every
//    scratch word before they read it (the prefix kernel's ticket counter is
//    reset by the first kernel of each call; the one-launch sort writes its
//    count matrix before its grid barrier), so nothing has to be cleared.
//  * The first call on a device looks up the array's device address there
//    (cudaGetSymbolAddress, with that device current) and caches it. Make that
//    first call before any stream capture on the device. The cached address
//    belongs to the device's context: do not use the library across a
//    cudaDeviceReset.
#include <mutex>

#include "common.cuh"

namespace {

// Host code may not use this name as a device address: on the host it is a
// stand-in, so kernels receive the address looked up per device below.
static __device__ __align__(256) unsigned char g_batching_scratch[MR_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.
mr_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MR_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MR_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_batching_scratch) != cudaSuccess || p == nullptr)
            return MR_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MR_OK;
}

}  // namespace

extern "C" mr_status ffnwb_batching_noalloc(
    const int32_t* expertIds, int32_t layerId, const void* tokenData, int64_t tokenRowStride,
    const void* scales, int64_t scaleStride, const int32_t* sessionIdsIn,
    const int32_t* microBatchIdsIn, const int32_t* tokenIdsIn, int64_t expertNum,
    const int64_t* maxOutShape, int64_t tokenDtype, int64_t needSchedule, int64_t layerNum,
    void* y, int64_t* groupList, int32_t* sessionIds, int32_t* microBatchIds, int32_t* tokenIds,
    int32_t* expertOffsets, float* dynamicScale, int64_t* actualTokenNum,
    int32_t* sortedIndicesOut, void* stream) {
    uint64_t need = 0;
    mr_status st = ffnwb_batching_get_workspace_size(expertNum, maxOutShape, tokenDtype,
                                                     needSchedule, layerNum, &need);
    if (st != MR_OK) return st;
    if (need > (uint64_t)MR_NOALLOC_SCRATCH_BYTES) return MR_ERR_WORKSPACE;
    void* scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != MR_OK) return st;
    return ffnwb_batching(expertIds, layerId, tokenData, tokenRowStride, scales, scaleStride,
                          sessionIdsIn, microBatchIdsIn, tokenIdsIn, expertNum, maxOutShape,
                          tokenDtype, needSchedule, layerNum, y, groupList, sessionIds,
                          microBatchIds, tokenIds, expertOffsets, dynamicScale, actualTokenNum,
                          sortedIndicesOut, scratch, (uint64_t)MR_NOALLOC_SCRATCH_BYTES, stream);
}
