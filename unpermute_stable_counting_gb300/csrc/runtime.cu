// Host utilities of the reorder library: device queries, status text and the
// per-thread timing hooks used by benchmarks.
#include "common.cuh"

namespace mr {

namespace {
int g_sm_count[64] = {0};
thread_local cudaEvent_t g_events[16] = {nullptr};
thread_local int g_num_events = 0;
}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kNumSMsHint;
    if (dev >= 0 && dev < 64 && g_sm_count[dev] > 0) return g_sm_count[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = kNumSMsHint;
    if (dev >= 0 && dev < 64) g_sm_count[dev] = n;
    return n;
}

AuxStream* aux_stream(cudaStream_t caller, cudaError_t* err) {
    static std::mutex create_mu;
    static AuxStream* table[64][kMaxAuxStreams] = {{nullptr}};
    *err = cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(create_mu);
    AuxStream** row = table[dev];
    int i = 0;
    for (; i < kMaxAuxStreams && row[i]; ++i)
        if (row[i]->caller == caller) return row[i];
    if (i == kMaxAuxStreams) return nullptr;  // table full: side work in line
    int lo = 0, hi = 0;
    e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (e != cudaSuccess) {
        *err = e;
        return nullptr;
    }
    AuxStream* a = new AuxStream();
    a->caller = caller;
    a->stream = nullptr;
    a->fork = a->join = nullptr;
    if ((e = cudaStreamCreateWithPriority(&a->stream, cudaStreamNonBlocking, hi)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&a->fork, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&a->join, cudaEventDisableTiming)) != cudaSuccess) {
        if (a->fork) cudaEventDestroy(a->fork);
        if (a->stream) cudaStreamDestroy(a->stream);
        delete a;
        *err = e;
        return nullptr;
    }
    row[i] = a;
    return a;
}

void profile_mark(cudaStream_t s, int event_index) {
    if (event_index < g_num_events && g_events[event_index]) cudaEventRecord(g_events[event_index], s);
}

}  // namespace mr

extern "C" const char* mr_status_string(mr_status status) {
    switch (status) {
        case MR_OK: return "ok";
        case MR_ERR_PARAM_NULLPTR: return "a required pointer is NULL";
        case MR_ERR_PARAM_INVALID: return "a dtype, shape or range is outside the supported set";
        case MR_ERR_INNER: return "topK_num > 512 or a probs shape outside the supported range";
        case MR_ERR_CUDA: return "the CUDA runtime reported an error";
        case MR_ERR_WORKSPACE: return "workspaceSize is smaller than required";
        case MR_ERR_UNSUPPORTED: return "a valid mode that this library does not implement";
    }
    return "unknown status";
}

#ifdef MR_CHECKED
namespace mr {
cudaError_t mr_check_words_batching(unsigned* out, bool reset);
cudaError_t mr_check_words_context(unsigned* out, bool reset);
cudaError_t mr_check_words_permute(unsigned* out, bool reset);
cudaError_t mr_check_words_unpermute(unsigned* out, bool reset);
cudaError_t mr_check_words_update_expert(unsigned* out, bool reset);
}  // namespace mr
#endif

extern "C" mr_status mr_checked_errors(uint32_t* failures, uint32_t* firstSite, int32_t reset) {
#ifdef MR_CHECKED
    if (!failures) return MR_ERR_PARAM_NULLPTR;
    cudaError_t (*readers[])(unsigned*, bool) = {mr::mr_check_words_batching, mr::mr_check_words_context,
                                                 mr::mr_check_words_permute, mr::mr_check_words_unpermute,
                                                 mr::mr_check_words_update_expert};
    uint32_t total = 0u, first = 0u;
    for (auto rd : readers) {
        unsigned w[2] = {0u, 0u};
        if (rd(w, reset != 0) != cudaSuccess) return MR_ERR_CUDA;
        if (w[0] != 0u && first == 0u) first = w[1];
        total += w[0];
    }
    *failures = total;
    if (firstSite) *firstSite = first;
    return MR_OK;
#else
    (void)reset;
    if (failures) *failures = 0u;
    if (firstSite) *firstSite = 0u;
    return MR_ERR_UNSUPPORTED;
#endif
}

extern "C" int32_t mr_version(void) { return 100; }

extern "C" mr_status mr_profile_set_events(void* const* events, int32_t count) {
    if (count < 0 || count > 16 || (count > 0 && !events)) return MR_ERR_PARAM_INVALID;
    for (int i = 0; i < 16; ++i) mr::g_events[i] = i < count ? reinterpret_cast<cudaEvent_t>(events[i]) : nullptr;
    mr::g_num_events = count;
    return MR_OK;
}
