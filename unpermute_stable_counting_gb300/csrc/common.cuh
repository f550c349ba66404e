// Shared device/host helpers of the GB300 reorder library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "../../include/moe_reorder.h"

namespace mr {

constexpr int kNumSMsHint = 152;  // GB300; the launch code queries the real count

// ---------------------------------------------------------------------------
// Programmatic dependent launch. Every kernel of the library starts with
// pdl_enter(): it waits for the previous kernel in the stream before its first
// global-memory access, so a kernel launched early (programmatic stream
// serialisation) never reads or writes memory that the previous kernel still
// uses.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Kernel prologue: wait for the previous kernel in the stream to finish (its
// memory is then visible). The next kernel is not triggered early: measured on
// GB300, letting the chain of small index kernels launch early made it slower.
__device__ __forceinline__ void pdl_enter() { grid_dependency_wait(); }

// ---------------------------------------------------------------------------
// Cache-hinted global accesses for streamed data (read once / written once).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ void st_stream_u32(void* p, uint32_t v) {
    asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ---------------------------------------------------------------------------
// Block-wide exclusive scan of one uint32 per thread (blockDim.x multiple of
// 32, at most 1024). `warp_sums` must hold 32 entries. Returns the exclusive
// prefix; *total receives the block sum.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums,
                                                         uint32_t* total) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t s = lane < nwarps ? warp_sums[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;  // inclusive prefix of warp sums
    }
    __syncthreads();
    const uint32_t warp_base = warp > 0 ? warp_sums[warp - 1] : 0u;
    if (total) *total = warp_sums[nwarps - 1];
    const uint32_t r = warp_base + x - v;
    __syncthreads();  // warp_sums may be reused by the caller
    return r;
}

// ---------------------------------------------------------------------------
// Element conversions (CUDA intrinsics: exact widening, RNE narrowing).
// ---------------------------------------------------------------------------
template <int DT> struct Elem;
template <> struct Elem<MR_DTYPE_F16> {
    using T = __half;
    static __device__ __forceinline__ float to_f32(uint16_t b) {
        return __half2float(__ushort_as_half(b));
    }
    static __device__ __forceinline__ uint16_t from_f32(float f) {
        return __half_as_ushort(__float2half_rn(f));
    }
};
template <> struct Elem<MR_DTYPE_BF16> {
    static __device__ __forceinline__ float to_f32(uint16_t b) {
        return __bfloat162float(__ushort_as_bfloat16(b));
    }
    static __device__ __forceinline__ uint16_t from_f32(float f) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(f));
    }
};

__device__ __forceinline__ float load_f32(const void* base, int64_t i, int dt) {
    if (dt == MR_DTYPE_F32) return reinterpret_cast<const float*>(base)[i];
    const uint16_t b = reinterpret_cast<const uint16_t*>(base)[i];
    return dt == MR_DTYPE_F16 ? Elem<MR_DTYPE_F16>::to_f32(b) : Elem<MR_DTYPE_BF16>::to_f32(b);
}

// ---------------------------------------------------------------------------
// Bounds-checked build (-DMR_CHECKED). Every gather index, row offset, CSR
// pointer and scatter destination that a kernel derives from data goes
// through MR_IN_RANGE(i, n, site): in a checked build it tests 0 <= i < n
// and, when that fails, counts the failure in this translation unit's error
// words (with the number of the first failing site) and yields false, so
// that the caller skips the access. In a regular build it is the constant
// true and costs nothing. mr_checked_errors() reads and clears the words of
// every translation unit; each .cu file that launches kernels defines its
// reader with MR_CHECK_ACCESSOR(name).
// ---------------------------------------------------------------------------
#ifdef MR_CHECKED
static __device__ unsigned int g_mr_check_words[2];  // failures, first failing site
__device__ __forceinline__ bool mr_in_range(int64_t i, int64_t n, unsigned site) {
    if (i >= 0 && i < n) return true;
    if (atomicAdd(&g_mr_check_words[0], 1u) == 0u) atomicExch(&g_mr_check_words[1], site);
    return false;
}
#define MR_IN_RANGE(i, n, site) ::mr::mr_in_range((int64_t)(i), (int64_t)(n), (unsigned)(site))
#define MR_CHECK_ACCESSOR(name)                                                              \
    cudaError_t mr_check_words_##name(unsigned* out, bool reset) {                           \
        cudaError_t e = cudaMemcpyFromSymbol(out, g_mr_check_words, 2 * sizeof(unsigned));    \
        if (e == cudaSuccess && reset) {                                                     \
            const unsigned zero[2] = {0u, 0u};                                               \
            e = cudaMemcpyToSymbol(g_mr_check_words, zero, sizeof(zero));                    \
        }                                                                                    \
        return e;                                                                            \
    }
#else
#define MR_IN_RANGE(i, n, site) true
#define MR_CHECK_ACCESSOR(name)
#endif

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
__host__ __device__ inline uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

int device_sm_count();                 // cached per device

// Auxiliary stream with fork/join events, one per (device, caller stream),
// created on first use and kept for the process lifetime. `mu` serialises the
// enqueue of one fork/join sequence, so host threads that share a caller
// stream do not interleave their records. Calls on different caller streams
// never share one: their side work overlaps, and a stream capture on one
// caller stream does not reach the auxiliary stream of another.
constexpr int kMaxAuxStreams = 64;  // caller streams per device
struct AuxStream {
    cudaStream_t caller;
    cudaStream_t stream;
    cudaEvent_t fork;
    cudaEvent_t join;
    std::mutex mu;
};
// The auxiliary stream of `caller` on the current device; nullptr when the
// device already has kMaxAuxStreams of them (the caller then runs the side
// work in line) or on a CUDA error (*err set).
AuxStream* aux_stream(cudaStream_t caller, cudaError_t* err);
void profile_mark(cudaStream_t s, int event_index);  // records a timing event if set

// Launch with programmatic stream serialisation (PDL) enabled, or (pdl =
// false) in plain stream order.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                 size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
    return launch_kernel(true, kernel, grid, block, smem, stream, args...);
}

}  // namespace mr

#define MR_TRY_CUDA(expr)                                   \
    do {                                                    \
        cudaError_t _e = (expr);                            \
        if (_e != cudaSuccess) return MR_ERR_CUDA;          \
    } while (0)
