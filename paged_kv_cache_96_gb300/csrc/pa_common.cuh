// pa_common.cuh -- host-side helpers shared by the library's entry points:
// status strings, the per-thread last CUDA error, alignment checks and the
// device error word.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "../../include/paged_attention.h"

namespace pa {

// Records `err` as this thread's last CUDA error and returns PA_ERR_CUDA
// (or PA_OK when err == cudaSuccess).
pa_status record_cuda(cudaError_t err);

// A wait of an attention kernel on staged data (a tile landing, a
// tensor-core result) gives up after this many nanoseconds and flags
// PA_DEVERR_TIMEOUT; the process-wide setting (pa_set_stage_wait_limit_ns)
// is read at each launch.  Waits that drain copies still in flight before a
// kernel exits always use the default.
constexpr uint64_t kDefaultStageWaitNs = 1000000000ull;  // one second
uint64_t stage_wait_limit_ns();
// Test hook of that time-out path (pa_debug_withhold_first_fill): 1 while
// every CTA of each attention launch leaves its first K/V fill unissued.
int withhold_first_fill();

inline bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialisation: it may begin while the kernel
// before it on the stream finishes, and waits in pdl_wait_primary() --
// before its first global read -- until that kernel's writes are visible.
// pdl_launch_dependents() lets the next kernel on the stream begin early.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline pa_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return record_cuda(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

// OR `bits` into the optional device error word.
__device__ __forceinline__ void flag_error(int32_t *error_word, int32_t bits)
{
    if (error_word != nullptr)
        atomicOr(error_word, bits);
}

} // namespace pa
