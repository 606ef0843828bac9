// pa_common.cuh -- host-side helpers shared by the library's entry points:
// status strings, the per-thread last CUDA error, alignment checks and the
// device error word.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/paged_attention.h"

namespace pa {

// Records `err` as this thread's last CUDA error and returns PA_ERR_CUDA
// (or PA_OK when err == cudaSuccess).
pa_status record_cuda(cudaError_t err);

inline bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// OR `bits` into the optional device error word.
__device__ __forceinline__ void flag_error(int32_t *error_word, int32_t bits)
{
    if (error_word != nullptr)
        atomicOr(error_word, bits);
}

} // namespace pa
