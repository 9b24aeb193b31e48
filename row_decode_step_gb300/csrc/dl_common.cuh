// Shared host/device helpers of the decode-step library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>
#include <cstddef>

#include "dl.h"

namespace dl {

// Record a failure for dl_last_error() and return `code`.
int fail(int code, const char *fmt, ...);
// Record a CUDA runtime failure and return DL_E_CUDA.
int cuda_fail(cudaError_t e, const char *what);
// Clear the calling thread's error text.
void clear_error();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// SM count of the current device (cached per device by the caller if needed).
int device_sm_count(int *out);

// Check the launch that was just issued; returns DL_OK or DL_E_CUDA.
int check_launch(const char *what);

}  // namespace dl

// Device side: OR bits into a status word (no trap, no assert).
__device__ __forceinline__ void dl_status_or(int32_t *status, int32_t bits)
{
    if (status) atomicOr(reinterpret_cast<int *>(status), bits);
}
