// Shared host/device helpers of the decode-step library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>
#include <cstddef>
#include <utility>

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

// Byte ranges a launch asks L2 to fetch on behalf of a later kernel (dl_l2_prefetch_next): every
// pointer 16-byte aligned, every size a multiple of 16.
constexpr int kMaxPrefetch = 16;
struct DlPrefetch {
    const char *p[kMaxPrefetch];
    uint64_t bytes[kMaxPrefetch];
    int n;
};

namespace dl {

// Move the calling thread's pending prefetch ranges into `out` (n = 0 if none) and clear them.
void take_prefetch(DlPrefetch *out);


// Launch `kern` on `st` as a programmatic dependent of the previous kernel in the
// stream (it may start before that kernel ends and must call dl_pdl_wait()
// before touching anything the previous kernel writes or reads).
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      const char *what, Args &&...args)
{
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&lc, kern, std::forward<Args>(args)...);
    if (e != cudaSuccess) return cuda_fail(e, what);
    return DL_OK;
}

}  // namespace dl

// Device side: wait for the previous kernel of the stream (no-op without PDL).
__device__ __forceinline__ void dl_pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Device side: let the next kernel of the stream begin launching.  Every kernel of the library
// calls this only after its own dl_pdl_wait(), so a kernel that starts early may rely on every
// kernel before its immediate predecessor having finished (the attention loads the cache slots
// that its predecessor does not write before waiting on it).
__device__ __forceinline__ void dl_pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
// Device side: ask L2 to fetch [p, p + bytes) (16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void dl_prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Device side: this CTA's share of every prefetch range (ranges split evenly over the grid in
// 16-byte units, at most 64 KB per request); one thread per CTA calls it.
__device__ __forceinline__ void dl_issue_prefetch(const DlPrefetch &pf)
{
    const uint64_t nb = (uint64_t)gridDim.x * gridDim.y * gridDim.z;
    const uint64_t b = blockIdx.x + (uint64_t)gridDim.x * (blockIdx.y + (uint64_t)gridDim.y * blockIdx.z);
    for (int i = 0; i < pf.n; ++i) {
        const uint64_t total = pf.bytes[i];
        const uint64_t per = ((total + nb - 1) / nb + 15) & ~(uint64_t)15;
        uint64_t off = per * b;
        const uint64_t end = off + per < total ? off + per : total;
        while (off < end) {
            const uint32_t len = (uint32_t)(end - off < 65536 ? end - off : 65536);
            dl_prefetch_l2(pf.p[i] + off, len);
            off += len;
        }
    }
}

// Device side: OR bits into a status word (no trap, no assert).
__device__ __forceinline__ void dl_status_or(int32_t *status, int32_t bits)
{
    if (status) atomicOr(reinterpret_cast<int *>(status), bits);
}
