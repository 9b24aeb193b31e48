// Host-side plumbing of the decode-step library: error text, status words,
// device queries, version.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "dl_common.cuh"

namespace dl {

static thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    snprintf(g_err, sizeof(g_err), "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
    return DL_E_CUDA;
}

void clear_error() { g_err[0] = 0; }

int device_sm_count(int *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    return DL_OK;
}

int check_launch(const char *what)
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, what);
    return DL_OK;
}

static thread_local DlPrefetch g_pf = {};

void take_prefetch(DlPrefetch *out)
{
    *out = g_pf;
    g_pf.n = 0;
}

}  // namespace dl

extern "C" {

const char *dl_last_error(void) { return dl::g_err; }

int dl_version(void) { return 100; }

int dl_l2_prefetch_next(int n, const void *const *ptrs, const size_t *bytes)
{
    dl::clear_error();
    dl::g_pf.n = 0;
    if (n < 0 || n > kMaxPrefetch) return dl::fail(DL_E_ARG, "dl_l2_prefetch_next: n=%d (0..%d)", n, kMaxPrefetch);
    if (n > 0 && (!ptrs || !bytes)) return dl::fail(DL_E_ARG, "dl_l2_prefetch_next: null pointer");
    DlPrefetch pf = {};
    for (int i = 0; i < n; ++i) {
        if (!ptrs[i] || !dl::aligned16(ptrs[i]) || bytes[i] % 16 != 0)
            return dl::fail(DL_E_ALIGN, "dl_l2_prefetch_next: range %d must start 16-byte aligned and span a "
                                        "multiple of 16 bytes", i);
        if (bytes[i] == 0) continue;
        pf.p[pf.n] = static_cast<const char *>(ptrs[i]);
        pf.bytes[pf.n] = bytes[i];
        ++pf.n;
    }
    dl::g_pf = pf;
    return DL_OK;
}

int dl_status_read(const int32_t *status_dev, int32_t *host_out)
{
    if (!status_dev || !host_out) return dl::fail(DL_E_ARG, "dl_status_read: null pointer");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_status_read: synchronize");
    e = cudaMemcpy(host_out, status_dev, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_status_read: copy");
    return DL_OK;
}

}  // extern "C"
