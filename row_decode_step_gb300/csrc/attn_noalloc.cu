// Decode attention whose partials live in a buffer the library owns, for callers
// that cannot allocate device memory.
//
// dl_decode_attn needs a workspace for the pieces' partial (o, lse), which the
// caller allocates.  Some callers cannot do that: a host that hands this code
// only the tensors of one step and keeps every other byte of device memory in
// its own pool; an engine whose device-memory budget is fixed once it has
// started serving; a caller on a latency-critical path where an allocation's
// implicit device synchronisation is not allowed.  For them this file keeps the
// partials in a fixed-size __device__ array inside the library instead.  Every
// GPU that loads the library holds the array until the process exits.
#include <mutex>

#include "dl_common.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)8 << 20;    // 8 MiB of partials

__device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_dev[256] = {};   // the array's device address asked last, per device ordinal

// Device address of the array on the current device.  In host code the array's
// name is only a host-side stand-in, so the address is asked of the runtime.  It is
// asked again on every call made outside stream capture (a cudaDeviceReset gives the
// device a new context and the array a new address); a call under capture uses the
// address asked last on that device.
int scratch_address(cudaStream_t st, void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_decode_attention_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= 256) return dl::fail(DL_E_ARG, "dl_decode_attention_noalloc: device %d", dev);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_decode_attention_noalloc: cudaStreamIsCapturing");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cs == cudaStreamCaptureStatusNone || !g_scratch_dev[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess) return dl::cuda_fail(e, "dl_decode_attention_noalloc: cudaGetSymbolAddress");
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return DL_OK;
}

}  // namespace

extern "C" {

size_t dl_decode_attention_noalloc_max_bytes(void) { return kScratchBytes; }

int dl_decode_attention_noalloc(const float *q, int64_t q_stride, const dl_kv_cache *kv,
                                const int32_t *seqlen, const dl_attn_plan *plan,
                                float *out, int64_t out_stride, float *lse,
                                int32_t *status, dl_stream_t stream)
{
    dl::clear_error();
    if (!plan) return dl::fail(DL_E_ARG, "dl_decode_attention_noalloc: null plan");
    if (plan->cluster > 0)
        return dl::fail(DL_E_ARG, "dl_decode_attention_noalloc: a cluster plan merges inside its clusters and keeps "
                                  "no partials; call dl_decode_attn_cluster, which needs no workspace either");
    if (plan->workspace_bytes > kScratchBytes)
        return dl::fail(DL_E_WORKSPACE,
                        "dl_decode_attention_noalloc: the plan needs %zu bytes of partials, the library's "
                        "fixed buffer holds %zu; use dl_decode_attn with a caller workspace",
                        plan->workspace_bytes, kScratchBytes);
    void *scratch = nullptr;
    int rc = scratch_address(static_cast<cudaStream_t>(stream), &scratch);
    if (rc != DL_OK) return rc;
    rc = dl_decode_attn(q, q_stride, kv, seqlen, plan, scratch, kScratchBytes, status, stream);
    if (rc != DL_OK) return rc;
    return dl_attn_merge(scratch, plan, seqlen, out, out_stride, lse, stream);
}

}  // extern "C"
