// Split-KV decode attention with GQA and its log-sum-exp merge, after daScript
// PR #4293 ("The decode attention's split follows the command's rows, not the
// planes' height"): a row's keys are cut into pieces sized so that the work
// items of the command fill the GPU, each piece yields a softmax partial
// (o, lse), and the partials are merged.
//
// Work item = (session, KV head, piece).  A session's rows share a region, so
// one CTA scores every query head of every session row that reads the KV head:
// each key is loaded from HBM once per session and step.  Stages of 32 keys of
// K and V reach shared memory through tensor maps (below); two inner products
// consume them: tensor cores for sessions of several rows, CUDA cores (lane = key
// for the scores, lanes over head dimensions for P.V) for a few queries.
//
// The attention kernel is in decode_attn_kernel.cuh; this unit holds its default instances
// (no in-launch merge), the merge kernel, the planner and the C entry points.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cmath>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "dl_common.cuh"
#include "dl_async.cuh"
#include "decode_attn_kernel.cuh"

namespace {

struct MergeArgs {
    const float *part_o, *part_lse;
    const int32_t *seqlen;
    float *out, *lse;
    int64_t out_stride;
    int rows, n_q, chunk, max_splits, capacity;
    int row_keys_max[DL_MAX_ROWS];
    DlPrefetch pf;       // L2 prefetches for a later kernel
};

// One CTA per (row, head); its eight warps take every eighth piece and issue the loads of
// their pieces' (lse, o) together, each warp keeping its own running maximum, so that the
// partials cross from L2 in one round; the warps' sums are combined in shared memory.

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(const __grid_constant__ MergeArgs a)
{
    constexpr int VPL = D / 32;              // values per lane
    __shared__ float s_acc[kMergeWarps][D];
    __shared__ float s_m[kMergeWarps], s_w[kMergeWarps];
    if (threadIdx.x == 0 && a.pf.n > 0) dl_issue_prefetch(a.pf);
    dl_pdl_wait();
    dl_pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x / a.n_q, h = blockIdx.x - (blockIdx.x / a.n_q) * a.n_q;
    const int L = clip_len(a.seqlen[r], a.row_keys_max[r], a.capacity, nullptr, false);
    const int np = (L + a.chunk - 1) / a.chunk;
    const float *pl = a.part_lse + ((int64_t)r * a.n_q + h) * a.max_splits;
    float *dst = a.out + r * a.out_stride + h * D;
    if (np == 0) {
        for (int d = threadIdx.x; d < D; d += kMergeWarps * 32) dst[d] = 0.f;
        if (a.lse && threadIdx.x == 0) a.lse[r * a.n_q + h] = -INFINITY;
        return;
    }
    const float *po = a.part_o + ((int64_t)r * a.n_q + h) * a.max_splits * D + lane * VPL;
    float Mw = -INFINITY, Ww = 0.f, acc[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) acc[i] = 0.f;
    for (int p0 = warp; p0 < np; p0 += kMergeWarps * kMergeBatch) {
        float lv[kMergeBatch], v[kMergeBatch][VPL];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            const int p = p0 + kMergeWarps * u;
            lv[u] = -INFINITY;
#pragma unroll
            for (int i = 0; i < VPL; ++i) v[u][i] = 0.f;
            if (p < np) {
                lv[u] = __ldcg(pl + p);
                if constexpr (VPL == 4) {
                    const float4 t = __ldcg(reinterpret_cast<const float4 *>(po + (int64_t)p * D));
                    v[u][0] = t.x; v[u][1] = t.y; v[u][2] = t.z; v[u][3] = t.w;
                } else {
                    const float2 t = __ldcg(reinterpret_cast<const float2 *>(po + (int64_t)p * D));
                    v[u][0] = t.x; v[u][1] = t.y;
                }
            }
        }
        float mb = Mw;
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) mb = fmaxf(mb, lv[u]);
        const float sc = Mw == -INFINITY ? 0.f : __expf(Mw - mb);
        Ww *= sc;
#pragma unroll
        for (int i = 0; i < VPL; ++i) acc[i] *= sc;
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            const float w = lv[u] == -INFINITY ? 0.f : __expf(lv[u] - mb);
            Ww += w;
#pragma unroll
            for (int i = 0; i < VPL; ++i) acc[i] = fmaf(w, v[u][i], acc[i]);
        }
        Mw = mb;
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) s_acc[warp][lane * VPL + i] = acc[i];
    if (lane == 0) {
        s_m[warp] = Mw;
        s_w[warp] = Ww;
    }
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, s_m[w]);
    float f[kMergeWarps], Wt = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
        f[w] = s_m[w] == -INFINITY ? 0.f : __expf(s_m[w] - M);
        Wt += f[w] * s_w[w];
    }
    const float inv = 1.f / Wt;
    for (int d = threadIdx.x; d < D; d += kMergeWarps * 32) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) t = fmaf(f[w], s_acc[w][d], t);
        dst[d] = t * inv;
    }
    if (a.lse && threadIdx.x == 0) a.lse[r * a.n_q + h] = M + logf(Wt);
}

// The driver's tensor-map encoder, looked up once through the runtime (no link against the driver).
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Tensor map of one cache plane as [region][kv_head * capacity + slot][head_dim] f16, read in
// boxes of 32 slots x 64 dims with the 128-byte swizzle; slots past the plane read as zero.
int make_kv_tmap(CUtensorMap *m, const void *plane, const dl_kv_cache *kv)
{
    const bool f32 = kv->elem_bytes == 4, q8 = kv->elem_bytes == 1;
    const cuuint64_t eb = f32 ? 4u : q8 ? 1u : 2u;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
    if (!enc) return dl::fail(DL_E_CUDA, "dl_decode_attn: the driver offers no tensor-map encoder");
    const cuuint64_t dims[3] = {(cuuint64_t)kv->head_dim, (cuuint64_t)kv->n_kv * (cuuint64_t)kv->capacity,
                                (cuuint64_t)kv->n_regions};
    const cuuint64_t strides[2] = {(cuuint64_t)kv->head_dim * eb, (cuuint64_t)kv->region_stride * eb};
    // box rows of 128 bytes (swizzled); the q8_0 mirror's rows are whole key rows of codes,
    // swizzled when they are 128 bytes (head_dim 128), plain when 64
    const cuuint32_t inner = q8 ? (cuuint32_t)kv->head_dim : (cuuint32_t)(128u / eb);
    const cuuint32_t box[3] = {inner, (cuuint32_t)kStKeys, 1u};
    const cuuint32_t es[3] = {1u, 1u, 1u};
    const CUtensorMapSwizzle swz = (q8 && kv->head_dim != 128) ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
    const CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                           const_cast<void *>(plane), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return dl::fail(DL_E_ARG, "dl_decode_attn: cache plane refused as a tensor map (%d)", (int)r);
    return DL_OK;
}

int check_plan(const dl_attn_plan *P)
{
    if (!P || P->rows < 1 || P->rows > DL_MAX_ROWS || P->n_sessions < 1 || P->n_sessions > DL_MAX_ROWS ||
        P->chunk < kTile || P->chunk % kTile != 0 || P->max_splits < 1 || P->n_work < 1 ||
        P->n_kv < 1 || P->n_q % P->n_kv != 0 || (P->head_dim != 64 && P->head_dim != 128))
        return dl::fail(DL_E_ARG, "dl attention: invalid plan");
    return DL_OK;
}

// The default instance for a head dimension and mirror (no in-launch merge): the tensor form, or
// the CUDA-core form with qm queries per warp.
template <int D, int EB>
const void *pick_attn_kernel(bool mma, int qm)
{
    if (mma) return reinterpret_cast<const void *>(decode_attn_tma_kernel<D, true, 8, EB>);
    if constexpr (EB == 2)
        if (qm == 3) return reinterpret_cast<const void *>(decode_attn_tma_kernel<D, false, 3, EB>);
    return qm <= 4 ? reinterpret_cast<const void *>(decode_attn_tma_kernel<D, false, 4, EB>)
         : qm == 6 ? reinterpret_cast<const void *>(decode_attn_tma_kernel<D, false, 6, EB>)
                   : reinterpret_cast<const void *>(decode_attn_tma_kernel<D, false, 8, EB>);
}

}  // namespace

namespace dl {
// The instance with the in-launch merges compiled in (its own translation unit).
const void *attn_kernel_merge_opts(int head_dim, int eb, bool mma, int qm);
}  // namespace dl

namespace dl {
// The f16/f32/q8_0 mirror plane as a tensor map (boxes of 32 slots): shared with the layer-step launch.
int make_kv_tmap(CUtensorMap *m, const void *plane, const dl_kv_cache *kv)
{
    return ::make_kv_tmap(m, plane, kv);
}
}  // namespace dl

extern "C" {

int dl_plan_groups(int n, int max_rows, int *sizes)
{
    if (n < 0 || max_rows <= 0 || !sizes) return dl::fail(DL_E_ARG, "dl_plan_groups: n=%d max_rows=%d", n, max_rows);
    if (n == 0) return 0;
    const int g = (n + max_rows - 1) / max_rows;
    const int base = n / g, rem = n % g;
    for (int i = 0; i < g; ++i) sizes[i] = base + (i < rem ? 1 : 0);
    return g;
}

// max_cluster == 0: pieces sized per session from the command's total keys (partials + merge);
// max_cluster > 0: every (session, KV head) gets the same C <= max_cluster pieces (one cluster).
static int plan_build(int rows, const int32_t *seqlen_host, const int32_t *region_host,
                      int n_q, int n_kv, int head_dim, int sm_count, int force_chunk, int max_cluster,
                      dl_attn_plan *out)
{
    if (!out || !seqlen_host) return dl::fail(DL_E_ARG, "dl_attn_plan_build: null pointer");
    if (rows < 1 || rows > DL_MAX_ROWS)
        return dl::fail(DL_E_SHAPE, "dl_attn_plan_build: rows=%d (a command steps 1..%d rows)", rows, DL_MAX_ROWS);
    if (n_kv < 1 || n_q < n_kv || n_q % n_kv != 0 || n_q / n_kv > kMaxQ)
        return dl::fail(DL_E_SHAPE, "dl_attn_plan_build: n_q=%d n_kv=%d", n_q, n_kv);
    if (head_dim != 64 && head_dim != 128)
        return dl::fail(DL_E_SHAPE, "dl_attn_plan_build: head_dim=%d (64 or 128)", head_dim);
    if (force_chunk < 0) return dl::fail(DL_E_ARG, "dl_attn_plan_build: force_chunk=%d", force_chunk);
    for (int r = 0; r < rows; ++r)
        if (seqlen_host[r] < 1) return dl::fail(DL_E_ARG, "dl_attn_plan_build: seqlen[%d]=%d", r, seqlen_host[r]);
    if (sm_count <= 0) {
        int rc = dl::device_sm_count(&sm_count);
        if (rc != DL_OK) return rc;
    }
    dl_attn_plan P;
    memset(&P, 0, sizeof(P));
    P.rows = rows;
    P.n_q = n_q;
    P.n_kv = n_kv;
    P.head_dim = head_dim;
    P.sm_count = sm_count;
    const int G = n_q / n_kv;
    const int max_sess_rows = kMaxQ / G;   // rows one work item can serve
    for (int r = 0; r < rows; ++r) {
        P.row_region[r] = region_host ? region_host[r] : 0;
        P.row_keys_max[r] = seqlen_host[r];
        if (P.row_region[r] < 0) return dl::fail(DL_E_ARG, "dl_attn_plan_build: region[%d]=%d", r, P.row_region[r]);
    }
    // sessions: rows sharing a region, in order of first appearance, at most max_sess_rows each
    bool taken[DL_MAX_ROWS] = {false};
    int ns = 0, nr = 0;
    for (int r = 0; r < rows; ++r) {
        if (taken[r]) continue;
        P.sess_begin[ns] = nr;
        int cnt = 0;
        for (int r2 = r; r2 < rows && cnt < max_sess_rows; ++r2) {
            if (taken[r2] || P.row_region[r2] != P.row_region[r]) continue;
            taken[r2] = true;
            P.sess_rows[nr++] = r2;
            ++cnt;
        }
        ++ns;
    }
    P.sess_begin[ns] = nr;
    P.n_sessions = ns;
    int lmax[DL_MAX_ROWS];
    int64_t total = 0;
    for (int s = 0; s < ns; ++s) {
        lmax[s] = 0;
        for (int i = P.sess_begin[s]; i < P.sess_begin[s + 1]; ++i) lmax[s] = std::max(lmax[s], seqlen_host[P.sess_rows[i]]);
        total += (int64_t)lmax[s] * n_kv;
    }
    if (max_cluster > 0) {
        // one cluster of C pieces per (session, KV head): about two work items per SM, the
        // longest session's keys in C pieces
        const int groups = ns * n_kv;
        int maxl = 1;
        for (int s = 0; s < ns; ++s) maxl = std::max(maxl, lmax[s]);
        int C = (int)std::min<int64_t>(max_cluster, std::max<int64_t>(1, dl::ceil_div(2LL * sm_count, groups)));
        const int chunk = (int)(dl::ceil_div(dl::ceil_div(maxl, C), kTile) * kTile);
        C = (int)dl::ceil_div(maxl, chunk);
        P.chunk = chunk;
        P.cluster = C;
        for (int s = 0; s < ns; ++s) {
            P.sess_splits[s] = C;
            P.sess_item0[s] = s * n_kv * C;
        }
        P.sess_item0[ns] = groups * C;
        P.n_work = groups * C;
        P.max_splits = C;
        P.workspace_bytes = 0;
        *out = P;
        return DL_OK;
    }
    // pieces sized from this command's own work: about two work items per SM
    int chunk;
    if (force_chunk > 0) {
        chunk = (int)dl::ceil_div(force_chunk, kTile) * kTile;
    } else {
        const int64_t target = 2LL * sm_count;
        chunk = (int)(dl::ceil_div(dl::ceil_div(total, target), kTile) * kTile);
        if (chunk < kTile) chunk = kTile;
    }
    P.chunk = chunk;
    int items = 0, ms = 0;
    for (int s = 0; s < ns; ++s) {
        P.sess_splits[s] = (int)dl::ceil_div(lmax[s], chunk);
        P.sess_item0[s] = items;
        items += n_kv * P.sess_splits[s];
        ms = std::max(ms, P.sess_splits[s]);
    }
    P.sess_item0[ns] = items;
    P.n_work = items;
    P.max_splits = ms;
    const size_t po = (size_t)rows * n_q * ms * head_dim * 4;
    const size_t pl = (size_t)rows * n_q * ms * 4;
    const size_t pc = (size_t)ns * n_kv * 4;          // the tail merge's piece counts
    P.workspace_bytes = ((po + 15) / 16) * 16 + ((pl + 15) / 16) * 16 + ((pc + 15) / 16) * 16;
    *out = P;
    return DL_OK;
}

int dl_attn_plan_build(int rows, const int32_t *seqlen_host, const int32_t *region_host,
                       int n_q, int n_kv, int head_dim, int sm_count, int force_chunk,
                       dl_attn_plan *out)
{
    dl::clear_error();
    return plan_build(rows, seqlen_host, region_host, n_q, n_kv, head_dim, sm_count, force_chunk, 0, out);
}

int dl_attn_plan_build_cluster(int rows, const int32_t *seqlen_host, const int32_t *region_host,
                               int n_q, int n_kv, int head_dim, int sm_count, int max_cluster,
                               dl_attn_plan *out)
{
    dl::clear_error();
    if (max_cluster < 0 || max_cluster > kMaxCluster)
        return dl::fail(DL_E_ARG, "dl_attn_plan_build_cluster: max_cluster=%d (0..%d)", max_cluster, kMaxCluster);
    return plan_build(rows, seqlen_host, region_host, n_q, n_kv, head_dim, sm_count, 0,
                      max_cluster == 0 ? kMaxCluster : max_cluster, out);
}

// The new rows of the fused form: raw k and v rows, optional bias, positions and the rope table.
struct FusedIn {
    const float *k, *v, *bias;
    int64_t k_stride, v_stride;
    const int32_t *pos;
    const dl_rope *rope;
};

// Results written by the attention launch itself: a cluster plan's, or the last piece's merge.
struct ClusterOut {
    float *out;
    int64_t out_stride;
    float *lse;
};

static int decode_attn_impl(const float *q, int64_t q_stride, const dl_kv_cache *kv, const int32_t *seqlen,
                            const dl_attn_plan *plan, void *workspace, size_t workspace_bytes,
                            int32_t *status, int path, dl_stream_t stream, const FusedIn *f = nullptr,
                            const ClusterOut *co = nullptr, bool tail = false)
{
    dl::clear_error();
    DlPrefetch pf;
    dl::take_prefetch(&pf);
    if (!q || !kv || !kv->k || !kv->v || !seqlen || ((!co || tail) && !workspace) || (co && !co->out))
        return dl::fail(DL_E_ARG, "dl_decode_attn: null pointer");
    int rc = check_plan(plan);
    if (rc != DL_OK) return rc;
    if (tail && plan->cluster > 0)
        return dl::fail(DL_E_ARG, "dl_decode_attn_merged: a cluster plan goes to dl_decode_attn_cluster");
    if (!tail && (plan->cluster > 0) != (co != nullptr))
        return dl::fail(DL_E_ARG, plan->cluster > 0 ? "dl_decode_attn: a cluster plan goes to dl_decode_attn_cluster"
                                                    : "dl_decode_attn_cluster: the plan has no clusters");
    if (co && !tail) {
        if (!co->out) return dl::fail(DL_E_ARG, "dl_decode_attn_cluster: null output");
        if (plan->cluster > kMaxCluster || plan->n_work != plan->n_sessions * plan->n_kv * plan->cluster)
            return dl::fail(DL_E_ARG, "dl_decode_attn_cluster: cluster of %d", plan->cluster);
        for (int si = 0; si < plan->n_sessions; ++si)
            if (plan->sess_splits[si] != plan->cluster || plan->sess_item0[si] != si * plan->n_kv * plan->cluster)
                return dl::fail(DL_E_ARG, "dl_decode_attn_cluster: session %d is not laid out in clusters", si);
        if (co->out_stride < (int64_t)plan->n_q * plan->head_dim || !dl::aligned16(co->out) || (co->out_stride % 4) != 0)
            return dl::fail(DL_E_ALIGN, "dl_decode_attn_cluster: out must be 16-byte aligned rows of n_q*head_dim");
    }
    if (kv->head_dim != plan->head_dim || kv->n_kv != plan->n_kv)
        return dl::fail(DL_E_SHAPE, "dl_decode_attn: cache heads/dim differ from the plan");
    if (kv->capacity <= 0 || kv->region_stride < (int64_t)kv->n_kv * kv->capacity * kv->head_dim)
        return dl::fail(DL_E_ARG, "dl_decode_attn: bad cache geometry");
    if (kv->elem_bytes != 0 && kv->elem_bytes != 1 && kv->elem_bytes != 2 && kv->elem_bytes != 4)
        return dl::fail(DL_E_ARG, "dl_decode_attn: elem_bytes=%d (1, 2 or 4)", kv->elem_bytes);
    if (kv->elem_bytes == 1) {
        if (!kv->k_scale || !kv->v_scale || !dl::aligned16(kv->k_scale) || !dl::aligned16(kv->v_scale))
            return dl::fail(DL_E_ALIGN, "dl_decode_attn: the q8_0 mirror wants 16-byte aligned scale planes");
        if (kv->capacity % 4 != 0 || kv->region_stride % 256 != 0)
            return dl::fail(DL_E_SHAPE, "dl_decode_attn: the q8_0 mirror wants capacity %% 4 == 0 and a region "
                                        "stride that is a multiple of 256 (capacity %d, stride %lld)",
                            kv->capacity, (long long)kv->region_stride);
    }
    for (int r = 0; r < plan->rows; ++r) {
        if (plan->row_region[r] >= kv->n_regions) return dl::fail(DL_E_ARG, "dl_decode_attn: plan region past the cache");
        if (plan->row_keys_max[r] > kv->capacity)
            return dl::fail(DL_E_ARG, "dl_decode_attn: plan covers %d keys of row %d, the cache holds %d",
                            plan->row_keys_max[r], r, kv->capacity);
    }
    const bool partials = !co || tail;           // pieces write partials to the workspace
    if (partials && workspace_bytes < plan->workspace_bytes)
        return dl::fail(DL_E_WORKSPACE, "dl_decode_attn: workspace %zu < %zu bytes", workspace_bytes, plan->workspace_bytes);
    if ((partials && !dl::aligned16(workspace)) || !dl::aligned16(kv->k) || !dl::aligned16(kv->v) || !dl::aligned16(q) ||
        (q_stride % 4) != 0 || (kv->region_stride * (kv->elem_bytes == 4 ? 4 : kv->elem_bytes == 1 ? 1 : 2)) % 16 != 0)
        return dl::fail(DL_E_ALIGN, "dl_decode_attn: q, cache planes and workspace must be 16-byte aligned");
    if (q_stride < (int64_t)plan->n_q * plan->head_dim) return dl::fail(DL_E_ARG, "dl_decode_attn: q_stride too small");

    AttnArgs a{};
    a.q = q;
    a.q_stride = q_stride;
    a.kc = kv->k;
    a.vc = kv->v;
    a.region_stride = kv->region_stride;
    a.capacity = kv->capacity;
    a.seqlen = seqlen;
    const size_t po = (size_t)plan->rows * plan->n_q * plan->max_splits * plan->head_dim * 4;
    const size_t pl = (size_t)plan->rows * plan->n_q * plan->max_splits * 4;
    if (partials) {
        a.part_o = static_cast<float *>(workspace);
        a.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + ((po + 15) / 16) * 16);
        a.counters = reinterpret_cast<int *>(static_cast<char *>(workspace) + ((po + 15) / 16) * 16 +
                                             ((pl + 15) / 16) * 16);
    }
    if (co) {
        if (co->out_stride < (int64_t)plan->n_q * plan->head_dim || !dl::aligned16(co->out) || co->out_stride % 4)
            return dl::fail(DL_E_ARG, "dl_decode_attn: out must be 16-byte aligned with a stride of at least "
                                      "n_q * head_dim (a multiple of 4)");
        a.out = co->out;
        a.out_stride = co->out_stride;
        a.lse_out = co->lse;
        a.tail_merge = tail ? 1 : 0;
    }
    a.status = status;
    a.qscale = (float)(1.4426950408889634 / std::sqrt((double)plan->head_dim));
    a.plan = *plan;
    a.pf = pf;
    if (f) {
        const int D = plan->head_dim;
        if (!f->k || !f->v || !f->pos || !f->rope || !f->rope->cos_sin)
            return dl::fail(DL_E_ARG, "dl_decode_attn_rope: null pointer");
        if (f->rope->rot_dim < 0 || f->rope->rot_dim % 2 != 0 || f->rope->rot_dim > D || f->rope->max_pos <= 0)
            return dl::fail(DL_E_SHAPE, "dl_decode_attn_rope: rot_dim=%d head_dim=%d", f->rope->rot_dim, D);
        if (f->k_stride < (int64_t)plan->n_kv * D || f->v_stride < (int64_t)plan->n_kv * D)
            return dl::fail(DL_E_ARG, "dl_decode_attn_rope: k/v strides below the row widths");
        if (!dl::aligned16(f->rope->cos_sin))
            return dl::fail(DL_E_ALIGN, "dl_decode_attn_rope: the rotary table must be 16-byte aligned");
        a.fused = 1;
        a.k_new = f->k;
        a.v_new = f->v;
        a.bias = f->bias;
        a.k_stride = f->k_stride;
        a.v_stride = f->v_stride;
        a.pos = f->pos;
        a.cs = reinterpret_cast<const float2 *>(f->rope->cos_sin);
        a.kc_w = kv->k;
        a.vc_w = kv->v;
        a.rot = f->rope->rot_dim;
        a.neox = f->rope->neox ? 1 : 0;
        a.max_pos = f->rope->max_pos;
    }
    if (path < 0 || path > 2) return dl::fail(DL_E_ARG, "dl_decode_attn: path=%d", path);
    int qmax = 0;
    for (int si = 0; si < plan->n_sessions; ++si)
        qmax = std::max(qmax, (plan->sess_begin[si + 1] - plan->sess_begin[si]) * (plan->n_q / plan->n_kv));
    if (tail && qmax > kTailMaxQ)
        return dl::fail(DL_E_SHAPE, "dl_decode_attn_merged: %d queries per work item (the last piece merges at "
                                    "most %d)", qmax, kTailMaxQ);
    const int eb = kv->elem_bytes == 0 ? 2 : kv->elem_bytes;
    const bool mma = path == 2 || (path == 0 && qmax > kCudaCoreMaxQ);
    a.ksc = static_cast<const uint16_t *>(kv->k_scale);
    a.vsc = static_cast<const uint16_t *>(kv->v_scale);
    a.ksc_w = static_cast<uint16_t *>(kv->k_scale);
    a.vsc_w = static_cast<uint16_t *>(kv->v_scale);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUtensorMap tk, tv;
    rc = make_kv_tmap(&tk, kv->k, kv);
    if (rc != DL_OK) return rc;
    rc = make_kv_tmap(&tv, kv->v, kv);
    if (rc != DL_OK) return rc;
    const size_t smem = attn_mma_smem_bytes(plan->head_dim, eb);
    // the CUDA-core form holds the queries of a warp in registers: 3 or 4 for one-row sessions
    // (3 on the f16 mirror for GQA groups of up to 3 heads, so that no query slot idles; the other
    // mirrors and the in-launch merges keep 4); 6 when a work item serves 17..24 queries (four
    // query groups keep all four consumer warps busy, where groups of 8 would leave one idle); else 8
    const int qm = qmax <= 3 ? 3 : qmax <= 4 ? 4 : (qmax > 16 && qmax <= 24) ? 6 : 8;
    // the in-launch merges (cluster, last piece) run in instances of their own
    const bool clustered = co && !tail;
    const void *kern = (co || tail) ? dl::attn_kernel_merge_opts(plan->head_dim, eb, mma, qm == 3 ? 4 : qm)
                     : eb == 4 ? (plan->head_dim == 128 ? pick_attn_kernel<128, 4>(mma, qm) : pick_attn_kernel<64, 4>(mma, qm))
                     : eb == 1 ? (plan->head_dim == 128 ? pick_attn_kernel<128, 1>(mma, qm) : pick_attn_kernel<64, 1>(mma, qm))
                               : (plan->head_dim == 128 ? pick_attn_kernel<128, 2>(mma, qm) : pick_attn_kernel<64, 2>(mma, qm));
    if (!kern) return dl::fail(DL_E_ARG, "dl_decode_attn: no instance for head_dim %d", plan->head_dim);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_decode_attn: set shared memory");
    // one thread-block cluster per (session, KV head): its pieces are consecutive work items
    if (clustered && plan->cluster > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return dl::cuda_fail(e, "dl_decode_attn_cluster: allow a large cluster");
    }
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)plan->n_work);
    lc.blockDim = dim3(kMmaThreads);
    lc.dynamicSmemBytes = smem;
    lc.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)plan->cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = clustered ? 2 : 1;
    if (clustered) {
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, kern, &lc);
        if (e != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            return dl::fail(DL_E_SHAPE, "dl_decode_attn_cluster: a cluster of %d does not fit on the device",
                            plan->cluster);
        }
    }
    void *args[3] = {&a, &tk, &tv};
    e = cudaLaunchKernelExC(&lc, kern, args);
    if (e != cudaSuccess) return dl::cuda_fail(e, clustered ? "dl_decode_attn_cluster: launch" : "dl_decode_attn: launch");
    return DL_OK;
}

int dl_decode_attn(const float *q, int64_t q_stride, const dl_kv_cache *kv, const int32_t *seqlen,
                   const dl_attn_plan *plan, void *workspace, size_t workspace_bytes,
                   int32_t *status, dl_stream_t stream)
{
    return decode_attn_impl(q, q_stride, kv, seqlen, plan, workspace, workspace_bytes, status, 0, stream);
}

int dl_decode_attn_ex(const float *q, int64_t q_stride, const dl_kv_cache *kv, const int32_t *seqlen,
                      const dl_attn_plan *plan, void *workspace, size_t workspace_bytes,
                      int32_t *status, int path, dl_stream_t stream)
{
    return decode_attn_impl(q, q_stride, kv, seqlen, plan, workspace, workspace_bytes, status, path, stream);
}

int dl_decode_attn_cluster(const float *q, int64_t q_stride, const dl_attn_rope_in *rope_in,
                           const dl_kv_cache *kv, const int32_t *seqlen, const dl_attn_plan *plan,
                           float *out, int64_t out_stride, float *lse, int32_t *status, int path,
                           dl_stream_t stream)
{
    const ClusterOut co{out, out_stride, lse};
    if (!rope_in)
        return decode_attn_impl(q, q_stride, kv, seqlen, plan, nullptr, 0, status, path, stream, nullptr, &co);
    const FusedIn f{rope_in->k, rope_in->v, rope_in->bias, rope_in->k_stride, rope_in->v_stride, rope_in->pos,
                    rope_in->rope};
    return decode_attn_impl(q, q_stride, kv, seqlen, plan, nullptr, 0, status, path, stream, &f, &co);
}

int dl_decode_attn_merged(const float *q, int64_t q_stride, const dl_attn_rope_in *rope_in,
                          const dl_kv_cache *kv, const int32_t *seqlen, const dl_attn_plan *plan,
                          void *workspace, size_t workspace_bytes, float *out, int64_t out_stride, float *lse,
                          int32_t *status, int path, dl_stream_t stream)
{
    const ClusterOut co{out, out_stride, lse};
    if (!rope_in)
        return decode_attn_impl(q, q_stride, kv, seqlen, plan, workspace, workspace_bytes, status, path, stream,
                                nullptr, &co, true);
    const FusedIn f{rope_in->k, rope_in->v, rope_in->bias, rope_in->k_stride, rope_in->v_stride, rope_in->pos,
                    rope_in->rope};
    return decode_attn_impl(q, q_stride, kv, seqlen, plan, workspace, workspace_bytes, status, path, stream, &f,
                            &co, true);
}

int dl_decode_attn_rope(const float *q, int64_t q_stride, const float *k, int64_t k_stride,
                        const float *v, int64_t v_stride, const float *bias, const int32_t *pos,
                        const dl_rope *rope, const dl_kv_cache *kv, const int32_t *seqlen,
                        const dl_attn_plan *plan, void *workspace, size_t workspace_bytes,
                        int32_t *status, int path, dl_stream_t stream)
{
    const FusedIn f{k, v, bias, k_stride, v_stride, pos, rope};
    return decode_attn_impl(q, q_stride, kv, seqlen, plan, workspace, workspace_bytes, status, path, stream, &f);
}

int dl_attn_merge(const void *workspace, const dl_attn_plan *plan, const int32_t *seqlen,
                  float *out, int64_t out_stride, float *lse, dl_stream_t stream)
{
    dl::clear_error();
    MergeArgs m{};
    dl::take_prefetch(&m.pf);
    if (!workspace || !seqlen || !out) return dl::fail(DL_E_ARG, "dl_attn_merge: null pointer");
    int rc = check_plan(plan);
    if (rc != DL_OK) return rc;
    if (plan->cluster > 0) return dl::fail(DL_E_ARG, "dl_attn_merge: a cluster plan merges inside its attention launch");
    if (out_stride < (int64_t)plan->n_q * plan->head_dim) return dl::fail(DL_E_ARG, "dl_attn_merge: out_stride too small");
    if (!dl::aligned16(out) || (out_stride % 4) != 0 || !dl::aligned16(workspace))
        return dl::fail(DL_E_ALIGN, "dl_attn_merge: out and workspace must be 16-byte aligned");
    const size_t po = (size_t)plan->rows * plan->n_q * plan->max_splits * plan->head_dim * 4;
    m.part_o = static_cast<const float *>(workspace);
    m.part_lse = reinterpret_cast<const float *>(static_cast<const char *>(workspace) + ((po + 15) / 16) * 16);
    m.seqlen = seqlen;
    m.out = out;
    m.lse = lse;
    m.out_stride = out_stride;
    m.rows = plan->rows;
    m.n_q = plan->n_q;
    m.chunk = plan->chunk;
    m.max_splits = plan->max_splits;
    m.capacity = 0x7fffffff;   // dl_decode_attn refuses plans that reach past the cache
    for (int r = 0; r < DL_MAX_ROWS; ++r) m.row_keys_max[r] = plan->row_keys_max[r];
    const unsigned grid = (unsigned)(plan->rows * plan->n_q);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto kern = plan->head_dim == 128 ? attn_merge_kernel<128> : attn_merge_kernel<64>;
    return dl::launch_pdl(kern, dim3(grid), dim3(kMergeWarps * 32), 0, st, "dl_attn_merge: launch", m);
}

}  // extern "C"
