// Fused RoPE and KV store, the GkRopeKvStore role of daScript PR #4293
// ("The decode rope-and-store rides one template on both homes"): bias rows
// added first, each q pair rotated in place, each k pair rotated into the f16 K
// mirror row of the token's slot, the v pair copied into the V mirror row, the
// stored halves clamped into the half range, channels past the rotated width
// copied through.
//
// One thread per channel pair of one head of one row.  q heads and KV heads
// share a launch: thread blocks cover 256 pairs, i.e. several heads of one row.
#include <cuda_fp16.h>
#include <cmath>

#include "dl_common.cuh"

namespace {

struct RopeArgs {
    float *q;
    const float *k, *v, *bias;
    int64_t q_stride, k_stride, v_stride;
    const int32_t *pos, *row_region;
    const float2 *cs;       // [max_pos][rot/2] (cos, sin)
    void *kc, *vc;           // f16 patterns, f32 values (f32) or int8 codes (q8)
    uint16_t *ks, *vs;       // q8: f16 scales, one per 32 values
    int64_t region_stride;
    int f32, q8;
    int32_t *status;
    int n_q, n_kv, D, rot, neox, max_pos, capacity, n_regions;
    DlPrefetch pf;           // L2 prefetches for a later kernel (first launch only)
};

__device__ __forceinline__ unsigned short to_half_clamped(float v)
{
    v = fminf(fmaxf(v, -65504.0f), 65504.0f);
    return __half_as_ushort(__float2half_rn(v));
}

__global__ void __launch_bounds__(256) rope_kv_store_kernel(const __grid_constant__ RopeArgs a)
{
    if (threadIdx.x == 0 && a.pf.n > 0) dl_issue_prefetch(a.pf);
    dl_pdl_wait();
    dl_pdl_launch_dependents();
    const int r = blockIdx.y;
    const int half = a.D >> 1;
    const int pairs_total = (a.n_q + a.n_kv) * half;
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= pairs_total) return;
    const int head = idx / half, j = idx - head * half;

    const int p = a.pos[r];
    const int reg = a.row_region ? a.row_region[r] : 0;
    if (p < 0 || p >= a.capacity || p >= a.max_pos) {
        if (idx == 0) dl_status_or(a.status, DL_STATUS_POS_RANGE);
        return;
    }
    if (reg < 0 || reg >= a.n_regions) {
        if (idx == 0) dl_status_or(a.status, DL_STATUS_REGION_RANGE);
        return;
    }

    // channels of this thread's pair
    const int rh = a.rot >> 1;
    int i0, i1;
    bool rotate = j < rh;
    if (rotate) {
        i0 = a.neox ? j : 2 * j;
        i1 = a.neox ? j + rh : 2 * j + 1;
    } else {
        i0 = a.rot + 2 * (j - rh);
        i1 = i0 + 1;
    }
    float c = 1.f, s = 0.f;
    if (rotate) {
        const float2 t = a.cs[(size_t)p * rh + j];
        c = t.x;
        s = t.y;
    }

    if (head < a.n_q) {
        float *qr = a.q + r * a.q_stride + head * a.D;
        float x0 = qr[i0], x1 = qr[i1];
        if (a.bias) {
            x0 += a.bias[head * a.D + i0];
            x1 += a.bias[head * a.D + i1];
        }
        if (rotate) {
            const float y0 = fmaf(x0, c, -x1 * s);
            const float y1 = fmaf(x0, s, x1 * c);
            x0 = y0;
            x1 = y1;
        }
        qr[i0] = x0;
        qr[i1] = x1;
    } else if (!a.q8) {
        const int h = head - a.n_q;
        const float *kr = a.k + r * a.k_stride + h * a.D;
        const float *vr = a.v + r * a.v_stride + h * a.D;
        float k0 = kr[i0], k1 = kr[i1];
        float v0 = vr[i0], v1 = vr[i1];
        if (a.bias) {
            const float *bk = a.bias + (a.n_q + h) * a.D;
            const float *bv = a.bias + (a.n_q + a.n_kv + h) * a.D;
            k0 += bk[i0];
            k1 += bk[i1];
            v0 += bv[i0];
            v1 += bv[i1];
        }
        if (rotate) {
            const float y0 = fmaf(k0, c, -k1 * s);
            const float y1 = fmaf(k0, s, k1 * c);
            k0 = y0;
            k1 = y1;
        }
        const int64_t base = (int64_t)reg * a.region_stride + ((int64_t)h * a.capacity + p) * a.D;
        if (a.f32) {
            // the f32 mirror: each value rounded once, nothing clamped
            float *kc = static_cast<float *>(a.kc), *vc = static_cast<float *>(a.vc);
            kc[base + i0] = k0;
            kc[base + i1] = k1;
            vc[base + i0] = v0;
            vc[base + i1] = v1;
        } else {
            uint16_t *kc = static_cast<uint16_t *>(a.kc), *vc = static_cast<uint16_t *>(a.vc);
            kc[base + i0] = to_half_clamped(k0);
            kc[base + i1] = to_half_clamped(k1);
            vc[base + i0] = to_half_clamped(v0);
            vc[base + i1] = to_half_clamped(v1);
        }
    }
}

// The q8_0 mirror's store: one warp per (row, KV head, k or v, block of 32 channels).  Lane l
// forms channel c = 32b + l: for k, bias first, then the rotation of its pair computed from the
// unrotated input (the partner is read, not written, so warps never race); the block's max|x|
// comes from the warp, d = max / 127 in f32, the code is x / d rounded half away from zero and
// clamped to +-127, the scale is stored as f16.
__global__ void __launch_bounds__(128) rope_kv_store_q8_kernel(RopeArgs a)
{
    dl_pdl_wait();
    dl_pdl_launch_dependents();
    const int r = blockIdx.y;
    const int nb = a.D / 32;
    const int unit = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (unit >= 2 * a.n_kv * nb) return;
    const int isv = unit / (a.n_kv * nb), rem = unit - isv * a.n_kv * nb;
    const int h = rem / nb, b = rem - (rem / nb) * nb;
    const int p = a.pos[r];
    const int reg = a.row_region ? a.row_region[r] : 0;
    if (p < 0 || p >= a.capacity || p >= a.max_pos) {
        if (unit == 0 && lane == 0) dl_status_or(a.status, DL_STATUS_POS_RANGE);
        return;
    }
    if (reg < 0 || reg >= a.n_regions) {
        if (unit == 0 && lane == 0) dl_status_or(a.status, DL_STATUS_REGION_RANGE);
        return;
    }
    const int c = 32 * b + lane;
    float x;
    if (isv) {
        x = a.v[r * a.v_stride + h * a.D + c];
        if (a.bias) x += a.bias[(a.n_q + a.n_kv + h) * a.D + c];
    } else {
        const float *kr = a.k + r * a.k_stride + h * a.D;
        const float *bk = a.bias ? a.bias + (a.n_q + h) * a.D : nullptr;
        x = kr[c] + (bk ? bk[c] : 0.f);
        const int rh = a.rot >> 1;
        if (c < a.rot) {
            // the pair (i0, i1) holding channel c and its angle index j
            const int j = a.neox ? (c < rh ? c : c - rh) : (c >> 1);
            const int i0 = a.neox ? j : 2 * j, i1 = a.neox ? j + rh : 2 * j + 1;
            const float x0 = kr[i0] + (bk ? bk[i0] : 0.f), x1 = kr[i1] + (bk ? bk[i1] : 0.f);
            const float2 t = a.cs[(size_t)p * rh + j];
            x = c == i0 ? fmaf(x0, t.x, -x1 * t.y) : fmaf(x0, t.y, x1 * t.x);
        }
    }
    float m = fabsf(x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float d32 = m / 127.0f;
    int code = 0;
    if (d32 > 0.f) {
        const float t = x / d32;
        const float rr = floorf(fabsf(t) + 0.5f);
        code = (int)(t < 0.f ? -rr : rr);
        code = max(-127, min(127, code));
    }
    const int64_t base = (int64_t)reg * a.region_stride + ((int64_t)h * a.capacity + p) * a.D;
    int8_t *codes = static_cast<int8_t *>(isv ? a.vc : a.kc);
    codes[base + c] = (int8_t)code;
    if (lane == 0) (isv ? a.vs : a.ks)[(base + 32 * b) / 32] = __half_as_ushort(__float2half_rn(d32));
}

}  // namespace

extern "C" {

int dl_rope_table_bytes(int rot_dim, int max_pos, size_t *bytes)
{
    if (rot_dim <= 0 || rot_dim % 2 != 0 || max_pos <= 0 || !bytes)
        return dl::fail(DL_E_ARG, "dl_rope_table_bytes: rot_dim=%d max_pos=%d", rot_dim, max_pos);
    *bytes = (size_t)max_pos * (size_t)(rot_dim / 2) * 2 * sizeof(float);
    return DL_OK;
}

int dl_rope_table_build(double theta, int rot_dim, int max_pos, float *host_out)
{
    dl::clear_error();
    if (!host_out || rot_dim <= 0 || rot_dim % 2 != 0 || max_pos <= 0 || !(theta > 1.0))
        return dl::fail(DL_E_ARG, "dl_rope_table_build: theta=%g rot_dim=%d max_pos=%d", theta, rot_dim, max_pos);
    const int rh = rot_dim / 2;
    for (int j = 0; j < rh; ++j) {
        // angle of pair j at position p: p * theta^(-2j/rot_dim), in double
        const double inv = std::pow(theta, -2.0 * (double)j / (double)rot_dim);
        for (int p = 0; p < max_pos; ++p) {
            const double ang = (double)p * inv;
            host_out[((size_t)p * rh + j) * 2 + 0] = (float)std::cos(ang);
            host_out[((size_t)p * rh + j) * 2 + 1] = (float)std::sin(ang);
        }
    }
    return DL_OK;
}

int dl_rope_kv_store(float *q, int64_t q_stride, const float *k, int64_t k_stride,
                     const float *v, int64_t v_stride, const float *bias, const int32_t *pos,
                     const int32_t *row_region, int rows, int n_q, const dl_rope *rope,
                     const dl_kv_cache *kv, int32_t *status, dl_stream_t stream)
{
    dl::clear_error();
    DlPrefetch pf;
    dl::take_prefetch(&pf);
    if (!q || !k || !v || !pos || !rope || !kv || !kv->k || !kv->v || !rope->cos_sin)
        return dl::fail(DL_E_ARG, "dl_rope_kv_store: null pointer");
    if (rows < 0 || n_q <= 0) return dl::fail(DL_E_ARG, "dl_rope_kv_store: rows=%d n_q=%d", rows, n_q);
    const int D = kv->head_dim;
    if (D <= 0 || D % 2 != 0 || D > 1024 || kv->n_kv <= 0 || n_q % kv->n_kv != 0)
        return dl::fail(DL_E_SHAPE, "dl_rope_kv_store: head_dim=%d n_q=%d n_kv=%d", D, n_q, kv->n_kv);
    if (rope->rot_dim < 0 || rope->rot_dim % 2 != 0 || rope->rot_dim > D || rope->max_pos <= 0)
        return dl::fail(DL_E_SHAPE, "dl_rope_kv_store: rot_dim=%d head_dim=%d", rope->rot_dim, D);
    if (kv->elem_bytes != 0 && kv->elem_bytes != 1 && kv->elem_bytes != 2 && kv->elem_bytes != 4)
        return dl::fail(DL_E_ARG, "dl_rope_kv_store: elem_bytes=%d (1, 2 or 4)", kv->elem_bytes);
    if (kv->elem_bytes == 1 && (!kv->k_scale || !kv->v_scale || D % 32 != 0 || kv->region_stride % 32 != 0))
        return dl::fail(DL_E_ARG, "dl_rope_kv_store: the q8_0 mirror wants scale planes, head_dim and region "
                                  "stride multiples of 32");
    if (kv->capacity <= 0 || kv->n_regions <= 0 ||
        kv->region_stride < (int64_t)kv->n_kv * kv->capacity * D)
        return dl::fail(DL_E_ARG, "dl_rope_kv_store: bad cache geometry");
    if (q_stride < (int64_t)n_q * D || k_stride < (int64_t)kv->n_kv * D || v_stride < (int64_t)kv->n_kv * D)
        return dl::fail(DL_E_ARG, "dl_rope_kv_store: strides below the row widths");
    if (rows == 0) return DL_OK;

    RopeArgs a{};
    a.q = q; a.k = k; a.v = v; a.bias = bias;
    a.q_stride = q_stride; a.k_stride = k_stride; a.v_stride = v_stride;
    a.pos = pos; a.row_region = row_region;
    a.cs = reinterpret_cast<const float2 *>(rope->cos_sin);
    a.kc = kv->k; a.vc = kv->v; a.region_stride = kv->region_stride;
    a.f32 = kv->elem_bytes == 4 ? 1 : 0;
    a.q8 = kv->elem_bytes == 1 ? 1 : 0;
    a.ks = static_cast<uint16_t *>(kv->k_scale);
    a.vs = static_cast<uint16_t *>(kv->v_scale);
    a.status = status;
    a.n_q = n_q; a.n_kv = kv->n_kv; a.D = D; a.rot = rope->rot_dim; a.neox = rope->neox ? 1 : 0;
    a.max_pos = rope->max_pos; a.capacity = kv->capacity; a.n_regions = kv->n_regions;
    a.pf = pf;
    // q heads and the f16 / f32 mirrors' k and v heads: one thread per channel pair
    const int pairs = (a.q8 ? n_q : n_q + kv->n_kv) * (D / 2);
    dim3 grid((unsigned)dl::ceil_div(pairs, 256), (unsigned)rows);
    int rc = dl::launch_pdl(rope_kv_store_kernel, grid, dim3(256), 0, static_cast<cudaStream_t>(stream),
                            "dl_rope_kv_store: launch", a);
    if (rc != DL_OK || !a.q8) return rc;
    a.pf.n = 0;
    // the q8_0 mirror's k and v: a warp per block of 32 channels, four warps a CTA
    dim3 grid8((unsigned)dl::ceil_div(2 * kv->n_kv * (D / 32), 4), (unsigned)rows);
    return dl::launch_pdl(rope_kv_store_q8_kernel, grid8, dim3(128), 0, static_cast<cudaStream_t>(stream),
                          "dl_rope_kv_store: q8_0 launch", a);
}

}  // extern "C"
