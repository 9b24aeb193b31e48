// The split-KV decode attention kernel (work item = session, KV head, piece), shared by the
// translation unit of the default instances and the one of the instances that carry the
// in-launch merges.  Everything here has internal linkage: each unit owns its instances.
#pragma once
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

namespace {

constexpr int kTile = 32;          // keys per tile
constexpr int kMaxQ = 32;          // queries one work item serves (session rows x group)
constexpr int kMaxCluster = 16;    // pieces of a (session, KV head) merged inside one cluster
constexpr int kCudaCoreMaxQ = 4;   // queries per work item up to which the CUDA-core form is used
constexpr int kMergeWarps = 8;     // the merge's warps per (row, head), as the merge kernel runs them
constexpr int kMergeBatch = 8;     // pieces a merge warp has in flight per pass
constexpr int kTailMaxQ = 8;       // queries per work item up to which the last piece may merge

struct AttnArgs {
    const float *q;
    int64_t q_stride;
    const void *kc, *vc;
    int64_t region_stride;
    int capacity;
    const int32_t *seqlen;
    float *part_o;       // [rows][n_q][max_splits][D]
    float *part_lse;     // [rows][n_q][max_splits]
    int32_t *status;
    float qscale;        // log2(e) / sqrt(D)
    dl_attn_plan plan;
    // rope and KV store fused into the launch (fused = 1): q holds the rows as projected, every
    // work item rotates its queries, and the item whose keys hold a row's position stores that
    // row's rotated k and its v into the mirror before reading them
    int fused;
    const float *k_new, *v_new, *bias;
    int64_t k_stride, v_stride;
    const int32_t *pos;
    const float2 *cs;    // [max_pos][rot/2] (cos, sin)
    void *kc_w, *vc_w;  // f16 patterns, or f32 values in the f32 mirror
    int rot, neox, max_pos;
    // the q8_0 mirror's f16 scale planes (one scale per 32 values of a key row)
    const uint16_t *ksc, *vsc;
    uint16_t *ksc_w, *vsc_w;    // the same planes, written by the fused store
    // merge inside the launch (plan.cluster = C > 0): the results go straight to out / lse_out
    float *out, *lse_out;
    int64_t out_stride;
    DlPrefetch pf;       // L2 prefetches for a later kernel (the producer issues its share)
    // merge by the last piece (tail_merge = 1): every piece writes its partials, counts itself in
    // counters[session][kv head] and the piece that completes the count merges the group's
    // partials into out / lse_out, then clears the count
    int tail_merge;
    int *counters;
};

// Signed bytes `lo`, `lo + 1` of w to floats: the byte flipped to u = q + 128 sits in the low
// mantissa of 2^23; one packed subtraction of 2^23 + 128 leaves q exactly.
__device__ __forceinline__ float2 s8x2_to_f32x2(uint32_t w, uint32_t lo)
{
    w ^= 0x80808080u;
    const float2 b = make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | lo)),
                                 __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541u | lo)));
    return __fadd2_rn(b, make_float2(-8388736.0f, -8388736.0f));
}

// Two signed codes as an f16 pair for the tensor form: `t` holds them flipped to u = q + 128 in
// bytes 0 and 2; with 0x64 above each, the halves read 1024 + u = 1152 + q, and one exact
// subtraction of 1152 leaves q.
__device__ __forceinline__ uint32_t q8_pair_h2(uint32_t t)
{
    const uint32_t b = (t & 0x00FF00FFu) ^ 0x64806480u;         // bytes 1, 3 <- 0x64; u = q ^ 0x80
    const __half2 h = __hsub2(*reinterpret_cast<const __half2 *>(&b), __half2half2(__ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ unsigned short attn_half_clamped(float v)
{
    v = fminf(fmaxf(v, -65504.0f), 65504.0f);
    return __half_as_ushort(__float2half_rn(v));
}

// Channels (i0, i1) of rotary pair j (pairs past rot/2 pass through two at a time).
__device__ __forceinline__ bool rope_pair(int j, int rot, int neox, int &i0, int &i1)
{
    const int rh = rot >> 1;
    if (j < rh) {
        i0 = neox ? j : 2 * j;
        i1 = neox ? j + rh : 2 * j + 1;
        return true;
    }
    i0 = rot + 2 * (j - rh);
    i1 = i0 + 1;
    return false;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Clip a row's device key count to what the plan and the cache cover.
__device__ __forceinline__ int clip_len(int L, int planned, int capacity, int32_t *status, bool report)
{
    const int hi = min(planned, capacity);
    if (L < 1 || L > hi) {
        if (report) dl_status_or(status, DL_STATUS_SEQLEN_RANGE);
        L = L < 1 ? 0 : hi;
    }
    return L;
}

// ---------------------------------------------------------------------------
// Tensor-core form for sessions of several rows (many queries per KV head):
// queries are the 16-row M side of 16x8x16 f16 products.  A producer warp
// streams 32-key stages of K and V through tensor maps (128-byte swizzle, so
// that the matrix loads below are conflict-free) into a ring of mbarrier-
// tracked shared-memory stages.  Stages whose keys all lie below the lowest
// position this command writes do not depend on the previous kernel and are
// issued before waiting on it.  Each consumer warp owns one 16-query tile and
// every KS-th stage (KS = 4 / query tiles), and keeps (m, l, O) for its queries
// in registers: scores S = Q K^T with Q split into two f16 terms (hi + lo,
// near-f32 exact), online softmax in the log2 domain on the accumulator
// fragments, then O += P V with P in f16 (the running maximum's own entry is
// exactly 1).  The warps holding the same queries combine their (m, l, O) in
// shared memory at the end.

__device__ __forceinline__ void ldsm_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two f32 values as bf16 pairs: hi = the values rounded to bf16, lo = the remainders rounded
// to bf16 (hi + lo carries 16 bits of each significand, over f32's whole exponent range).
__device__ __forceinline__ void bf16x2_split(float x, float y, uint32_t &hi, uint32_t &lo)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ uint32_t h2_bits(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 2^x and log2 x through the special-function unit (PTX ex2.approx / lg2.approx: relative error
// about 2^-22, far below the f16 probabilities and the tolerances of the partials)
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_log2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr int kStKeys = 32;                  // keys per stage
constexpr int kMmaConsumers = 4;             // consumer warps
constexpr int kMmaThreads = (kMmaConsumers + 1) * 32;
constexpr int kMmaMaxStages = 8;
constexpr int kHalfTile = kStKeys * 128;     // bytes of 32 keys x 64 dims (one swizzled box)
constexpr int kAttnPreWaitStages = 1;        // stages requested before the wait on the previous kernel
                                             // (more delay the query fetch that follows the wait)

// Ring depth per head dimension: two CTAs fit on an SM.
__host__ __device__ constexpr int mma_stages(int D) { return D == 128 ? 4 : 8; }
// Stages of the ring.  Stage i sits in slot i % S and the consumer warps' stage groups take
// stages round robin, so S must be at least the number of groups (kMmaConsumers): a warp must
// never wait on a slot two fills ahead of what it holds (a parity wait cannot tell the phases
// apart).  The f32 mirror keeps four stages of twice the bytes (one CTA per SM at D = 128).
__host__ __device__ constexpr int attn_stages(int D, int eb) { return eb != 2 ? 4 : mma_stages(D); }
// Bytes of one ring slot: K and V of 32 keys; for the q8_0 mirror the codes, then the K and V
// scales, padded to 1024 bytes (the swizzled destinations' alignment).
__host__ __device__ constexpr uint32_t attn_slot_bytes(int D, int eb)
{
    return eb == 1 ? ((uint32_t)(2 * kStKeys * D + 2 * kStKeys * (D / 16)) + 1023u) & ~1023u
                   : (uint32_t)(2 * kStKeys * D * eb);
}

size_t attn_mma_smem_bytes(int D, int eb = 2)
{
    const size_t stage = attn_slot_bytes(D, eb);                         // K and V of 32 keys
    const size_t qf = (size_t)2 * (D / 16) * 32 * 32;                    // query fragments, 2 tiles
    const size_t qr = (size_t)kMaxQ * D * 4;                             // the queries as they arrive
    const size_t cs = (size_t)DL_MAX_ROWS * (D / 2) * 8;                 // rotary rows (fused form)
    return 1024 + (size_t)attn_stages(D, eb) * stage + qf + qr + cs;    // + alignment slack
}

// OR of `flag` over the consumer warps (uniform result).
__device__ __forceinline__ bool attn_consumers_any(bool flag)
{
    uint32_t r;
    asm volatile("{\n .reg .pred pin, pout;\n setp.ne.u32 pin, %1, 0;\n"
                 " bar.red.or.pred pout, 1, %2, pin;\n selp.u32 %0, 1, 0, pout;\n}"
                 : "=r"(r) : "r"((uint32_t)flag), "r"((uint32_t)(kMmaConsumers * 32)) : "memory");
    return r != 0;
}

// EB: bytes per element of the mirror: 2 the f16 mirror, 4 the f32 mirror, 1 the q8_0 mirror
// (codes; the scales ride along). In the tensor form the f32 mirror's values and the
// probabilities enter as bf16 hi + lo pairs (f32's range, about 16 bits of each significand),
// and the q8_0 codes as exact f16 operands, with each key's block scales applied to the score
// sums and to the V operand.
// MO: the in-launch merges (cluster merge, merge by the last piece) are compiled in; the default
// instances leave them out and are launched only for plans and calls that use neither.
template <int D, bool MMA, int QM, int EB = 2, bool MO = false>
__global__ void __launch_bounds__(kMmaThreads, 2)
decode_attn_tma_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv)
{
    constexpr int NKS = D / 16;     // k-steps of the score product
    constexpr int NDT = D / 8;      // 8-wide column tiles of the output

    constexpr bool KV32 = EB == 4, KVQ8 = EB == 1;
    constexpr int EPB = KVQ8 ? D : 128 / EB;  // elements per box row (q8_0: the whole key row)
    constexpr int NH = D / EPB;               // boxes per key row
    constexpr int S = attn_stages(D, EB);
    static_assert(S >= kMmaConsumers, "every stage group needs a slot of its own in flight");
    static_assert((size_t)kTailMaxQ * kMergeWarps * (D + 2) * 4 <= (size_t)S * attn_slot_bytes(D, EB),
                  "the tail merge's per-warp sums fit in the idle ring");
    constexpr uint32_t kStageBytes = attn_slot_bytes(D, EB);
    constexpr uint32_t kCodeBytes = kStKeys * D;                  // q8_0: codes of 32 keys
    constexpr uint32_t kScaleBytes = kStKeys * (D / 16);          // q8_0: scales of 32 keys
    constexpr uint32_t kVOff = KVQ8 ? kCodeBytes : kStageBytes / 2;   // V within a slot
    constexpr int kRowB = KVQ8 ? D : 128;    // bytes of a box row in shared memory
    constexpr bool kSwz = kRowB == 128;      // 128-byte rows are swizzled, 64-byte rows are not
    const dl_attn_plan &P = a.plan;
    const int cluster = MO ? P.cluster : 0;        // pieces merged inside one cluster (0: none)
    const bool tail = MO && a.tail_merge;          // the last piece merges

    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full[kMmaMaxStages], empty[kMmaMaxStages], qbar, csbar;
    __shared__ int s_len[DL_MAX_ROWS], s_row[DL_MAX_ROWS], s_pos[DL_MAX_ROWS];
    __shared__ unsigned char s_qrow[kMaxQ], s_qhead[kMaxQ];   // query -> (session row, head in group)
    __shared__ float s_plse[kMaxQ], s_mM[kMaxQ], s_mW[kMaxQ];   // cluster merge: this piece's lse, weights
    __shared__ int s_last;                                      // tail merge: this piece completes the count
    // the swizzled boxes want 1024-byte aligned destinations
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~static_cast<uintptr_t>(1023));

    const int item = blockIdx.x;
    int s = 0;
    while (s + 1 < P.n_sessions && item >= P.sess_item0[s + 1]) ++s;
    const int local = item - P.sess_item0[s];
    const int splits = P.sess_splits[s];
    const int h = local / splits, piece = local - h * splits;
    const int rb = P.sess_begin[s], nrows = P.sess_begin[s + 1] - rb;
    const int G = P.n_q / P.n_kv;
    const int Q = nrows * G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const bool producer = warp == kMmaConsumers;

    // warps: NT query tiles (16 queries, tensor form; 8, CUDA-core form) x NS stage groups
    constexpr int TL = MMA ? 16 : QM;
    const int NT = (Q + TL - 1) / TL;
    const int NS = kMmaConsumers / NT;
    const int MT = NT, KS = NS;
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            dla::mbar_init(&full[i], 1);
            dla::mbar_init(&empty[i], (uint32_t)NT);   // released by the warps of one stage group
        }
        dla::mbar_init(&qbar, 1);                       // the session's queries have arrived
        dla::mbar_init(&csbar, 1);                      // the rows' rotary table rows have arrived (fused)
        dla::mbar_init_fence();
    }
    // the key counts come from the caller, not from the previous kernel: read them now
    if (tid < nrows) {
        const int r = P.sess_rows[rb + tid];
        s_row[tid] = r;
        s_len[tid] = clip_len(a.seqlen[r], P.row_keys_max[r], a.capacity, a.status, piece == 0 && h == 0);
        s_pos[tid] = a.fused ? a.pos[r] : 0;            // a caller input as well
    }
    if (tid < Q) {
        s_qrow[tid] = (unsigned char)(tid / G);
        s_qhead[tid] = (unsigned char)(tid - (tid / G) * G);
    }
    __syncthreads();
    int lmax = 0, lmin = 0x7fffffff;
    for (int i = 0; i < nrows; ++i) {
        lmax = max(lmax, s_len[i]);
        lmin = min(lmin, s_len[i]);
    }
    const int k0 = piece * P.chunk;
    const int k1 = min(k0 + P.chunk, lmax);
    const bool idle = k0 >= k1;                 // nothing of this piece is attended
    // (no barrier pending; with a cluster merge the CTA stays to merge its share of the group)
    if (idle && !cluster) {
        // tail merge with no keys in any row of the session: no piece counts, so the first one
        // writes the merge's empty result (out = 0, lse = -inf)
        if (tail && piece == 0 && lmax == 0) {
            for (int e = tid; e < Q * D; e += kMmaThreads) {
                const int qi = e / D, d = e - qi * D;
                const int r = s_row[s_qrow[qi]], hq = h * G + s_qhead[qi];
                a.out[(int64_t)r * a.out_stride + (int64_t)hq * D + d] = 0.f;
                if (d == 0 && a.lse_out) a.lse_out[(int64_t)r * P.n_q + hq] = -INFINITY;
            }
        }
        return;
    }
    const int nst = idle ? 0 : (k1 - k0 + kStKeys - 1) / kStKeys;

    const int reg = P.row_region[s_row[0]];
    unsigned char *ring = smem;
    unsigned char *qfrag = smem + (size_t)S * kStageBytes;
    float *qraw = reinterpret_cast<float *>(qfrag + (size_t)2 * (D / 16) * 32 * 32);   // [Q][D] as stored
    float2 *s_cs = reinterpret_cast<float2 *>(qraw + (size_t)kMaxQ * D);              // [rows][rot/2] (fused)
    // the fused form copies each row's table row (rot/2 (cos, sin) pairs) into shared memory when
    // it is a whole number of 16-byte units; otherwise the rotations read the table in place
    const int rh = a.rot >> 1;
    const bool cs_staged = a.fused && (rh % 2) == 0 && rh > 0;
    auto cs_at = [&](int i, int p, int jp) -> float2 {
        return cs_staged ? s_cs[i * rh + jp] : a.cs[(size_t)p * rh + jp];
    };
    const uint32_t ring_s = dla::smem_u32(ring);
    bool bad = false;

    // the session's queries of this KV head: row r's G heads are contiguous in q
    auto issue_queries = [&]() {
        dla::mbar_expect_tx(&qbar, (uint32_t)(Q * D * 4));
        for (int r = 0; r < nrows; ++r)
            dla::bulk_g2s(qraw + r * G * D, a.q + (int64_t)s_row[r] * a.q_stride + (int64_t)h * G * D,
                          (uint32_t)(G * D * 4), &qbar);
    };
    // fused form: this piece stores the new rows whose positions fall in its keys (a position past
    // every piece goes to the last one); every thread of the CTA a share of the (row, channel pair)
    // elements, each fencing its writes so that the copies issued after the CTA barrier that
    // follows read them
    auto store_new_rows = [&]() {
        const int owner_last = (lmax - 1) / P.chunk;
        const int hp = D / 2;
        if (cs_staged && !dla::mbar_wait(&csbar, 0u)) bad = true;
        if (KVQ8 && !bad) {
            // the q8_0 mirror: a warp per (row, k or v, block of 32 channels), lane = channel, with
            // the separate store's arithmetic (bias, then the rotation of the channel's pair from
            // the unrotated input; d = max|x| / 127 in f32, codes rounded half away from zero)
            constexpr int NB = D / 32;
            for (int t = warp; t < nrows * 2 * NB; t += kMmaConsumers + 1) {
                const int i = t / (2 * NB), rem = t - i * (2 * NB), isv = rem / NB, b = rem - isv * NB;
                const int p = s_pos[i];
                if (min(max(p, 0) / P.chunk, owner_last) != piece) continue;
                if (p < 0 || p >= a.capacity || p >= a.max_pos) {
                    if (rem == 0 && lane == 0) dl_status_or(a.status, DL_STATUS_POS_RANGE);
                    continue;
                }
                const int r = s_row[i];
                const int c = 32 * b + lane;
                float x;
                if (isv) {
                    x = a.v_new[(int64_t)r * a.v_stride + (int64_t)h * D + c];
                    if (a.bias) x += a.bias[(int64_t)(P.n_q + P.n_kv + h) * D + c];
                } else {
                    const float *kr = a.k_new + (int64_t)r * a.k_stride + (int64_t)h * D;
                    const float *bk = a.bias ? a.bias + (int64_t)(P.n_q + h) * D : nullptr;
                    x = kr[c] + (bk ? bk[c] : 0.f);
                    if (c < a.rot) {
                        const int j = a.neox ? (c < rh ? c : c - rh) : (c >> 1);
                        const int i0 = a.neox ? j : 2 * j, i1 = a.neox ? j + rh : 2 * j + 1;
                        const float x0 = kr[i0] + (bk ? bk[i0] : 0.f), x1 = kr[i1] + (bk ? bk[i1] : 0.f);
                        const float2 cs = cs_at(i, p, j);
                        x = c == i0 ? fmaf(x0, cs.x, -x1 * cs.y) : fmaf(x0, cs.y, x1 * cs.x);
                    }
                }
                float m = fabsf(x);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                const float d32 = m / 127.0f;
                int code = 0;
                if (d32 > 0.f) {
                    const float tq = x / d32;
                    const float rr = floorf(fabsf(tq) + 0.5f);
                    code = (int)(tq < 0.f ? -rr : rr);
                    code = max(-127, min(127, code));
                }
                const int64_t base = (int64_t)reg * a.region_stride + ((int64_t)h * a.capacity + p) * D;
                static_cast<int8_t *>(isv ? a.vc_w : a.kc_w)[base + c] = (int8_t)code;
                if (lane == 0) (isv ? a.vsc_w : a.ksc_w)[(base + 32 * b) / 32] = __half_as_ushort(__float2half_rn(d32));
            }
        } else if (!bad) {
#pragma unroll 4
            for (int e = tid; e < nrows * hp; e += kMmaThreads) {
                const int i = e / hp, jp = e - i * hp;
                const int p = s_pos[i];
                if (min(max(p, 0) / P.chunk, owner_last) != piece) continue;
                if (p < 0 || p >= a.capacity || p >= a.max_pos) {
                    if (jp == 0) dl_status_or(a.status, DL_STATUS_POS_RANGE);
                    continue;
                }
                const int r = s_row[i];
                const float *kr = a.k_new + (int64_t)r * a.k_stride + (int64_t)h * D;
                const float *vr = a.v_new + (int64_t)r * a.v_stride + (int64_t)h * D;
                int i0, i1;
                const bool rotate = rope_pair(jp, a.rot, a.neox, i0, i1);
                float k0 = kr[i0], k1 = kr[i1], v0 = vr[i0], v1 = vr[i1];
                if (a.bias) {
                    const float *bk = a.bias + (int64_t)(P.n_q + h) * D;
                    const float *bv = a.bias + (int64_t)(P.n_q + P.n_kv + h) * D;
                    k0 += bk[i0];
                    k1 += bk[i1];
                    v0 += bv[i0];
                    v1 += bv[i1];
                }
                if (rotate) {
                    const float2 t = cs_at(i, p, jp);
                    const float y0 = fmaf(k0, t.x, -k1 * t.y);
                    const float y1 = fmaf(k0, t.y, k1 * t.x);
                    k0 = y0;
                    k1 = y1;
                }
                const int64_t base = (int64_t)reg * a.region_stride + ((int64_t)h * a.capacity + p) * D;
                if constexpr (KV32) {
                    float *kcw = static_cast<float *>(a.kc_w), *vcw = static_cast<float *>(a.vc_w);
                    kcw[base + i0] = k0;
                    kcw[base + i1] = k1;
                    vcw[base + i0] = v0;
                    vcw[base + i1] = v1;
                } else {
                    uint16_t *kcw = static_cast<uint16_t *>(a.kc_w), *vcw = static_cast<uint16_t *>(a.vc_w);
                    kcw[base + i0] = attn_half_clamped(k0);
                    kcw[base + i1] = attn_half_clamped(k1);
                    vcw[base + i0] = attn_half_clamped(v0);
                    vcw[base + i1] = attn_half_clamped(v1);
                }
            }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
    };
    if (producer && idle) {
        if (lane == 0 && a.pf.n > 0) dl_issue_prefetch(a.pf);
        dl_pdl_wait();
        dl_pdl_launch_dependents();
        if (cluster) {                                   // the group's two cluster barriers
            dla::cluster_sync_all();
            dla::cluster_sync_relaxed();
        }
        return;
    }
    if (producer) {
        // keys below the lowest slot this command writes are final before the previous kernel ends:
        // the first few such stages are requested before waiting on it; after the wait come the
        // session's queries (one bulk copy per row: the G heads of this KV head are contiguous),
        // then the rest of the ring, so that those latency-critical lines go first
        const int stable = lmin - 1;
        const int nstable = k1 <= stable ? nst : max(0, (stable - k0) / kStKeys);
        const int npre = min(min(nstable, kAttnPreWaitStages), min(nst, S));
        auto issue_stage = [&](int i) {
            const int st = i % S;
            unsigned char *kd = ring + (size_t)st * kStageBytes;
            unsigned char *vd = kd + kVOff;
            const int key0 = k0 + i * kStKeys;
            const int y = h * a.capacity + key0;
            if constexpr (KVQ8) {
                // codes: one box per key row (keys past the cache read as zero); scales: the
                // stage's keys up to the capacity (a multiple of 4: whole 16-byte units)
                const int nk = min(kStKeys, a.capacity - key0);
                const uint32_t sb = (uint32_t)nk * (D / 16);
                const int64_t s0 = ((int64_t)reg * a.region_stride + (int64_t)y * D) / 32;
                dla::mbar_expect_tx(&full[st], 2 * kCodeBytes + 2 * sb);
                dla::tma_g2s_3d(kd, &tk, 0, y, reg, &full[st]);
                dla::tma_g2s_3d(vd, &tv, 0, y, reg, &full[st]);
                dla::bulk_g2s(kd + 2 * kCodeBytes, a.ksc + s0, sb, &full[st]);
                dla::bulk_g2s(kd + 2 * kCodeBytes + kScaleBytes, a.vsc + s0, sb, &full[st]);
            } else {
                dla::mbar_expect_tx(&full[st], kStageBytes);
#pragma unroll
                for (int hf = 0; hf < NH; ++hf) {
                    dla::tma_g2s_3d(kd + hf * kHalfTile, &tk, hf * EPB, y, reg, &full[st]);
                    dla::tma_g2s_3d(vd + hf * kHalfTile, &tv, hf * EPB, y, reg, &full[st]);
                }
            }
        };
        if (lane == 0) {
            dla::prefetch_tmap(&tk);
            dla::prefetch_tmap(&tv);
            if (cs_staged) {
                // the rows' table rows (a caller input, not the previous kernel's): one bulk copy
                // each; a row whose position is outside the table gets none (and no rotation)
                uint32_t bytes = 0;
                for (int i = 0; i < nrows; ++i)
                    if (s_pos[i] >= 0 && s_pos[i] < a.max_pos) bytes += (uint32_t)rh * 8u;
                dla::mbar_expect_tx(&csbar, bytes);
                for (int i = 0; i < nrows; ++i)
                    if (s_pos[i] >= 0 && s_pos[i] < a.max_pos)
                        dla::bulk_g2s(s_cs + i * rh, a.cs + (size_t)s_pos[i] * rh, (uint32_t)rh * 8u, &csbar);
            }
            for (int i = 0; i < npre; ++i) issue_stage(i);      // npre <= S: every slot is free
            if (a.pf.n > 0) dl_issue_prefetch(a.pf);
        }
        dl_pdl_wait();
        if (lane == 0) issue_queries();
        if (a.fused) {                                       // (an idle piece returned above)
            store_new_rows();
            dla::named_sync(2, kMmaThreads);                 // every new row is stored and fenced
        }
        if (lane == 0) {
            int i = npre;
            for (; i < nst; ++i) {
                const int st = i % S;
                if (i >= S && !dla::mbar_wait(&empty[st], (uint32_t)(((i / S) - 1) & 1))) {
                    bad = true;
                    break;
                }
                issue_stage(i);
            }
            if (bad) {
                // leave no copy in flight: wait (bounded) for the queries, the table rows and the
                // stages issued last
                dla::mbar_wait(&qbar, 0u);
                if (cs_staged) dla::mbar_wait(&csbar, 0u);
                for (int j = max(0, i - S); j < i; ++j) dla::mbar_wait(&full[j % S], (uint32_t)((j / S) & 1));
            }
        }
        dl_pdl_launch_dependents();
        __syncwarp();
        if (cluster) {                                   // the group's two cluster barriers
            dla::cluster_sync_all();
            dla::cluster_sync_relaxed();
        }
        return;
    }

    dl_pdl_wait();
    dl_pdl_launch_dependents();
    if (a.fused && !idle) {
        store_new_rows();
        dla::named_sync(2, kMmaThreads);
    }

    const int mt = warp % MT, grp = warp / MT;
    const int ms = P.max_splits;
    // a stage never arrived: this piece's partials are marked invalid (NaN) for the merge
    auto poison_partials = [&]() {
        for (int e = tid; e < Q * D; e += kMmaConsumers * 32) {
            const int qi = e / D, d = e - qi * D;
            const int rq = s_qrow[qi], gq = s_qhead[qi];
            if (s_len[rq] <= k0) continue;
            if (cluster) {
                qraw[qi * D + d] = __int_as_float(0x7fc00000);
                if (d == 0) s_plse[qi] = __int_as_float(0x7fc00000);
                continue;
            }
            const int64_t pidx = ((int64_t)s_row[rq] * P.n_q + h * G + gq) * ms + piece;
            a.part_o[pidx * D + d] = __int_as_float(0x7fc00000);
            if (d == 0) a.part_lse[pidx] = __int_as_float(0x7fc00000);
        }
    };
    // cluster merge: every piece of the group holds (o, lse) of the rows it covers in its shared
    // memory (o in the query area, lse in s_plse); after the release/acquire cluster barrier each
    // CTA (rank = piece) merges the queries' weights over the pieces that hold keys of their row,
    // then writes every C-th (query, 4-dimension) element; the closing barrier keeps this CTA's
    // results alive until its peers have read them
    auto cluster_merge = [&]() {
        const int C = P.cluster;                     // (called only where cluster != 0)
        __syncwarp();                                // the barrier instructions are warp-aligned
        dla::cluster_sync_all();
        for (int qi = tid; qi < Q; qi += kMmaConsumers * 32) {
            const int rq = s_qrow[qi];
            const int np = min(C, (s_len[rq] + P.chunk - 1) / P.chunk);
            float M = -INFINITY;
            for (int pp = 0; pp < np; ++pp) M = fmaxf(M, dla::ld_dsmem_f32(&s_plse[qi], (uint32_t)pp));
            float W = 0.f;
            for (int pp = 0; pp < np; ++pp) {
                const float l = dla::ld_dsmem_f32(&s_plse[qi], (uint32_t)pp);
                W += l == -INFINITY ? 0.f : __expf(l - M);
            }
            s_mM[qi] = M;
            s_mW[qi] = W;
            if (a.lse_out && qi % C == piece)
                a.lse_out[(int64_t)s_row[rq] * P.n_q + h * G + s_qhead[qi]] = np == 0 ? -INFINITY : M + logf(W);
        }
        dla::named_sync(1, kMmaConsumers * 32);
        for (int e = piece + C * tid; e < Q * (D / 4); e += C * kMmaConsumers * 32) {
            const int qi = e / (D / 4), d4 = e - qi * (D / 4);
            const int rq = s_qrow[qi];
            const int np = min(C, (s_len[rq] + P.chunk - 1) / P.chunk);
            const float M = s_mM[qi];
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int pp = 0; pp < np; ++pp) {
                const float l = dla::ld_dsmem_f32(&s_plse[qi], (uint32_t)pp);
                const float w = l == -INFINITY ? 0.f : __expf(l - M);
                const float4 v = dla::ld_dsmem_f32x4(qraw + qi * D + d4 * 4, (uint32_t)pp);
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
            const float inv = np == 0 ? 0.f : 1.f / s_mW[qi];
            *reinterpret_cast<float4 *>(a.out + (int64_t)s_row[rq] * a.out_stride +
                                        (int64_t)(h * G + s_qhead[qi]) * D + d4 * 4) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
        dla::cluster_sync_relaxed();
    };
    // tail merge: after this piece's partials are written and fenced, one thread counts the piece
    // in; the piece that completes the count of the (session, KV head) (its pieces with keys)
    // clears it for the next launch and merges the group's partials with the merge kernel's
    // arithmetic, operation for operation: per query, eight virtual merge warps (each on every
    // eighth piece, in batches of eight, with its own running maximum) in the ring's shared
    // memory, then their combination
    auto tail_merge = [&]() {
        __threadfence();
        dla::named_sync(1, kMmaConsumers * 32);
        if (tid == 0) {
            const int np_act = min(splits, (lmax + P.chunk - 1) / P.chunk);
            int *cnt = a.counters + ((int64_t)s * P.n_kv + h);
            const int prev = atomicAdd(cnt, 1);
            s_last = prev == np_act - 1 ? 1 : 0;
            if (s_last) atomicExch(cnt, 0);
        }
        dla::named_sync(1, kMmaConsumers * 32);
        if (!s_last) return;
        __threadfence();
        constexpr int VPL = D / 32;
        float *t_acc = reinterpret_cast<float *>(smem);             // [Q][8][D]
        float *t_m = t_acc + (size_t)kTailMaxQ * kMergeWarps * D;   // [Q][8]
        float *t_w = t_m + kTailMaxQ * kMergeWarps;
        for (int pr = warp; pr < Q * kMergeWarps; pr += kMmaConsumers) {
            const int qi = pr / kMergeWarps, vw = pr - qi * kMergeWarps;
            const int rq = s_qrow[qi];
            const int hq = h * G + s_qhead[qi];
            const int np = (s_len[rq] + P.chunk - 1) / P.chunk;
            const float *pl = a.part_lse + ((int64_t)s_row[rq] * P.n_q + hq) * ms;
            const float *po = a.part_o + ((int64_t)s_row[rq] * P.n_q + hq) * ms * D + lane * VPL;
            float Mw = -INFINITY, Ww = 0.f, acc[VPL];
#pragma unroll
            for (int i = 0; i < VPL; ++i) acc[i] = 0.f;
            for (int p0 = vw; p0 < np; p0 += kMergeWarps * kMergeBatch) {
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
            for (int i = 0; i < VPL; ++i) t_acc[((size_t)qi * kMergeWarps + vw) * D + lane * VPL + i] = acc[i];
            if (lane == 0) {
                t_m[qi * kMergeWarps + vw] = Mw;
                t_w[qi * kMergeWarps + vw] = Ww;
            }
        }
        dla::named_sync(1, kMmaConsumers * 32);
        for (int e = tid; e < Q * D; e += kMmaConsumers * 32) {
            const int qi = e / D, d = e - qi * D;
            const int rq = s_qrow[qi];
            const int r = s_row[rq], hq = h * G + s_qhead[qi];
            float *dst = a.out + (int64_t)r * a.out_stride + (int64_t)hq * D;
            if (s_len[rq] == 0) {
                dst[d] = 0.f;
                if (d == 0 && a.lse_out) a.lse_out[(int64_t)r * P.n_q + hq] = -INFINITY;
                continue;
            }
            const float *mq = t_m + qi * kMergeWarps, *wq = t_w + qi * kMergeWarps;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, mq[w]);
            float f[kMergeWarps], Wt = 0.f;
#pragma unroll
            for (int w = 0; w < kMergeWarps; ++w) {
                f[w] = mq[w] == -INFINITY ? 0.f : __expf(mq[w] - M);
                Wt += f[w] * wq[w];
            }
            const float inv = 1.f / Wt;
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < kMergeWarps; ++w) t = fmaf(f[w], t_acc[((size_t)qi * kMergeWarps + w) * D + d], t);
            dst[d] = t * inv;
            if (d == 0 && a.lse_out) a.lse_out[(int64_t)r * P.n_q + hq] = M + logf(Wt);
        }
    };
    if (idle) {                                      // (cluster plans only: the others returned)
        cluster_merge();
        return;
    }
    // fused form: rotate the session's queries in shared memory (bias first), every consumer
    // thread a share of the (query, channel pair) elements, before any of them is read
    auto rotate_queries = [&](bool qok) {
        if (a.fused && qok && cs_staged && !__all_sync(0xffffffffu, dla::mbar_wait(&csbar, 0u))) {
            qok = false;
            bad = true;
        }
        if (a.fused && qok) {
            for (int e = tid; e < Q * (D / 2); e += kMmaConsumers * 32) {
                const int qi = e / (D / 2), jp = e - qi * (D / 2);
                const int ri = s_qrow[qi], head = h * G + s_qhead[qi];
                const int p = s_pos[ri];
                int i0, i1;
                const bool rotate = rope_pair(jp, a.rot, a.neox, i0, i1);
                float *qv = qraw + qi * D;
                float x0 = qv[i0], x1 = qv[i1];
                if (a.bias) {
                    x0 += a.bias[(int64_t)head * D + i0];
                    x1 += a.bias[(int64_t)head * D + i1];
                }
                if (rotate && p >= 0 && p < a.max_pos) {
                    const float2 t = cs_at(ri, p, jp);
                    const float y0 = fmaf(x0, t.x, -x1 * t.y);
                    const float y1 = fmaf(x0, t.y, x1 * t.x);
                    x0 = y0;
                    x1 = y1;
                }
                qv[i0] = x0;
                qv[i1] = x1;
            }
        }
        if (a.fused) dla::named_sync(1, kMmaConsumers * 32);
    };
    // combine area (the ring, idle once every stage is consumed): [4 warps][16 rows][CP], m, l
    constexpr int CP = D + 8;                          // padded row: the fragment stores spread over banks
    float *co = reinterpret_cast<float *>(smem);
    float *cm = co + kMmaConsumers * 16 * CP;
    float *cl = cm + kMmaConsumers * 16;
    if constexpr (MMA) {
        // ---- query operand fragments (log2-domain scaled, hi + lo f16 terms) in shared memory:
        // [query tile][k-step][hi, lo][lane] 16 bytes = a0..a3.  On the f32 mirror the terms are
        // bf16 (f32's exponent range) and the lane quad c of k-step ks holds dimensions
        // 16 ks + 4c .. 16 ks + 4c + 3 (one 16-byte read of a key row).  On the q8_0 mirror the
        // dimensions are permuted within each 32-dimension block (the order of a sum is free when
        // both operands follow it): k-step 2b + e, column pair p of lane quad c holds dimensions
        // 32b + 8c + 4e + 2p + {0, 1}, so that a key's codes of both k-steps of block b are the 8
        // contiguous bytes at 32b + 8c of its row
        const bool qok = __all_sync(0xffffffffu, dla::mbar_wait(&qbar, 0u));
        if (!qok) bad = true;
        rotate_queries(qok);
        for (int fi = tid; fi < MT * NKS * 32; fi += kMmaConsumers * 32) {
            const int t = fi & 31, ks = (fi >> 5) % NKS, qt = (fi >> 5) / NKS;
            const int gg = t >> 2, cc = t & 3;
            const int q0i = qt * 16 + gg, q1i = q0i + 8;
            const float *q0 = q0i < Q ? qraw + q0i * D : nullptr;
            const float *q1 = q1i < Q ? qraw + q1i * D : nullptr;
            uint32_t hv[4], lv[4];
    #pragma unroll
            for (int part = 0; part < 4; ++part) {
                const float *src = (part & 1) ? q1 : q0;
                const int col = KVQ8 ? 32 * (ks >> 1) + 8 * cc + 4 * (ks & 1) + (part >> 1) * 2
                              : KV32 ? ks * 16 + 4 * cc + (part >> 1) * 2
                                     : ks * 16 + 2 * cc + (part >> 1) * 8;
                float2 v = make_float2(0.f, 0.f);
                if (src) v = *reinterpret_cast<const float2 *>(src + col);
                v.x *= a.qscale;
                v.y *= a.qscale;
                if constexpr (KV32) {
                    bf16x2_split(v.x, v.y, hv[part], lv[part]);
                } else {
                    const __half2 hq = __floats2half2_rn(v.x, v.y);
                    const float2 hf = __half22float2(hq);
                    hv[part] = *reinterpret_cast<const uint32_t *>(&hq);
                    lv[part] = h2_bits(v.x - hf.x, v.y - hf.y);
                }
            }
            uint4 *dst = reinterpret_cast<uint4 *>(qfrag + (size_t)(fi >> 5) * 1024 + t * 16);
            dst[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            dst[32] = make_uint4(lv[0], lv[1], lv[2], lv[3]);
        }
        dla::named_sync(1, kMmaConsumers * 32);
        const unsigned char *myq = qfrag + (size_t)mt * NKS * 1024 + lane * 16;
        const int r0 = mt * 16 + g, r1 = r0 + 8;
        const int len0 = r0 < Q ? s_len[s_qrow[r0]] : 0;
        const int len1 = r1 < Q ? s_len[s_qrow[r1]] : 0;

        float o[NDT][4];
    #pragma unroll
        for (int i = 0; i < NDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

        for (int i = grp; i < nst; i += KS) {
            const int st = i % S;
            if (!__all_sync(0xffffffffu, dla::mbar_wait(&full[st], (uint32_t)((i / S) & 1)))) {
                bad = true;
                break;
            }
            const uint32_t ksm = ring_s + (uint32_t)st * kStageBytes;
            const uint32_t vsm = ksm + kVOff;
            const int kb0 = k0 + i * kStKeys;
            if (kb0 + kStKeys > k1) {
                // keys past the piece may hold anything (even NaN) in the V rows: zero them (the
                // q8_0 mirror's codes are finite; zeroing their scales is enough)
                if constexpr (KVQ8) {
                    uint16_t *vs = reinterpret_cast<uint16_t *>(ring + (size_t)st * kStageBytes + 2 * kCodeBytes +
                                                                kScaleBytes);
                    for (int e = lane; e < kStKeys * (D / 32); e += 32)
                        if (kb0 + e / (D / 32) >= k1) vs[e] = 0;
                } else {
                    unsigned char *vrow = ring + (size_t)st * kStageBytes + kStageBytes / 2;
                    for (int e = lane; e < NH * kStKeys * 8; e += 32) {
                        const int hf = e / (kStKeys * 8), rem = e - hf * kStKeys * 8;
                        const int key = rem >> 3;
                        if (kb0 + key >= k1)
                            *reinterpret_cast<uint4 *>(vrow + hf * kHalfTile + rem * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                dla::fence_proxy_async();
                __syncwarp();
            }

            // scores of 32 keys: four 8-key column tiles, hi and lo terms in independent chains
            float sc[4][4], sl[4][4];
    #pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
                sl[nt][0] = sl[nt][1] = sl[nt][2] = sl[nt][3] = 0.f;
            }
            if constexpr (KV32) {
                // lane (g, c) reads key g's four dimensions 16 ks + 4c .. + 3 (one 16-byte chunk
                // of its swizzled 128-byte box row) and splits them into bf16 hi + lo; the products
                // q_hi k_hi, q_lo k_hi and q_hi k_lo keep about 16 bits of each operand
                const unsigned char *kst = ring + (size_t)st * kStageBytes;
    #pragma unroll
                for (int ks = 0; ks < NKS; ++ks) {
                    const uint4 qa = *reinterpret_cast<const uint4 *>(myq + ks * 1024);
                    const uint4 qb = *reinterpret_cast<const uint4 *>(myq + ks * 1024 + 512);
                    const uint32_t qh[4] = {qa.x, qa.y, qa.z, qa.w}, ql[4] = {qb.x, qb.y, qb.z, qb.w};
                    const int chunk = 4 * (ks & 1) + c;
    #pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        const int key = nt * 8 + g;
                        const float4 kf = *reinterpret_cast<const float4 *>(
                            kst + (ks >> 1) * kHalfTile + key * 128 + ((chunk ^ (key & 7)) << 4));
                        uint32_t h0, l0, h1, l1;
                        bf16x2_split(kf.x, kf.y, h0, l0);
                        bf16x2_split(kf.z, kf.w, h1, l1);
                        mma_bf16(sc[nt], qh, h0, h1);
                        mma_bf16(sl[nt], ql, h0, h1);
                        mma_bf16(sl[nt], qh, l0, l1);
                    }
                }
            } else if constexpr (KVQ8) {
                // per 32-dimension block b: lane (g, c) takes key g's 8 codes at 32b + 8c (both
                // k-steps of the block), the block's products accumulate apart and are scaled by
                // the key's scale of that block (the columns 2c, 2c + 1 of the fragment)
                const unsigned char *kcs = ring + (size_t)st * kStageBytes;
                const uint16_t *ksc = reinterpret_cast<const uint16_t *>(kcs + 2 * kCodeBytes);
    #pragma unroll
                for (int b = 0; b < D / 32; ++b) {
                    const uint4 qa = *reinterpret_cast<const uint4 *>(myq + (2 * b) * 1024);
                    const uint4 qb = *reinterpret_cast<const uint4 *>(myq + (2 * b) * 1024 + 512);
                    const uint4 qc = *reinterpret_cast<const uint4 *>(myq + (2 * b + 1) * 1024);
                    const uint4 qd = *reinterpret_cast<const uint4 *>(myq + (2 * b + 1) * 1024 + 512);
                    const uint32_t qh0[4] = {qa.x, qa.y, qa.z, qa.w}, ql0[4] = {qb.x, qb.y, qb.z, qb.w};
                    const uint32_t qh1[4] = {qc.x, qc.y, qc.z, qc.w}, ql1[4] = {qd.x, qd.y, qd.z, qd.w};
                    const int byte = 32 * b + 8 * c, ch = byte >> 4;
    #pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        const int key = nt * 8 + g;
                        const uint2 w = *reinterpret_cast<const uint2 *>(
                            kcs + key * kRowB + ((kSwz ? (ch ^ (key & 7)) : ch) << 4) + (byte & 8));
                        const uint32_t b0 = q8_pair_h2(__byte_perm(w.x, 0u, 0x3120u));   // dims +0, +1
                        const uint32_t b1 = q8_pair_h2(__byte_perm(w.x, 0u, 0x1302u));   // dims +2, +3
                        const uint32_t b2 = q8_pair_h2(__byte_perm(w.y, 0u, 0x3120u));
                        const uint32_t b3 = q8_pair_h2(__byte_perm(w.y, 0u, 0x1302u));
                        float th[4] = {0.f, 0.f, 0.f, 0.f}, tl[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_f16(th, qh0, b0, b1);
                        mma_f16(tl, ql0, b0, b1);
                        mma_f16(th, qh1, b2, b3);
                        mma_f16(tl, ql1, b2, b3);
                        const int kc0 = nt * 8 + 2 * c;
                        const float d0 = __half2float(__ushort_as_half(ksc[kc0 * (D / 32) + b]));
                        const float d1 = __half2float(__ushort_as_half(ksc[(kc0 + 1) * (D / 32) + b]));
                        sc[nt][0] = fmaf(d0, th[0] + tl[0], sc[nt][0]);
                        sc[nt][1] = fmaf(d1, th[1] + tl[1], sc[nt][1]);
                        sc[nt][2] = fmaf(d0, th[2] + tl[2], sc[nt][2]);
                        sc[nt][3] = fmaf(d1, th[3] + tl[3], sc[nt][3]);
                    }
                }
            } else
    #pragma unroll
            for (int ks = 0; ks < NKS; ks += 2) {
                const uint4 qa = *reinterpret_cast<const uint4 *>(myq + ks * 1024);
                const uint4 qb = *reinterpret_cast<const uint4 *>(myq + ks * 1024 + 512);
                const uint4 qc = *reinterpret_cast<const uint4 *>(myq + (ks + 1) * 1024);
                const uint4 qd = *reinterpret_cast<const uint4 *>(myq + (ks + 1) * 1024 + 512);
                const uint32_t qh0[4] = {qa.x, qa.y, qa.z, qa.w}, ql0[4] = {qb.x, qb.y, qb.z, qb.w};
                const uint32_t qh1[4] = {qc.x, qc.y, qc.z, qc.w}, ql1[4] = {qd.x, qd.y, qd.z, qd.w};
                const int ch = 2 * ks + (lane >> 3);                 // 16-byte chunk of the key row
                const uint32_t half_off = (uint32_t)(ch >> 3) * kHalfTile;
    #pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int key = nt * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(b0, b1, b2, b3, ksm + half_off + (uint32_t)(key * 128 + (((ch & 7) ^ (key & 7)) << 4)));
                    mma_f16(sc[nt], qh0, b0, b1);
                    mma_f16(sl[nt], ql0, b0, b1);
                    mma_f16(sc[nt], qh1, b2, b3);
                    mma_f16(sl[nt], ql1, b2, b3);
                }
            }
            // mask keys past each row's count, online softmax per row (quad of lanes = one row)
            float mx0 = -INFINITY, mx1 = -INFINITY;
    #pragma unroll
            for (int nt = 0; nt < 4; ++nt)
    #pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = kb0 + nt * 8 + 2 * c + e;
                    const float v0 = sc[nt][e] + sl[nt][e], v1 = sc[nt][2 + e] + sl[nt][2 + e];
                    sc[nt][e] = key < len0 ? v0 : -INFINITY;
                    sc[nt][2 + e] = key < len1 ? v1 : -INFINITY;
                    mx0 = fmaxf(mx0, sc[nt][e]);
                    mx1 = fmaxf(mx1, sc[nt][2 + e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float al0 = (mn0 == -INFINITY) ? 1.f : fast_exp2(m0 - mn0);
            const float al1 = (mn1 == -INFINITY) ? 1.f : fast_exp2(m1 - mn1);
    #pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                sc[nt][0] = sc[nt][0] == -INFINITY ? 0.f : fast_exp2(sc[nt][0] - mn0);
                sc[nt][1] = sc[nt][1] == -INFINITY ? 0.f : fast_exp2(sc[nt][1] - mn0);
                sc[nt][2] = sc[nt][2] == -INFINITY ? 0.f : fast_exp2(sc[nt][2] - mn1);
                sc[nt][3] = sc[nt][3] == -INFINITY ? 0.f : fast_exp2(sc[nt][3] - mn1);
            }
            float ps0 = 0.f, ps1 = 0.f;
    #pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                ps0 += sc[nt][0] + sc[nt][1];
                ps1 += sc[nt][2] + sc[nt][3];
            }
            l0 = l0 * al0 + ps0;
            l1 = l1 * al1 + ps1;
            m0 = mn0;
            m1 = mn1;
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
    #pragma unroll
                for (int j = 0; j < NDT; ++j) {
                    o[j][0] *= al0;
                    o[j][1] *= al0;
                    o[j][2] *= al1;
                    o[j][3] *= al1;
                }
            }
            // O += P V over two 16-key steps: two 8-wide output tiles per transposed 4-matrix load
            if constexpr (KV32) {
                // output column n of tile j is dimension (D / 8) n + j: lane (g, c) reads the D / 8
                // contiguous values at (D / 8) g of its keys 2c, 2c + 1, 2c + 8, 2c + 9, four at a
                // time, and P and V enter as bf16 hi + lo (P_hi V_hi + P_lo V_hi + P_hi V_lo)
                const unsigned char *vst = ring + (size_t)st * kStageBytes + kVOff;
                constexpr int VB = D / 8;
                const int d0 = VB * g;
                const unsigned char *vbox = vst + (d0 >> 5) * kHalfTile;
                const int ch0 = (d0 & 31) >> 2;
    #pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    uint32_t ph[4], pl[4];
                    bf16x2_split(sc[2 * kk][0], sc[2 * kk][1], ph[0], pl[0]);
                    bf16x2_split(sc[2 * kk][2], sc[2 * kk][3], ph[1], pl[1]);
                    bf16x2_split(sc[2 * kk + 1][0], sc[2 * kk + 1][1], ph[2], pl[2]);
                    bf16x2_split(sc[2 * kk + 1][2], sc[2 * kk + 1][3], ph[3], pl[3]);
    #pragma unroll
                    for (int m = 0; m < VB / 4; ++m) {
                        float4 w[4];
    #pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int key = kk * 16 + 2 * c + (u & 1) + (u >> 1) * 8;
                            w[u] = *reinterpret_cast<const float4 *>(vbox + key * 128 + (((ch0 + m) ^ (key & 7)) << 4));
                        }
                        const float v0[4] = {w[0].x, w[0].y, w[0].z, w[0].w}, v1[4] = {w[1].x, w[1].y, w[1].z, w[1].w};
                        const float v2[4] = {w[2].x, w[2].y, w[2].z, w[2].w}, v3[4] = {w[3].x, w[3].y, w[3].z, w[3].w};
    #pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            uint32_t bh0, bl0, bh1, bl1;
                            bf16x2_split(v0[jj], v1[jj], bh0, bl0);
                            bf16x2_split(v2[jj], v3[jj], bh1, bl1);
                            float (&oj)[4] = o[4 * m + jj];
                            mma_bf16(oj, ph, bh0, bh1);
                            mma_bf16(oj, pl, bh0, bh1);
                            mma_bf16(oj, ph, bl0, bl1);
                        }
                    }
                }
            } else if constexpr (KVQ8) {
                // output column n of tile j is dimension (D / 8) n + j, so that lane (g, c) reads
                // the D / 8 contiguous codes at (D / 8) g of its keys 2c, 2c + 1, 2c + 8, 2c + 9 (all
                // in block g / (256 / D)) and takes byte j of them for tile j; each pair is scaled
                // by its keys' scales of that block as it becomes an f16 operand
                const unsigned char *vcs = ring + (size_t)st * kStageBytes + kCodeBytes;
                const uint16_t *vsc =
                    reinterpret_cast<const uint16_t *>(ring + (size_t)st * kStageBytes + 2 * kCodeBytes + kScaleBytes);
                constexpr int VB = D / 8;                 // codes per lane and key
                const int blk = (VB * g) >> 5;
    #pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const uint32_t pa[4] = {h2_bits(sc[2 * kk][0], sc[2 * kk][1]), h2_bits(sc[2 * kk][2], sc[2 * kk][3]),
                                            h2_bits(sc[2 * kk + 1][0], sc[2 * kk + 1][1]),
                                            h2_bits(sc[2 * kk + 1][2], sc[2 * kk + 1][3])};
                    uint32_t wv[4][VB / 4];
                    __half2 dv[2];
    #pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int key = kk * 16 + 2 * c + (u & 1) + (u >> 1) * 8;
                        const unsigned char *row = vcs + key * kRowB;
                        if constexpr (VB == 16) {
                            const uint4 w = *reinterpret_cast<const uint4 *>(row + ((kSwz ? (g ^ (key & 7)) : g) << 4));
                            wv[u][0] = w.x; wv[u][1] = w.y; wv[u][2] = w.z; wv[u][3] = w.w;
                        } else {
                            const uint2 w = *reinterpret_cast<const uint2 *>(row + VB * g);
                            wv[u][0] = w.x; wv[u][1] = w.y;
                        }
                    }
    #pragma unroll
                    for (int u2 = 0; u2 < 2; ++u2) {
                        const int key = kk * 16 + 2 * c + u2 * 8;
                        dv[u2] = __halves2half2(__ushort_as_half(vsc[key * (D / 32) + blk]),
                                                __ushort_as_half(vsc[(key + 1) * (D / 32) + blk]));
                    }
    #pragma unroll
                    for (int j = 0; j < NDT; ++j) {
                        const uint32_t sel = (uint32_t)(j & 3) | ((uint32_t)(4 + (j & 3)) << 8);
                        uint32_t b01 = q8_pair_h2(__byte_perm(wv[0][j >> 2], wv[1][j >> 2], sel));
                        uint32_t b23 = q8_pair_h2(__byte_perm(wv[2][j >> 2], wv[3][j >> 2], sel));
                        const __half2 v01 = __hmul2(*reinterpret_cast<const __half2 *>(&b01), dv[0]);
                        const __half2 v23 = __hmul2(*reinterpret_cast<const __half2 *>(&b23), dv[1]);
                        mma_f16(o[j], pa, *reinterpret_cast<const uint32_t *>(&v01),
                                *reinterpret_cast<const uint32_t *>(&v23));
                    }
                }
            } else
    #pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const uint32_t pa[4] = {h2_bits(sc[2 * kk][0], sc[2 * kk][1]), h2_bits(sc[2 * kk][2], sc[2 * kk][3]),
                                        h2_bits(sc[2 * kk + 1][0], sc[2 * kk + 1][1]),
                                        h2_bits(sc[2 * kk + 1][2], sc[2 * kk + 1][3])};
                const int vkey = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    #pragma unroll
                for (int j = 0; j < NDT / 2; ++j) {
                    const int ch = 2 * j + (lane >> 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(b0, b1, b2, b3, vsm + (uint32_t)(ch >> 3) * kHalfTile +
                                                  (uint32_t)(vkey * 128 + (((ch & 7) ^ (vkey & 7)) << 4)));
                    mma_f16(o[2 * j], pa, b0, b1);
                    mma_f16(o[2 * j + 1], pa, b2, b3);
                }
            }
            __syncwarp();
            if (lane == 0) dla::mbar_arrive(&empty[st]);      // the stage is free for the producer
        }
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

        if (attn_consumers_any(bad)) {
            poison_partials();
            if (cluster) cluster_merge();
            else if (tail) tail_merge();
            return;
        }
    #pragma unroll
        for (int j = 0; j < NDT; ++j) {
            if constexpr (KVQ8 || KV32) {            // column n of tile j is dimension (D / 8) n + j
                const int d0 = (D / 8) * 2 * c + j, d1 = d0 + D / 8;
                co[(warp * 16 + g) * CP + d0] = o[j][0];
                co[(warp * 16 + g) * CP + d1] = o[j][1];
                co[(warp * 16 + g + 8) * CP + d0] = o[j][2];
                co[(warp * 16 + g + 8) * CP + d1] = o[j][3];
            } else {
                *reinterpret_cast<float2 *>(co + (warp * 16 + g) * CP + j * 8 + 2 * c) = make_float2(o[j][0], o[j][1]);
                *reinterpret_cast<float2 *>(co + (warp * 16 + g + 8) * CP + j * 8 + 2 * c) =
                    make_float2(o[j][2], o[j][3]);
            }
        }
        if (c == 0) {
            cm[warp * 16 + g] = m0;
            cm[warp * 16 + g + 8] = m1;
            cl[warp * 16 + g] = l0;
            cl[warp * 16 + g + 8] = l1;
        }
    } else {
        // ---- CUDA-core form: warp (query group qg of up to QM queries, stage group sg); lane = key
        // for the scores, lanes over the dimensions for P.V
        constexpr int DPL = D / 32;                 // dimensions per lane
        const int qg = warp % NT, sg = warp / NT;
        const int qb = qg * QM, nq = min(QM, Q - qb);
        const float *qs = qraw;                      // [Q][D] f32 as stored; the scale goes on the score
        float *pb = reinterpret_cast<float *>(qfrag) + warp * QM * kStKeys;   // this warp's probabilities
        if (!__all_sync(0xffffffffu, dla::mbar_wait(&qbar, 0u))) bad = true;
        rotate_queries(!bad);
        int lenq[QM];
#pragma unroll
        for (int q = 0; q < QM; ++q) lenq[q] = q < nq ? s_len[s_qrow[qb + q]] : 0;
        float2 o[QM][DPL];                           // (even keys, odd keys) of each dimension
        float mq[QM], lq[QM];
#pragma unroll
        for (int q = 0; q < QM; ++q) {
            mq[q] = -INFINITY;
            lq[q] = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[q][e] = make_float2(0.f, 0.f);
        }
        const int d0 = DPL * lane, dch = d0 / (16 / EB);     // 16-byte chunk of the lane's dimensions
        for (int i = sg; sg < NS && i < nst; i += NS) {
            const int st = i % S;
            if (!__all_sync(0xffffffffu, dla::mbar_wait(&full[st], (uint32_t)((i / S) & 1)))) {
                bad = true;
                break;
            }
            const unsigned char *kst = ring + (size_t)st * kStageBytes;
            const unsigned char *vst = kst + kVOff;
            const int kb0 = k0 + i * kStKeys;
            if (kb0 + kStKeys > k1) {
                // keys past the piece may hold anything (even NaN) in the V rows: zero them (the
                // q8_0 mirror's codes are finite; zeroing their scales is enough)
                if constexpr (KVQ8) {
                    uint16_t *vs = reinterpret_cast<uint16_t *>(ring + (size_t)st * kStageBytes + 2 * kCodeBytes +
                                                                kScaleBytes);
                    for (int e = lane; e < kStKeys * (D / 32); e += 32)
                        if (kb0 + e / (D / 32) >= k1) vs[e] = 0;
                } else {
                    unsigned char *vrow = ring + (size_t)st * kStageBytes + kVOff;
                    for (int e = lane; e < NH * kStKeys * 8; e += 32) {
                        const int hf = e / (kStKeys * 8), rem = e - hf * kStKeys * 8;
                        if (kb0 + (rem >> 3) >= k1)
                            *reinterpret_cast<uint4 *>(vrow + hf * kHalfTile + rem * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                dla::fence_proxy_async();
                __syncwarp();
            }
            // scores: lane = key, its row read 16 bytes at a time through the swizzle
            float2 sc[QM], sd[QM];                 // partial sums per score: even, odd chunks x
#pragma unroll                                     // even, odd dimensions
            for (int q = 0; q < QM; ++q) sc[q] = sd[q] = make_float2(0.f, 0.f);
            if constexpr (KVQ8) {
                // the key's row of D codes, 16 per chunk, two chunks per block of 32; each block's
                // dot product is scaled by the key's scale of that block
                const unsigned char *krow = kst + lane * kRowB;
                const uint16_t *ksr = reinterpret_cast<const uint16_t *>(kst + 2 * kCodeBytes) + lane * (D / 32);
#pragma unroll 1
                for (int b = 0; b < D / 32; ++b) {
                    float2 tq[QM];
#pragma unroll
                    for (int q = 0; q < QM; ++q) tq[q] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int ch = 2 * b + hh;
                        const uint4 w = *reinterpret_cast<const uint4 *>(
                            krow + ((kSwz ? (ch ^ (lane & 7)) : ch) << 4));
                        const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
                        float2 kf[8];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            kf[2 * u] = s8x2_to_f32x2(wd[u], 0);
                            kf[2 * u + 1] = s8x2_to_f32x2(wd[u], 2);
                        }
#pragma unroll
                        for (int q = 0; q < QM; ++q) {
                            if (q < nq) {
                                const float *qv = qs + (qb + q) * D + ch * 16;
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const float4 qa = *reinterpret_cast<const float4 *>(qv + 4 * u);
                                    tq[q] = __ffma2_rn(make_float2(qa.x, qa.y), kf[2 * u], tq[q]);
                                    tq[q] = __ffma2_rn(make_float2(qa.z, qa.w), kf[2 * u + 1], tq[q]);
                                }
                            }
                        }
                    }
                    const float dk = __half2float(__ushort_as_half(ksr[b]));
#pragma unroll
                    for (int q = 0; q < QM; ++q) sc[q] = __ffma2_rn(make_float2(dk, dk), tq[q], sc[q]);
                }
            } else if constexpr (KV32) {
                // 16 bytes = 4 dimensions per chunk
#pragma unroll 2
                for (int ch = 0; ch < D / 4; ++ch) {
                    const float4 kf = *reinterpret_cast<const float4 *>(kst + (ch >> 3) * kHalfTile + lane * 128 +
                                                                        (((ch & 7) ^ (lane & 7)) << 4));
#pragma unroll
                    for (int q = 0; q < QM; ++q) {
                        if (q < nq) {
                            const float4 qa = *reinterpret_cast<const float4 *>(qs + (qb + q) * D + ch * 4);
                            float2 t = (ch & 1) ? sd[q] : sc[q];
                            t = __ffma2_rn(make_float2(qa.x, qa.y), make_float2(kf.x, kf.y), t);
                            t = __ffma2_rn(make_float2(qa.z, qa.w), make_float2(kf.z, kf.w), t);
                            if (ch & 1) sd[q] = t; else sc[q] = t;
                        }
                    }
                }
            } else
#pragma unroll 4
            for (int ch = 0; ch < D / 8; ++ch) {
                const uint4 kv = *reinterpret_cast<const uint4 *>(kst + (ch >> 3) * kHalfTile + lane * 128 +
                                                                  (((ch & 7) ^ (lane & 7)) << 4));
                const float2 k01 = __half22float2(*reinterpret_cast<const __half2 *>(&kv.x));
                const float2 k23 = __half22float2(*reinterpret_cast<const __half2 *>(&kv.y));
                const float2 k45 = __half22float2(*reinterpret_cast<const __half2 *>(&kv.z));
                const float2 k67 = __half22float2(*reinterpret_cast<const __half2 *>(&kv.w));
#pragma unroll
                for (int q = 0; q < QM; ++q) {
                    if (q < nq) {
                        const float4 qa = *reinterpret_cast<const float4 *>(qs + (qb + q) * D + ch * 8);
                        const float4 qc = *reinterpret_cast<const float4 *>(qs + (qb + q) * D + ch * 8 + 4);
                        float2 t = (ch & 1) ? sd[q] : sc[q];
                        t = __ffma2_rn(make_float2(qa.x, qa.y), k01, t);
                        t = __ffma2_rn(make_float2(qa.z, qa.w), k23, t);
                        t = __ffma2_rn(make_float2(qc.x, qc.y), k45, t);
                        t = __ffma2_rn(make_float2(qc.z, qc.w), k67, t);
                        if (ch & 1) sd[q] = t; else sc[q] = t;
                    }
                }
            }
            // online softmax per query over the stage's 32 keys: the queries' maxima reduced
            // side by side, each lane keeping its own part of the sums (reduced after the loop)
            const int key = kb0 + lane;
            float ps[QM], mx[QM];
#pragma unroll
            for (int q = 0; q < QM; ++q) {
                ps[q] = q < nq && key < lenq[q] ? ((sc[q].x + sd[q].x) + (sc[q].y + sd[q].y)) * a.qscale : -INFINITY;
                mx[q] = ps[q];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int q = 0; q < QM; ++q) mx[q] = fmaxf(mx[q], __shfl_xor_sync(0xffffffffu, mx[q], off));
#pragma unroll
            for (int q = 0; q < QM; ++q) {
                const float mn = fmaxf(mq[q], mx[q]);
                // rescale of what is summed so far: 1 while no key is attended, 0 at the first one
                const float al = mn == -INFINITY ? 1.f : mq[q] == -INFINITY ? 0.f : fast_exp2(mq[q] - mn);
                ps[q] = ps[q] == -INFINITY ? 0.f : fast_exp2(ps[q] - mn);
                lq[q] = lq[q] * al + ps[q];
                mq[q] = mn;
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[q][e] = __fmul2_rn(o[q][e], make_float2(al, al));
            }
            // O += P V: lane holds dimensions d0 .. d0 + DPL - 1; the probabilities go through this
            // warp's shared buffer and come back four keys per broadcast load
            for (int q = 0; q < QM; ++q)
                if (q < nq) pb[q * kStKeys + lane] = ps[q];
            __syncwarp();
            const unsigned char *vcol = KVQ8 ? vst + (d0 & 15) : vst + (dch >> 3) * kHalfTile + (d0 & (16 / EB - 1)) * EB;
            const uint16_t *vsr = reinterpret_cast<const uint16_t *>(kst + 2 * kCodeBytes + kScaleBytes) + d0 / 32;
#pragma unroll 4
            for (int j4 = 0; j4 < kStKeys; j4 += 4) {
                float v[4][DPL];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int j = j4 + kk;
                    const unsigned char *vp = KVQ8 ? vcol + j * kRowB + ((kSwz ? ((d0 >> 4) ^ (j & 7)) : (d0 >> 4)) << 4)
                                                   : vcol + j * 128 + (((dch & 7) ^ (j & 7)) << 4);
                    if constexpr (KVQ8) {
                        // DPL codes of key j, times the key's scale of their block
                        const float dv = __half2float(__ushort_as_half(vsr[j * (D / 32)]));
                        if constexpr (DPL == 4) {
                            const uint32_t w = *reinterpret_cast<const uint32_t *>(vp);
                            const float2 c01 = s8x2_to_f32x2(w, 0), c23 = s8x2_to_f32x2(w, 2);
                            v[kk][0] = dv * c01.x; v[kk][1] = dv * c01.y; v[kk][2] = dv * c23.x; v[kk][3] = dv * c23.y;
                        } else {
                            const uint32_t w = *reinterpret_cast<const uint16_t *>(vp);
                            const float2 c01 = s8x2_to_f32x2(w, 0);
                            v[kk][0] = dv * c01.x; v[kk][1] = dv * c01.y;
                        }
                    } else if constexpr (KV32 && DPL == 4) {
                        const float4 w = *reinterpret_cast<const float4 *>(vp);
                        v[kk][0] = w.x; v[kk][1] = w.y; v[kk][2] = w.z; v[kk][3] = w.w;
                    } else if constexpr (KV32) {
                        const float2 w = *reinterpret_cast<const float2 *>(vp);
                        v[kk][0] = w.x; v[kk][1] = w.y;
                    } else if constexpr (DPL == 4) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(vp);
                        const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
                        const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
                        v[kk][0] = v01.x; v[kk][1] = v01.y; v[kk][2] = v23.x; v[kk][3] = v23.y;
                    } else {
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(vp);
                        const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&w));
                        v[kk][0] = v01.x; v[kk][1] = v01.y;
                    }
                }
#pragma unroll
                for (int q = 0; q < QM; ++q) {
                    if (q < nq) {
                        const float4 p4 = *reinterpret_cast<const float4 *>(pb + q * kStKeys + j4);
                        const float2 p01 = make_float2(p4.x, p4.y), p23 = make_float2(p4.z, p4.w);
#pragma unroll
                        for (int e = 0; e < DPL; ++e) {
                            o[q][e] = __ffma2_rn(p01, make_float2(v[0][e], v[1][e]), o[q][e]);
                            o[q][e] = __ffma2_rn(p23, make_float2(v[2][e], v[3][e]), o[q][e]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) dla::mbar_arrive(&empty[st]);      // the stage is free for the producer
        }
        if (attn_consumers_any(bad)) {
            poison_partials();
            if (cluster) cluster_merge();
            else if (tail) tail_merge();
            return;
        }
#pragma unroll
        for (int q = 0; q < QM; ++q) lq[q] = warp_sum(lq[q]);
        if (sg < NS) {
#pragma unroll
            for (int q = 0; q < QM; ++q) {
                if (q < nq) {
#pragma unroll
                    for (int e = 0; e < DPL; ++e) co[(warp * 16 + q) * CP + d0 + e] = o[q][e].x + o[q][e].y;
                    if (lane == 0) {
                        cm[warp * 16 + q] = mq[q];
                        cl[warp * 16 + q] = lq[q];
                    }
                }
            }
        }
    }
    dla::named_sync(1, kMmaConsumers * 32);
    // per query: the warps' weights and the normaliser (one thread each), then the weighted
    // sums with every thread on independent (query, 4 dimensions) elements
    float *cf = cl + kMmaConsumers * 16;               // [kMaxQ][kMmaConsumers + 1]: weights, 1/sum
    if (tid < Q) {
        const int qi = tid;
        const int qt = qi / TL, row = qi - qt * TL;
        float M = -INFINITY;
        for (int kq = 0; kq < KS; ++kq) M = fmaxf(M, cm[(kq * MT + qt) * 16 + row]);
        float wsum = 0.f;
        for (int kq = 0; kq < kMmaConsumers; ++kq) {
            float f = 0.f;
            if (kq < KS) {
                const float mw = cm[(kq * MT + qt) * 16 + row];
                f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
                wsum += f * cl[(kq * MT + qt) * 16 + row];
            }
            cf[qi * (kMmaConsumers + 1) + kq] = f;
        }
        cf[qi * (kMmaConsumers + 1) + kMmaConsumers] = 1.f / wsum;
        const int rq = s_qrow[qi];
        if (s_len[rq] > k0) {
            const float lse_piece = (M + fast_log2(wsum)) * 0.69314718055994530942f;
            if (cluster)
                s_plse[qi] = lse_piece;
            else
                a.part_lse[((int64_t)s_row[rq] * P.n_q + h * G + s_qhead[qi]) * ms + piece] = lse_piece;
        }
    }
    dla::named_sync(1, kMmaConsumers * 32);
    for (int e = tid; e < Q * (D / 4); e += kMmaConsumers * 32) {
        const int qi = e / (D / 4), d4 = e - qi * (D / 4);
        const int rq = s_qrow[qi];
        if (s_len[rq] <= k0) continue;
        const int qt = qi / TL, row = qi - qt * TL;
        const float *f = cf + qi * (kMmaConsumers + 1);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int kq = 0; kq < kMmaConsumers; ++kq) {
            if (kq < KS) {
                const float4 v = *reinterpret_cast<const float4 *>(co + ((kq * MT + qt) * 16 + row) * CP + d4 * 4);
                acc.x = fmaf(f[kq], v.x, acc.x);
                acc.y = fmaf(f[kq], v.y, acc.y);
                acc.z = fmaf(f[kq], v.z, acc.z);
                acc.w = fmaf(f[kq], v.w, acc.w);
            }
        }
        const float inv = f[kMmaConsumers];
        const float4 res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (cluster) {
            *reinterpret_cast<float4 *>(qraw + qi * D + d4 * 4) = res;
        } else {
            const int64_t pidx = ((int64_t)s_row[rq] * P.n_q + h * G + s_qhead[qi]) * ms + piece;
            *reinterpret_cast<float4 *>(a.part_o + pidx * D + d4 * 4) = res;
        }
    }
    if (cluster) cluster_merge();
    else if (tail) tail_merge();
}

}  // namespace
