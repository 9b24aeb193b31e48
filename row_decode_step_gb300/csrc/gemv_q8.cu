// Q8_0 projection GEMV over 1..8 rows per command (the router/projection
// "enc_cols" role of daScript PR #4473, commit "cud_router_enc_cols tiles every
// router launch": eight activation columns per launch, longer launches tiled).
//
// Device weight form: tiles of 16 output rows x 32 inputs (one Q8_0 block per
// row), 512 bytes each, in the A-operand order of the 16x8x32 int8 tensor-core
// product: lane t = 4g + c owns 16 bytes = row g at inputs 4c..4c+3, row g+8 at
// the same inputs, row g at 16+4c..16+4c+3, row g+8 at those.  The tiles of one
// row tile are contiguous along K.  Scales: per 16 rows and 4 tiles, 128 bytes;
// lane group g reads 16 bytes = (d[g], d[g+8]) for the 4 tiles.
//
// Kernel shape:
//  * a CTA = one producer warp + 8 consumer warps owns a run of row tiles and one
//    K-slice; the producer streams one row tile's slice (weights, then scales: two
//    contiguous bulk copies) into each stage of a shared-memory ring, tracked by
//    mbarriers, and issues the first stages before waiting on the previous kernel
//    (programmatic dependent launch);
//  * each consumer warp owns an eighth of the slice's k-tiles; its activations are
//    loaded once and kept in registers as operands for the whole launch;
//  * per row tile each warp adds its k-tiles into a 16x8 accumulator and parks it
//    in shared memory; the warps' partials are summed once at the end in a fixed
//    order, and the K-slices of a thread-block cluster through distributed shared
//    memory in rank order (no atomics: results do not depend on timing).
// Two inner products share this shape.  Tensor path: the int8 weights enter
// 16x8x32 int8 products as they are; each activation row is quantised per warp to
// two int8 terms, x ~ s (h + l/254) with s = max|x|/127, so that both products are
// exact in int32 and 254 h-sum + l-sum is formed exactly before one conversion to
// f32 (activation error <= max|x| / 64516 per element).  CUDA-core path: the
// weights are widened to f32 and multiplied with the f32 activations by FMAs.
#include <cuda_fp16.h>
#include <cstdio>
#include <type_traits>

#include "dl_common.cuh"

namespace {

enum { PATH_AUTO = 0, PATH_CUDA_CORE = 1, PATH_TENSOR = 2 };

struct GemvArgs {
    const uint4 *qs;        // packed weight tiles
    const uint32_t *d;      // packed scales as (d[g], d[g+8]) pairs
    const float *x;
    float *y;
    int64_t x_stride, y_stride;
    int n_out, n_in;
    int nr;                 // rows of this command, 1..8
    int KT;                 // k-tiles, padded to a multiple of 4
    int RT;                 // row tiles
    int cs;                 // K-slices (= cluster size)
    int ksl;                // k-tiles per K-slice (multiple of 4)
    int rpr;                // row tiles per CTA
    int stages;             // ring depth
};

constexpr int kConsumers = 8;                        // consumer warps, each a share of the K-slice
constexpr int kThreads = (kConsumers + 1) * 32;      // and one producer warp
constexpr int kMaxStages = 8;

// ---- cluster and shared-memory helpers
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(const float *local, uint32_t rank)
{
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// ---- asynchronous bulk copies into shared memory, tracked by mbarriers
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait: false if the phase never completed (the caller then stops using the stage).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    for (int spin = 0; spin < (1 << 22); ++spin)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ---- arithmetic helpers
// stored weight byte `sel` of w (int8) to float, through the biased byte q + 128 placed in
// the low mantissa of 2^23 (2^23 + 128 subtracted)
__device__ __forceinline__ float s8_to_f32(uint32_t w, uint32_t sel)
{
    return __uint_as_float(__byte_perm(w ^ 0x80808080u, 0x4B000000u, 0x7540u | sel)) - 8388736.0f;
}
__device__ __forceinline__ void imma16832(int &c0, int &c1, int &c2, int &c3, const uint4 &a, uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+r"(c0), "+r"(c1), "+r"(c2), "+r"(c3)
                 : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_s8x4(int a, int b, int c, int d)
{
    return (uint32_t)(a & 0xFF) | ((uint32_t)(b & 0xFF) << 8) | ((uint32_t)(c & 0xFF) << 16) | ((uint32_t)(d & 0xFF) << 24);
}

// Shared-memory bytes of a launch: a ring of `stages` row-tile stages of `ksl` k-tiles (weights
// then scales), per-warp partials of `rpr` row tiles, and the cluster partials.
size_t gemv_smem(int ksl, int stages, int rpr)
{
    const size_t sb = (size_t)ksl * 512 + (size_t)ksl * 32;
    return (size_t)stages * sb + (size_t)rpr * kConsumers * 128 * 4 + (size_t)rpr * 128 * 4;
}

template <bool MMA, int NRC, int KWM>
__global__ void __launch_bounds__(kThreads, 2) gemv_q8_kernel(const __grid_constant__ GemvArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages];
    __shared__ int s_fail;

    const int S = a.stages;
    const int slice = blockIdx.x % a.cs;
    const int rt0 = (blockIdx.x / a.cs) * a.rpr;
    const int nrt = max(0, min(a.rpr, a.RT - rt0));      // row tiles of this CTA
    const int kt0 = slice * a.ksl, kt1 = min(a.KT, kt0 + a.ksl);
    const int nkt = kt1 - kt0;
    const uint32_t wbytes = (uint32_t)nkt * 512u, dbytes = (uint32_t)nkt * 32u;
    const size_t SB = (size_t)a.ksl * 544;
    unsigned char *ring = smem;
    float *red = reinterpret_cast<float *>(smem + S * SB);          // [kConsumers][rpr][128]
    float *cpart = red + kConsumers * a.rpr * 128;                  // [rpr][128]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int KG = a.KT >> 2;
    const bool producer = warp == kConsumers;
    const unsigned char *qs = reinterpret_cast<const unsigned char *>(a.qs);
    const unsigned char *dp = reinterpret_cast<const unsigned char *>(a.d);

    if (threadIdx.x == 0) {
        for (int st = 0; st < S; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], kConsumers);
        }
        s_fail = 0;
        mbar_init_fence();
    }
    __syncthreads();

    // stage j: row tile rt0 + j, this slice's k-tiles (contiguous), then their scales (contiguous)
    auto issue = [&](int j) {
        const int st = j % S;
        const int rt = rt0 + j;
        unsigned char *dst = ring + st * SB;
        mbar_expect_tx(&full[st], wbytes + dbytes);
        bulk_g2s(dst, qs + ((size_t)rt * a.KT + kt0) * 512, wbytes, &full[st]);
        bulk_g2s(dst + (size_t)a.ksl * 512, dp + ((size_t)rt * KG + (kt0 >> 2)) * 128, dbytes, &full[st]);
    };
    // the weights do not depend on the previous kernel: start the ring before waiting on it
    if (producer && lane == 0)
        for (int j = 0; j < S && j < nrt; ++j) issue(j);
    dl_pdl_launch_dependents();
    dl_pdl_wait();

    // ---- this warp's share of the slice and its activations, kept in registers
    const int wk0 = (warp * nkt) / kConsumers, wk1 = ((warp + 1) * nkt) / kConsumers;   // slice-local
    const int nw = producer ? 0 : min(wk1 - wk0, KWM);
    if (!producer && lane == 0 && wk1 - wk0 > KWM) atomicExch(&s_fail, 1);   // launch shape broken: poison
    float xv[KWM][NRC][8];
#pragma unroll
    for (int j = 0; j < KWM; ++j) {
        const int kt = kt0 + wk0 + j;
        const bool live = j < nw && kt * 32 < a.n_in;
#pragma unroll
        for (int r = 0; r < NRC; ++r) {
            const int row = MMA ? g : r;
            const bool ok = live && row < a.nr;
            float4 lo4 = make_float4(0.f, 0.f, 0.f, 0.f), hi4 = lo4;
            if (ok) {
                const float *xr = a.x + (int64_t)row * a.x_stride + kt * 32;
                lo4 = __ldg(reinterpret_cast<const float4 *>(xr + 4 * c));
                hi4 = __ldg(reinterpret_cast<const float4 *>(xr + 16 + 4 * c));
            }
            xv[j][r][0] = lo4.x; xv[j][r][1] = lo4.y; xv[j][r][2] = lo4.z; xv[j][r][3] = lo4.w;
            xv[j][r][4] = hi4.x; xv[j][r][5] = hi4.y; xv[j][r][6] = hi4.z; xv[j][r][7] = hi4.w;
        }
    }
    // tensor path: activation row g quantised over this warp's inputs to two int8 terms,
    // x ~ s (h + l/254); the products' scale s/254 is applied per accumulator column at the end
    uint32_t bh[KWM][2], bl[KWM][2];
    float cs0 = 0.f, cs1 = 0.f;
    if constexpr (MMA) {
        float m = 0.f;
#pragma unroll
        for (int j = 0; j < KWM; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(xv[j][0][e]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const float s = m / 127.f;
        const float inv = m > 0.f ? 127.f / m : 0.f;
#pragma unroll
        for (int j = 0; j < KWM; ++j)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                int hq[4], lq[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float t = fminf(fmaxf(xv[j][0][4 * half + e] * inv, -127.f), 127.f);
                    const float hr = rintf(t);
                    hq[e] = (int)hr;
                    lq[e] = (int)rintf((t - hr) * 254.f);
                }
                bh[j][half] = pack_s8x4(hq[0], hq[1], hq[2], hq[3]);
                bl[j][half] = pack_s8x4(lq[0], lq[1], lq[2], lq[3]);
            }
        // accumulator columns of this lane are rows 2c and 2c+1 (held by lanes 8c and 8c+4)
        const float sc = s / 254.f;
        cs0 = __shfl_sync(0xffffffffu, sc, 8 * c);
        cs1 = __shfl_sync(0xffffffffu, sc, 8 * c + 4);
    }

    if (producer) {
        // refill each stage once every consumer warp has released it
        if (lane == 0) {
            for (int j = S; j < nrt; ++j) {
                const int st = j % S;
                if (!mbar_wait(&empty[st], (uint32_t)(((j / S) - 1) & 1))) {
                    atomicExch(&s_fail, 1);
                    break;
                }
                issue(j);
            }
        }
    } else {
        for (int i = 0; i < nrt; ++i) {
            const int st = i % S;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (uint32_t)((i / S) & 1)))) {
                if (lane == 0) atomicExch(&s_fail, 1);
                break;
            }
            const unsigned char *sw = ring + st * SB;
            const unsigned char *sd = sw + (size_t)a.ksl * 512;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            float accg[NRC], acch[NRC];
#pragma unroll
            for (int r = 0; r < NRC; ++r) accg[r] = acch[r] = 0.f;
#pragma unroll
            for (int j = 0; j < KWM; ++j) {
                if (j >= nw) break;
                const int kl = wk0 + j;                                  // slice-local k-tile
                const uint4 w = *reinterpret_cast<const uint4 *>(sw + kl * 512 + lane * 16);
                const uint32_t sp = *reinterpret_cast<const uint32_t *>(sd + (kl >> 2) * 128 + g * 16 + (kl & 3) * 4);
                const float dg = __half2float(__ushort_as_half((unsigned short)(sp & 0xFFFFu)));
                const float dh = __half2float(__ushort_as_half((unsigned short)(sp >> 16)));
                if constexpr (MMA) {
                    int h0 = 0, h1 = 0, h2 = 0, h3 = 0, l0 = 0, l1 = 0, l2 = 0, l3 = 0;
                    imma16832(h0, h1, h2, h3, w, bh[j][0], bh[j][1]);
                    imma16832(l0, l1, l2, l3, w, bl[j][0], bl[j][1]);
                    // 254 h-sum + l-sum is exact in int32 (|h-sum| <= 32*127*127)
                    acc[0] = fmaf(dg, (float)(h0 * 254 + l0), acc[0]);
                    acc[1] = fmaf(dg, (float)(h1 * 254 + l1), acc[1]);
                    acc[2] = fmaf(dh, (float)(h2 * 254 + l2), acc[2]);
                    acc[3] = fmaf(dh, (float)(h3 * 254 + l3), acc[3]);
                } else {
                    // row g: words 0 and 2; row g+8: words 1 and 3
                    float wg[8], wh[8];
                    wg[0] = s8_to_f32(w.x, 0); wg[1] = s8_to_f32(w.x, 1); wg[2] = s8_to_f32(w.x, 2); wg[3] = s8_to_f32(w.x, 3);
                    wg[4] = s8_to_f32(w.z, 0); wg[5] = s8_to_f32(w.z, 1); wg[6] = s8_to_f32(w.z, 2); wg[7] = s8_to_f32(w.z, 3);
                    wh[0] = s8_to_f32(w.y, 0); wh[1] = s8_to_f32(w.y, 1); wh[2] = s8_to_f32(w.y, 2); wh[3] = s8_to_f32(w.y, 3);
                    wh[4] = s8_to_f32(w.w, 0); wh[5] = s8_to_f32(w.w, 1); wh[6] = s8_to_f32(w.w, 2); wh[7] = s8_to_f32(w.w, 3);
#pragma unroll
                    for (int r = 0; r < NRC; ++r) {
                        float sg = wg[0] * xv[j][r][0], sh = wh[0] * xv[j][r][0];
#pragma unroll
                        for (int e = 1; e < 8; ++e) {
                            sg = fmaf(wg[e], xv[j][r][e], sg);
                            sh = fmaf(wh[e], xv[j][r][e], sh);
                        }
                        accg[r] = fmaf(dg, sg, accg[r]);
                        acch[r] = fmaf(dh, sh, acch[r]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);            // the stage is free for the producer
            float *rw = red + (warp * a.rpr + i) * 128;
            if constexpr (MMA) {
                *reinterpret_cast<float2 *>(rw + g * 8 + 2 * c) = make_float2(acc[0] * cs0, acc[1] * cs1);
                *reinterpret_cast<float2 *>(rw + (g + 8) * 8 + 2 * c) = make_float2(acc[2] * cs0, acc[3] * cs1);
            } else {
#pragma unroll
                for (int r = 0; r < NRC; ++r) {
                    float vg = accg[r], vh = acch[r];
                    vg += __shfl_xor_sync(0xffffffffu, vg, 1);
                    vg += __shfl_xor_sync(0xffffffffu, vg, 2);
                    vh += __shfl_xor_sync(0xffffffffu, vh, 1);
                    vh += __shfl_xor_sync(0xffffffffu, vh, 2);
                    if (c == 0) {
                        rw[g * 8 + r] = vg;
                        rw[(g + 8) * 8 + r] = vh;
                    }
                }
            }
        }
    }
    __syncthreads();
    const bool failed = s_fail != 0;

    // ---- sum the warps' partials in a fixed order; finish here or hand to the cluster
    for (int e = threadIdx.x; e < nrt * 128; e += kThreads) {
        const int i = e >> 7, el = e & 127;
        const int row = el >> 3, col = el & 7;
        if (col >= a.nr) continue;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) sum += red[(w * a.rpr + i) * 128 + el];
        if (failed) sum = __int_as_float(0x7fc00000);
        if (a.cs == 1) {
            const int o = (rt0 + i) * 16 + row;
            if (o < a.n_out) a.y[(int64_t)col * a.y_stride + o] = sum;
        } else {
            cpart[e] = sum;
        }
    }
    if (a.cs > 1) {
        // every K-slice of this run of row tiles holds its partials in shared memory: sum in rank order
        cluster_sync_all();
        for (int e = threadIdx.x; e < nrt * 128; e += kThreads) {
            if ((e >> 3) % a.cs != slice) continue;      // each rank finishes a share of the rows
            const int col = e & 7;
            if (col >= a.nr) continue;
            float sum = 0.f;
            for (int q = 0; q < a.cs; ++q) sum += ld_dsmem_f32(cpart + e, (uint32_t)q);
            const int o = rt0 * 16 + (e >> 3);
            if (o < a.n_out) a.y[(int64_t)col * a.y_stride + o] = sum;
        }
        cluster_sync_all();   // keep this CTA's shared memory alive until every peer has read it
    }
}

// ---------------------------------------------------------------- packing

__device__ __forceinline__ uint32_t q8_byte(const uint8_t *blocks, int64_t n_out, int64_t n_in,
                                            int64_t o, int64_t k)
{
    if (o >= n_out || k >= n_in) return 0u;
    return blocks[(o * (n_in / 32) + k / 32) * 34 + 2 + (k % 32)];
}

// lane t = 4g + c of tile (rt, kt): word 0 = row g at inputs 4c..4c+3, word 1 = row g+8 there,
// words 2 and 3 = the same rows at 16+4c..16+4c+3
__global__ void q8_pack_qs_kernel(const uint8_t *blocks, int64_t n_out, int64_t n_in, int KT,
                                  int64_t units, uint4 *qs)
{
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= units) return;
    const int lane = (int)(u & 31);
    const int64_t t = u >> 5;
    const int64_t kt = t % KT, rt = t / KT;
    const int g = lane >> 2, c = lane & 3;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int row = g + (q & 1) * 8;
        const int k0 = 4 * c + (q >> 1) * 16;
        uint32_t v = 0u;
#pragma unroll
        for (int b = 0; b < 4; ++b) v |= q8_byte(blocks, n_out, n_in, rt * 16 + row, kt * 32 + k0 + b) << (8 * b);
        w[q] = v;
    }
    qs[u] = make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void q8_pack_d_kernel(const uint8_t *blocks, int64_t n_out, int64_t n_in, int KG,
                                 int64_t units, uint4 *d)
{
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= units) return;
    const int g = (int)(u & 7);
    const int64_t t = u >> 3;
    const int64_t kg = t % KG, rt = t / KG;
    const int64_t nb = n_in / 32;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t pair = 0u;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t o = rt * 16 + g + h * 8;
            const int64_t b = kg * 4 + q;
            uint32_t v = 0u;
            if (o < n_out && b < nb) {
                const uint8_t *blk = blocks + (o * nb + b) * 34;
                v = (uint32_t)blk[0] | ((uint32_t)blk[1] << 8);
            }
            pair |= v << (16 * h);
        }
        w[q] = pair;
    }
    d[u] = make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------- launch

struct GemvCfg {
    bool mma;
    int nrc, kwm, cs, ksl, rpr, stages, grid;
    size_t smem;
};

template <bool MMA, int NRC, int KWM>
void *kptr() { return reinterpret_cast<void *>(gemv_q8_kernel<MMA, NRC, KWM>); }

void *pick_kernel(bool mma, int nrc, int kwm)
{
    switch (kwm) {
    case 1: return mma ? kptr<true, 1, 1>() : nrc == 1 ? kptr<false, 1, 1>() : kptr<false, 2, 1>();
    case 2: return mma ? kptr<true, 1, 2>() : nrc == 1 ? kptr<false, 1, 2>() : kptr<false, 2, 2>();
    case 4: return mma ? kptr<true, 1, 4>() : nrc == 1 ? kptr<false, 1, 4>() : kptr<false, 2, 4>();
    case 6: return mma ? kptr<true, 1, 6>() : nullptr;
    case 8: return mma ? kptr<true, 1, 8>() : nrc == 1 ? kptr<false, 1, 8>() : nullptr;
    }
    return nullptr;
}

// The dynamic shared-memory limit is a per-function attribute shared by every launch of the
// kernel (graph nodes and profilers re-launch against it): set it once to the largest size any
// launch shape may use, never to one launch's own size.
constexpr int kSmemLimit = 200 * 1024;

int prepare_kernel(const void *kern, int cs)
{
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8: set shared memory");
    if (cs > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8: allow a large cluster");
    }
    return DL_OK;
}

// Clusters of `cs` CTAs of this shape that are resident at once.
int resident_clusters(const void *kern, int cs, size_t smem)
{
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)cs);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &lc) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return clusters;
}

// Launch shape.  K is cut into cs slices of ksl k-tiles (whole groups of 4); each CTA takes
// rpr consecutive row tiles of one slice and streams them one row tile per ring stage.  The
// shape with the least work per CTA whose grid is resident in one wave wins (near-ties go
// to fewer slices).
int choose_cfg(int nr, int RT, int KT, int sm, int path, GemvCfg *out)
{
    const bool mma = path == PATH_TENSOR || (path == PATH_AUTO && nr > 2);
    if (!mma && nr > 2) return dl::fail(DL_E_SHAPE, "dl_gemv_q8: the CUDA-core path serves 1 or 2 rows per command");
    const int nrc = mma ? 1 : nr;
    const int kw_max = (!mma && nrc == 2) ? 4 : 8;
    GemvCfg best{};
    long best_cost = -1;
    for (int cs = 1; cs <= 16; ++cs) {
        const int ksl = (int)dl::ceil_div(dl::ceil_div(KT, cs), 4) * 4;
        if ((int)dl::ceil_div(KT, ksl) != cs) continue;
        const int kw = (int)dl::ceil_div(ksl, kConsumers);             // k-tiles per consumer warp
        if (kw > kw_max || (size_t)ksl * 544 > 48 * 1024) continue;
        const int kwm = kw <= 1 ? 1 : kw <= 2 ? 2 : kw <= 4 ? 4 : (mma && kw <= 6) ? 6 : 8;
        const size_t sb = (size_t)ksl * 544;
        // two CTAs per SM when shared memory allows, else one; the ring takes what the
        // partials leave (2 to 8 stages)
        for (int per_sm = 2; per_sm >= 1; --per_sm) {
            const int ranges = (per_sm * sm) / cs;
            if (ranges < 1) continue;
            const int rpr = (int)dl::ceil_div(RT, ranges);
            const size_t limit = per_sm == 2 ? (size_t)112 * 1024 : (size_t)kSmemLimit;
            const size_t fixed = gemv_smem(ksl, 0, rpr);
            if (fixed + 2 * sb > limit) continue;
            int stages = (int)((limit - fixed) / sb);
            if (stages > kMaxStages) stages = kMaxStages;
            const size_t smem = gemv_smem(ksl, stages, rpr);
            const long cost = (long)rpr * ksl * 100 + cs;        // bytes per CTA, then fewer slices
            if (best_cost < 0 || cost * 100 < best_cost * 95) {
                best_cost = cost;
                best = GemvCfg{mma, nrc, kwm, cs, ksl, rpr, stages, (int)dl::ceil_div(RT, rpr) * cs, smem};
            }
            break;
        }
    }
    if (best_cost < 0) {
        // no single-wave shape (very many row tiles): CTAs of as many row tiles as shared memory
        // holds, in several waves
        for (int cs = 1; cs <= 16 && best_cost < 0; ++cs) {
            const int ksl = (int)dl::ceil_div(dl::ceil_div(KT, cs), 4) * 4;
            if ((int)dl::ceil_div(KT, ksl) != cs) continue;
            const int kw = (int)dl::ceil_div(ksl, kConsumers);
            if (kw > kw_max || (size_t)ksl * 544 > 48 * 1024) continue;
            const int kwm = kw <= 1 ? 1 : kw <= 2 ? 2 : kw <= 4 ? 4 : (mma && kw <= 6) ? 6 : 8;
            const size_t sb = (size_t)ksl * 544;
            const int stages = 3;
            int rpr = (int)(((size_t)112 * 1024 - stages * sb) / ((size_t)kConsumers * 512 + 512));
            if (rpr < 1) continue;
            if (rpr > RT) rpr = RT;
            best_cost = 0;
            best = GemvCfg{mma, nrc, kwm, cs, ksl, rpr, stages, (int)dl::ceil_div(RT, rpr) * cs,
                           gemv_smem(ksl, stages, rpr)};
        }
        if (best_cost < 0) return dl::fail(DL_E_SHAPE, "dl_gemv_q8: no launch shape for %d k-tiles", KT);
    }
    const void *kern = pick_kernel(best.mma, best.nrc, best.kwm);
    if (!kern) return dl::fail(DL_E_SHAPE, "dl_gemv_q8: no kernel for this shape");
    int rc = prepare_kernel(kern, best.cs);
    if (rc != DL_OK) return rc;
    if (best.cs > 1 && best_cost > 0) {
        // a one-wave shape stays one wave with clusters: grow the row tiles per CTA until every
        // cluster is resident at once, within the shared-memory limit
        while (resident_clusters(kern, best.cs, best.smem) < best.grid / best.cs && best.rpr < RT) {
            const size_t smem = gemv_smem(best.ksl, best.stages, best.rpr + 1);
            if (smem > (size_t)kSmemLimit) break;
            best.rpr += 1;
            best.smem = smem;
            best.grid = (int)dl::ceil_div(RT, best.rpr) * best.cs;
        }
    }
    *out = best;
    return DL_OK;
}

int gemv_group(GemvArgs a, int nr, int sm, int path, cudaStream_t st)
{
    GemvCfg cfg;
    int rc = choose_cfg(nr, a.RT, a.KT, sm, path, &cfg);
    if (rc != DL_OK) return rc;
    a.nr = nr;
    a.cs = cfg.cs;
    a.ksl = cfg.ksl;
    a.rpr = cfg.rpr;
    a.stages = cfg.stages;
    const void *kern = pick_kernel(cfg.mma, cfg.nrc, cfg.kwm);
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)cfg.grid);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = cfg.smem;
    lc.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cfg.cs > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)cfg.cs;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    lc.attrs = attr;
    lc.numAttrs = na;
    void *args[1] = {&a};
    cudaError_t e = cudaLaunchKernelExC(&lc, kern, args);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8: launch");
    return DL_OK;
}

int gemv_impl(const dl_q8_weight *W, const float *x, int rows, int64_t x_stride, float *y, int64_t y_stride,
              int path, dl_stream_t stream)
{
    dl::clear_error();
    if (!W || !x || !y || !W->qs || !W->d) return dl::fail(DL_E_ARG, "dl_gemv_q8: null pointer");
    if (rows < 0) return dl::fail(DL_E_ARG, "dl_gemv_q8: rows=%d", rows);
    if (path < PATH_AUTO || path > PATH_TENSOR) return dl::fail(DL_E_ARG, "dl_gemv_q8: path=%d", path);
    int rc = dl_q8_packed_size(W->n_out, W->n_in, nullptr, nullptr);
    if (rc != DL_OK) return rc;
    if (rows == 0) return DL_OK;
    if (x_stride < W->n_in || y_stride < W->n_out)
        return dl::fail(DL_E_ARG, "dl_gemv_q8: strides %lld/%lld below the row widths",
                        (long long)x_stride, (long long)y_stride);
    if (!dl::aligned16(x) || (x_stride % 4) != 0 || !dl::aligned16(W->qs) || !dl::aligned16(W->d))
        return dl::fail(DL_E_ALIGN, "dl_gemv_q8: x, its stride and the weight planes must be 16-byte aligned");
    const char *xb = reinterpret_cast<const char *>(x), *yb = reinterpret_cast<const char *>(y);
    const char *xe = xb + ((size_t)(rows - 1) * x_stride + W->n_in) * 4;
    const char *ye = yb + ((size_t)(rows - 1) * y_stride + W->n_out) * 4;
    if (xb < ye && yb < xe) return dl::fail(DL_E_ARG, "dl_gemv_q8: y overlaps x");
    int sm = 0;
    rc = dl::device_sm_count(&sm);
    if (rc != DL_OK) return rc;

    GemvArgs a{};
    a.qs = static_cast<const uint4 *>(W->qs);
    a.d = static_cast<const uint32_t *>(W->d);
    a.x_stride = x_stride;
    a.y_stride = y_stride;
    a.n_out = (int)W->n_out;
    a.n_in = (int)W->n_in;
    a.KT = (int)(dl::ceil_div(W->n_in, 128) * 4);
    a.RT = (int)dl::ceil_div(W->n_out, 16);

    int sizes[64];
    int done = 0;
    while (done < rows) {
        // commands of at most eight rows, in the fewest balanced groups
        const int chunk = rows - done > 8 * 64 ? 8 * 64 : rows - done;
        const int ng = dl_plan_groups(chunk, DL_MAX_ROWS, sizes);
        if (ng < 0) return ng;
        for (int gi = 0; gi < ng; ++gi) {
            a.x = x + (size_t)done * x_stride;
            a.y = y + (size_t)done * y_stride;
            rc = gemv_group(a, sizes[gi], sm, path, static_cast<cudaStream_t>(stream));
            if (rc != DL_OK) return rc;
            done += sizes[gi];
        }
    }
    return DL_OK;
}

}  // namespace

extern "C" {

int dl_q8_packed_size(int64_t n_out, int64_t n_in, size_t *qs_bytes, size_t *d_bytes)
{
    if (n_out <= 0 || n_in <= 0 || n_in % 32 != 0)
        return dl::fail(DL_E_SHAPE, "dl_q8_packed_size: n_out=%lld n_in=%lld (n_in must be a positive multiple of 32)",
                        (long long)n_out, (long long)n_in);
    if (n_out > (1LL << 30) || n_in > (1LL << 24))
        return dl::fail(DL_E_SHAPE, "dl_q8_packed_size: matrix too large");
    const int64_t RT = dl::ceil_div(n_out, 16), KT = dl::ceil_div(n_in, 128) * 4;
    if (qs_bytes) *qs_bytes = (size_t)(RT * KT * 512);
    if (d_bytes) *d_bytes = (size_t)(RT * KT * 32);
    return DL_OK;
}

int dl_q8_pack(const uint8_t *blocks, int64_t n_out, int64_t n_in, void *qs, void *d, dl_stream_t stream)
{
    dl::clear_error();
    size_t qb = 0, db = 0;
    int rc = dl_q8_packed_size(n_out, n_in, &qb, &db);
    if (rc != DL_OK) return rc;
    if (!blocks || !qs || !d) return dl::fail(DL_E_ARG, "dl_q8_pack: null pointer");
    if (!dl::aligned16(qs) || !dl::aligned16(d)) return dl::fail(DL_E_ALIGN, "dl_q8_pack: planes must be 16-byte aligned");
    const int KT = (int)(dl::ceil_div(n_in, 128) * 4);
    const int64_t units_q = (int64_t)(qb / 16), units_d = (int64_t)(db / 16);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    q8_pack_qs_kernel<<<(unsigned)dl::ceil_div(units_q, 256), 256, 0, st>>>(blocks, n_out, n_in, KT, units_q,
                                                                          static_cast<uint4 *>(qs));
    rc = dl::check_launch("dl_q8_pack: qs");
    if (rc != DL_OK) return rc;
    q8_pack_d_kernel<<<(unsigned)dl::ceil_div(units_d, 256), 256, 0, st>>>(blocks, n_out, n_in, KT / 4, units_d,
                                                                         static_cast<uint4 *>(d));
    return dl::check_launch("dl_q8_pack: d");
}

int dl_gemv_q8(const dl_q8_weight *W, const float *x, int rows, int64_t x_stride,
               float *y, int64_t y_stride, dl_stream_t stream)
{
    return gemv_impl(W, x, rows, x_stride, y, y_stride, PATH_AUTO, stream);
}

int dl_gemv_q8_ex(const dl_q8_weight *W, const float *x, int rows, int64_t x_stride,
                  float *y, int64_t y_stride, int path, dl_stream_t stream)
{
    return gemv_impl(W, x, rows, x_stride, y, y_stride, path, stream);
}

}  // extern "C"
