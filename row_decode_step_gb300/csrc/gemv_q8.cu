// Q8_0 projection GEMV over 1..8 rows per command (the router/projection
// "enc_cols" role of daScript PR #4473, commit "cud_router_enc_cols tiles every
// router launch": eight activation columns per launch, longer launches tiled).
//
// Device weight form: tiles of 16 output rows x 32 inputs (one Q8_0 block per
// row), 512 bytes each, lane t of a warp owning the 16 bytes at 16*t; a lane
// holds rows g = t/4 and g+8 at the eight inputs {2c, 2c+1, 2c+8, 2c+9} and the
// same +16, c = t%4 (the A-operand order of a 16x8x16 tensor-core product).
// Scales: per 16 rows and 4 tiles, 128 bytes; lane group g reads 16 bytes.
//
// Kernel shape (2-D tiling of the matrix):
//  * a CTA of 8 warps owns a run of row tiles and one K-slice of 8*KW k-tiles;
//    warp w owns KW consecutive k-tiles of the slice for every row tile of the
//    CTA, so its share of the activations is loaded from global memory once and
//    kept in registers for the whole launch;
//  * the warps stream their weight tiles with 16-byte L1-bypassing loads, two
//    groups in flight; partial sums of a group of row tiles are reduced across
//    the warps in shared memory in a fixed order;
//  * the K-slices of one run of row tiles form a thread-block cluster whose
//    partials are summed through distributed shared memory in rank order (no
//    atomics: results do not depend on timing);
//  * before waiting on the previous kernel (programmatic dependent launch) each
//    CTA asks L2 to prefetch all of its weights, so weight streaming overlaps the
//    previous kernel's tail.
// Two inner products share this shape: f32 CUDA-core FMAs (few rows) and
// 16x8x16 f16 tensor-core products on exact int8 weights with the activations
// split into two f16 terms (hi + lo) per power-of-two-scaled block, f32
// accumulation (more rows, where FMAs would bound the kernel).
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
    int ksl;                // k-tiles per K-slice
};

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

// byte `sel` of wx (a stored weight byte, q + 128) to float q: the byte becomes the low
// mantissa bits of 2^23 and 2^23 + 128 is subtracted.
__device__ __forceinline__ float s8_to_f32(uint32_t wx, uint32_t sel)
{
    return __uint_as_float(__byte_perm(wx, 0x4B000000u, 0x7540u | sel)) - 8388736.0f;
}

// bytes (0,1) or (2,3) of wx (stored weight bytes, q + 128) to an f16x2 pair of exact
// integers: each byte becomes the low mantissa of 1024 (f16 0x64xx) and 1024 + 128 is
// subtracted.
__device__ __forceinline__ uint32_t s8x2_to_h2(uint32_t wx, uint32_t sel)
{
    const uint32_t v = __byte_perm(wx, 0x64646464u, sel);
    __half2 h = __hsub2(*reinterpret_cast<const __half2 *>(&v), __halves2half2(__ushort_as_half(0x6480),
                                                                               __ushort_as_half(0x6480)));
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void mma16816(float &c0, float &c1, float &c2, float &c3, uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c0), "+f"(c1), "+f"(c2), "+f"(c3)
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// power-of-two scale bringing a block maximum m into [2^13, 2^14), and its inverse
__device__ __forceinline__ void block_scale(float m, float &s, float &sinv)
{
    const uint32_t bits = __float_as_uint(m);
    int e = (int)((bits >> 23) & 0xFF) - 126;          // m = f * 2^e, f in [0.5, 1)
    if (m == 0.f || !(m < INFINITY)) e = 14;           // zero, inf, nan: no scaling
    int es = 14 - e, ei = e - 14;
    es = max(-126, min(127, es));
    ei = max(-126, min(127, ei));
    s = __uint_as_float((uint32_t)(es + 127) << 23);
    sinv = __uint_as_float((uint32_t)(ei + 127) << 23);
}

// Offsets (in floats) of the 8 inputs a lane of quad position c holds inside a 32-input block.
__device__ __forceinline__ int lane_k(int c, int j)
{
    return 2 * c + (j & 1) + ((j >> 1) & 1) * 8 + (j >> 2) * 16;
}

// ---- asynchronous bulk copies into shared memory, tracked by mbarriers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
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

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

constexpr int kConsumers = 8;                        // consumer warps, one row tile each
constexpr int kThreads5 = (kConsumers + 1) * 32;     // and one producer warp
constexpr int kStages = 3;                           // ring depth, in groups of 4 k-tiles
constexpr int kStageBytes = kConsumers * 4 * 512;    // one group of the CTA's 8 row tiles

// Shared-memory bytes of a launch: weight ring, activation fragments, cluster partials.
size_t gemv_smem(bool mma, int nrc, int ksl)
{
    const size_t fb = mma ? 32 : (size_t)nrc * 32;
    return (size_t)kStages * kStageBytes + (size_t)ksl * 32 * fb + (size_t)kConsumers * 128 * 4;
}

template <bool MMA, int NRC>
__global__ void __launch_bounds__(kThreads5, 2) gemv_q8_kernel(const __grid_constant__ GemvArgs a)
{
    constexpr int FB = MMA ? 32 : NRC * 32;          // fragment bytes per lane and k-tile
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
    __shared__ int s_rowmax[8];
    __shared__ int s_fail;

    unsigned char *ring = smem;
    unsigned char *xf = smem + kStages * kStageBytes;
    float *cpart = reinterpret_cast<float *>(xf + (size_t)a.ksl * 32 * FB);

    const int slice = blockIdx.x % a.cs;
    const int rt0 = (blockIdx.x / a.cs) * kConsumers;
    const int kt0 = slice * a.ksl, kt1 = min(a.KT, kt0 + a.ksl);
    const int nkt = kt1 - kt0, ng = nkt >> 2, gb = kt0 >> 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int nrt = min(kConsumers, a.RT - rt0);
    const int KG = a.KT >> 2;
    const bool producer = warp == kConsumers;
    const unsigned char *qs = reinterpret_cast<const unsigned char *>(a.qs);

    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], kConsumers);
        }
        for (int r = 0; r < 8; ++r) s_rowmax[r] = 0;
        s_fail = 0;
        mbar_init_fence();
    }
    __syncthreads();

    // group j of this slice: the CTA's row tiles at k-tiles 4(gb+j) .. 4(gb+j)+3, 2 KB each
    auto issue = [&](int j) {
        const int st = j % kStages;
        mbar_expect_tx(&full[st], (uint32_t)nrt * 2048u);
        for (int i = 0; i < nrt; ++i)
            bulk_g2s(ring + st * kStageBytes + i * 2048, qs + ((size_t)(rt0 + i) * a.KT + 4 * (size_t)(gb + j)) * 512,
                     2048u, &full[st]);
    };
    // the weights do not depend on the previous kernel: start the ring before waiting on it
    if (producer && lane == 0)
        for (int j = 0; j < kStages && j < ng; ++j) issue(j);
    if (producer && lane < nrt && ng > kStages)
        dl_prefetch_l2(qs + ((size_t)(rt0 + lane) * a.KT + 4 * (size_t)(gb + kStages)) * 512,
                       (uint32_t)(ng - kStages) * 2048u);
    dl_pdl_launch_dependents();
    dl_pdl_wait();

    // ---- the slice's activations, as operand fragments in shared memory (every thread).
    // One pass over global memory: each (k-tile, lane) slot first receives the lane's raw f32
    // inputs (the CUDA-core operand); the tensor path then rewrites it in place as f16 hi/lo
    // terms scaled by one power of two per activation row.
    const int npairs = nkt * 32;                     // (k-tile, lane) pairs
    {
        constexpr int PB = 4;                        // slots per thread per batch, loads issued together
        for (int base = threadIdx.x; base < npairs; base += PB * kThreads5) {
            float v[PB][NRC][8];
#pragma unroll
            for (int u = 0; u < PB; ++u) {
                const int pi = base + u * kThreads5;
                const int kt = kt0 + (pi >> 5), t = pi & 31, cc = t & 3;
#pragma unroll
                for (int r = 0; r < NRC; ++r) {
                    const int row = MMA ? (t >> 2) : r;
                    const bool ok = pi < npairs && row < a.nr && kt * 32 < a.n_in;
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        float2 w = make_float2(0.f, 0.f);
                        if (ok) w = __ldg(reinterpret_cast<const float2 *>(a.x + (int64_t)row * a.x_stride + kt * 32 + lane_k(cc, e)));
                        v[u][r][e] = w.x;
                        v[u][r][e + 1] = w.y;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < PB; ++u) {
                const int pi = base + u * kThreads5;
                if (pi >= npairs) break;
                float4 *dst = reinterpret_cast<float4 *>(xf + (size_t)pi * FB);
#pragma unroll
                for (int r = 0; r < NRC; ++r) {
                    dst[2 * r] = make_float4(v[u][r][0], v[u][r][1], v[u][r][2], v[u][r][3]);
                    dst[2 * r + 1] = make_float4(v[u][r][4], v[u][r][5], v[u][r][6], v[u][r][7]);
                }
                if constexpr (MMA) {
                    const int gg = (pi & 31) >> 2;
                    float m = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[u][0][e]));
                    if (gg < a.nr && m > 0.f) atomicMax(&s_rowmax[gg], __float_as_int(m));
                }
            }
        }
    }
    __syncthreads();
    if constexpr (MMA) {
        for (int pi = threadIdx.x; pi < npairs; pi += kThreads5) {
            const int gg = (pi & 31) >> 2;
            float sc, si;
            block_scale(__int_as_float(s_rowmax[gg]), sc, si);
            uint4 *slot = reinterpret_cast<uint4 *>(xf + (size_t)pi * FB);
            const uint4 r0 = slot[0], r1 = slot[1];
            const float x[8] = {__uint_as_float(r0.x), __uint_as_float(r0.y), __uint_as_float(r0.z), __uint_as_float(r0.w),
                                __uint_as_float(r1.x), __uint_as_float(r1.y), __uint_as_float(r1.z), __uint_as_float(r1.w)};
            uint32_t hv[4], lv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x0 = x[2 * e] * sc, x1 = x[2 * e + 1] * sc;
                const __half2 h = __floats2half2_rn(x0, x1);
                const float2 hf = __half22float2(h);
                hv[e] = *reinterpret_cast<const uint32_t *>(&h);
                lv[e] = pack_h2(x0 - hf.x, x1 - hf.y);
            }
            slot[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            slot[1] = make_uint4(lv[0], lv[1], lv[2], lv[3]);
        }
        __syncthreads();
    }

    float acc[4] = {0.f, 0.f, 0.f, 0.f};             // tensor path: C fragment
    float accg[NRC], acch[NRC];                      // CUDA-core path: rows g, g+8
#pragma unroll
    for (int r = 0; r < NRC; ++r) accg[r] = acch[r] = 0.f;

    if (producer) {
        // refill each stage once every consumer warp has released it
        if (lane == 0) {
            for (int j = kStages; j < ng; ++j) {
                const int st = j % kStages;
                if (!mbar_wait(&empty[st], (uint32_t)(((j / kStages) - 1) & 1))) {
                    atomicExch(&s_fail, 1);
                    break;
                }
                issue(j);
            }
        }
    } else {
        const int rt = rt0 + warp;
        const bool live = warp < nrt;
        const uint4 *dsc = reinterpret_cast<const uint4 *>(a.d);
        uint4 scn = make_uint4(0u, 0u, 0u, 0u);
        if (live && ng > 0) scn = __ldg(dsc + ((size_t)rt * KG + gb) * 8 + g);
        for (int j = 0; j < ng; ++j) {
            const int st = j % kStages;
            const uint4 sc4 = scn;
            if (live && j + 1 < ng) scn = __ldg(dsc + ((size_t)rt * KG + gb + j + 1) * 8 + g);
            if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (uint32_t)((j / kStages) & 1)))) {
                if (lane == 0) atomicExch(&s_fail, 1);
                break;
            }
            if (live) {
                const unsigned char *sw = ring + st * kStageBytes + warp * 2048;
                const uint32_t sp[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(sw + q * 512 + lane * 16);
                    const float dg = __half2float(__ushort_as_half((unsigned short)(sp[q] & 0xFFFFu)));
                    const float dh = __half2float(__ushort_as_half((unsigned short)(sp[q] >> 16)));
                    const unsigned char *fr = xf + ((size_t)(4 * j + q) * 32 + lane) * FB;
                    if constexpr (MMA) {
                        const uint4 bh = *reinterpret_cast<const uint4 *>(fr);
                        const uint4 bl = *reinterpret_cast<const uint4 *>(fr + 16);
                        const uint32_t a0 = s8x2_to_h2(w.x, 0x5150), a1 = s8x2_to_h2(w.x, 0x5352);
                        const uint32_t a2 = s8x2_to_h2(w.y, 0x5150), a3 = s8x2_to_h2(w.y, 0x5352);
                        const uint32_t a4 = s8x2_to_h2(w.z, 0x5150), a5 = s8x2_to_h2(w.z, 0x5352);
                        const uint32_t a6 = s8x2_to_h2(w.w, 0x5150), a7 = s8x2_to_h2(w.w, 0x5352);
                        float h0 = 0.f, h1 = 0.f, h2 = 0.f, h3 = 0.f;    // hi terms
                        float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;    // lo terms (independent chain)
                        mma16816(h0, h1, h2, h3, a0, a1, a2, a3, bh.x, bh.y);
                        mma16816(l0, l1, l2, l3, a0, a1, a2, a3, bl.x, bl.y);
                        mma16816(h0, h1, h2, h3, a4, a5, a6, a7, bh.z, bh.w);
                        mma16816(l0, l1, l2, l3, a4, a5, a6, a7, bl.z, bl.w);
                        acc[0] = fmaf(dg, h0 + l0, acc[0]);
                        acc[1] = fmaf(dg, h1 + l1, acc[1]);
                        acc[2] = fmaf(dh, h2 + l2, acc[2]);
                        acc[3] = fmaf(dh, h3 + l3, acc[3]);
                    } else {
                        float wg[8], wh[8];
                        wg[0] = s8_to_f32(w.x, 0); wg[1] = s8_to_f32(w.x, 1);
                        wg[2] = s8_to_f32(w.y, 0); wg[3] = s8_to_f32(w.y, 1);
                        wg[4] = s8_to_f32(w.z, 0); wg[5] = s8_to_f32(w.z, 1);
                        wg[6] = s8_to_f32(w.w, 0); wg[7] = s8_to_f32(w.w, 1);
                        wh[0] = s8_to_f32(w.x, 2); wh[1] = s8_to_f32(w.x, 3);
                        wh[2] = s8_to_f32(w.y, 2); wh[3] = s8_to_f32(w.y, 3);
                        wh[4] = s8_to_f32(w.z, 2); wh[5] = s8_to_f32(w.z, 3);
                        wh[6] = s8_to_f32(w.w, 2); wh[7] = s8_to_f32(w.w, 3);
#pragma unroll
                        for (int r = 0; r < NRC; ++r) {
                            const float4 xa = *reinterpret_cast<const float4 *>(fr + r * 32);
                            const float4 xb = *reinterpret_cast<const float4 *>(fr + r * 32 + 16);
                            float sg = wg[0] * xa.x, sh = wh[0] * xa.x;
                            sg = fmaf(wg[1], xa.y, sg); sh = fmaf(wh[1], xa.y, sh);
                            sg = fmaf(wg[2], xa.z, sg); sh = fmaf(wh[2], xa.z, sh);
                            sg = fmaf(wg[3], xa.w, sg); sh = fmaf(wh[3], xa.w, sh);
                            sg = fmaf(wg[4], xb.x, sg); sh = fmaf(wh[4], xb.x, sh);
                            sg = fmaf(wg[5], xb.y, sg); sh = fmaf(wh[5], xb.y, sh);
                            sg = fmaf(wg[6], xb.z, sg); sh = fmaf(wh[6], xb.z, sh);
                            sg = fmaf(wg[7], xb.w, sg); sh = fmaf(wh[7], xb.w, sh);
                            accg[r] = fmaf(dg, sg, accg[r]);
                            acch[r] = fmaf(dh, sh, acch[r]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
    }
    __syncthreads();
    const bool failed = s_fail != 0;

    // ---- results: each consumer warp holds complete sums of its row tile over the slice
    const int rt = rt0 + warp;
    const bool mine = !producer && warp < nrt;
    auto emit = [&](int o, int col, float v) {         // o: output row, col: activation row
        if (failed) v = __int_as_float(0x7fc00000);
        if (a.cs == 1) {
            if (o < a.n_out) a.y[(int64_t)col * a.y_stride + o] = v;
        } else {
            cpart[(warp * 16 + (o - rt * 16)) * 8 + col] = v;
        }
    };
    if (mine) {
        if constexpr (MMA) {
            float s0, si0, s1, si1;
            block_scale(__int_as_float(s_rowmax[2 * c]), s0, si0);
            block_scale(__int_as_float(s_rowmax[2 * c + 1]), s1, si1);
            if (2 * c < a.nr) {
                emit(rt * 16 + g, 2 * c, acc[0] * si0);
                emit(rt * 16 + g + 8, 2 * c, acc[2] * si0);
            }
            if (2 * c + 1 < a.nr) {
                emit(rt * 16 + g, 2 * c + 1, acc[1] * si1);
                emit(rt * 16 + g + 8, 2 * c + 1, acc[3] * si1);
            }
        } else {
#pragma unroll
            for (int r = 0; r < NRC; ++r) {
                float vg = accg[r], vh = acch[r];
                vg += __shfl_xor_sync(0xffffffffu, vg, 1);
                vg += __shfl_xor_sync(0xffffffffu, vg, 2);
                vh += __shfl_xor_sync(0xffffffffu, vh, 1);
                vh += __shfl_xor_sync(0xffffffffu, vh, 2);
                if (c == 0 && r < a.nr) {
                    emit(rt * 16 + g, r, vg);
                    emit(rt * 16 + g + 8, r, vh);
                }
            }
        }
    }
    if (a.cs > 1) {
        // every K-slice of this run of row tiles holds its partials in shared memory: sum in rank order
        cluster_sync_all();
        for (int e = threadIdx.x; e < nrt * 128; e += kThreads5) {
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
    if (o >= n_out || k >= n_in) return 0x80u;       // a zero weight, stored biased
    return blocks[(o * (n_in / 32) + k / 32) * 34 + 2 + (k % 32)] ^ 0x80u;   // q + 128
}

__global__ void q8_pack_qs_kernel(const uint8_t *blocks, int64_t n_out, int64_t n_in, int KT,
                                  int64_t units, uint4 *qs)
{
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= units) return;
    const int lane = (int)(u & 31);
    const int64_t t = u >> 5;
    const int64_t kt = t % KT, rt = t / KT;
    const int g = lane >> 2, c = lane & 3;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int h = j >> 3, p = (j >> 1) & 3, e = j & 1;
        const int row = g + (p & 1) * 8;
        const int kk = 2 * c + (p >> 1) * 8 + h * 16 + e;
        const uint32_t b = q8_byte(blocks, n_out, n_in, rt * 16 + row, kt * 32 + kk);
        w[j >> 2] |= b << (8 * (j & 3));
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
    int nrc, cs, ksl, grid;
    size_t smem;
};

void *pick_kernel(bool mma, int nrc)
{
    if (mma) return reinterpret_cast<void *>(gemv_q8_kernel<true, 1>);
    if (nrc == 1) return reinterpret_cast<void *>(gemv_q8_kernel<false, 1>);
    return reinterpret_cast<void *>(gemv_q8_kernel<false, 2>);
}

// The dynamic shared-memory limit is a per-function attribute shared by every launch of the
// kernel (graph nodes and profilers re-launch against it): set it once to the largest size any
// launch shape may use, never to one launch's own size.
constexpr int kSmemLimit = 200 * 1024;

int prepare_kernel(const void *kern, size_t smem, int cs)
{
    if (smem > (size_t)kSmemLimit) return dl::fail(DL_E_SHAPE, "dl_gemv_q8: %zu bytes of shared memory", smem);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8: set shared memory");
    if (cs > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8: allow a large cluster");
    }
    return DL_OK;
}

// CTAs of one launch shape that are resident at once (clusters counted whole).
int resident_ctas(const void *kern, int cs, size_t smem, int sm)
{
    if (cs <= 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads5, smem) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        return per_sm * sm;
    }
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)cs);
    lc.blockDim = dim3(kThreads5);
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
    return clusters * cs;
}

// Launch shape: K split into cs slices of whole groups of 4 k-tiles, 8 row tiles per CTA;
// the smallest slice whose grid is resident in one wave, then the fewest slices.
int choose_cfg(int nr, int RT, int KT, int sm, int path, GemvCfg *out)
{
    const bool mma = path == PATH_TENSOR || (path == PATH_AUTO && nr > 2);
    if (!mma && nr > 2) return dl::fail(DL_E_SHAPE, "dl_gemv_q8: the CUDA-core path serves 1 or 2 rows per command");
    const int nrc = mma ? 1 : nr;
    const void *kern = pick_kernel(mma, nrc);
    const int mgroups = (int)dl::ceil_div(RT, kConsumers);
    GemvCfg best{};
    int best_ksl = -1;
    for (int cs = 1; cs <= 16; ++cs) {
        const int ksl = (int)dl::ceil_div(dl::ceil_div(KT, cs), 4) * 4;
        if ((int)dl::ceil_div(KT, ksl) != cs) continue;
        const size_t smem = gemv_smem(mma, nrc, ksl);
        if (smem > (size_t)kSmemLimit) continue;
        if (prepare_kernel(kern, smem, cs) != DL_OK) return DL_E_CUDA;
        const int grid = mgroups * cs;
        if (grid > resident_ctas(kern, cs, smem, sm)) continue;
        if (best_ksl < 0 || ksl < best_ksl) {
            best_ksl = ksl;
            best = GemvCfg{mma, nrc, cs, ksl, grid, smem};
        }
    }
    if (best_ksl < 0) {
        // more row tiles than one wave holds: whole-K CTAs in several waves, or the
        // smallest slices that fit shared memory
        for (int cs = 1; cs <= 16 && best_ksl < 0; ++cs) {
            const int ksl = (int)dl::ceil_div(dl::ceil_div(KT, cs), 4) * 4;
            if ((int)dl::ceil_div(KT, ksl) != cs) continue;
            const size_t smem = gemv_smem(mma, nrc, ksl);
            if (smem > (size_t)kSmemLimit) continue;
            if (prepare_kernel(kern, smem, cs) != DL_OK) return DL_E_CUDA;
            best_ksl = ksl;
            best = GemvCfg{mma, nrc, cs, ksl, mgroups * cs, smem};
        }
        if (best_ksl < 0) return dl::fail(DL_E_SHAPE, "dl_gemv_q8: no launch shape for %d k-tiles", KT);
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
    const void *kern = pick_kernel(cfg.mma, cfg.nrc);
    rc = prepare_kernel(kern, cfg.smem, cfg.cs);     // the shape search left another candidate's limit
    if (rc != DL_OK) return rc;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)cfg.grid);
    lc.blockDim = dim3(kThreads5);
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
