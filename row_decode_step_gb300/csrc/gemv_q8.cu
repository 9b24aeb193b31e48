// Q8_0 projection GEMV over 1..8 rows per command (the router/projection
// "enc_cols" role of daScript PR #4473, commit "cud_router_enc_cols tiles every
// router launch": eight activation columns per launch, longer launches tiled).
//
// Device weight form: tiles of 16 output rows x 32 inputs (one Q8_0 block per
// row), 512 bytes each, in the A-operand order of two 16x8x16 f16 tensor-core
// products, as biased bytes u = q + 128.  Lane t = 4g + c owns 16 bytes; word p
// (p = 0..3) covers inputs kb = 16(p/2) + 8(p%2) + 2c and kb + 1 of row g (bytes
// 0, 1) and of row g + 8 (bytes 2, 3).  One byte permute turns two bytes into the
// f16 pair (1024 + u) = (1152 + q), exact.  The tiles of one row tile are
// contiguous along K.  Scales: per 16 rows and 4 tiles, 128 bytes; lane group g
// reads 16 bytes = (d[g], d[g+8]) for the 4 tiles.
//
// The same kernel serves f16 weights (the halfword-weight reference lane of the same PR's
// description): 1024-byte tiles of 16 rows x 32 inputs in the same A-operand order, no scales.
//
// Kernel shape (two CTAs per SM, one wave):
//  * a CTA of 8 warps owns a run of row tiles and one K-slice; each stage of a shared-memory
//    ring (about 80 KB, mbarrier-tracked) holds one row tile's slice (weights, then scales: two
//    contiguous bulk copies; f16 weights: one).  Thread 0 requests two stages before waiting on
//    the previous kernel (programmatic dependent launch: the weights do not depend on it) and the
//    rest right after the warps have requested their activations;
//  * each warp owns an eighth of the slice's k-tiles; its activations are loaded once, per lane
//    from L2, and kept in registers as operands for the whole launch;
//  * warps run free over the stages: each keeps its partials of a batch of 4 row tiles in
//    registers, the last warp done with a stage refills its slot, one CTA-wide reduction per batch
//    sums the 8 warps' 16x8 partials in warp order; the K-slices of a thread-block cluster are
//    summed through distributed shared memory in rank order at the end (no atomics: results do
//    not depend on timing).
// Two inner products share this shape.  Tensor path: the f16 weights (1152 + q for Q8_0, as
// stored for f16 weights) enter 16x8x16 f16 products with f32 accumulation; each activation row
// is scaled per warp by a power of two (largest |x| into [2^14, 2^15)) and split into two f16
// terms hi + lo (about 22 significant bits); for Q8_0 the products' bias 1152 * sum(x) is taken
// off per block and column; the scale is undone per column at the end.  CUDA-core path (1 or 2
// rows): the weights are widened to f32 and multiplied with the f32 activations by packed FMAs.
#include <cuda_fp16.h>
#include <cstdio>
#include <algorithm>
#include <mutex>

#include "dl_common.cuh"
#include "dl_async.cuh"

namespace {

enum { PATH_AUTO = 0, PATH_CUDA_CORE = 1, PATH_TENSOR = 2 };

struct GemvArgs {
    const unsigned char *qs;   // packed weight tiles
    const unsigned char *d;    // packed scales as (d[g], d[g+8]) pairs
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
    int pre;                // ring stages requested before waiting on the previous kernel
    DlPrefetch pf;          // L2 prefetches for a later kernel, issued after those stages
};

constexpr int kConsumers = 8;                        // warps, each a share of the K-slice
constexpr int kThreads = kConsumers * 32;
constexpr int kMaxStages = 8;
constexpr int kTileBytesQ8 = 512 + 32;               // Q8_0: weights and scales of one k-tile
constexpr int kTileBytesF16 = 1024;                  // f16 weights of one k-tile
constexpr int kRowBatch = 4;                         // row tiles whose partials a warp holds at once
constexpr size_t kRedBytes = (size_t)kRowBatch * kConsumers * 128 * 4;   // one batch of per-warp partials

// Shared-memory bytes of a launch: the ring, the per-stage partials and, with clusters,
// this CTA's K-slice sums of its row tiles.
size_t gemv_smem(int ksl, int stages, int rpr, int cs, int tile_bytes)
{
    return (size_t)stages * ksl * tile_bytes + kRedBytes + (cs > 1 ? (size_t)rpr * 128 * 4 : 0);
}

// ---- arithmetic helpers
// biased weight bytes `lo`, `lo + 1` of w (u = q + 128) to the float pair (q, q'): each u is placed
// in the low mantissa of 2^23, and one packed subtraction takes 2^23 + 128 off both
__device__ __forceinline__ float2 u8x2_to_f32x2(uint32_t w, uint32_t lo)
{
    const float2 b = make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | lo)),
                                 __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541u | lo)));
    return __fadd2_rn(b, make_float2(-8388736.0f, -8388736.0f));
}
// two biased bytes (0, 1 or 2, 3) of w to the f16 pair (1024 + u)
__device__ __forceinline__ uint32_t u8x2_to_h2(uint32_t w, uint32_t sel)
{
    return __byte_perm(w, 0x64646464u, sel);
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// W16: the weights are f16 (the halfword-weight lane) instead of Q8_0 biased bytes and scales.
template <bool W16, bool MMA, int NRC, int KWM>
__global__ void __launch_bounds__(kThreads, 2) gemv_q8_kernel(const __grid_constant__ GemvArgs a)
{
    constexpr int RB = kRowBatch;
    constexpr int TB = W16 ? kTileBytesF16 : kTileBytesQ8;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ int s_shape_bad, s_issued;
    __shared__ int s_cnt[kMaxStages];                 // warps done with the stage in each slot

    const int S = a.stages;
    const int slice = blockIdx.x % a.cs;
    const int rt0 = (blockIdx.x / a.cs) * a.rpr;
    const int nrt = max(0, min(a.rpr, a.RT - rt0));      // row tiles of this CTA
    const int kt0 = slice * a.ksl, kt1 = min(a.KT, kt0 + a.ksl);
    const int nkt = max(0, kt1 - kt0);
    const uint32_t wbytes = (uint32_t)nkt * (W16 ? 1024u : 512u), dbytes = W16 ? 0u : (uint32_t)nkt * 32u;
    const size_t SB = (size_t)a.ksl * TB;
    unsigned char *ring = smem;
    float *red = reinterpret_cast<float *>(smem + S * SB);          // [kRowBatch][kConsumers][128]
    float *part = red + kRowBatch * kConsumers * 128;                // [rpr][128] (clusters)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int KG = a.KT >> 2;

    if (threadIdx.x == 0) {
        for (int st = 0; st < S; ++st) {
            dla::mbar_init(&full[st], 1);
            s_cnt[st] = 0;
        }
        s_shape_bad = 0;
        s_issued = min(S, nrt);
        dla::mbar_init_fence();
    }
    // a slice shorter than the stage (the last one of K): the missing k-tiles' scales (Q8_0) or
    // weights (f16, where stale bytes could read as Inf or NaN and poison 0 * w) read as zero, so
    // that they contribute nothing (the copies carry this slice's k-tiles only, so these bytes
    // are never overwritten)
    if (nkt < a.ksl) {
        const int zw = (a.ksl - nkt) * (W16 ? 256 : 8);              // words per slot
        const size_t z0 = W16 ? (size_t)nkt * 1024 : (size_t)a.ksl * 512 + (size_t)nkt * 32;
        for (int e = threadIdx.x; e < S * zw; e += kThreads) {
            const int st = e / zw, w = e - st * zw;
            reinterpret_cast<uint32_t *>(ring + st * SB + z0)[w] = 0u;
        }
    }
    __syncthreads();

    // stage j: row tile rt0 + j, this slice's k-tiles (contiguous), then their scales (contiguous)
    auto issue = [&](int j) {
        const int st = j % S;
        const int rt = rt0 + j;
        unsigned char *dst = ring + st * SB;
        dla::mbar_expect_tx(&full[st], wbytes + dbytes);
        if constexpr (W16) {
            dla::bulk_g2s(dst, a.qs + ((size_t)rt * a.KT + kt0) * 1024, wbytes, &full[st]);
        } else {
            dla::bulk_g2s(dst, a.qs + ((size_t)rt * a.KT + kt0) * 512, wbytes, &full[st]);
            dla::bulk_g2s(dst + (size_t)a.ksl * 512, a.d + ((size_t)rt * KG + (kt0 >> 2)) * 128, dbytes,
                          &full[st]);
        }
    };
    // the weights do not depend on the previous kernel: the first stages are requested before
    // waiting on it, the rest once the activations are requested (an SM's requests are served
    // roughly in order, and the activations gate every stage)
    if (threadIdx.x == 0) {
        for (int j = 0; j < a.pre && j < S && j < nrt; ++j) issue(j);
        if (a.pf.n > 0) dl_issue_prefetch(a.pf);
    }
    auto issue_rest = [&]() {
        if (threadIdx.x == 0)
            for (int j = a.pre; j < S && j < nrt; ++j) issue(j);
    };
    // every thread waits before the next kernel may launch: kernels after this one can rely
    // on everything before this one having finished
    dl_pdl_wait();
    dl_pdl_launch_dependents();
    const int xfl = max(0, min(nkt * 32, a.n_in - kt0 * 32));   // valid inputs of the slice

    // ---- this warp's window of KWM k-tiles of the slice and its activations, kept in registers;
    // k-tiles past the slice (the last slice of K may be short) have zero activations and scales
    const int wk0 = warp * KWM;                                  // slice-local
    const int nw = max(0, min(KWM, nkt - wk0));
    if (lane == 0 && kConsumers * KWM != a.ksl) atomicExch(&s_shape_bad, 1);   // broken launch shape
    // lane (g, c) holds inputs 8c .. 8c + 7 of each k-tile (pairs 8c + 2p, 8c + 2p + 1): the packed
    // weights put the same inputs in the MMA slots 2c, 2c+1 / 2c+8, 2c+9 / 16+2c, 17+2c / 24+2c, 25+2c
    uint32_t bh[MMA ? KWM : 1][4], bl[MMA ? KWM : 1][4];
    float2 ncorr[MMA && !W16 ? KWM : 1];         // -1152 * sum(x) of columns 2c, 2c+1 per k-tile (Q8_0)
    float xv[MMA ? 1 : KWM][NRC][8];
    float us0 = 1.f, us1 = 1.f;
    if constexpr (MMA) {
        float2 v[KWM][4];
        float m = 0.f;
        float mj[KWM];
#pragma unroll
        for (int j = 0; j < KWM; ++j) {
            const int kl = wk0 + j;
            const bool live = kl * 32 < xfl && g < a.nr;
            const float4 *xr = reinterpret_cast<const float4 *>(a.x + (int64_t)g * a.x_stride + (kt0 + kl) * 32 + 8 * c);
            const float4 lo = live ? __ldcg(xr) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 hi = live ? __ldcg(xr + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
            v[j][0] = make_float2(lo.x, lo.y);
            v[j][1] = make_float2(lo.z, lo.w);
            v[j][2] = make_float2(hi.x, hi.y);
            v[j][3] = make_float2(hi.z, hi.w);
        }
        issue_rest();
#pragma unroll
        for (int j = 0; j < KWM; ++j) {
            mj[j] = fmaxf(fmaxf(fmaxf(fabsf(v[j][0].x), fabsf(v[j][0].y)), fmaxf(fabsf(v[j][1].x), fabsf(v[j][1].y))),
                          fmaxf(fmaxf(fabsf(v[j][2].x), fabsf(v[j][2].y)), fmaxf(fabsf(v[j][3].x), fabsf(v[j][3].y))));
        }
#pragma unroll
        for (int j = 0; j < KWM; ++j) m = fmaxf(m, mj[j]);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        // power-of-two scale of activation row g over this warp's inputs: largest |x| into [2^14, 2^15),
        // built from the exponent field of m (m in [2^(E-127), 2^(E-126)) -> scale 2^(141-E), at most
        // 2^126; m = 0 keeps 1)
        const int ebits = (int)((__float_as_uint(m) >> 23) & 0xFFu);
        const int sexp = m > 0.f ? min(268 - ebits, 253) : 127;
        const float sig = __uint_as_float((uint32_t)sexp << 23);
        const float inv = __uint_as_float((uint32_t)(254 - sexp) << 23);
#pragma unroll
        for (int j = 0; j < KWM; ++j) {
            float colsum = 0.f;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float tx = v[j][p].x * sig, ty = v[j][p].y * sig;
                const __half2 h = __floats2half2_rn(tx, ty);
                const float2 hf = __half22float2(h);
                const __half2 l = __floats2half2_rn(tx - hf.x, ty - hf.y);
                const float2 lf = __half22float2(l);
                bh[j][p] = h2_bits(h);
                bl[j][p] = h2_bits(l);
                colsum += (hf.x + lf.x) + (hf.y + lf.y);
            }
            if constexpr (!W16) {
                colsum += __shfl_xor_sync(0xffffffffu, colsum, 1);
                colsum += __shfl_xor_sync(0xffffffffu, colsum, 2);
                // accumulator columns of this lane are activation rows 2c and 2c+1 (lanes 8c, 8c+4)
                ncorr[j] = make_float2(-1152.f * __shfl_sync(0xffffffffu, colsum, 8 * c),
                                       -1152.f * __shfl_sync(0xffffffffu, colsum, 8 * c + 4));
            }
        }
        us0 = __shfl_sync(0xffffffffu, inv, 8 * c);
        us1 = __shfl_sync(0xffffffffu, inv, 8 * c + 4);
    } else {
#pragma unroll
        for (int j = 0; j < KWM; ++j) {
            const int kl = wk0 + j;
#pragma unroll
            for (int r = 0; r < NRC; ++r) {
                const bool live = kl * 32 < xfl && r < a.nr;
                const float4 *xr = reinterpret_cast<const float4 *>(a.x + (int64_t)r * a.x_stride + (kt0 + kl) * 32 + 8 * c);
                const float4 lo = live ? __ldcg(xr) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 hi = live ? __ldcg(xr + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                xv[j][r][0] = lo.x;
                xv[j][r][1] = lo.y;
                xv[j][r][2] = lo.z;
                xv[j][r][3] = lo.w;
                xv[j][r][4] = hi.x;
                xv[j][r][5] = hi.y;
                xv[j][r][6] = hi.z;
                xv[j][r][7] = hi.w;
            }
        }
        issue_rest();
    }

    // ---- stages in batches of RB row tiles: each warp keeps its partial of every row tile of
    // the batch in registers; no barrier between stages (the last warp done with a stage refills
    // its slot), one CTA-wide reduction per batch
    bool bad = false;
    for (int b0 = 0; b0 < nrt; b0 += RB) {
        const int nb = min(RB, nrt - b0);
        float2 acc01[RB], acc23[RB];                 // tensor path: rows g, g+8 x columns 2c, 2c+1
        float2 accg[RB][NRC], acch[RB][NRC];         // CUDA-core path: rows g, g+8 x activation rows
                                                     // (even and odd inputs summed apart)
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            acc01[r] = acc23[r] = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NRC; ++q) accg[r][q] = acch[r][q] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            if (r >= nb) break;                                      // CTA-uniform
            const int i = b0 + r, st = i % S;
            const bool ok = __all_sync(0xffffffffu, dla::mbar_wait(&full[st], (uint32_t)((i / S) & 1)));
            if (!ok) bad = true;
            const unsigned char *sw = ring + st * SB;
            const unsigned char *sd = sw + (size_t)a.ksl * 512;
            if (ok) {
#pragma unroll
                for (int j = 0; j < KWM; ++j) {
                    const int kl = wk0 + j;                                  // slice-local k-tile
                    if constexpr (W16) {
                        // lane's 32 bytes: the A operands of the two 16x8x16 products, f16 as stored
                        const uint4 w0 = *reinterpret_cast<const uint4 *>(sw + kl * 1024 + lane * 32);
                        const uint4 w1 = *reinterpret_cast<const uint4 *>(sw + kl * 1024 + lane * 32 + 16);
                        if constexpr (MMA) {
                            float t[4] = {acc01[r].x, acc01[r].y, acc23[r].x, acc23[r].y};
                            mma16816(t, w0.x, w0.y, w0.z, w0.w, bh[j][0], bh[j][1]);
                            mma16816(t, w0.x, w0.y, w0.z, w0.w, bl[j][0], bl[j][1]);
                            mma16816(t, w1.x, w1.y, w1.z, w1.w, bh[j][2], bh[j][3]);
                            mma16816(t, w1.x, w1.y, w1.z, w1.w, bl[j][2], bl[j][3]);
                            acc01[r] = make_float2(t[0], t[1]);
                            acc23[r] = make_float2(t[2], t[3]);
                        } else {
                            // word 2p: row g, inputs of pair p; word 2p + 1: row g + 8
                            const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                            float2 wg[4], wh[4];
#pragma unroll
                            for (int p = 0; p < 4; ++p) {
                                wg[p] = __half22float2(*reinterpret_cast<const __half2 *>(&wd[2 * p]));
                                wh[p] = __half22float2(*reinterpret_cast<const __half2 *>(&wd[2 * p + 1]));
                            }
#pragma unroll
                            for (int q = 0; q < NRC; ++q) {
                                float2 sg = accg[r][q], sh = acch[r][q];
#pragma unroll
                                for (int p = 0; p < 4; ++p) {
                                    const float2 xp = make_float2(xv[j][q][2 * p], xv[j][q][2 * p + 1]);
                                    sg = __ffma2_rn(wg[p], xp, sg);
                                    sh = __ffma2_rn(wh[p], xp, sh);
                                }
                                accg[r][q] = sg;
                                acch[r][q] = sh;
                            }
                        }
                    } else {
                        const uint4 w = *reinterpret_cast<const uint4 *>(sw + kl * 512 + lane * 16);
                        const __half2 sp = *reinterpret_cast<const __half2 *>(sd + (kl >> 2) * 128 + g * 16 + (kl & 3) * 4);
                        const float2 dgh = __half22float2(sp);          // (d[g], d[g+8])
                        const float dg = dgh.x, dh = dgh.y;
                        if constexpr (MMA) {
                            float t[4] = {0.f, 0.f, 0.f, 0.f};
                            const uint32_t a0 = u8x2_to_h2(w.x, 0x4140u), a1 = u8x2_to_h2(w.x, 0x4342u);
                            const uint32_t a2 = u8x2_to_h2(w.y, 0x4140u), a3 = u8x2_to_h2(w.y, 0x4342u);
                            mma16816(t, a0, a1, a2, a3, bh[j][0], bh[j][1]);
                            mma16816(t, a0, a1, a2, a3, bl[j][0], bl[j][1]);
                            const uint32_t a4 = u8x2_to_h2(w.z, 0x4140u), a5 = u8x2_to_h2(w.z, 0x4342u);
                            const uint32_t a6 = u8x2_to_h2(w.w, 0x4140u), a7 = u8x2_to_h2(w.w, 0x4342u);
                            mma16816(t, a4, a5, a6, a7, bh[j][2], bh[j][3]);
                            mma16816(t, a4, a5, a6, a7, bl[j][2], bl[j][3]);
                            acc01[r] = __ffma2_rn(make_float2(dg, dg), __fadd2_rn(make_float2(t[0], t[1]), ncorr[j]), acc01[r]);
                            acc23[r] = __ffma2_rn(make_float2(dh, dh), __fadd2_rn(make_float2(t[2], t[3]), ncorr[j]), acc23[r]);
                        } else {
                            // row g: bytes 0, 1 of each word; row g+8: bytes 2, 3 (inputs 2p, 2p+1 of
                            // the lane's eight), multiplied pairwise with the activation pairs
                            const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
                            float2 wg[4], wh[4];
#pragma unroll
                            for (int p = 0; p < 4; ++p) {
                                wg[p] = u8x2_to_f32x2(wd[p], 0);
                                wh[p] = u8x2_to_f32x2(wd[p], 2);
                            }
#pragma unroll
                            for (int q = 0; q < NRC; ++q) {
                                const float2 x0 = make_float2(xv[j][q][0], xv[j][q][1]);
                                float2 sg = __fmul2_rn(wg[0], x0), sh = __fmul2_rn(wh[0], x0);
#pragma unroll
                                for (int p = 1; p < 4; ++p) {
                                    const float2 xp = make_float2(xv[j][q][2 * p], xv[j][q][2 * p + 1]);
                                    sg = __ffma2_rn(wg[p], xp, sg);
                                    sh = __ffma2_rn(wh[p], xp, sh);
                                }
                                accg[r][q] = __ffma2_rn(make_float2(dg, dg), sg, accg[r][q]);
                                acch[r][q] = __ffma2_rn(make_float2(dh, dh), sh, acch[r][q]);
                            }
                        }
                    }
                }
            }
            // the last warp done with this stage refills its slot (every warp has read it: the
            // values sit in registers)
            __syncwarp();
            if (lane == 0 && atomicAdd(&s_cnt[st], 1) == kConsumers - 1) {
                s_cnt[st] = 0;
                if (i + S < nrt) {
                    issue(i + S);
                    s_issued = i + S + 1;
                }
            }
        }
        // this warp's partials of the batch: [row tile][warp][row 0..15][column 0..7]
        __syncthreads();                                   // the previous batch's reduction is done
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            if (r >= nb) break;
            float *rw = red + (r * kConsumers + warp) * 128;
            if constexpr (MMA) {
                *reinterpret_cast<float2 *>(rw + g * 8 + 2 * c) = make_float2(acc01[r].x * us0, acc01[r].y * us1);
                *reinterpret_cast<float2 *>(rw + (g + 8) * 8 + 2 * c) = make_float2(acc23[r].x * us0, acc23[r].y * us1);
            } else {
#pragma unroll
                for (int q = 0; q < NRC; ++q) {
                    float vg = accg[r][q].x + accg[r][q].y, vh = acch[r][q].x + acch[r][q].y;
                    vg += __shfl_xor_sync(0xffffffffu, vg, 1);
                    vg += __shfl_xor_sync(0xffffffffu, vg, 2);
                    vh += __shfl_xor_sync(0xffffffffu, vh, 1);
                    vh += __shfl_xor_sync(0xffffffffu, vh, 2);
                    if (c == 0) {
                        rw[g * 8 + q] = vg;
                        rw[(g + 8) * 8 + q] = vh;
                    }
                }
            }
        }
        if (__syncthreads_or(bad)) {                       // a stage that never arrived: stop
            bad = true;
            break;
        }
        // sum the 8 warps' partials in warp order: thread -> 4 consecutive elements of a row tile
        for (int e4 = threadIdx.x; e4 < nb * 32; e4 += kThreads) {
            const int r = e4 >> 5, el = (e4 & 31) * 4;
            const float *rb = red + r * kConsumers * 128 + el;
            float4 sum = *reinterpret_cast<const float4 *>(rb);
#pragma unroll
            for (int w = 1; w < kConsumers; ++w) {
                const float4 t = *reinterpret_cast<const float4 *>(rb + w * 128);
                sum.x += t.x;
                sum.y += t.y;
                sum.z += t.z;
                sum.w += t.w;
            }
            const int i = b0 + r;
            if (a.cs == 1) {
                const int o = (rt0 + i) * 16 + (el >> 3), col0 = el & 7;
                if (o < a.n_out) {
                    const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (col0 + q < a.nr) a.y[(int64_t)(col0 + q) * a.y_stride + o] = sv[q];
                }
            } else {
                *reinterpret_cast<float4 *>(part + i * 128 + el) = sum;
            }
        }
    }
    if (bad && threadIdx.x == 0) {
        // do not leave with copies in flight: wait (bounded) for every stage that may still land
        const int hi = s_issued;
        for (int j = max(0, hi - S); j < hi; ++j) dla::mbar_wait(&full[j % S], (uint32_t)((j / S) & 1));
    }
    const bool failed = __syncthreads_or(bad || s_shape_bad) != 0;

    if (a.cs > 1) {
        // every K-slice of this run of row tiles holds its sums in shared memory: add them in rank order
        if (failed)
            for (int e = threadIdx.x; e < nrt * 128; e += kThreads) part[e] = __int_as_float(0x7fc00000);
        dla::cluster_sync_all();
        for (int e4 = threadIdx.x; e4 < nrt * 32; e4 += kThreads) {
            const int i = e4 >> 5;
            if (i % a.cs != slice) continue;                 // each rank finishes a share of the row tiles
            float4 s = dla::ld_dsmem_f32x4(part + e4 * 4, 0);
            for (int q = 1; q < a.cs; ++q) {
                const float4 t = dla::ld_dsmem_f32x4(part + e4 * 4, (uint32_t)q);
                s.x += t.x;
                s.y += t.y;
                s.z += t.z;
                s.w += t.w;
            }
            const int o = (rt0 + i) * 16 + ((e4 & 31) >> 1), col0 = (e4 & 1) * 4;
            if (o < a.n_out) {
                const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (col0 + q < a.nr) a.y[(int64_t)(col0 + q) * a.y_stride + o] = sv[q];
            }
        }
        // keep this CTA's shared memory alive until every peer has read it (no ordering of the
        // output stores is needed, so the arrive does not wait for them)
        dla::cluster_sync_relaxed();
    } else if (failed) {
        for (int e = threadIdx.x; e < nrt * 128; e += kThreads) {
            const int o = rt0 * 16 + (e >> 3), col = e & 7;
            if (o < a.n_out && col < a.nr) a.y[(int64_t)col * a.y_stride + o] = __int_as_float(0x7fc00000);
        }
    }
}

// ---------------------------------------------------------------- packing

__device__ __forceinline__ uint32_t q8_byte(const uint8_t *blocks, int64_t n_out, int64_t n_in,
                                            int64_t o, int64_t k)
{
    if (o >= n_out || k >= n_in) return 0u;
    return blocks[(o * (n_in / 32) + k / 32) * 34 + 2 + (k % 32)];
}

// lane t = 4g + c of tile (rt, kt), word p: inputs kb, kb + 1 (kb = 8c + 2p) of row g, then of
// row g + 8, as biased bytes q + 128 (padding: q = 0).  In the tensor path word p fills the MMA
// A slots of pair p of the lane (2c, 2c+1 / 2c+8, 2c+9 / 16+2c, 17+2c / 24+2c, 25+2c): the order
// of the 32 inputs inside a k-tile is permuted alike for the weights and the activations, so a
// lane's activations are eight consecutive floats (two 16-byte loads)
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
    for (int p = 0; p < 4; ++p) {
        const int kb = 8 * c + 2 * p;
        const int64_t k = kt * 32 + kb, o = rt * 16 + g;
        const uint32_t b0 = q8_byte(blocks, n_out, n_in, o, k) ^ 0x80u;
        const uint32_t b1 = q8_byte(blocks, n_out, n_in, o, k + 1) ^ 0x80u;
        const uint32_t b2 = q8_byte(blocks, n_out, n_in, o + 8, k) ^ 0x80u;
        const uint32_t b3 = q8_byte(blocks, n_out, n_in, o + 8, k + 1) ^ 0x80u;
        w[p] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
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

// ---------------------------------------------------------------- chained GEMVs
// A sequence of Q8_0 GEMVs (say O -> gate/up -> down) in one persistent launch: the grid is
// exactly the CTAs resident at once (two per SM), the phases are separated by grid barriers
// (phase p + 1 may read phase p's outputs), and each CTA's stages of all phases form one
// sequence through its ring, so the weights of phase p + 1 stream while phase p finishes and
// the barrier settles.  Every slice is 32 k-tiles (four per warp); the K-slices of a row tile
// add their sums into outputs zeroed before the first barrier.
constexpr int kChainKWM = 4;
constexpr int kChainKsl = kConsumers * kChainKWM;
constexpr int kChainMaxPhases = 4;
constexpr int kBarrierSpins = 1 << 20;               // x 256 ns: a barrier gives up after ~0.3 s

struct ChainPhase {
    const unsigned char *qs, *d;
    const float *x;
    float *y;
    int64_t x_stride, y_stride;
    int n_out, n_in, KT, RT, cs, rpr;
};

struct ChainArgs {
    ChainPhase ph[kChainMaxPhases];
    int nph, nr, stages;
    unsigned *sync;                                  // [0] arrivals, [1] generation
    int32_t *status;
};

template <bool MMA, int NRC>
__global__ void __launch_bounds__(kThreads, 2) gemv_chain_kernel(const __grid_constant__ ChainArgs a)
{
    constexpr int RB = kRowBatch, KWM = kChainKWM;
    constexpr size_t SB = (size_t)kChainKsl * kTileBytesQ8;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ int s_issued, s_fail;
    __shared__ int s_cnt[kMaxStages];
    __shared__ int s_off[kChainMaxPhases + 1], s_rt0[kChainMaxPhases], s_slice[kChainMaxPhases];

    const int S = a.stages;
    unsigned char *ring = smem;
    float *red = reinterpret_cast<float *>(smem + S * SB);          // [kRowBatch][kConsumers][128]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const unsigned G = gridDim.x;

    if (threadIdx.x == 0) {
        int off = 0;
        for (int p = 0; p < a.nph; ++p) {
            const ChainPhase &P = a.ph[p];
            const int rt0 = (int)(blockIdx.x / P.cs) * P.rpr;
            s_off[p] = off;
            s_rt0[p] = rt0;
            s_slice[p] = (int)(blockIdx.x % P.cs);
            off += max(0, min(P.rpr, P.RT - rt0));
        }
        s_off[a.nph] = off;
        for (int st = 0; st < S; ++st) {
            dla::mbar_init(&full[st], 1);
            s_cnt[st] = 0;
        }
        s_issued = min(S, off);
        s_fail = 0;
        dla::mbar_init_fence();
    }
    __syncthreads();
    const int total = s_off[a.nph];

    // stage gi of this CTA's sequence: phase p's row tile, its slice's k-tiles, then their scales
    auto issue = [&](int gi) {
        int p = 0;
        while (gi >= s_off[p + 1]) ++p;
        const ChainPhase &P = a.ph[p];
        const int rt = s_rt0[p] + (gi - s_off[p]);
        const int kt0 = s_slice[p] * kChainKsl;
        unsigned char *dst = ring + (size_t)(gi % S) * SB;
        dla::mbar_expect_tx(&full[gi % S], (uint32_t)(kChainKsl * kTileBytesQ8));
        dla::bulk_g2s(dst, P.qs + ((size_t)rt * P.KT + kt0) * 512, kChainKsl * 512u, &full[gi % S]);
        dla::bulk_g2s(dst + kChainKsl * 512, P.d + ((size_t)rt * (P.KT >> 2) + (kt0 >> 2)) * 128, kChainKsl * 32u,
                      &full[gi % S]);
    };
    // grid barrier (every CTA resident: the grid is the resident capacity); bounded: a CTA that
    // waits too long records the failure and the launch winds down
    auto grid_barrier = [&]() -> bool {
        __syncthreads();
        if (threadIdx.x == 0) {
            volatile unsigned *gen = a.sync + 1;
            const unsigned g0 = *gen;
            __threadfence();
            const unsigned arrived = atomicAdd(a.sync, 1u);
            bool ok = true;
            if (arrived == G - 1) {
                atomicExch(a.sync, 0u);
                __threadfence();
                atomicAdd(a.sync + 1, 1u);
            } else {
                for (int it = 0; *gen == g0; ++it) {
                    if (it > kBarrierSpins) {
                        ok = false;
                        break;
                    }
                    __nanosleep(256);
                }
            }
            __threadfence();
            if (!ok) {
                s_fail = 1;
                dl_status_or(a.status, DL_STATUS_SYNC_TIMEOUT);
            }
        }
        __syncthreads();
        return s_fail == 0;
    };

    if (threadIdx.x == 0)
        for (int gi = 0; gi < S && gi < total; ++gi) issue(gi);     // weights: not the previous kernel's
    dl_pdl_wait();
    // every phase's outputs start at zero (the K-slices add into them)
    for (int p = 0; p < a.nph; ++p) {
        const ChainPhase &P = a.ph[p];
        const int n4 = P.n_out / 4;
        for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < (int64_t)a.nr * n4;
             e += (int64_t)G * kThreads) {
            const int r = (int)(e / n4), o4 = (int)(e - (int64_t)r * n4);
            reinterpret_cast<float4 *>(P.y + r * P.y_stride)[o4] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    bool bad = !grid_barrier();
    for (int p = 0; p < a.nph && !bad; ++p) {
        if (p > 0 && !grid_barrier()) {
            bad = true;
            break;
        }
        const ChainPhase &P = a.ph[p];
        const int base = s_off[p], nrt = s_off[p + 1] - base;
        const int kt0 = s_slice[p] * kChainKsl;
        const int wk0 = warp * KWM;
        // this warp's activations (every slice is whole: K is a multiple of 32 k-tiles)
        uint32_t bh[MMA ? KWM : 1][4], bl[MMA ? KWM : 1][4];
        float2 ncorr[MMA ? KWM : 1];
        float xv[MMA ? 1 : KWM][NRC][8];
        float us0 = 1.f, us1 = 1.f;
        if constexpr (MMA) {
            float2 v[KWM][4];
#pragma unroll
            for (int j = 0; j < KWM; ++j) {
                const float4 *xr = reinterpret_cast<const float4 *>(P.x + (int64_t)g * P.x_stride + (kt0 + wk0 + j) * 32 + 8 * c);
                const float4 lo = g < a.nr ? __ldcg(xr) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 hi = g < a.nr ? __ldcg(xr + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                v[j][0] = make_float2(lo.x, lo.y);
                v[j][1] = make_float2(lo.z, lo.w);
                v[j][2] = make_float2(hi.x, hi.y);
                v[j][3] = make_float2(hi.z, hi.w);
            }
            float m = 0.f;
#pragma unroll
            for (int j = 0; j < KWM; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(fabsf(v[j][q].x), fabsf(v[j][q].y)));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            const int ebits = (int)((__float_as_uint(m) >> 23) & 0xFFu);
            const int sexp = m > 0.f ? min(268 - ebits, 253) : 127;
            const float sig = __uint_as_float((uint32_t)sexp << 23);
            const float inv = __uint_as_float((uint32_t)(254 - sexp) << 23);
#pragma unroll
            for (int j = 0; j < KWM; ++j) {
                float colsum = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float tx = v[j][q].x * sig, ty = v[j][q].y * sig;
                    const __half2 hh = __floats2half2_rn(tx, ty);
                    const float2 hf = __half22float2(hh);
                    const __half2 ll = __floats2half2_rn(tx - hf.x, ty - hf.y);
                    const float2 lf = __half22float2(ll);
                    bh[j][q] = h2_bits(hh);
                    bl[j][q] = h2_bits(ll);
                    colsum += (hf.x + lf.x) + (hf.y + lf.y);
                }
                colsum += __shfl_xor_sync(0xffffffffu, colsum, 1);
                colsum += __shfl_xor_sync(0xffffffffu, colsum, 2);
                ncorr[j] = make_float2(-1152.f * __shfl_sync(0xffffffffu, colsum, 8 * c),
                                       -1152.f * __shfl_sync(0xffffffffu, colsum, 8 * c + 4));
            }
            us0 = __shfl_sync(0xffffffffu, inv, 8 * c);
            us1 = __shfl_sync(0xffffffffu, inv, 8 * c + 4);
        } else {
#pragma unroll
            for (int j = 0; j < KWM; ++j)
#pragma unroll
                for (int r = 0; r < NRC; ++r) {
                    const float4 *xr = reinterpret_cast<const float4 *>(P.x + (int64_t)r * P.x_stride + (kt0 + wk0 + j) * 32 + 8 * c);
                    const float4 lo = r < a.nr ? __ldcg(xr) : make_float4(0.f, 0.f, 0.f, 0.f);
                    const float4 hi = r < a.nr ? __ldcg(xr + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                    xv[j][r][0] = lo.x;
                    xv[j][r][1] = lo.y;
                    xv[j][r][2] = lo.z;
                    xv[j][r][3] = lo.w;
                    xv[j][r][4] = hi.x;
                    xv[j][r][5] = hi.y;
                    xv[j][r][6] = hi.z;
                    xv[j][r][7] = hi.w;
                }
        }
        for (int b0 = 0; b0 < nrt && !bad; b0 += RB) {
            const int nb = min(RB, nrt - b0);
            float2 acc01[RB], acc23[RB];
            float2 accg[RB][NRC], acch[RB][NRC];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                acc01[r] = acc23[r] = make_float2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < NRC; ++q) accg[r][q] = acch[r][q] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                if (r >= nb) break;                                     // CTA-uniform
                const int gi = base + b0 + r, st = gi % S;
                const bool ok = __all_sync(0xffffffffu, dla::mbar_wait(&full[st], (uint32_t)((gi / S) & 1)));
                if (!ok) bad = true;
                const unsigned char *sw = ring + (size_t)st * SB;
                const unsigned char *sd = sw + kChainKsl * 512;
                if (ok) {
#pragma unroll
                    for (int j = 0; j < KWM; ++j) {
                        const int kl = wk0 + j;
                        const uint4 w = *reinterpret_cast<const uint4 *>(sw + kl * 512 + lane * 16);
                        const __half2 sp = *reinterpret_cast<const __half2 *>(sd + (kl >> 2) * 128 + g * 16 + (kl & 3) * 4);
                        const float2 dgh = __half22float2(sp);
                        if constexpr (MMA) {
                            float t[4] = {0.f, 0.f, 0.f, 0.f};
                            const uint32_t a0 = u8x2_to_h2(w.x, 0x4140u), a1 = u8x2_to_h2(w.x, 0x4342u);
                            const uint32_t a2 = u8x2_to_h2(w.y, 0x4140u), a3 = u8x2_to_h2(w.y, 0x4342u);
                            mma16816(t, a0, a1, a2, a3, bh[j][0], bh[j][1]);
                            mma16816(t, a0, a1, a2, a3, bl[j][0], bl[j][1]);
                            const uint32_t a4 = u8x2_to_h2(w.z, 0x4140u), a5 = u8x2_to_h2(w.z, 0x4342u);
                            const uint32_t a6 = u8x2_to_h2(w.w, 0x4140u), a7 = u8x2_to_h2(w.w, 0x4342u);
                            mma16816(t, a4, a5, a6, a7, bh[j][2], bh[j][3]);
                            mma16816(t, a4, a5, a6, a7, bl[j][2], bl[j][3]);
                            acc01[r] = __ffma2_rn(make_float2(dgh.x, dgh.x), __fadd2_rn(make_float2(t[0], t[1]), ncorr[j]), acc01[r]);
                            acc23[r] = __ffma2_rn(make_float2(dgh.y, dgh.y), __fadd2_rn(make_float2(t[2], t[3]), ncorr[j]), acc23[r]);
                        } else {
                            const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
                            float2 wg[4], wh[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                wg[q] = u8x2_to_f32x2(wd[q], 0);
                                wh[q] = u8x2_to_f32x2(wd[q], 2);
                            }
#pragma unroll
                            for (int q = 0; q < NRC; ++q) {
                                float2 sg = __fmul2_rn(wg[0], make_float2(xv[j][q][0], xv[j][q][1]));
                                float2 sh = __fmul2_rn(wh[0], make_float2(xv[j][q][0], xv[j][q][1]));
#pragma unroll
                                for (int u = 1; u < 4; ++u) {
                                    const float2 xp = make_float2(xv[j][q][2 * u], xv[j][q][2 * u + 1]);
                                    sg = __ffma2_rn(wg[u], xp, sg);
                                    sh = __ffma2_rn(wh[u], xp, sh);
                                }
                                accg[r][q] = __ffma2_rn(make_float2(dgh.x, dgh.x), sg, accg[r][q]);
                                acch[r][q] = __ffma2_rn(make_float2(dgh.y, dgh.y), sh, acch[r][q]);
                            }
                        }
                    }
                }
                // the last warp done with this stage refills its slot, possibly with the next
                // phase's weights
                __syncwarp();
                if (lane == 0 && atomicAdd(&s_cnt[st], 1) == kConsumers - 1) {
                    s_cnt[st] = 0;
                    if (gi + S < total) {
                        issue(gi + S);
                        s_issued = gi + S + 1;
                    }
                }
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                if (r >= nb) break;
                float *rw = red + (r * kConsumers + warp) * 128;
                if constexpr (MMA) {
                    *reinterpret_cast<float2 *>(rw + g * 8 + 2 * c) = make_float2(acc01[r].x * us0, acc01[r].y * us1);
                    *reinterpret_cast<float2 *>(rw + (g + 8) * 8 + 2 * c) = make_float2(acc23[r].x * us0, acc23[r].y * us1);
                } else {
#pragma unroll
                    for (int q = 0; q < NRC; ++q) {
                        float vg = accg[r][q].x + accg[r][q].y, vh = acch[r][q].x + acch[r][q].y;
                        vg += __shfl_xor_sync(0xffffffffu, vg, 1);
                        vg += __shfl_xor_sync(0xffffffffu, vg, 2);
                        vh += __shfl_xor_sync(0xffffffffu, vh, 1);
                        vh += __shfl_xor_sync(0xffffffffu, vh, 2);
                        if (c == 0) {
                            rw[g * 8 + q] = vg;
                            rw[(g + 8) * 8 + q] = vh;
                        }
                    }
                }
            }
            if (__syncthreads_or(bad)) {
                bad = true;
                break;
            }
            // this slice's sums, four consecutive outputs of one activation row per thread, added
            // into the phase's outputs
            for (int e = threadIdx.x; e < nb * 32; e += kThreads) {
                const int r = e >> 5, col = (e & 31) >> 2, o4 = (e & 3) * 4;
                if (col >= a.nr) continue;
                const float *rb = red + r * kConsumers * 128 + col;
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int w = 0; w < kConsumers; ++w)
#pragma unroll
                    for (int i2 = 0; i2 < 4; ++i2) s4[i2] += rb[w * 128 + (o4 + i2) * 8];
                const int o = (s_rt0[p] + b0 + r) * 16 + o4;
                atomicAdd(reinterpret_cast<float4 *>(P.y + (int64_t)col * P.y_stride + o),
                          make_float4(s4[0], s4[1], s4[2], s4[3]));
            }
        }
    }
    // a failure: leave no copy in flight (bounded waits on the stages issued last)
    if (__syncthreads_or(bad) && threadIdx.x == 0) {
        dl_status_or(a.status, DL_STATUS_SYNC_TIMEOUT);
        const int hi = s_issued;
        for (int j = max(0, hi - S); j < hi; ++j) dla::mbar_wait(&full[j % S], (uint32_t)((j / S) & 1));
    }
    // the next kernel may only launch now: before this, a later kernel's CTAs could take the slots
    // of CTAs of this grid not yet resident, which the barriers wait for
    dl_pdl_launch_dependents();
}

// ---------------------------------------------------------------- launch

struct GemvCfg {
    bool w16, mma;
    int nrc, kwm, cs, ksl, rpr, stages, grid;
    size_t smem;
};

template <bool W16, bool MMA, int NRC, int KWM>
void *kptr() { return reinterpret_cast<void *>(gemv_q8_kernel<W16, MMA, NRC, KWM>); }

void *pick_kernel(bool w16, bool mma, int nrc, int kwm)
{
    if (w16) {
        // a k-tile is 1 KB: windows of up to 4 k-tiles per warp keep two stages per CTA in reach
        switch (kwm) {
        case 1: return mma ? kptr<true, true, 1, 1>() : nrc == 1 ? kptr<true, false, 1, 1>() : kptr<true, false, 2, 1>();
        case 2: return mma ? kptr<true, true, 1, 2>() : nrc == 1 ? kptr<true, false, 1, 2>() : kptr<true, false, 2, 2>();
        case 4: return mma ? kptr<true, true, 1, 4>() : nrc == 1 ? kptr<true, false, 1, 4>() : kptr<true, false, 2, 4>();
        }
        return nullptr;
    }
    if (mma) {
        switch (kwm) {
        case 1: return kptr<false, true, 1, 1>();
        case 2: return kptr<false, true, 1, 2>();
        case 4: return kptr<false, true, 1, 4>();
        case 6: return kptr<false, true, 1, 6>();
        }
        return nullptr;
    }
    switch (kwm) {
    case 1: return nrc == 1 ? kptr<false, false, 1, 1>() : kptr<false, false, 2, 1>();
    case 2: return nrc == 1 ? kptr<false, false, 1, 2>() : kptr<false, false, 2, 2>();
    case 4: return nrc == 1 ? kptr<false, false, 1, 4>() : kptr<false, false, 2, 4>();
    case 8: return nrc == 1 ? kptr<false, false, 1, 8>() : nullptr;
    }
    return nullptr;
}

// The dynamic shared-memory limit is a per-function attribute shared by every launch of the
// kernel (graph nodes and profilers re-launch against it): set it once to the largest size any
// launch shape may use, never to one launch's own size.
constexpr int kSmemLimit = 200 * 1024;
// Two CTAs share an SM (registers are capped for it): ring bytes aimed at per CTA and the
// largest footprint with which two fit.
constexpr size_t kRingBudget = 64 * 1024;
constexpr size_t kShareLimit = 110 * 1024;

int prepare_kernel(const void *kern, int cs)
{
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8: set shared memory");
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8: shared-memory carveout");
    if (cs > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8: allow a large cluster");
    }
    return DL_OK;
}

// Clusters of `cs` CTAs resident at once with one CTA per SM (asked with a shared-memory
// footprint that no two CTAs can share), cached per device and cluster size.
int clusters_one_per_sm(const void *kern, int cs)
{
    static std::mutex mu;
    static int cache[16][17];
    static bool init = false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!init) {
        for (auto &row : cache)
            for (int &v : row) v = -1;
        init = true;
    }
    if (cache[dev][cs] >= 0) return cache[dev][cs];
    if (prepare_kernel(kern, cs) != DL_OK) return 0;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)cs);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = (size_t)150 * 1024;
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
        clusters = 0;
    }
    cache[dev][cs] = clusters;
    return clusters;
}

// Whether two CTAs of this kernel fit on an SM at the largest shared footprint the launch shapes
// use (registers decide), cached per device and kernel.
bool two_per_sm(const void *kern)
{
    static std::mutex mu;
    static const void *keys[16][32];
    static int vals[16][32];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < 32; ++i) {
        if (keys[dev][i] == kern) return vals[dev][i] >= 2;
        if (!keys[dev][i]) {
            int n = 0;
            if (prepare_kernel(kern, 1) != DL_OK ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, kShareLimit) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
            keys[dev][i] = kern;
            vals[dev][i] = n;
            return n >= 2;
        }
    }
    return false;
}

// Clusters of `csz` CTAs with `smem` bytes each that are resident at once, cached per device.
int max_clusters(const void *kern, int csz, size_t smem)
{
    struct Key { int dev; const void *kern; int csz; size_t smem; int val; };
    static std::mutex mu;
    static Key cache[64];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].dev == dev && cache[i].kern == kern && cache[i].csz == csz && cache[i].smem == smem)
            return cache[i].val;
    int clusters = 0;
    if (prepare_kernel(kern, csz) == DL_OK) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3((unsigned)csz);
        lc.blockDim = dim3(kThreads);
        lc.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)csz;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &lc) != cudaSuccess) {
            cudaGetLastError();
            clusters = 0;
        }
    }
    if (used < 64) cache[used++] = Key{dev, kern, csz, smem, clusters};
    return clusters;
}

// Launch shape.  K is cut into cs slices of ksl = 8 x kwm k-tiles (every warp holds the
// activations of its kwm k-tiles in registers; the last slice may be short); each CTA takes rpr
// consecutive row tiles of one slice and streams them one row tile per ring stage.  Among the
// shapes that run in one wave with two CTAs per SM, the least bytes per CTA wins (near-ties go
// to fewer slices).  Matrices too tall for one wave run in several.
int choose_cfg(bool w16, int nr, int RT, int KT, int sm, int path, GemvCfg *out)
{
    const bool mma = path == PATH_TENSOR || (path == PATH_AUTO && nr > 2);
    if (!mma && nr > 2) return dl::fail(DL_E_SHAPE, "dl_gemv_q8: the CUDA-core path serves 1 or 2 rows per command");
    const int nrc = mma ? 1 : nr;
    const int tb = w16 ? kTileBytesF16 : kTileBytesQ8;
    GemvCfg best{};
    long best_cost = -1;
    for (int kwm : {8, 6, 4, 2, 1}) {                           // fewer slices first
        // Q8_0: a window of six or eight k-tiles per warp when one fits (timed against the byte
        // count below, which prefers narrower windows: 3B step 64.1 -> 60.8 us at 8 rows, 54.0 ->
        // 49.4 at 1 row, 1B 34.3 -> 29.9); narrower windows only when no wider one fits
        if (!w16 && kwm < 6 && best_cost >= 0) break;
        const void *kern = pick_kernel(w16, mma, nrc, kwm);
        if (!kern) continue;
        const int ksl = kConsumers * kwm;
        const int cs = (int)dl::ceil_div(KT, ksl);
        if (cs > 16) continue;
        const size_t sb = (size_t)ksl * tb;
        const int per_sm = two_per_sm(kern) ? 2 : 1;
        if (cs > 1 && clusters_one_per_sm(kern, cs) < 1) continue;
        // footprint for an even spread of the row tiles over per_sm CTAs per SM, then the real
        // number of resident clusters at that footprint
        int stages = (int)(kRingBudget / sb);
        stages = stages < 2 ? 2 : stages > kMaxStages ? kMaxStages : stages;
        int rpr = (int)dl::ceil_div(RT, std::max(1, (per_sm * sm) / cs));
        const size_t limit = per_sm == 2 ? kShareLimit : (size_t)kSmemLimit;
        while (stages > 2 && gemv_smem(ksl, stages, rpr, cs, tb) > limit) --stages;
        size_t smem = gemv_smem(ksl, stages, rpr, cs, tb);
        if (smem > (size_t)kSmemLimit) continue;
        const int nclu = cs == 1 ? per_sm * sm : max_clusters(kern, cs, smem);
        if (nclu < 1) continue;
        rpr = (int)dl::ceil_div(RT, nclu);
        smem = gemv_smem(ksl, stages, rpr, cs, tb);
        if (smem > (size_t)kSmemLimit) continue;
        const int ctas = (int)dl::ceil_div(RT, rpr) * cs;
        const int ctas_per_sm = (int)dl::ceil_div(ctas, sm);
        const long cost = (long)ctas_per_sm * rpr * ksl * 100 + cs;   // bytes per SM, then fewer slices
        if (best_cost < 0 || cost * 100 < best_cost * 95) {
            best_cost = cost;
            best = GemvCfg{w16, mma, nrc, kwm, cs, ksl, rpr, stages, ctas, smem};
        }
    }
    if (best_cost < 0) {
        // no one-wave shape (very many row tiles): CTAs of as many row tiles as shared memory
        // holds, in several waves
        for (int kwm : {8, 6, 4, 2, 1}) {
            if (best_cost >= 0) break;
            if (!pick_kernel(w16, mma, nrc, kwm)) continue;
            const int ksl = kConsumers * kwm;
            const int cs = (int)dl::ceil_div(KT, ksl);
            if (cs > 16) continue;
            const size_t sb = (size_t)ksl * tb;
            int stages = (int)(kRingBudget / sb);
            stages = stages < 2 ? 2 : stages > kMaxStages ? kMaxStages : stages;
            const size_t fixed = gemv_smem(ksl, stages, 0, cs, tb);
            if (fixed >= (size_t)kSmemLimit) continue;
            int rpr = cs > 1 ? (int)(((size_t)kSmemLimit - fixed) / 512) : (int)dl::ceil_div(RT, sm);
            if (rpr < 1) continue;
            if (rpr > RT) rpr = RT;
            best_cost = 0;
            best = GemvCfg{w16, mma, nrc, kwm, cs, ksl, rpr, stages, (int)dl::ceil_div(RT, rpr) * cs,
                           gemv_smem(ksl, stages, rpr, cs, tb)};
        }
        if (best_cost < 0) return dl::fail(DL_E_SHAPE, "dl_gemv_q8: no launch shape for %d k-tiles", KT);
    }
    const void *kern = pick_kernel(best.w16, best.mma, best.nrc, best.kwm);
    const int rc = prepare_kernel(kern, best.cs);
    if (rc != DL_OK) return rc;
    *out = best;
    return DL_OK;
}

int gemv_group(GemvArgs a, bool w16, int nr, int sm, int path, cudaStream_t st)
{
    GemvCfg cfg;
    int rc = choose_cfg(w16, nr, a.RT, a.KT, sm, path, &cfg);
    if (rc != DL_OK) return rc;
    a.nr = nr;
    a.cs = cfg.cs;
    a.ksl = cfg.ksl;
    a.rpr = cfg.rpr;
    a.stages = cfg.stages;
    // one stage per CTA ahead of the activations (measured: more delay the activation fetch that
    // follows the wait, none leaves the SM idle while the previous kernel drains)
    a.pre = 1;
    const void *kern = pick_kernel(cfg.w16, cfg.mma, cfg.nrc, cfg.kwm);
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

// Shared launch path of both weight kinds (the caller has checked the matrix shape).
int gemv_run(const char *name, const void *wq, const void *wd, int64_t n_out, int64_t n_in, bool w16,
             const float *x, int rows, int64_t x_stride, float *y, int64_t y_stride, int path, dl_stream_t stream,
             const DlPrefetch &pf)
{
    if (!x || !y) return dl::fail(DL_E_ARG, "%s: null pointer", name);
    if (rows < 0) return dl::fail(DL_E_ARG, "%s: rows=%d", name, rows);
    if (path < PATH_AUTO || path > PATH_TENSOR) return dl::fail(DL_E_ARG, "%s: path=%d", name, path);
    if (rows == 0) return DL_OK;
    if (x_stride < n_in || y_stride < n_out)
        return dl::fail(DL_E_ARG, "%s: strides %lld/%lld below the row widths", name,
                        (long long)x_stride, (long long)y_stride);
    if (!dl::aligned16(x) || (x_stride % 4) != 0 || !dl::aligned16(wq) || (wd && !dl::aligned16(wd)))
        return dl::fail(DL_E_ALIGN, "%s: x, its stride and the weight planes must be 16-byte aligned", name);
    const char *xb = reinterpret_cast<const char *>(x), *yb = reinterpret_cast<const char *>(y);
    const char *xe = xb + ((size_t)(rows - 1) * x_stride + n_in) * 4;
    const char *ye = yb + ((size_t)(rows - 1) * y_stride + n_out) * 4;
    if (xb < ye && yb < xe) return dl::fail(DL_E_ARG, "%s: y overlaps x", name);
    int sm = 0;
    int rc = dl::device_sm_count(&sm);
    if (rc != DL_OK) return rc;

    GemvArgs a{};
    a.qs = static_cast<const unsigned char *>(wq);
    a.d = static_cast<const unsigned char *>(wd);
    a.x_stride = x_stride;
    a.y_stride = y_stride;
    a.n_out = (int)n_out;
    a.n_in = (int)n_in;
    a.KT = (int)(dl::ceil_div(n_in, 128) * 4);
    a.RT = (int)dl::ceil_div(n_out, 16);

    a.pf = pf;                                 // the first command's launch issues them
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
            rc = gemv_group(a, w16, sizes[gi], sm, path, static_cast<cudaStream_t>(stream));
            if (rc != DL_OK) return rc;
            a.pf.n = 0;
            done += sizes[gi];
        }
    }
    return DL_OK;
}

int gemv_impl(const dl_q8_weight *W, const float *x, int rows, int64_t x_stride, float *y, int64_t y_stride,
              int path, dl_stream_t stream)
{
    dl::clear_error();
    DlPrefetch pf;
    dl::take_prefetch(&pf);
    if (!W || !W->qs || !W->d) return dl::fail(DL_E_ARG, "dl_gemv_q8: null pointer");
    const int rc = dl_q8_packed_size(W->n_out, W->n_in, nullptr, nullptr);
    if (rc != DL_OK) return rc;
    return gemv_run("dl_gemv_q8", W->qs, W->d, W->n_out, W->n_in, false, x, rows, x_stride, y, y_stride, path,
                    stream, pf);
}

int gemv_f16w_impl(const dl_f16_weight *W, const float *x, int rows, int64_t x_stride, float *y,
                   int64_t y_stride, int path, dl_stream_t stream)
{
    dl::clear_error();
    DlPrefetch pf;
    dl::take_prefetch(&pf);
    if (!W || !W->w) return dl::fail(DL_E_ARG, "dl_gemv_f16w: null pointer");
    const int rc = dl_f16w_packed_size(W->n_out, W->n_in, nullptr);
    if (rc != DL_OK) return rc;
    return gemv_run("dl_gemv_f16w", W->w, nullptr, W->n_out, W->n_in, true, x, rows, x_stride, y, y_stride, path,
                    stream, pf);
}

// Chained GEMVs: grid = the CTAs resident at once (the grid barriers need every CTA running).
int gemv_chain_impl(const dl_q8_weight *const *W, const float *const *x, const int64_t *x_stride,
                    float *const *y, const int64_t *y_stride, int nph, int rows, uint32_t *sync,
                    int32_t *status, int path, dl_stream_t stream)
{
    dl::clear_error();
    if (!W || !x || !x_stride || !y || !y_stride || !sync) return dl::fail(DL_E_ARG, "dl_gemv_q8_chain: null pointer");
    if (nph < 1 || nph > kChainMaxPhases) return dl::fail(DL_E_ARG, "dl_gemv_q8_chain: %d phases", nph);
    if (rows < 1 || rows > DL_MAX_ROWS) return dl::fail(DL_E_SHAPE, "dl_gemv_q8_chain: rows=%d (1..%d)", rows, DL_MAX_ROWS);
    if (path < PATH_AUTO || path > PATH_TENSOR) return dl::fail(DL_E_ARG, "dl_gemv_q8_chain: path=%d", path);
    const bool mma = path == PATH_TENSOR || (path == PATH_AUTO && rows > 2);
    if (!mma && rows > 2) return dl::fail(DL_E_SHAPE, "dl_gemv_q8_chain: the CUDA-core path serves 1 or 2 rows");
    if (!dl::aligned16(sync)) return dl::fail(DL_E_ALIGN, "dl_gemv_q8_chain: sync must be 16-byte aligned");
    ChainArgs a{};
    for (int p = 0; p < nph; ++p) {
        const dl_q8_weight *w = W[p];
        if (!w || !w->qs || !w->d || !x[p] || !y[p]) return dl::fail(DL_E_ARG, "dl_gemv_q8_chain: null pointer");
        int rc = dl_q8_packed_size(w->n_out, w->n_in, nullptr, nullptr);
        if (rc != DL_OK) return rc;
        if (w->n_in % 1024 != 0 || w->n_out % 16 != 0)
            return dl::fail(DL_E_SHAPE, "dl_gemv_q8_chain: phase %d is %lld x %lld (n_in a multiple of 1024, n_out of 16)",
                            p, (long long)w->n_out, (long long)w->n_in);
        if (x_stride[p] < w->n_in || y_stride[p] < w->n_out || x_stride[p] % 4 || y_stride[p] % 4)
            return dl::fail(DL_E_ARG, "dl_gemv_q8_chain: phase %d strides", p);
        if (!dl::aligned16(x[p]) || !dl::aligned16(y[p]) || !dl::aligned16(w->qs) || !dl::aligned16(w->d))
            return dl::fail(DL_E_ALIGN, "dl_gemv_q8_chain: phase %d pointers must be 16-byte aligned", p);
        ChainPhase &P = a.ph[p];
        P.qs = static_cast<const unsigned char *>(w->qs);
        P.d = static_cast<const unsigned char *>(w->d);
        P.x = x[p];
        P.y = y[p];
        P.x_stride = x_stride[p];
        P.y_stride = y_stride[p];
        P.n_out = (int)w->n_out;
        P.n_in = (int)w->n_in;
        P.KT = (int)(w->n_in / 32);
        P.RT = (int)(w->n_out / 16);
        P.cs = P.KT / kChainKsl;
    }
    for (int p = 0; p < nph; ++p)
        for (int q = 0; q < nph; ++q) {
            const char *yb = reinterpret_cast<const char *>(a.ph[p].y), *xb = reinterpret_cast<const char *>(a.ph[q].x);
            const char *ye = yb + ((size_t)(rows - 1) * a.ph[p].y_stride + a.ph[p].n_out) * 4;
            const char *xe = xb + ((size_t)(rows - 1) * a.ph[q].x_stride + a.ph[q].n_in) * 4;
            if (q <= p && xb < ye && yb < xe)
                return dl::fail(DL_E_ARG, "dl_gemv_q8_chain: phase %d's output overlaps phase %d's input", p, q);
        }
    int sm = 0;
    int rc = dl::device_sm_count(&sm);
    if (rc != DL_OK) return rc;
    const void *kern = mma ? reinterpret_cast<const void *>(gemv_chain_kernel<true, 1>)
                           : rows == 1 ? reinterpret_cast<const void *>(gemv_chain_kernel<false, 1>)
                                       : reinterpret_cast<const void *>(gemv_chain_kernel<false, 2>);
    const size_t sb = (size_t)kChainKsl * kTileBytesQ8;
    const int stages = std::min(kMaxStages, std::max(2, (int)(kRingBudget / sb)));
    const size_t smem = (size_t)stages * sb + kRedBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8_chain: set shared memory");
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8_chain: shared-memory carveout");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        return dl::fail(DL_E_SHAPE, "dl_gemv_q8_chain: no CTA fits an SM");
    }
    per_sm = std::min(per_sm, 2);
    const int G = per_sm * sm;
    for (int p = 0; p < nph; ++p) {
        ChainPhase &P = a.ph[p];
        if (P.cs > G) return dl::fail(DL_E_SHAPE, "dl_gemv_q8_chain: phase %d needs %d K-slices", p, P.cs);
        const int runs = G / P.cs;
        P.rpr = (int)dl::ceil_div(P.RT, runs);
    }
    a.nph = nph;
    a.nr = rows;
    a.stages = stages;
    a.sync = reinterpret_cast<unsigned *>(sync);
    a.status = status;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)G);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = smem;
    lc.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    void *args[1] = {&a};
    e = cudaLaunchKernelExC(&lc, kern, args);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8_chain: launch");
    return DL_OK;
}

// f16 weights [n_out][n_in] (row-major) to the tile form: one thread per 16 bytes, the half
// `hf` of lane t's 32 bytes = words 4hf .. 4hf + 3; word m holds inputs kb, kb + 1
// (kb = 16(p/2) + 8(p%2) + 2c, p = m/2) of row g + 8(m%2).  Out-of-range weights are zero.
__global__ void f16w_pack_kernel(const uint16_t *w, int64_t n_out, int64_t n_in, int KT, int64_t units, uint4 *out)
{
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= units) return;
    const int hf = (int)(u & 1), lane = (int)((u >> 1) & 31);
    const int64_t t = u >> 6;
    const int64_t kt = t % KT, rt = t / KT;
    const int g = lane >> 2, c = lane & 3;
    uint32_t word[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int m = 4 * hf + e, p = m >> 1;
        const int64_t o = rt * 16 + g + 8 * (m & 1);
        const int64_t k = kt * 32 + 8 * c + 2 * p;
        uint32_t lo = 0u, hi = 0u;
        if (o < n_out && k < n_in) lo = w[o * n_in + k];
        if (o < n_out && k + 1 < n_in) hi = w[o * n_in + k + 1];
        word[e] = lo | (hi << 16);
    }
    out[u] = make_uint4(word[0], word[1], word[2], word[3]);
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

int dl_gemv_q8_chain(const dl_q8_weight *const *W, const float *const *x, const int64_t *x_stride,
                     float *const *y, const int64_t *y_stride, int n_phases, int rows,
                     uint32_t *sync, int32_t *status, int path, dl_stream_t stream)
{
    return gemv_chain_impl(W, x, x_stride, y, y_stride, n_phases, rows, sync, status, path, stream);
}

int dl_f16w_packed_size(int64_t n_out, int64_t n_in, size_t *bytes)
{
    if (n_out <= 0 || n_in <= 0 || n_in % 32 != 0)
        return dl::fail(DL_E_SHAPE, "dl_f16w_packed_size: n_out=%lld n_in=%lld (n_in must be a positive multiple of 32)",
                        (long long)n_out, (long long)n_in);
    if (n_out > (1LL << 30) || n_in > (1LL << 24))
        return dl::fail(DL_E_SHAPE, "dl_f16w_packed_size: matrix too large");
    const int64_t RT = dl::ceil_div(n_out, 16), KT = dl::ceil_div(n_in, 128) * 4;
    if (bytes) *bytes = (size_t)(RT * KT * 1024);
    return DL_OK;
}

int dl_f16w_pack(const uint16_t *w, int64_t n_out, int64_t n_in, void *packed, dl_stream_t stream)
{
    dl::clear_error();
    size_t bytes = 0;
    const int rc = dl_f16w_packed_size(n_out, n_in, &bytes);
    if (rc != DL_OK) return rc;
    if (!w || !packed) return dl::fail(DL_E_ARG, "dl_f16w_pack: null pointer");
    if (!dl::aligned16(packed)) return dl::fail(DL_E_ALIGN, "dl_f16w_pack: the packed plane must be 16-byte aligned");
    const int KT = (int)(dl::ceil_div(n_in, 128) * 4);
    const int64_t units = (int64_t)(bytes / 16);
    f16w_pack_kernel<<<(unsigned)dl::ceil_div(units, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        w, n_out, n_in, KT, units, static_cast<uint4 *>(packed));
    return dl::check_launch("dl_f16w_pack");
}

int dl_gemv_f16w(const dl_f16_weight *W, const float *x, int rows, int64_t x_stride,
                 float *y, int64_t y_stride, dl_stream_t stream)
{
    return gemv_f16w_impl(W, x, rows, x_stride, y, y_stride, PATH_AUTO, stream);
}

int dl_gemv_f16w_ex(const dl_f16_weight *W, const float *x, int rows, int64_t x_stride,
                    float *y, int64_t y_stride, int path, dl_stream_t stream)
{
    return gemv_f16w_impl(W, x, rows, x_stride, y, y_stride, path, stream);
}

}  // extern "C"
