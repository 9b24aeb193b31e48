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
// Kernel shape: a CTA of 8 warps owns RTC row tiles and one K-slice; the
// slice's activations are staged once in shared memory, the warps split the
// slice's k-tiles, each streaming 16-byte weight loads (L1 bypass) straight into
// registers.  Partial sums are reduced across warps in shared memory and, when
// K is split over several CTAs, across a thread-block cluster through
// distributed shared memory (fixed order: deterministic).
#include <cuda_fp16.h>
#include <cstdio>

#include "dl_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr size_t kXsBudget = 96 * 1024;   // bytes of staged activations per CTA

struct GemvArgs {
    const uint4 *qs;        // packed weight tiles
    const uint32_t *d;      // packed scales as (d[g], d[g+8]) pairs
    const float *x;
    float *y;
    int64_t x_stride, y_stride;
    int n_out, n_in;
    int KT;                 // k-tiles, padded to a multiple of 4
    int RT;                 // row tiles
    int cs;                 // K-slices (= cluster size)
    int ksl;                // k-tiles per slice (multiple of 4)
};

__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// int8 byte `sel` of w (already XOR-ed with 0x80 so it reads as q + 128) to float q:
// the byte becomes the low mantissa bits of 2^23, and 2^23 + 128 is subtracted.
__device__ __forceinline__ float s8_to_f32(uint32_t wx, uint32_t sel)
{
    uint32_t bits = __byte_perm(wx, 0x4B000000u, 0x7540u | sel);
    return __uint_as_float(bits) - 8388736.0f;
}

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

template <int NR, int RTC>
__global__ void __launch_bounds__(kThreads, 2) gemv_q8_cc_kernel(GemvArgs a)
{
    constexpr int U = (8 / RTC) > 0 ? (8 / RTC) : 1;   // k-tiles in flight per step
    extern __shared__ __align__(16) unsigned char smem[];

    const int slice = blockIdx.x % a.cs;
    const int rt0 = (blockIdx.x / a.cs) * RTC;
    const int kt0 = slice * a.ksl;
    const int nkt = min(a.KT, kt0 + a.ksl) - kt0;

    float *xs = reinterpret_cast<float *>(smem);           // [ksl][NR][4 quads][8]
    float *red = xs + (size_t)a.ksl * NR * 32;             // [8 warps][RTC*16*NR]
    float *cpart = red + kWarps * RTC * 16 * NR;           // [RTC*16*NR]

    // ---- stage this slice's activations in lane order
    {
        const int k4n = nkt * 8;                           // float4 per row
        for (int idx = threadIdx.x; idx < NR * k4n; idx += kThreads) {
            const int r = idx / k4n;
            const int k4 = idx - r * k4n;
            const int k = (kt0 * 32) + k4 * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < a.n_in) v = *reinterpret_cast<const float4 *>(a.x + r * a.x_stride + k);
            const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int kk = k4 * 4 + q;            // slice-local input
                const int ktl = kk >> 5, m32 = kk & 31;
                const int h = m32 >> 4, m = m32 & 15;
                const int c = (m & 7) >> 1;
                const int j = h * 4 + ((m >> 3) << 1) + (m & 1);
                xs[((ktl * NR + r) * 4 + c) * 8 + j] = e[q];
            }
        }
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int per = nkt / kWarps, rem = nkt % kWarps;
    const int wk0 = warp * per + min(warp, rem);
    const int wk1 = wk0 + per + (warp < rem ? 1 : 0);

    float acc[RTC][2][NR];
#pragma unroll
    for (int i = 0; i < RTC; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int r = 0; r < NR; ++r) acc[i][h][r] = 0.f;

    const int KG = a.KT >> 2;
    for (int kt = wk0; kt < wk1; kt += U) {
        uint4 wv[U][RTC];
        uint32_t sp[U][RTC];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int i = 0; i < RTC; ++i) {
                const int rt = rt0 + i;
                const int ktg = kt0 + kt + u;
                if (kt + u < wk1 && rt < a.RT) {
                    wv[u][i] = ld_stream(a.qs + ((size_t)rt * a.KT + ktg) * 32 + lane);
                    sp[u][i] = __ldg(a.d + (((size_t)rt * KG + (ktg >> 2)) * 8 + g) * 4 + (ktg & 3));
                } else {
                    wv[u][i] = make_uint4(0u, 0u, 0u, 0u);
                    sp[u][i] = 0u;
                }
            }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (kt + u >= wk1) break;
            const float *xk = xs + ((size_t)(kt + u) * NR * 4 + c) * 8;
#pragma unroll
            for (int i = 0; i < RTC; ++i) {
                const uint32_t w0 = wv[u][i].x ^ 0x80808080u, w1 = wv[u][i].y ^ 0x80808080u;
                const uint32_t w2 = wv[u][i].z ^ 0x80808080u, w3 = wv[u][i].w ^ 0x80808080u;
                // row g: bytes 0,1 of each word; row g+8: bytes 2,3
                float wg[8], wh[8];
                wg[0] = s8_to_f32(w0, 0); wg[1] = s8_to_f32(w0, 1);
                wg[2] = s8_to_f32(w1, 0); wg[3] = s8_to_f32(w1, 1);
                wg[4] = s8_to_f32(w2, 0); wg[5] = s8_to_f32(w2, 1);
                wg[6] = s8_to_f32(w3, 0); wg[7] = s8_to_f32(w3, 1);
                wh[0] = s8_to_f32(w0, 2); wh[1] = s8_to_f32(w0, 3);
                wh[2] = s8_to_f32(w1, 2); wh[3] = s8_to_f32(w1, 3);
                wh[4] = s8_to_f32(w2, 2); wh[5] = s8_to_f32(w2, 3);
                wh[6] = s8_to_f32(w3, 2); wh[7] = s8_to_f32(w3, 3);
                const float dg = __half2float(__ushort_as_half((unsigned short)(sp[u][i] & 0xFFFFu)));
                const float dh = __half2float(__ushort_as_half((unsigned short)(sp[u][i] >> 16)));
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    const float4 xa = *reinterpret_cast<const float4 *>(xk + r * 32);
                    const float4 xb = *reinterpret_cast<const float4 *>(xk + r * 32 + 4);
                    float sg = wg[0] * xa.x;
                    sg = fmaf(wg[1], xa.y, sg); sg = fmaf(wg[2], xa.z, sg); sg = fmaf(wg[3], xa.w, sg);
                    sg = fmaf(wg[4], xb.x, sg); sg = fmaf(wg[5], xb.y, sg);
                    sg = fmaf(wg[6], xb.z, sg); sg = fmaf(wg[7], xb.w, sg);
                    float sh = wh[0] * xa.x;
                    sh = fmaf(wh[1], xa.y, sh); sh = fmaf(wh[2], xa.z, sh); sh = fmaf(wh[3], xa.w, sh);
                    sh = fmaf(wh[4], xb.x, sh); sh = fmaf(wh[5], xb.y, sh);
                    sh = fmaf(wh[6], xb.z, sh); sh = fmaf(wh[7], xb.w, sh);
                    acc[i][0][r] = fmaf(dg, sg, acc[i][0][r]);
                    acc[i][1][r] = fmaf(dh, sh, acc[i][1][r]);
                }
            }
        }
    }

    // ---- reduce the quad (the four lanes holding one row's 32 inputs)
#pragma unroll
    for (int i = 0; i < RTC; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                float v = acc[i][h][r];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                acc[i][h][r] = v;
            }
    if (c == 0) {
#pragma unroll
        for (int i = 0; i < RTC; ++i)
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                red[warp * RTC * 16 * NR + (i * 16 + g) * NR + r] = acc[i][0][r];
                red[warp * RTC * 16 * NR + (i * 16 + g + 8) * NR + r] = acc[i][1][r];
            }
    }
    __syncthreads();

    // ---- reduce the warps (fixed order), then the cluster's K-slices
    constexpr int E = RTC * 16 * NR;
    for (int e = threadIdx.x; e < E; e += kThreads) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[w * E + e];
        if (a.cs == 1) {
            const int i = e / (16 * NR), row = (e / NR) % 16, r = e % NR;
            const int o = (rt0 + i) * 16 + row;
            if (o < a.n_out) a.y[r * a.y_stride + o] = s;
        } else {
            cpart[e] = s;
        }
    }
    if (a.cs > 1) {
        cluster_sync_all();
        for (int e = threadIdx.x; e < E; e += kThreads) {
            if (e % a.cs != slice) continue;
            float s = 0.f;
            for (int q = 0; q < a.cs; ++q) s += ld_dsmem_f32(cpart + e, (uint32_t)q);
            const int i = e / (16 * NR), row = (e / NR) % 16, r = e % NR;
            const int o = (rt0 + i) * 16 + row;
            if (o < a.n_out) a.y[r * a.y_stride + o] = s;
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
    int rtc, cs, ksl;
    size_t smem;
    int grid;
};

size_t gemv_smem(int NR, int rtc, int ksl)
{
    return (size_t)ksl * NR * 32 * 4 + (size_t)kWarps * rtc * 16 * NR * 4 + (size_t)rtc * 16 * NR * 4;
}

GemvCfg gemv_choose(int NR, int RT, int KT, int sm)
{
    GemvCfg best{0, 0, 0, 0, 0};
    const int rtcs[4] = {8, 4, 2, 1};
    for (int ri = 0; ri < 4; ++ri) {
        const int rtc = rtcs[ri];
        if (rtc * NR > 16) continue;
        for (int cs = 1; cs <= 8; ++cs) {
            const int ksl = (int)dl::ceil_div(dl::ceil_div(KT, cs), 4) * 4;
            if ((int)dl::ceil_div(KT, ksl) != cs) continue;          // every slice holds k-tiles
            if ((size_t)NR * ksl * 128 > kXsBudget) continue;
            const int grid = (int)dl::ceil_div(RT, rtc) * cs;
            GemvCfg cfg{rtc, cs, ksl, gemv_smem(NR, rtc, ksl), grid};
            if (grid >= 2 * sm) return cfg;                          // enough CTAs: keep reuse
            if (grid > best.grid) best = cfg;
        }
    }
    return best;
}

template <int NR, int RTC>
int launch_cc(const GemvArgs &a, const GemvCfg &cfg, cudaStream_t st)
{
    auto kern = gemv_q8_cc_kernel<NR, RTC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.smem);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8: set shared memory");
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)cfg.grid);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = cfg.smem;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    lc.attrs = attr;
    lc.numAttrs = 0;
    if (cfg.cs > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cfg.cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        lc.numAttrs = 1;
    }
    e = cudaLaunchKernelEx(&lc, kern, a);
    if (e != cudaSuccess) return dl::cuda_fail(e, "dl_gemv_q8: launch");
    return DL_OK;
}

template <int NR>
int launch_rows(const GemvArgs &a, const GemvCfg &cfg, cudaStream_t st)
{
    switch (cfg.rtc) {
    case 1: return launch_cc<NR, 1>(a, cfg, st);
    case 2: return launch_cc<NR, 2>(a, cfg, st);
    case 4: if constexpr (NR <= 4) return launch_cc<NR, 4>(a, cfg, st); break;
    case 8: if constexpr (NR <= 2) return launch_cc<NR, 8>(a, cfg, st); break;
    }
    return dl::fail(DL_E_SHAPE, "dl_gemv_q8: no kernel for %d rows x %d row tiles", NR, cfg.rtc);
}

int gemv_group(const GemvArgs &a, int nr, int sm, cudaStream_t st)
{
    const GemvCfg cfg = gemv_choose(nr, a.RT, a.KT, sm);
    if (cfg.grid == 0) return dl::fail(DL_E_SHAPE, "dl_gemv_q8: no launch shape for n_in=%d", a.n_in);
    GemvArgs b = a;
    b.cs = cfg.cs;
    b.ksl = cfg.ksl;
    switch (nr) {
    case 1: return launch_rows<1>(b, cfg, st);
    case 2: return launch_rows<2>(b, cfg, st);
    case 3: return launch_rows<3>(b, cfg, st);
    case 4: return launch_rows<4>(b, cfg, st);
    case 5: return launch_rows<5>(b, cfg, st);
    case 6: return launch_rows<6>(b, cfg, st);
    case 7: return launch_rows<7>(b, cfg, st);
    case 8: return launch_rows<8>(b, cfg, st);
    }
    return dl::fail(DL_E_SHAPE, "dl_gemv_q8: bad group size %d", nr);
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
    dl::clear_error();
    if (!W || !x || !y || !W->qs || !W->d) return dl::fail(DL_E_ARG, "dl_gemv_q8: null pointer");
    if (rows < 0) return dl::fail(DL_E_ARG, "dl_gemv_q8: rows=%d", rows);
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
            rc = gemv_group(a, sizes[gi], sm, static_cast<cudaStream_t>(stream));
            if (rc != DL_OK) return rc;
            done += sizes[gi];
        }
    }
    return DL_OK;
}

}  // extern "C"
