/*
 * Decode-step oracle: a plain, slow, double-precision CPU statement of what the
 * one-row / N-row decode step computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg may load this library.  It shares no code, header,
 * table or helper with the CUDA library; the two meet only in the seeded inputs
 * they are both handed.
 *
 * Sources (the pages are pull-request texts; they print no formulas):
 *  - daScript PR #4473 "dasLLAMA: the audio towers on the CUDA home ...", commit
 *    "cud_router_enc_cols tiles every router launch": the projection GEMV serves up
 *    to eight activation columns per launch and longer launches are tiled, each
 *    row's result equal to the row stepped alone.
 *  - daScript PR #4293 "dasLLAMA llama leg ...", commit "The decode rope-and-store
 *    rides one template on both homes" (GkRopeKvStore): bias rows added first, the
 *    q pair roped in place, the k pair roped into the f16 K mirror row, the v pair
 *    copied into the V mirror row, values clamped into the half range, channels past
 *    the rotated width copied through.
 *  - the same PR, commits "The Vulkan batched step past eight rows runs in groups"
 *    (fewest balanced groups of at most eight rows) and "The decode attention's
 *    split follows the command's rows" (keys split into pieces whose partial
 *    results are merged).  The merge is the log-sum-exp combination of softmax
 *    partials; with exact arithmetic any split equals one split.
 *
 * Every function works in double precision with plain loops.  The Q8_0 block is
 * read in its interchange form: 34 bytes per 32 weights, an f16 scale
 * (little-endian) then 32 int8 values.  Caches are f16 planes laid out
 * [region][kv_head][capacity][head_dim].
 *
 * Parity pins (checked by the CPU tests): brute-force dequantise-then-matmul,
 * one-hot and all-ones GEMV cases, rotation norm preservation, position-0
 * identity, rotation composition, full-softmax attention, seqlen-1 and equal-key
 * attention, and split invariance of the merge.  No function here is "parity
 * unpinned".
 *
 * Threads: built with OpenMP, the GEMV runs its (row, output) pairs and the split
 * attention its (row, head) pairs on several threads (orc_set_threads; one by
 * default).  Each result is still computed by one thread in the order above, so
 * the values do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EARG (-1)

/* Threads the parallel loops use from now on (at least 1); returns the number in effect
 * (always 1 without OpenMP). */
int orc_set_threads(int n)
{
#ifdef _OPENMP
    omp_set_num_threads(n < 1 ? 1 : n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ---------------------------------------------------------------- f16 ---- */

/* IEEE 754 binary16 -> double: sign, 5-bit exponent (bias 15), 10-bit fraction. */
double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* double -> binary16, round to nearest, ties to even (overflow -> inf, NaN -> 0x7E00). */
uint16_t orc_double_to_half(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x))
        return 0x7E00;
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7C00);
    int E;
    frexp(a, &E);              /* a in [2^(E-1), 2^E) */
    int u = E - 1;             /* unbiased exponent of a */
    int qexp = (u < -14) ? -24 : u - 10;   /* exponent of one unit in the last place */
    double n = ldexp(a, -qexp);            /* a measured in ulps; exact */
    double fl = floor(n);
    double fr = n - fl;
    double r = fl;
    if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) != 0.0))
        r = fl + 1.0;
    if (u < -14) {
        /* subnormal range; r == 1024 is exactly the smallest normal 0x0400 */
        return (uint16_t)(sign | (uint16_t)r);
    }
    if (r >= 2048.0) {         /* rounding carried into the next binade */
        r = 1024.0;
        u += 1;
    }
    if (u + 15 >= 31)
        return (uint16_t)(sign | 0x7C00);
    return (uint16_t)(sign | ((u + 15) << 10) | ((int)r - 1024));
}

/*
 * Decoded value of every binary16 pattern, filled on first use from
 * orc_half_to_double (a speed-up of the attention and f16-weight loops only; same values).
 */
static double orc_h2d_table[65536];
static int orc_h2d_ready = 0;

static double orc_h2d(uint16_t h)
{
    if (!orc_h2d_ready) {
        for (int i = 0; i < 65536; ++i)
            orc_h2d_table[i] = orc_half_to_double((uint16_t)i);
        orc_h2d_ready = 1;
    }
    return orc_h2d_table[h];
}

/* ---------------------------------------------------------------- Q8_0 --- */

static int orc_s8(uint8_t b)   /* two's complement byte -> int, without relying on char signedness */
{
    return (b & 0x80) ? (int)b - 256 : (int)b;
}

static double orc_block_scale(const uint8_t *blk)
{
    return orc_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
}

/*
 * Q8_0 GEMV, the method's form: y[r][o] = sum_b d[o][b] * sum_i q[o][b][i] * x[r][32b+i].
 * blocks: [n_out][n_in/32] blocks of 34 bytes.  x: rows of n_in floats, row stride x_stride.
 */
int orc_gemv_q8(const uint8_t *blocks, int64_t n_out, int64_t n_in,
                const float *x, int rows, int64_t x_stride,
                double *y, int64_t y_stride)
{
    if (!blocks || !x || !y || n_in % 32 != 0 || rows < 0)
        return ORC_EARG;
    int64_t nb = n_in / 32;
#pragma omp parallel for collapse(2) schedule(static)
    for (int r = 0; r < rows; ++r) {
        for (int64_t o = 0; o < n_out; ++o) {
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *blk = blocks + (o * nb + b) * 34;
                double s = 0.0;
                for (int i = 0; i < 32; ++i)
                    s += (double)orc_s8(blk[2 + i]) * (double)x[r * x_stride + b * 32 + i];
                acc += orc_block_scale(blk) * s;
            }
            y[r * y_stride + o] = acc;
        }
    }
    return ORC_OK;
}

/* Dequantise every weight to double: w[o][i] = d[o][i/32] * q[o][i]. */
int orc_q8_dequant(const uint8_t *blocks, int64_t n_out, int64_t n_in, double *w)
{
    if (!blocks || !w || n_in % 32 != 0)
        return ORC_EARG;
    int64_t nb = n_in / 32;
    for (int64_t o = 0; o < n_out; ++o)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = blocks + (o * nb + b) * 34;
            double d = orc_block_scale(blk);
            for (int i = 0; i < 32; ++i)
                w[o * n_in + b * 32 + i] = d * (double)orc_s8(blk[2 + i]);
        }
    return ORC_OK;
}

/* Plain dense product y[r][o] = sum_i w[o][i] * x[r][i] (the brute-force side of the GEMV pin). */
int orc_matmul(const double *w, int64_t n_out, int64_t n_in,
               const float *x, int rows, int64_t x_stride, double *y, int64_t y_stride)
{
    if (!w || !x || !y)
        return ORC_EARG;
    for (int r = 0; r < rows; ++r)
        for (int64_t o = 0; o < n_out; ++o) {
            double acc = 0.0;
            for (int64_t i = 0; i < n_in; ++i)
                acc += w[o * n_in + i] * (double)x[r * x_stride + i];
            y[r * y_stride + o] = acc;
        }
    return ORC_OK;
}

/*
 * f16-weight GEMV (the halfword-weight "reference lane" of daScript PR #4473, where a
 * lane reads half-precision weights and accumulates in f32): y[r][o] = sum_i w[o][i] * x[r][i]
 * with w the binary16 values of a row-major [n_out][n_in] array, every product and sum in double
 * (the values come from the decode table of orc_half_to_double).
 */
int orc_gemv_f16w(const uint16_t *w, int64_t n_out, int64_t n_in,
                  const float *x, int rows, int64_t x_stride,
                  double *y, int64_t y_stride)
{
    if (!w || !x || !y || n_in <= 0 || rows < 0)
        return ORC_EARG;
    for (int r = 0; r < rows; ++r)
        for (int64_t o = 0; o < n_out; ++o) {
            double acc = 0.0;
            for (int64_t i = 0; i < n_in; ++i)
                acc += orc_h2d(w[o * n_in + i]) * (double)x[r * x_stride + i];
            y[r * y_stride + o] = acc;
        }
    return ORC_OK;
}

void orc_q8_encode_block(const float *x, int8_t *q, uint16_t *d);   /* the q8_0 mirror's encoder, below */

/* ---------------------------------------------------------------- RoPE --- */

/*
 * Rotate one head vector in place at position pos.  Pair j (j < rot/2) turns by
 * angle pos * theta^(-2j/rot).  NeoX pairing couples channels (j, j + rot/2);
 * the interleaved ("NORM") pairing couples (2j, 2j+1).  Channels >= rot pass.
 */
void orc_rope_vec(double *x, int rot_dim, int neox, double theta, double pos)
{
    int half = rot_dim / 2;
    for (int j = 0; j < half; ++j) {
        double inv = pow(theta, -2.0 * (double)j / (double)rot_dim);
        double a = pos * inv;
        double c = cos(a), s = sin(a);
        int i0 = neox ? j : 2 * j;
        int i1 = neox ? j + half : 2 * j + 1;
        double x0 = x[i0], x1 = x[i1];
        x[i0] = x0 * c - x1 * s;
        x[i1] = x0 * s + x1 * c;
    }
}

static double orc_clamp_half(double v)
{
    if (v > 65504.0) return 65504.0;
    if (v < -65504.0) return -65504.0;
    return v;
}

/*
 * Fused rope and KV store for `rows` token rows.
 *   q_in  [rows][n_q*D]  (row stride q_stride)   -> q_out [rows][n_q*D] doubles, roped
 *   k_in  [rows][n_kv*D]                           -> K mirror, roped, clamped, f16
 *   v_in  [rows][n_kv*D]                           -> V mirror, clamped, f16
 *   bias  NULL or [(n_q + 2*n_kv)*D]: q bias, then k bias, then v bias, added first.
 * Row r writes slot pos[r] of region row_region[r] (NULL: region 0) of each KV head:
 *   K[(reg*region_stride) + (h*capacity + pos)*D + d].
 */
static int orc_rope_kv_store_any(const float *q_in, int64_t q_stride,
                                 const float *k_in, int64_t k_stride,
                                 const float *v_in, int64_t v_stride,
                                 const float *bias, const int32_t *pos, const int32_t *row_region, int rows,
                                 int n_q, int n_kv, int head_dim, int rot_dim, int neox, double theta,
                                 double *q_out, int64_t qo_stride,
                                 void *kcache, void *vcache, int elem, int64_t region_stride, int capacity)
{
    if (!q_in || !k_in || !v_in || !pos || !q_out || !kcache || !vcache)
        return ORC_EARG;
    if (rot_dim < 0 || rot_dim > head_dim || rot_dim % 2 != 0)
        return ORC_EARG;
    int D = head_dim;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)D);
    if (!tmp)
        return ORC_EARG;
    for (int r = 0; r < rows; ++r) {
        int p = pos[r];
        int reg = row_region ? row_region[r] : 0;
        if (p < 0 || p >= capacity) {
            free(tmp);
            return ORC_EARG;
        }
        for (int h = 0; h < n_q; ++h) {
            for (int d = 0; d < D; ++d)
                tmp[d] = (double)q_in[r * q_stride + h * D + d] + (bias ? (double)bias[h * D + d] : 0.0);
            orc_rope_vec(tmp, rot_dim, neox, theta, (double)p);
            for (int d = 0; d < D; ++d)
                q_out[r * qo_stride + h * D + d] = tmp[d];
        }
        for (int h = 0; h < n_kv; ++h) {
            int64_t base = (int64_t)reg * region_stride + ((int64_t)h * capacity + p) * D;
            for (int d = 0; d < D; ++d)
                tmp[d] = (double)k_in[r * k_stride + h * D + d] + (bias ? (double)bias[(n_q + h) * D + d] : 0.0);
            orc_rope_vec(tmp, rot_dim, neox, theta, (double)p);
            for (int d = 0; d < D; ++d) {
                if (elem == 4)
                    ((float *)kcache)[base + d] = (float)tmp[d];      /* f32 mirror: round to nearest */
                else
                    ((uint16_t *)kcache)[base + d] = orc_double_to_half(orc_clamp_half(tmp[d]));
            }
            for (int d = 0; d < D; ++d) {
                double v = (double)v_in[r * v_stride + h * D + d] + (bias ? (double)bias[(n_q + n_kv + h) * D + d] : 0.0);
                if (elem == 4)
                    ((float *)vcache)[base + d] = (float)v;
                else
                    ((uint16_t *)vcache)[base + d] = orc_double_to_half(orc_clamp_half(v));
            }
        }
    }
    free(tmp);
    return ORC_OK;
}

/* The rope-and-store into the f16 mirror (clamped into the half range, round to nearest even). */
int orc_rope_kv_store(const float *q_in, int64_t q_stride, const float *k_in, int64_t k_stride,
                      const float *v_in, int64_t v_stride, const float *bias, const int32_t *pos,
                      const int32_t *row_region, int rows, int n_q, int n_kv, int head_dim, int rot_dim,
                      int neox, double theta, double *q_out, int64_t qo_stride,
                      uint16_t *kcache, uint16_t *vcache, int64_t region_stride, int capacity)
{
    return orc_rope_kv_store_any(q_in, q_stride, k_in, k_stride, v_in, v_stride, bias, pos, row_region, rows,
                                 n_q, n_kv, head_dim, rot_dim, neox, theta, q_out, qo_stride, kcache, vcache, 2,
                                 region_stride, capacity);
}

/* The same into the f32 mirror (each value rounded once to f32). */
int orc_rope_kv_store_f32(const float *q_in, int64_t q_stride, const float *k_in, int64_t k_stride,
                          const float *v_in, int64_t v_stride, const float *bias, const int32_t *pos,
                          const int32_t *row_region, int rows, int n_q, int n_kv, int head_dim, int rot_dim,
                          int neox, double theta, double *q_out, int64_t qo_stride,
                          float *kcache, float *vcache, int64_t region_stride, int capacity)
{
    return orc_rope_kv_store_any(q_in, q_stride, k_in, k_stride, v_in, v_stride, bias, pos, row_region, rows,
                                 n_q, n_kv, head_dim, rot_dim, neox, theta, q_out, qo_stride, kcache, vcache, 4,
                                 region_stride, capacity);
}

/*
 * The same into the q8_0 mirror: every stored value is first rounded to f32 (the values the
 * rope produces), then each block of 32 channels of a key row is encoded by orc_q8_encode_block
 * into the code plane (laid out as the f16 mirror) and the scale plane (one per 32 values).
 */
int orc_rope_kv_store_q8(const float *q_in, int64_t q_stride, const float *k_in, int64_t k_stride,
                         const float *v_in, int64_t v_stride, const float *bias, const int32_t *pos,
                         const int32_t *row_region, int rows, int n_q, int n_kv, int head_dim, int rot_dim,
                         int neox, double theta, double *q_out, int64_t qo_stride,
                         int8_t *kq, uint16_t *kd, int8_t *vq, uint16_t *vd, int64_t region_stride, int capacity)
{
    if (!q_in || !k_in || !v_in || !pos || !q_out || !kq || !kd || !vq || !vd)
        return ORC_EARG;
    if (rot_dim < 0 || rot_dim > head_dim || rot_dim % 2 != 0 || head_dim % 32 != 0 || region_stride % 32 != 0)
        return ORC_EARG;
    int D = head_dim;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)D);
    if (!tmp)
        return ORC_EARG;
    float blk[32];
    for (int r = 0; r < rows; ++r) {
        int p = pos[r];
        int reg = row_region ? row_region[r] : 0;
        if (p < 0 || p >= capacity) {
            free(tmp);
            return ORC_EARG;
        }
        for (int h = 0; h < n_q; ++h) {
            for (int d = 0; d < D; ++d)
                tmp[d] = (double)q_in[r * q_stride + h * D + d] + (bias ? (double)bias[h * D + d] : 0.0);
            orc_rope_vec(tmp, rot_dim, neox, theta, (double)p);
            for (int d = 0; d < D; ++d)
                q_out[r * qo_stride + h * D + d] = tmp[d];
        }
        for (int h = 0; h < n_kv; ++h) {
            int64_t base = (int64_t)reg * region_stride + ((int64_t)h * capacity + p) * D;
            for (int d = 0; d < D; ++d)
                tmp[d] = (double)k_in[r * k_stride + h * D + d] + (bias ? (double)bias[(n_q + h) * D + d] : 0.0);
            orc_rope_vec(tmp, rot_dim, neox, theta, (double)p);
            for (int b = 0; b < D / 32; ++b) {
                for (int i = 0; i < 32; ++i) blk[i] = (float)tmp[32 * b + i];
                orc_q8_encode_block(blk, kq + base + 32 * b, kd + (base + 32 * b) / 32);
            }
            for (int b = 0; b < D / 32; ++b) {
                for (int i = 0; i < 32; ++i) {
                    int d = 32 * b + i;
                    blk[i] = (float)((double)v_in[r * v_stride + h * D + d] +
                                     (bias ? (double)bias[(n_q + n_kv + h) * D + d] : 0.0));
                }
                orc_q8_encode_block(blk, vq + base + 32 * b, vd + (base + 32 * b) / 32);
            }
        }
    }
    free(tmp);
    return ORC_OK;
}

/* ----------------------------------------------------------- attention --- */

/* Score of query q (D doubles) against cached key (kv head h, slot j): (q . k_j) / sqrt(D). */
/*
 * A KV plane of either mirror: binary16 patterns (elem = 2, the default f16 mirror) or f32
 * values (elem = 4, the f32 mirror of the same rope-and-store template).
 */

/*
 * The block-codec (q8_0) mirror: a plane of int8 codes shaped like the f16 mirror and a plane
 * of f16 scales, one per 32 consecutive values of a key row (scale index = value index / 32).
 * Value i = scale[i / 32] * code[i].
 */
typedef struct { const int8_t *q; const uint16_t *d; } orc_q8kv;

static double orc_q8kv_get(orc_q8kv p, int64_t i)
{
    return orc_h2d(p.d[i / 32]) * (double)p.q[i];
}

/* Value i of a KV plane: f16 (elem 2), f32 (elem 4) or q8_0 (elem 1, `plane` an orc_q8kv). */
static double orc_kv_get(const void *plane, int elem, int64_t i)
{
    if (elem == 1)
        return orc_q8kv_get(*(const orc_q8kv *)plane, i);
    return elem == 4 ? (double)((const float *)plane)[i] : orc_h2d(((const uint16_t *)plane)[i]);
}

/*
 * Q8_0 encoding of one block of 32 f32 values, decided in f32 (the stored precision of the
 * values): d = max|x| / 127, code = x / d rounded half away from zero and clamped to +-127,
 * the scale stored as f16 (round to nearest even); an all-zero block has d = 0 and codes 0.
 */
void orc_q8_encode_block(const float *x, int8_t *q, uint16_t *d)
{
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d32 = amax / 127.0f;
    for (int i = 0; i < 32; ++i) {
        int c = 0;
        if (d32 > 0.0f) {
            float t = x[i] / d32;
            float r = floorf(fabsf(t) + 0.5f);
            c = (int)(t < 0.0f ? -r : r);
            if (c > 127) c = 127;
            if (c < -127) c = -127;
        }
        q[i] = (int8_t)c;
    }
    *d = orc_double_to_half((double)d32);
}

static double orc_score(const double *q, const void *kc, int elem, int64_t kbase, int D)
{
    double s = 0.0;
    for (int d = 0; d < D; ++d)
        s += q[d] * orc_kv_get(kc, elem, kbase + d);
    return s / sqrt((double)D);
}

/*
 * Split-KV decode attention, the method's form.  Query head h of row r reads KV head
 * h / (n_q/n_kv) of region row_region[r] (NULL: 0), keys 0..seqlen[r]-1.  Keys are cut
 * into pieces [s*chunk, (s+1)*chunk) for s < n_splits; piece s of (r, h) yields
 *   m = max score, l = sum exp(score - m), o = sum exp(score - m) v / l, lse = m + ln l,
 * and an empty piece yields lse = -inf, o = 0.
 *   q        [rows][n_q*D] doubles (row stride q_stride)
 *   part_o   [rows][n_q][n_splits][D]
 *   part_lse [rows][n_q][n_splits]
 */
static int orc_attn_split_any(const double *q, int64_t q_stride, int rows, int n_q, int n_kv, int head_dim,
                   const void *kcache, const void *vcache, int elem, int64_t region_stride, int capacity,
                   const int32_t *row_region, const int32_t *seqlen, int chunk, int n_splits,
                   double *part_o, double *part_lse)
{
    if (!q || !kcache || !vcache || !seqlen || !part_o || !part_lse)
        return ORC_EARG;
    if (n_kv <= 0 || n_q % n_kv != 0 || chunk <= 0 || n_splits <= 0)
        return ORC_EARG;
    int D = head_dim, G = n_q / n_kv;
    for (int r = 0; r < rows; ++r) {
        int L = seqlen[r];
        if (L < 1 || L > capacity || (int64_t)n_splits * chunk < L)
            return ORC_EARG;
    }
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < n_q; ++h) {
            int reg = row_region ? row_region[r] : 0;
            int L = seqlen[r];
            int kvh = h / G;
            int64_t hbase = (int64_t)reg * region_stride + (int64_t)kvh * capacity * D;
            const double *qv = q + r * q_stride + (int64_t)h * D;
            for (int s = 0; s < n_splits; ++s) {
                double *o = part_o + (((int64_t)r * n_q + h) * n_splits + s) * D;
                double *lse = part_lse + ((int64_t)r * n_q + h) * n_splits + s;
                int k0 = s * chunk, k1 = (s + 1) * chunk;
                if (k1 > L) k1 = L;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                if (k0 >= k1) {
                    *lse = -INFINITY;
                    continue;
                }
                double m = -INFINITY;
                for (int j = k0; j < k1; ++j) {
                    double sc = orc_score(qv, kcache, elem, hbase + (int64_t)j * D, D);
                    if (sc > m) m = sc;
                }
                double l = 0.0;
                for (int j = k0; j < k1; ++j) {
                    double w = exp(orc_score(qv, kcache, elem, hbase + (int64_t)j * D, D) - m);
                    l += w;
                    for (int d = 0; d < D; ++d)
                        o[d] += w * orc_kv_get(vcache, elem, hbase + (int64_t)j * D + d);
                }
                for (int d = 0; d < D; ++d) o[d] /= l;
                *lse = m + log(l);
            }
        }
    }
    return ORC_OK;
}

/*
 * Log-sum-exp merge of the pieces of each (row, head):
 *   M = max_s lse_s, w_s = exp(lse_s - M), out = sum w_s o_s / sum w_s, LSE = M + ln sum w_s.
 * Pieces with lse = -inf weigh nothing.
 */
int orc_attn_merge(const double *part_o, const double *part_lse, int rows, int n_q, int n_splits,
                   int head_dim, double *out, int64_t out_stride, double *lse)
{
    if (!part_o || !part_lse || !out || !lse)
        return ORC_EARG;
    int D = head_dim;
    for (int r = 0; r < rows; ++r)
        for (int h = 0; h < n_q; ++h) {
            const double *pl = part_lse + ((int64_t)r * n_q + h) * n_splits;
            double M = -INFINITY;
            for (int s = 0; s < n_splits; ++s)
                if (pl[s] > M) M = pl[s];
            double *ov = out + r * out_stride + (int64_t)h * D;
            for (int d = 0; d < D; ++d) ov[d] = 0.0;
            double W = 0.0;
            for (int s = 0; s < n_splits; ++s) {
                if (pl[s] == -INFINITY) continue;
                double w = exp(pl[s] - M);
                W += w;
                const double *po = part_o + (((int64_t)r * n_q + h) * n_splits + s) * D;
                for (int d = 0; d < D; ++d) ov[d] += w * po[d];
            }
            for (int d = 0; d < D; ++d) ov[d] /= W;
            lse[(int64_t)r * n_q + h] = M + log(W);
        }
    return ORC_OK;
}

/*
 * Brute force: softmax over all seqlen[r] keys at once,
 *   out = sum_j softmax(s)_j v_j,  LSE = ln sum_j exp(s_j).
 * Written without the running maximum of the split form: the scores are first
 * collected, then exponentiated against their exact maximum.
 */
static int orc_attn_full_any(const double *q, int64_t q_stride, int rows, int n_q, int n_kv, int head_dim,
                  const void *kcache, const void *vcache, int elem, int64_t region_stride, int capacity,
                  const int32_t *row_region, const int32_t *seqlen,
                  double *out, int64_t out_stride, double *lse)
{
    if (!q || !kcache || !vcache || !seqlen || !out || !lse)
        return ORC_EARG;
    if (n_kv <= 0 || n_q % n_kv != 0)
        return ORC_EARG;
    int D = head_dim, G = n_q / n_kv;
    for (int r = 0; r < rows; ++r) {
        int reg = row_region ? row_region[r] : 0;
        int L = seqlen[r];
        if (L < 1 || L > capacity)
            return ORC_EARG;
        double *sc = (double *)malloc(sizeof(double) * (size_t)L);
        if (!sc)
            return ORC_EARG;
        for (int h = 0; h < n_q; ++h) {
            int64_t hbase = (int64_t)reg * region_stride + (int64_t)(h / G) * capacity * D;
            const double *qv = q + r * q_stride + (int64_t)h * D;
            double M = -INFINITY;
            for (int j = 0; j < L; ++j) {
                sc[j] = orc_score(qv, kcache, elem, hbase + (int64_t)j * D, D);
                if (sc[j] > M) M = sc[j];
            }
            double Z = 0.0;
            for (int j = 0; j < L; ++j) Z += exp(sc[j] - M);
            for (int j = 0; j < L; ++j) sc[j] = exp(sc[j] - M) / Z;     /* softmax weights */
            double *ov = out + r * out_stride + (int64_t)h * D;
            for (int d = 0; d < D; ++d) ov[d] = 0.0;
            for (int j = 0; j < L; ++j)
                for (int d = 0; d < D; ++d)
                    ov[d] += sc[j] * orc_kv_get(vcache, elem, hbase + (int64_t)j * D + d);
            lse[(int64_t)r * n_q + h] = M + log(Z);
        }
        free(sc);
    }
    return ORC_OK;
}

int orc_attn_split(const double *q, int64_t q_stride, int rows, int n_q, int n_kv, int head_dim,
                   const uint16_t *kcache, const uint16_t *vcache, int64_t region_stride, int capacity,
                   const int32_t *row_region, const int32_t *seqlen, int chunk, int n_splits,
                   double *part_o, double *part_lse)
{
    return orc_attn_split_any(q, q_stride, rows, n_q, n_kv, head_dim, kcache, vcache, 2, region_stride, capacity,
                              row_region, seqlen, chunk, n_splits, part_o, part_lse);
}

int orc_attn_split_f32(const double *q, int64_t q_stride, int rows, int n_q, int n_kv, int head_dim,
                       const float *kcache, const float *vcache, int64_t region_stride, int capacity,
                       const int32_t *row_region, const int32_t *seqlen, int chunk, int n_splits,
                       double *part_o, double *part_lse)
{
    return orc_attn_split_any(q, q_stride, rows, n_q, n_kv, head_dim, kcache, vcache, 4, region_stride, capacity,
                              row_region, seqlen, chunk, n_splits, part_o, part_lse);
}

int orc_attn_full(const double *q, int64_t q_stride, int rows, int n_q, int n_kv, int head_dim,
                  const uint16_t *kcache, const uint16_t *vcache, int64_t region_stride, int capacity,
                  const int32_t *row_region, const int32_t *seqlen, double *out, int64_t out_stride, double *lse)
{
    return orc_attn_full_any(q, q_stride, rows, n_q, n_kv, head_dim, kcache, vcache, 2, region_stride, capacity,
                             row_region, seqlen, out, out_stride, lse);
}

int orc_attn_full_f32(const double *q, int64_t q_stride, int rows, int n_q, int n_kv, int head_dim,
                      const float *kcache, const float *vcache, int64_t region_stride, int capacity,
                      const int32_t *row_region, const int32_t *seqlen, double *out, int64_t out_stride, double *lse)
{
    return orc_attn_full_any(q, q_stride, rows, n_q, n_kv, head_dim, kcache, vcache, 4, region_stride, capacity,
                             row_region, seqlen, out, out_stride, lse);
}

int orc_attn_split_q8(const double *q, int64_t q_stride, int rows, int n_q, int n_kv, int head_dim,
                      const int8_t *kq, const uint16_t *kd, const int8_t *vq, const uint16_t *vd,
                      int64_t region_stride, int capacity, const int32_t *row_region, const int32_t *seqlen,
                      int chunk, int n_splits, double *part_o, double *part_lse)
{
    const orc_q8kv K = {kq, kd}, V = {vq, vd};
    if (!kq || !kd || !vq || !vd)
        return ORC_EARG;
    return orc_attn_split_any(q, q_stride, rows, n_q, n_kv, head_dim, &K, &V, 1, region_stride, capacity,
                              row_region, seqlen, chunk, n_splits, part_o, part_lse);
}

int orc_attn_full_q8(const double *q, int64_t q_stride, int rows, int n_q, int n_kv, int head_dim,
                     const int8_t *kq, const uint16_t *kd, const int8_t *vq, const uint16_t *vd,
                     int64_t region_stride, int capacity, const int32_t *row_region, const int32_t *seqlen,
                     double *out, int64_t out_stride, double *lse)
{
    const orc_q8kv K = {kq, kd}, V = {vq, vd};
    if (!kq || !kd || !vq || !vd)
        return ORC_EARG;
    return orc_attn_full_any(q, q_stride, rows, n_q, n_kv, head_dim, &K, &V, 1, region_stride, capacity,
                             row_region, seqlen, out, out_stride, lse);
}

/* ------------------------------------------------------------- grouping --- */

/*
 * Rows past the command's width run in the fewest balanced groups: g = ceil(n / max_rows)
 * groups whose sizes differ by at most one, the larger groups first.
 */
int orc_plan_groups(int n, int max_rows, int *sizes)
{
    if (n < 0 || max_rows <= 0 || !sizes)
        return ORC_EARG;
    if (n == 0)
        return 0;
    int g = (n + max_rows - 1) / max_rows;
    int base = n / g, rem = n % g;
    for (int i = 0; i < g; ++i)
        sizes[i] = base + (i < rem ? 1 : 0);
    return g;
}
