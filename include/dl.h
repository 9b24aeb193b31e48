/*
 * dl.h - C ABI of the GB300 decode-step library (libdl_gb300.so).
 *
 * The library runs the data-parallel hot path of a one-row / N-row transformer
 * decode step over a resident f16 KV cache, one hand-written sm_103a CUDA kernel
 * per call:
 *
 *   dl_gemv_q8        block-quantised (Q8_0) projection GEMV over 1..8 rows per
 *                     command, longer launches tiled by eight rows
 *   dl_rope_kv_store  fused RoPE of q (in place) and k, with the K/V store into
 *                     the f16 mirror
 *   dl_decode_attn    split-KV decode attention with GQA, the split sized by the
 *                     command's rows
 *   dl_attn_merge     log-sum-exp merge of the split pieces
 *   dl_gemv_f16w      the same projection GEMV on f16 weights (the reference lane)
 *   dl_layer_step     the whole layer step of one command as one launch (an option:
 *                     it reads the same bytes and is not yet faster than the calls)
 *
 * plus host-side helpers (weight packing, RoPE tables, the row-grouping and
 * split planner, status words).
 *
 * Conventions shared by every call:
 *  - Every pointer argument documented as "device" is caller-owned device
 *    memory; the library allocates nothing and keeps no global mutable state.
 *  - Every GPU call is asynchronous on the caller's stream (`stream` is a
 *    cudaStream_t; NULL means the legacy default stream) and never synchronises.
 *  - Every call returns an int status: DL_OK or a negative DL_E_* code.  On a
 *    non-OK return nothing was launched and no memory was touched.  The text of
 *    the last failure on the calling thread is available from dl_last_error().
 *  - Conditions only the GPU can see (a position outside the cache, a key
 *    count past what the plan covers) are never trapped: the kernel skips the
 *    offending write and ORs a DL_STATUS_* bit into a caller-provided device
 *    status word, which dl_status_read() (or any device-to-host copy) reports.
 *  - f16 values travel as uint16_t bit patterns (IEEE 754 binary16).
 *
 * Sources (pull-request texts; no formulas are printed there):
 *  [ENC]  daScript PR #4473 "dasLLAMA: the audio towers on the CUDA home, q8 + f16
 *         on every GPU home", commit "cud_router_enc_cols tiles every router
 *         launch": a projection launch holds eight activation columns, longer
 *         launches are tiled, every row equal to the row stepped alone.
 *  [F16W] the same PR #4473, its description: every GPU home serves two weight
 *         lanes, q8 by default and f16 (halfword weights, f32 accumulate) as the
 *         reference lane.
 *  [CLU]  TensorFold PR #926 "drama: the tower's one-row projections ...": a CTA
 *         cluster shares a head, its CTAs exchanging their pieces' results over
 *         distributed shared memory instead of a separate merge pass.
 *  [KV32] daScript PR #4293, "Tests": the rope-and-store template also serves an
 *         f32 mirror (RopeKvStore's f32 stamp) beside the default f16 one.  With
 *         it every stored value is rounded once to f32 (no clamp).  The
 *         attention's tensor form splits the values (and the probabilities)
 *         into bf16 hi + lo pairs, keeping f32's exponent range.
 *  [KVQ8] daScript PR #4293 ("_regions_q8kv" and the block-codec mirror): K and V
 *         kept as Q8_0 blocks of 32 values.  Here: per block the scale d = max|x| / 127
 *         (f32, stored as f16) and codes round(x / d) half away from zero, both decided
 *         in f32; the attention decodes d * code on CUDA cores, or on tensor cores
 *         with the codes as exact f16 operands, each key's block scale applied to
 *         its 32-dimension score sums (f32) and to the V operand (rounded once to
 *         f16).  The rope/store inside the attention launch encodes the new rows
 *         exactly as dl_rope_kv_store does.  Requires capacity % 4 == 0 and the
 *         region stride a multiple of 256 values (16-byte aligned scale rows).
 *  [ROPE] daScript PR #4293 "dasLLAMA llama leg ...", commit "The decode
 *         rope-and-store rides one template on both homes" (GkRopeKvStore).
 *  [GRP]  the same PR, commit "The Vulkan batched step past eight rows runs in
 *         groups, never a row at a time", and the PR body's twelve-stream line.
 *  [SPL]  the same PR, commit "The decode attention's split follows the
 *         command's rows, not the planes' height", and the "Not done" note on
 *         one-row and N-row commands summing keys alike.
 *  [Q8]   the same pages' "q8" lane: Q8_0 blocks of 32 int8 values and one f16
 *         scale.
 */
#ifndef DL_GB300_H
#define DL_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
#define DL_OK            0
#define DL_E_ARG        (-1)  /* null pointer, bad stride, bad count */
#define DL_E_SHAPE      (-2)  /* unsupported head_dim / group / row count / width */
#define DL_E_ALIGN      (-3)  /* a pointer or stride breaks the 16-byte rule */
#define DL_E_WORKSPACE  (-4)  /* caller's workspace smaller than required */
#define DL_E_CUDA       (-5)  /* a CUDA runtime call failed (see dl_last_error) */
#define DL_E_RANGE      (-6)  /* a device status word reports an out-of-range value */

/* bits a kernel ORs into a device status word */
#define DL_STATUS_POS_RANGE     0x1  /* rope/store: pos < 0 or pos >= capacity (row skipped) */
#define DL_STATUS_REGION_RANGE  0x2  /* rope/store: region outside the cache (row skipped) */
#define DL_STATUS_SEQLEN_RANGE  0x4  /* attention: seqlen < 1 or past the plan (keys clipped) */
#define DL_STATUS_SYNC_TIMEOUT  0x8  /* a bounded wait of a persistent launch gave up (outputs invalid) */

#define DL_MAX_ROWS 8          /* rows one command steps at once */

typedef void *dl_stream_t;     /* a cudaStream_t */

/* Text of the calling thread's last failure ("" if none).  Host only. */
const char *dl_last_error(void);

/* Library version as an integer MMmmpp. */
int dl_version(void);

/*
 * Copy a device status word to the host.  Synchronises the device (test and
 * debug use).  Returns DL_OK and stores the word, or DL_E_CUDA.
 */
int dl_status_read(const int32_t *status_dev, int32_t *host_out);

/*
 * L2 prefetch on behalf of a later kernel.  No page defines this: it is a
 * scheduling hint of this library.  The decode step's launches are latency
 * bound, so HBM idles while they run.  The step can use that time to bring the
 * weights or keys of the kernels after them into L2.
 *
 * The next launching call this host thread makes among dl_gemv_q8,
 * dl_gemv_q8_ex, dl_gemv_f16w, dl_gemv_f16w_ex, dl_rope_kv_store, dl_decode_attn,
 * dl_decode_attn_ex, dl_decode_attn_rope, dl_decode_attn_cluster,
 * dl_decode_attn_merged and dl_attn_merge takes the ranges, whether or not it launches.  Its kernel then
 * splits them over its CTAs and issues bulk L2 prefetches for them before
 * waiting on the previous kernel.
 *
 *   n       0..16 ranges (0 clears what is pending)
 *   ptrs    host array of n device pointers, each 16-byte aligned
 *   bytes   host array of n sizes, each a multiple of 16 (0 skips the range)
 *
 * Results do not change.  The ranges must lie inside live device allocations
 * until that kernel ends; the library keeps no reference past it.  A new call
 * replaces what is pending.
 * Errors: DL_E_ARG (n out of range, null arrays), DL_E_ALIGN (a range breaks
 * the 16-byte rule); either leaves nothing pending.  Host only, no CUDA call.
 */
int dl_l2_prefetch_next(int n, const void *const *ptrs, const size_t *bytes);

/* ------------------------------------------------------------ Q8_0 weights
 *
 * Interchange form [Q8]: a row-major [n_out][n_in/32] array of 34-byte blocks,
 * each an f16 scale d (little-endian) followed by 32 int8 values q; weight
 * (o, 32b+i) is d[o][b] * q[o][b][i].
 *
 * Device form (written by dl_q8_pack, read by dl_gemv_q8): two planes.
 *  qs: tiles of 16 output rows x 32 inputs (512 bytes), tile (rt, kt) at byte
 *      ((rt * KT) + kt) * 512 with KT = 4 * ceil(n_in / 128); inside a tile the
 *      16 bytes of lane t = 4g + c are four words, word p holding inputs kb and
 *      kb + 1 (kb = 16*(p/2) + 8*(p%2) + 2c) of row g, then of row g + 8 (the
 *      A-operand order of two 16x8x16 f16 tensor-core products), each weight as
 *      the biased byte q + 128.
 *  d:  per 16 rows and 4 consecutive tiles, 128 bytes: lane group g's 16 bytes
 *      hold (d[g], d[g+8]) for those 4 tiles.
 * Rows past n_out and inputs past n_in hold q = 0 and d = 0.  Both planes must be
 * 16-byte aligned.
 */
typedef struct dl_q8_weight {
    const void *qs;     /* device, packed int8 tiles */
    const void *d;      /* device, packed f16 scales */
    int64_t n_out;      /* output features */
    int64_t n_in;       /* input features, a multiple of 32 */
} dl_q8_weight;

/* Sizes in bytes of the two device planes for an [n_out][n_in] weight.  Host only. */
int dl_q8_packed_size(int64_t n_out, int64_t n_in, size_t *qs_bytes, size_t *d_bytes);

/*
 * Convert interchange blocks (device, n_out * n_in/32 * 34 bytes, any alignment)
 * into the device form (qs, d: device, sizes from dl_q8_packed_size, 16-byte
 * aligned).  One-time preparation, not part of a decode step.
 */
int dl_q8_pack(const uint8_t *blocks, int64_t n_out, int64_t n_in,
               void *qs, void *d, dl_stream_t stream);

/*
 * Q8_0 GEMV [ENC][Q8]:  y[r][o] = sum_b d[o][b] * sum_{i<32} q[o][b][i] * x[r][32b+i]
 * for r < rows, o < n_out.
 *   W        host struct describing the device planes
 *   x        device f32, row r at x + r*x_stride (x_stride >= n_in, in elements)
 *   y        device f32, row r at y + r*y_stride (y_stride >= n_out); must not alias x
 * Rows are stepped eight at a time: the weights are read once per group of up
 * to eight rows, and a row's result does not depend on the rows stepped with it.
 * x and the planes must be 16-byte aligned and x_stride a multiple of 4.
 * Arithmetic: see dl_gemv_q8_ex (path 0).
 */
int dl_gemv_q8(const dl_q8_weight *W, const float *x, int rows, int64_t x_stride,
               float *y, int64_t y_stride, dl_stream_t stream);

/*
 * dl_gemv_q8 with the inner product chosen by the caller (testing and
 * measurement): path 0 = automatic (what dl_gemv_q8 does: CUDA cores for
 * commands of 1 or 2 rows, tensor cores for 3 to 8), 1 = f32 CUDA-core FMAs on
 * the widened weights (commands of 1 or 2 rows only, else DL_E_SHAPE), 2 =
 * 16x8x16 f16 tensor-core products with f32 accumulation on the weights as
 * 1152 + q (exact in f16), each activation row scaled per block of inputs by a
 * power of two and split into two f16 terms (about 22 significant bits), the
 * bias 1152 * sum(x) removed per block.  Same result contract.
 */
int dl_gemv_q8_ex(const dl_q8_weight *W, const float *x, int rows, int64_t x_stride,
                  float *y, int64_t y_stride, int path, dl_stream_t stream);

/*
 * Chained Q8_0 GEMVs in one persistent launch: phase p computes
 * y_p[r] = W_p x_p[r] (as dl_gemv_q8) for r < rows (1..8), the phases in order,
 * each complete before the next starts (x_{p+1} may be y_p).  The weights of a
 * phase stream while the previous one finishes.  Requirements: 1 <= n_phases <= 4,
 * every n_in a multiple of 1024 and every n_out of 16, x/y 16-byte aligned with
 * strides multiples of 4, y_p overlapping no x_q.
 *   sync     device uint32[2], zero before the first call; every successful call
 *            leaves it ready for the next (its own grid barrier's words)
 *   status   device int32 or NULL: DL_STATUS_SYNC_TIMEOUT if a bounded wait gave up
 *   path     as dl_gemv_q8_ex
 * The K-slices of a row tile are added into the outputs (zeroed by the launch), so
 * the summation order, and the last bits of a result, may vary from call to call.
 */
int dl_gemv_q8_chain(const dl_q8_weight *const *W, const float *const *x, const int64_t *x_stride,
                     float *const *y, const int64_t *y_stride, int n_phases, int rows,
                     uint32_t *sync, int32_t *status, int path, dl_stream_t stream);

/* ------------------------------------------------- f16 weights (reference lane)
 *
 * The halfword-weight lane [F16W]: y[r][o] = sum_i w[o][i] * x[r][i] with w in
 * binary16, accumulated in f32.
 *
 * Interchange form: a row-major [n_out][n_in] array of f16 bit patterns.
 * Device form (written by dl_f16w_pack, read by dl_gemv_f16w): tiles of 16 output
 * rows x 32 inputs, 1024 bytes, tile (rt, kt) at byte ((rt * KT) + kt) * 1024 with
 * KT = 4 * ceil(n_in / 128); the 32 bytes of lane t = 4g + c are eight words,
 * word m holding inputs kb and kb + 1 (kb = 16*(p/2) + 8*(p%2) + 2c, p = m/2) of
 * row g + 8*(m%2) (the A operands of two 16x8x16 f16 tensor-core products).
 * Rows past n_out and inputs past n_in hold 0.  The plane must be 16-byte aligned.
 */
typedef struct dl_f16_weight {
    const void *w;      /* device, packed f16 tiles */
    int64_t n_out;      /* output features */
    int64_t n_in;       /* input features, a multiple of 32 */
} dl_f16_weight;

/* Size in bytes of the device plane for an [n_out][n_in] f16 weight.  Host only. */
int dl_f16w_packed_size(int64_t n_out, int64_t n_in, size_t *bytes);

/*
 * Convert an interchange f16 matrix (device, n_out * n_in halves, 2-byte aligned)
 * into the device form (packed: device, dl_f16w_packed_size bytes, 16-byte
 * aligned).  One-time preparation, not part of a decode step.
 */
int dl_f16w_pack(const uint16_t *w, int64_t n_out, int64_t n_in, void *packed, dl_stream_t stream);

/*
 * f16-weight GEMV [F16W]: y[r][o] = sum_i w[o][i] * x[r][i] for r < rows, o < n_out.
 * Arguments, strides, alignment, row grouping and error codes as dl_gemv_q8.
 * Arithmetic: CUDA cores for commands of 1 or 2 rows (the f16 weights widened
 * to f32, f32 FMAs); tensor cores for 3 to 8 (16x8x16 f16 products of the
 * weights as stored with each activation row scaled per warp by a power of two
 * and split into two f16 terms, f32 accumulation).
 */
int dl_gemv_f16w(const dl_f16_weight *W, const float *x, int rows, int64_t x_stride,
                 float *y, int64_t y_stride, dl_stream_t stream);

/* dl_gemv_f16w with the inner product chosen by the caller: path 0 automatic,
 * 1 CUDA cores (1 or 2 rows only, else DL_E_SHAPE), 2 tensor cores. */
int dl_gemv_f16w_ex(const dl_f16_weight *W, const float *x, int rows, int64_t x_stride,
                    float *y, int64_t y_stride, int path, dl_stream_t stream);

/* ---------------------------------------------------------------- KV cache */

/*
 * The f16 KV mirror: K and V planes laid out [region][kv_head][slot][head_dim];
 * element (reg, h, slot, d) of a plane P sits at P[reg*region_stride +
 * (h*capacity + slot)*head_dim + d].  A token at position p lives in slot p.
 * Each session (stream) owns one region.
 */
typedef struct dl_kv_cache {
    void *k;                  /* device K plane: f16 patterns, or f32 values (elem_bytes 4) */
    void *v;                  /* device V plane, same element type */
    int64_t region_stride;    /* elements between regions, >= n_kv*capacity*head_dim */
    int n_regions;
    int n_kv;                 /* KV heads */
    int head_dim;             /* 64 or 128 */
    int capacity;             /* slots per head and region */
    int elem_bytes;           /* 2 (or 0): the f16 mirror; 4: the f32 mirror [KV32];
                                 1: the q8_0 mirror [KVQ8]: k and v hold int8 codes */
    void *k_scale;            /* q8_0 mirror only: device f16 scales of K, one per 32 values: */
    void *v_scale;            /*   scale of value index i (as above) at index i / 32 */
} dl_kv_cache;

/* ------------------------------------------------------------------- RoPE */

/*
 * Rotary embedding table: f32 [max_pos][rot_dim/2][2] holding (cos a, sin a),
 * a = p * theta^(-2j/rot_dim), evaluated in double precision on the host and
 * rounded to f32.  The caller copies it to the device.
 */
typedef struct dl_rope {
    const float *cos_sin;     /* device table from dl_rope_table_build */
    int max_pos;              /* table rows */
    int rot_dim;              /* rotated channels: even, <= head_dim */
    int neox;                 /* 1: pairs (j, j + rot_dim/2); 0: pairs (2j, 2j+1) */
} dl_rope;

/* Bytes of a table (host only). */
int dl_rope_table_bytes(int rot_dim, int max_pos, size_t *bytes);
/* Fill host_out (rot_dim/2 * 2 * max_pos floats) (host only). */
int dl_rope_table_build(double theta, int rot_dim, int max_pos, float *host_out);

/*
 * Fused RoPE and KV store [ROPE], one launch for `rows` token rows:
 *  - the bias rows (optional) are added first: bias = [q bias (n_q*D) | k bias
 *    (n_kv*D) | v bias (n_kv*D)];
 *  - every q head is rotated in place (f32);
 *  - every k head is rotated, clamped into +-65504 and stored as f16 (round to
 *    nearest even) in slot pos[r] of its KV head in region row_region[r];
 *  - every v head is clamped and stored as f16 the same way;
 *  - channels >= rot_dim pass through unrotated.
 * On the f32 mirror [KV32] k and v are rounded once to f32 (no clamp); on the
 * q8_0 mirror [KVQ8] each block of 32 values of k (rotated) and v is encoded
 * as codes and a scale.
 *   q        device f32, row r at q + r*q_stride, n_q heads of head_dim
 *   k, v     device f32, rows at k + r*k_stride / v + r*v_stride, n_kv heads
 *   bias     device f32 or NULL
 *   pos      device int32 [rows]
 *   row_region device int32 [rows] or NULL (all rows in region 0)
 *   status   device int32 status word or NULL; a row whose pos or region is out of
 *            range is skipped and DL_STATUS_POS_RANGE / _REGION_RANGE is set
 * pos must be < rope->max_pos.
 */
int dl_rope_kv_store(float *q, int64_t q_stride,
                     const float *k, int64_t k_stride,
                     const float *v, int64_t v_stride,
                     const float *bias, const int32_t *pos, const int32_t *row_region,
                     int rows, int n_q, const dl_rope *rope, const dl_kv_cache *kv,
                     int32_t *status, dl_stream_t stream);

/* --------------------------------------------------------------- planning */

/*
 * Row grouping [GRP]: n rows run as the fewest groups of at most `max_rows`
 * rows whose sizes differ by at most one, larger groups first (12 -> 6+6,
 * 9 -> 5+4).  Writes the sizes into sizes[] (capacity >= ceil(n/max_rows)) and
 * returns the group count (>= 0) or DL_E_ARG.  Host only.
 */
int dl_plan_groups(int n, int max_rows, int *sizes);

/*
 * Split plan of one attention command (at most DL_MAX_ROWS rows) [SPL].
 * Rows in the same region form a session: one work item serves all of a
 * session's query heads that share a KV head, so each key is read once per
 * session and step.  The keys are cut into pieces of `chunk` keys; the piece
 * count is chosen from the command's own rows and the SM count so that the
 * work items fill the GPU (not from the planes' height).
 */
typedef struct dl_attn_plan {
    int rows;                      /* rows of the command, 1..8 */
    int n_q, n_kv, head_dim;
    int chunk;                     /* keys per piece (a multiple of 32) */
    int max_splits;                /* pieces of the longest row; partial stride */
    int n_sessions;
    int n_work;                    /* work items (CTAs) of dl_decode_attn */
    int sm_count;                  /* SMs the plan was sized for */
    int cluster;                   /* 0: pieces write partials for dl_attn_merge; C > 0: the C pieces
                                      of every (session, KV head) form one thread-block cluster that
                                      merges itself (dl_decode_attn_cluster) */
    int row_region[DL_MAX_ROWS];   /* region of each row */
    int row_keys_max[DL_MAX_ROWS]; /* planned key bound of each row (host seqlen) */
    int sess_rows[DL_MAX_ROWS];    /* rows sorted by session */
    int sess_begin[DL_MAX_ROWS + 1];  /* session s owns sess_rows[sess_begin[s] .. sess_begin[s+1]) */
    int sess_splits[DL_MAX_ROWS];  /* pieces of session s */
    int sess_item0[DL_MAX_ROWS + 1];  /* first work item of session s (items = n_kv * splits) */
    size_t workspace_bytes;        /* bytes of the workspace: partials (o, lse), then the
                                      last-piece merge's counters */
} dl_attn_plan;

/*
 * Build a plan.
 *   seqlen_host   host int32 [rows]: keys each row attends (>= 1); the device
 *                 seqlen passed later must not exceed these
 *   region_host   host int32 [rows] or NULL (all rows region 0)
 *   sm_count      SMs to fill; 0 = query the current device
 *   force_chunk   0 = automatic; otherwise the piece length (rounded up to 32)
 * Host only (plus one device attribute query when sm_count == 0).
 */
int dl_attn_plan_build(int rows, const int32_t *seqlen_host, const int32_t *region_host,
                       int n_q, int n_kv, int head_dim, int sm_count, int force_chunk,
                       dl_attn_plan *out);

/*
 * A plan for dl_decode_attn_cluster [SPL][CLU]: every (session, KV head) gets the
 * same number C <= max_cluster (<= 16; 0 = 16) of pieces, sized like
 * dl_attn_plan_build's (about two work items per SM, the longest session's keys
 * split into C pieces of a multiple of 32 keys); sessions with fewer keys leave
 * their last pieces empty.  No workspace is needed (workspace_bytes = 0).
 * Host only (plus one device attribute query when sm_count == 0).
 */
int dl_attn_plan_build_cluster(int rows, const int32_t *seqlen_host, const int32_t *region_host,
                               int n_q, int n_kv, int head_dim, int sm_count, int max_cluster,
                               dl_attn_plan *out);

/*
 * Split-KV decode attention [SPL].  For row r, query head h (KV head
 * h / (n_q/n_kv)) and piece p covering keys [p*chunk, (p+1)*chunk) of
 * [0, seqlen[r]) of region plan->row_region[r]: scores s_j = q.k_j / sqrt(D),
 * m = max s_j, l = sum exp(s_j - m), o = sum exp(s_j - m) v_j / l, lse = m + ln l.
 *   q          device f32, row r at q + r*q_stride (n_q heads of head_dim)
 *   seqlen     device int32 [rows], 1 <= seqlen[r] <= plan->row_keys_max[r] and
 *              <= kv->capacity; violations clip and set DL_STATUS_SEQLEN_RANGE
 *   workspace  device, >= plan->workspace_bytes, 16-byte aligned: the pieces'
 *              (o, lse), read by dl_attn_merge
 * Pieces past a row's last key are neither computed nor written.
 */
int dl_decode_attn(const float *q, int64_t q_stride, const dl_kv_cache *kv,
                   const int32_t *seqlen, const dl_attn_plan *plan,
                   void *workspace, size_t workspace_bytes,
                   int32_t *status, dl_stream_t stream);

/*
 * dl_decode_attn with the inner product chosen by the caller (testing and
 * measurement): path 0 = automatic (what dl_decode_attn does: CUDA cores when a
 * work item serves at most 4 queries, tensor cores above), 1 = f32 CUDA-core
 * dot products, 2 = 16x8x16 f16 tensor-core products with q split into two f16
 * terms (hi + lo) and probabilities in f16, f32 accumulation and softmax.  On
 * the f32 mirror path 2 takes q, the keys, the probabilities and the values as
 * bf16 hi + lo pairs (three products per pair of operands, f32 accumulation);
 * on the q8_0 mirror the codes are exact f16 operands, each key's block scale
 * multiplies its score sums (f32) and its values (rounded once to f16).
 */
int dl_decode_attn_ex(const float *q, int64_t q_stride, const dl_kv_cache *kv,
                      const int32_t *seqlen, const dl_attn_plan *plan,
                      void *workspace, size_t workspace_bytes,
                      int32_t *status, int path, dl_stream_t stream);

/*
 * Split-KV decode attention with the rope and KV store fused in: one launch does
 * what dl_rope_kv_store followed by dl_decode_attn_ex do, for a command whose
 * rows carry their new token [ROPE][SPL].  The bias (optional, laid out as for
 * dl_rope_kv_store) is added first; every work item rotates its queries in
 * shared memory (q itself is only read, never rotated in place); the work item
 * whose keys hold pos[r] (the last one, for a position past every row's keys)
 * rotates k and stores k and v in slot pos[r] of region plan->row_region[r] as
 * dl_rope_kv_store does for the mirror (f16: clamped into +-65504, round to
 * nearest even; f32: rounded once; q8_0: block-encoded), then reads them back
 * from the mirror after its own stores.  The stored values, the queries and the
 * results equal those of the two separate calls.
 *   q        device f32, row r at q + r*q_stride: n_q heads as projected (unrotated)
 *   k, v     device f32 rows, n_kv heads each; k_stride, v_stride >= n_kv*head_dim
 *   bias     device f32 [(n_q + 2*n_kv) * head_dim] or NULL
 *   pos      device int32 [rows]: the new token's slot; a row whose pos is outside
 *            the cache or the table is not stored and DL_STATUS_POS_RANGE is set
 *   rope     rotary table (16-byte aligned) and pairing (rot_dim even, <= head_dim)
 * The other arguments, the path and the error codes are those of dl_decode_attn_ex.
 */
int dl_decode_attn_rope(const float *q, int64_t q_stride, const float *k, int64_t k_stride,
                        const float *v, int64_t v_stride, const float *bias, const int32_t *pos,
                        const dl_rope *rope, const dl_kv_cache *kv, const int32_t *seqlen,
                        const dl_attn_plan *plan, void *workspace, size_t workspace_bytes,
                        int32_t *status, int path, dl_stream_t stream);

/* The new rows of a command for the attention launches that store them: as dl_decode_attn_rope. */
typedef struct dl_attn_rope_in {
    const float *k;
    int64_t k_stride;
    const float *v;
    int64_t v_stride;
    const float *bias;             /* or NULL */
    const int32_t *pos;            /* device int32 [rows] */
    const dl_rope *rope;           /* table 16-byte aligned */
} dl_attn_rope_in;

/*
 * Split-KV decode attention with the merge inside the launch [SPL][CLU]: the C
 * pieces of a (session, KV head) (plan from dl_attn_plan_build_cluster) run as one
 * thread-block cluster; each keeps its (o, lse) in shared memory, and after a
 * cluster barrier every CTA merges a share of the group's outputs by reading its
 * peers' pieces through distributed shared memory, with the arithmetic of
 * dl_attn_merge (pieces holding none of a row's keys weigh nothing; a row with
 * no keys gets out = 0, lse = -inf).  No partials reach global memory.
 *   rope_in  NULL: q is already rotated and the new rows stored (dl_rope_kv_store);
 *            else the rope and store happen in the launch, as in dl_decode_attn_rope
 *   out      device f32, row r at out + r*out_stride, n_q*head_dim values
 *   lse      device f32 [rows][n_q] or NULL
 * Other arguments, the path and the error codes as dl_decode_attn_ex; a plan
 * without clusters is refused (DL_E_ARG), as is a cluster plan handed to
 * dl_decode_attn / dl_decode_attn_rope.
 */
int dl_decode_attn_cluster(const float *q, int64_t q_stride, const dl_attn_rope_in *rope_in,
                           const dl_kv_cache *kv, const int32_t *seqlen, const dl_attn_plan *plan,
                           float *out, int64_t out_stride, float *lse, int32_t *status, int path,
                           dl_stream_t stream);

/*
 * Split-KV decode attention with the merge done by the last piece [SPL]: every
 * piece writes its (o, lse) to the workspace as dl_decode_attn does, then counts
 * itself in a per-(session, KV head) counter kept in the workspace; the piece
 * that completes the count merges the group's partials into out / lse with the
 * arithmetic of dl_attn_merge, operation for operation (the results are
 * bit-identical to dl_decode_attn_ex + dl_attn_merge), and clears the counter.
 * One launch instead of two; for commands of few queries per KV head (the
 * merge of a group runs in one CTA).
 *   plan       from dl_attn_plan_build; at most 8 queries per work item (rows of
 *              a session x n_q / n_kv), else DL_E_SHAPE
 *   workspace  plan->workspace_bytes, 16-byte aligned; its counters (the last
 *              16-byte-rounded n_sessions * n_kv int32) must be zero before the
 *              first call (zero the whole workspace once); every call leaves
 *              them zero
 *   rope_in, out, lse   as dl_decode_attn_cluster
 * Other arguments, the path and the error codes as dl_decode_attn_ex.
 */
int dl_decode_attn_merged(const float *q, int64_t q_stride, const dl_attn_rope_in *rope_in,
                          const dl_kv_cache *kv, const int32_t *seqlen, const dl_attn_plan *plan,
                          void *workspace, size_t workspace_bytes, float *out, int64_t out_stride,
                          float *lse, int32_t *status, int path, dl_stream_t stream);

/*
 * Log-sum-exp merge of the pieces of every (row, head):
 *   M = max_p lse_p, w_p = exp(lse_p - M), out = sum w_p o_p / sum w_p,
 *   LSE = M + ln sum w_p  (natural log of the scaled scores' exp-sum).
 * Reads only the pieces dl_decode_attn wrote for the same seqlen.
 *   out   device f32, row r at out + r*out_stride, n_q*head_dim values
 *   lse   device f32 [rows][n_q] or NULL
 */
int dl_attn_merge(const void *workspace, const dl_attn_plan *plan, const int32_t *seqlen,
                  float *out, int64_t out_stride, float *lse, dl_stream_t stream);

/* ------------------------------------------------------------- whole layer step
 *
 * One decoder layer's decode step for one command (1..8 rows) in a single
 * launch [ENC][ROPE][SPL][GRP]: the QKV projection, the rope and store of the
 * rows' new k and v into the f16 mirror, split-KV attention over the plan's
 * pieces, their log-sum-exp merge, then the O, gate/up and down projections.
 * Each part has the arithmetic of its separate call (dl_gemv_q8_ex,
 * dl_decode_attn_rope, dl_attn_merge); the projections' K is cut into parts of
 * 1024 inputs whose sums are added (atomically, in the order they arrive) into
 * outputs the launch zeroes first, so a projection's last bits may differ from
 * dl_gemv_q8's and, with three or more parts, from one call to the next; the
 * stored k and v rows follow them within one f16 ulp.
 *
 * The launch holds one CTA per SM for the whole step.  A CTA streams its share
 * of every projection's weights and of the keys ahead of use, and each part
 * waits only for the outputs it reads: the attention for the whole QKV
 * projection, the merge for every piece, O for every merged head, gate/up for
 * the whole O output and down for the whole gate/up output (in a decoder layer
 * a norm reads all of O's output and the SwiGLU all of gate/up's, between
 * them; neither is computed here).
 */
typedef struct dl_layer_weights {
    dl_q8_weight qkv;    /* [(n_q + 2 n_kv) head_dim][hidden]: q, then k, then v rows */
    dl_q8_weight o;      /* [hidden][n_q head_dim] */
    dl_q8_weight gu;     /* [2 ffn][hidden] (gate and up concatenated); qs == NULL: no FFN */
    dl_q8_weight down;   /* [hidden][ffn] (ignored without FFN) */
} dl_layer_weights;

/* Row buffers of a layer step: device f32, row r of a buffer at ptr + r*stride (in elements). */
typedef struct dl_layer_bufs {
    const float *x;      int64_t x_stride;       /* layer input [rows][hidden], read by QKV */
    float *qkv;          int64_t qkv_stride;     /* QKV output (q | k | v), unrotated */
    float *attn;         int64_t attn_stride;    /* merged attention [rows][n_q head_dim]: O's input */
    float *lse;                                  /* [rows][n_q] or NULL */
    float *o;            int64_t o_stride;       /* O output [rows][hidden] */
    const float *x_ffn;  int64_t x_ffn_stride;   /* gate/up input; may be o */
    float *gu;           int64_t gu_stride;      /* gate/up output [rows][2 ffn] */
    const float *x_down; int64_t x_down_stride;  /* down input [rows][ffn]; may point into gu */
    float *down;         int64_t down_stride;    /* down output [rows][hidden] */
} dl_layer_bufs;

/*
 * Bytes of the workspace dl_layer_step needs for these weights and plan: its
 * own counters and the attention pieces' (o, lse).
 * Host only.
 */
int dl_layer_step_workspace_size(const dl_layer_weights *W, const dl_attn_plan *plan, size_t *bytes);

/*
 * The layer step of one command.
 *   W, B      weights (device planes) and row buffers as above; the inputs x,
 *             x_ffn, x_down, the planes and qkv/attn must be 16-byte aligned with
 *             strides a multiple of 4; every output apart from every other, from
 *             its own input and from the workspace
 *   bias, pos, rope, kv, seqlen, plan    as dl_decode_attn_rope; the plan from
 *             dl_attn_plan_build for this command (about one work item per SM
 *             fills the launch: build it with sm_count = SMs / 2), no cluster
 *   workspace device, >= dl_layer_step_workspace_size bytes, 16-byte aligned,
 *             zero before the first call (zero it once); every completed call
 *             leaves its counters zero again
 *   status    device int32 or NULL: the bits of the separate calls, plus
 *             DL_STATUS_SYNC_TIMEOUT if a bounded wait gave up (outputs invalid;
 *             zero the workspace again before the next call)
 *   path      0 automatic (tensor-core projections for 3..8 rows, CUDA cores for
 *             1..2), 1 CUDA-core projections (3..8 rows at head_dim 128 only:
 *             slower, kept to compare the two), 2 tensor cores;
 *             the attention takes tensor cores for work items of more than four
 *             queries, CUDA cores otherwise
 * The f16 mirror only (elem_bytes 0 or 2), head_dim 64 or 128.  The launch holds
 * every SM until it ends and its CTAs wait on one another: never run two of
 * these launches (or one beside other work that fills SMs and waits on it) at
 * the same time; issue a step's commands one after another on one stream.
 */
int dl_layer_step(const dl_layer_weights *W, const dl_layer_bufs *B, const float *bias, const int32_t *pos,
                  const dl_rope *rope, const dl_kv_cache *kv, const int32_t *seqlen, const dl_attn_plan *plan,
                  void *workspace, size_t workspace_bytes, int32_t *status, int path, dl_stream_t stream);

/* ------------------------------------------------------------- no-allocation form
 *
 * (No counterpart on the pages: an addition for callers that cannot allocate
 * device memory, e.g. a host that passes only one step's tensors and owns all
 * other device memory through its own pool, or an engine whose device budget is
 * fixed once serving starts.)
 *
 * dl_decode_attn followed by dl_attn_merge, with the pieces' partials kept in a
 * fixed array inside the library (dl_decode_attention_noalloc_max_bytes() bytes,
 * 8 MiB, held by every GPU that loads the library until the process exits)
 * instead of a caller workspace.  Same arguments and results as those two calls;
 * allocates nothing.
 *  - The first call on a device looks up the array's device address on that
 *    device (current device at the call); make that first call before any
 *    stream capture.
 *  - Every call shares the one array and it keeps the last call's contents.
 *    Nothing in it has to start at zero: a call writes every partial it reads.
 *    Calls whose kernels overlap on the GPU (other streams, other threads) race
 *    on the array; serialise them.
 *  - A plan whose workspace_bytes exceeds the array is refused with
 *    DL_E_WORKSPACE before anything is launched.  A cluster plan
 *    (dl_attn_plan_build_cluster: no partials) is refused with DL_E_ARG; it
 *    goes to dl_decode_attn_cluster, which needs no workspace either.
 *  - The array's device address is asked of the runtime on every call made
 *    outside stream capture; a call under capture uses the address asked last
 *    on that device.  After cudaDeviceReset (a new context, so a new address)
 *    make one call outside capture before capturing another.
 */
size_t dl_decode_attention_noalloc_max_bytes(void);
int dl_decode_attention_noalloc(const float *q, int64_t q_stride, const dl_kv_cache *kv,
                                const int32_t *seqlen, const dl_attn_plan *plan,
                                float *out, int64_t out_stride, float *lse,
                                int32_t *status, dl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DL_GB300_H */
