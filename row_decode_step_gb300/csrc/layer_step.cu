// One decoder layer's decode step as a single persistent launch: the QKV projection, the rope and
// KV store, split-KV attention, the log-sum-exp merge and the O, gate/up and down projections of
// one command (at most eight rows), the same arithmetic as the separate calls (daScript PR #4293:
// the N-row token command reads every weight once per command and sums each row's keys in
// pieces sized by the command's rows; PR #4473: the projection GEMV over at most eight activation
// columns).
//
// Why one launch: every separate launch of the step pays a fixed start (wait for its
// predecessor, fetch its activations, fill its ring) and a drain, and with each kernel filling
// every SM the next one cannot start streaming until the previous one leaves.  Here each SM holds
// one CTA for the whole step:
//  * a producer warp streams, in a fixed order, every byte the CTA will consume over the step
//    (its share of each projection's Q8_0 tiles and of the attention's K/V stages) through a ring
//    of ten 17 KB shared-memory slots (bulk and tensor-map copies, mbarrier-tracked).  Nothing it
//    streams depends on another CTA, so it keeps HBM busy while the consumers wait;
//  * eight consumer warps work the CTA's units phase by phase and wait, with bounded spins, only
//    on the counters of the phase whose outputs they read (data-flow, no grid barrier);
//  * the weights of the first units are requested before waiting on the previous kernel of the
//    stream (programmatic dependent launch), the keys only after it (that kernel may have stored
//    them).
//
// Work of a phase is split evenly over the CTAs in a fixed order:
//  * projections: units of (K-part of 1024 inputs, row tile of 16 outputs); with no more parts
//    than CTAs, each CTA takes a run of one part's row tiles (its activations are prepared once).
//    Each warp multiplies 4 k-tiles of the unit (tensor cores on f16 weights 1152 + q against
//    hi + lo activation terms with f32 accumulation for 3..8 rows, f32 CUDA-core FMAs for 1..2
//    rows or when asked), the CTA sums its warps in warp order every four units; a unit over the
//    whole K stores its row tile, a unit over a K-part adds it (red.add) into outputs zeroed at
//    the start, so with three or more parts the last bits depend on the order the parts arrive;
//  * attention: the plan's work items (session, KV head, piece); the item whose keys hold a
//    row's position rotates and stores that row's k and v before the producer requests the stages
//    that hold them; queries are rotated in shared memory; tensor cores for items of more than
//    four queries, CUDA cores otherwise; the consumer warps' partial softmax states are combined
//    pairwise in shared memory and written as the piece's (o, lse);
//  * merge: one (row, query head) per unit, the pieces' (o, lse) combined as the merge kernel does.
//
// Phase order and what each waits for: QKV -> attention (every QKV row tile) -> merge (every
// piece) -> O (every merged head) -> gate/up (every O row tile: a norm of the O output sits
// between them in a decoder layer) -> down (every gate/up row tile: the SwiGLU of the gate/up
// output).  Norms, SwiGLU and residual adds are not computed here; the gate/up and down inputs are
// caller buffers, which may be the O and gate/up outputs themselves.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <climits>
#include <cmath>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "dl_common.cuh"
#include "dl_async.cuh"

namespace dl {
int make_kv_tmap(CUtensorMap *m, const void *plane, const dl_kv_cache *kv);
}

namespace {

constexpr int kCW = 8;                               // consumer warps
constexpr int kCT = kCW * 32;                        // consumer threads
constexpr int kThreads = kCT + 128;                  // and a producer warpgroup (one thread of it issues)
constexpr int kConsRegs = 232;                       // registers of a consumer thread after the split
constexpr int kProdRegs = 40;                        // registers of a producer thread after the split
static_assert(kCW * 32 * kConsRegs + 128 * kProdRegs <= kThreads * 168,
              "the split draws on the registers the CTA was launched with (168 a thread at 384 threads)");
constexpr int kMaxIt = 8;                            // attention work items per CTA
constexpr int kKWM = 4;                              // k-tiles of a slot per warp
constexpr int kKsl = kCW * kKWM;                     // k-tiles per slot (1024 inputs)
constexpr uint32_t kUnitW = kKsl * 512;              // weight bytes of a whole slot
constexpr uint32_t kSlot = kUnitW + kKsl * 32;       // ring slot: weights + scales (17 KB)
constexpr int kPartSlots = 1;                        // slots of a projection unit at most
constexpr int kPartKT = kPartSlots * kKsl;           // k-tiles of a unit's K part (4096 inputs)
constexpr int kStages = 10;                          // ring slots
constexpr int kRBMax = 8;                            // units per CTA-wide reduction, at most
constexpr int kStKeys = 32;                          // keys per attention stage
constexpr int kMaxQ = 32;                            // queries per work item
constexpr int kCCMaxQ = 4;                           // CUDA-core attention up to this many queries
constexpr int kHalfTile = kStKeys * 128;             // one swizzled box: 32 keys x 128 bytes
constexpr uint32_t kScratch = 48 * 1024;             // per-phase scratch (reduction, activations, queries, combine)
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kSlot + kScratch;
constexpr int kSpinLimit = 1 << 22;                  // dependency polls (about a second) before giving up
static_assert(kSlot % 1024 == 0, "swizzled stage boxes want 1024-byte aligned slots");
static_assert(2 * kStKeys * 128 * 2 <= (int)kSlot, "an attention stage of head_dim 128 fits a slot");

enum { PH_QKV = 0, PH_ATTN, PH_MERGE, PH_O, PH_GU, PH_DOWN, PH_N };
// sync words (uint32) at the head of the workspace; the per-row-tile arrival counts follow
enum { SY_DONE = 0, SY_FINISH = 8, SY_ABORTED = 9, SY_ZEROED = 10, SY_WORDS = 16 };

struct SGemv {
    const unsigned char *qs, *d;       // packed Q8_0 planes
    const float *x;
    float *y;
    int64_t x_stride, y_stride;
    int n_out, n_in, KT, RT, cs;       // KT padded to a multiple of 4, cs = K parts of kPartKT k-tiles
};

struct StepArgs {
    SGemv g[4];                        // QKV, O, gate/up, down
    int n_gemv;                        // 2 (no FFN) or 4
    int nr;                            // rows of the command
    const float *bias;                 // [(n_q + 2 n_kv) D] or null
    const int32_t *pos;
    const float2 *cs;                  // rotary table [max_pos][rot/2]
    int rot, neox, max_pos;
    uint16_t *kc, *vc;                 // the f16 mirror's planes
    int64_t region_stride;
    int capacity;
    const int32_t *seqlen;
    float *part_o, *part_lse;          // the pieces' partials
    float *attn;                       // merged attention output (the O projection's input)
    int64_t attn_stride;
    float *lse;                        // [rows][n_q] or null
    float qscale;                      // log2(e) / sqrt(D)
    dl_attn_plan plan;
    unsigned *sync;
    int32_t *status;
};

// ---------------------------------------------------------------- arithmetic helpers

__device__ __forceinline__ float2 u8x2_to_f32x2(uint32_t w, uint32_t lo)
{
    const float2 b = make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | lo)),
                                 __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541u | lo)));
    return __fadd2_rn(b, make_float2(-8388736.0f, -8388736.0f));
}
__device__ __forceinline__ uint32_t u8x2_to_h2(uint32_t w, uint32_t sel) { return __byte_perm(w, 0x64646464u, sel); }
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ uint32_t h2_bits(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// the same product as plain (non-volatile) assembly: the compiler may interleave independent ones
__device__ __forceinline__ void mma16816p(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    mma16816(c, a[0], a[1], a[2], a[3], b0, b1);
}
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
// 2^x and log2 x through the special-function unit (relative error about 2^-22)
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
__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ unsigned short half_clamped(float v)
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
__device__ __forceinline__ int clip_len(int L, int planned, int capacity, int32_t *status, bool report)
{
    const int hi = min(planned, capacity);
    if (L < 1 || L > hi) {
        if (report) dl_status_or(status, DL_STATUS_SEQLEN_RANGE);
        L = L < 1 ? 0 : hi;
    }
    return L;
}

// ---------------------------------------------------------------- synchronisation helpers

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t *bar, uint32_t cnt)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(dla::smem_u32(bar)), "r"(cnt) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// barrier of the eight consumer warps (a named barrier; the producer warpgroup never takes part)
__device__ __forceinline__ void csync() { dla::named_sync(1, kCT); }
// consumer barrier that returns the OR of `flag` over the consumer threads (the same value in all)
__device__ __forceinline__ bool csync_or(bool flag)
{
    uint32_t r;
    asm volatile("{\n .reg .pred pin, pout;\n setp.ne.u32 pin, %1, 0;\n"
                 " bar.red.or.pred pout, 1, %2, pin;\n selp.u32 %0, 1, 0, pout;\n}"
                 : "=r"(r) : "r"((uint32_t)flag), "r"((uint32_t)kCT) : "memory");
    return r != 0;
}

// Even share [b, e) of n units for CTA c of C.
__device__ __forceinline__ void share(int64_t n, int c, int C, int &b, int &e)
{
    b = (int)(n * c / C);
    e = (int)(n * (c + 1) / C);
}

// This CTA's projection units [b, e) of RT row tiles x cs K-parts (unit u = row tile u % RT of part
// u / RT).  With no more parts than CTAs, the CTAs split into one run per part and each takes an even
// share of its part's row tiles, so that no CTA spans two parts (a part's activations are prepared
// once per CTA); with more parts, an even share of all units.
__device__ __forceinline__ void unit_share(int RT, int cs, int c, int C, int &b, int &e)
{
    if (cs > C) {
        share((int64_t)RT * cs, c, C, b, e);
        return;
    }
    const int s = (int)((int64_t)c * cs / C);                     // this CTA's part
    const int f = (int)(((int64_t)s * C + cs - 1) / cs);          // the part's first CTA
    const int l = (int)(((int64_t)(s + 1) * C + cs - 1) / cs);    // the next part's first CTA
    int rb, re;
    share(RT, c - f, l - f, rb, re);
    b = s * RT + rb;
    e = s * RT + re;
}

// ---------------------------------------------------------------- attention work items

struct Item {
    int s, h, piece, rb, nrows, G, Q, k0, k1, nst, reg, lmin, lmax, own_min;
    unsigned own;                      // rows whose new k/v this item stores
    int row[DL_MAX_ROWS], len[DL_MAX_ROWS], pos[DL_MAX_ROWS];
};

// seq, posr: the rows' key counts and positions (copied to shared memory at the start)
__device__ __forceinline__ void item_meta(const StepArgs &a, const int *seq, const int *posr, int item, Item &m, bool report)
{
    const dl_attn_plan &P = a.plan;
    int s = 0;
    while (s + 1 < P.n_sessions && item >= P.sess_item0[s + 1]) ++s;
    const int local = item - P.sess_item0[s];
    const int splits = P.sess_splits[s];
    m.s = s;
    m.h = local / splits;
    m.piece = local - m.h * splits;
    m.rb = P.sess_begin[s];
    m.nrows = P.sess_begin[s + 1] - m.rb;
    m.G = P.n_q / P.n_kv;
    m.Q = m.nrows * m.G;
    int lmax = 0, lmin = INT_MAX;
    for (int i = 0; i < m.nrows; ++i) {
        const int r = P.sess_rows[m.rb + i];
        m.row[i] = r;
        m.len[i] = clip_len(seq[r], P.row_keys_max[r], a.capacity, a.status, report && m.piece == 0 && m.h == 0);
        m.pos[i] = posr[r];
        lmax = max(lmax, m.len[i]);
        lmin = min(lmin, m.len[i]);
    }
    m.lmax = lmax;
    m.lmin = lmin;
    m.k0 = m.piece * P.chunk;
    m.k1 = min(m.k0 + P.chunk, lmax);
    m.nst = m.k0 >= m.k1 ? 0 : (m.k1 - m.k0 + kStKeys - 1) / kStKeys;
    m.reg = P.row_region[m.row[0]];
    m.own = 0u;
    m.own_min = INT_MAX;
    if (m.nst > 0) {
        // the piece whose keys hold a row's position stores that row (a position past every
        // piece goes to the last one)
        const int owner_last = (lmax - 1) / P.chunk;
        for (int i = 0; i < m.nrows; ++i) {
            const int p = m.pos[i];
            if (min(max(p, 0) / P.chunk, owner_last) != m.piece) continue;
            if (p < 0 || p >= a.capacity || p >= a.max_pos) continue;      // refused: not stored
            m.own |= 1u << i;
            m.own_min = min(m.own_min, p);
        }
    }
}


// ---------------------------------------------------------------- the kernel

template <int D, bool GMMA, int NRC>
__global__ void __launch_bounds__(kThreads, 1)
layer_step_kernel(const __grid_constant__ StepArgs ap, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv)
{
    // the arguments in shared memory: reached through references and run-time indices (the phase's
    // projection, a session's items), parameter-space reads would go the slow generic way and be
    // repeated after every global store the compiler cannot tell apart from them
    __shared__ __align__(16) StepArgs s_a;
    static_assert(sizeof(StepArgs) % 4 == 0, "copied as words");
    for (int i = threadIdx.x; i < (int)(sizeof(StepArgs) / 4); i += blockDim.x)
        reinterpret_cast<int *>(&s_a)[i] = reinterpret_cast<const int *>(&ap)[i];
    __syncthreads();
    const StepArgs &a = s_a;
    constexpr int NKS = D / 16;                  // k-steps of the score product
    constexpr int NDT = D / 8;                   // 8-wide output column tiles
    constexpr int NH = D / 64;                   // boxes per key row
    constexpr uint32_t kVOff = kStKeys * D * 2;  // V within an attention stage
    constexpr int DPL = D / 32;                  // dimensions per lane (CUDA-core attention)
    const dl_attn_plan &P = a.plan;

    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
    __shared__ int s_iss[kStages];               // stages issued into each slot
    __shared__ int s_items_ready;                // this CTA's work items are described (producer waits)
    __shared__ int s_abort;
    __shared__ int s_seq[DL_MAX_ROWS], s_posr[DL_MAX_ROWS];   // the rows' key counts and positions
    // this CTA's attention work items (shared: every consumer thread reads them, and per-thread copies
    // with run-time indices would live in local memory, which the small L1 beside this shared memory
    // cannot hold)
    __shared__ Item s_items[kMaxIt];
    // aligned by an offset into the shared array (not through an integer cast), so that every pointer
    // derived from it stays a shared-memory pointer: the compiler then knows its accesses cannot
    // touch global memory and overlaps them with global loads
    unsigned char *smem = smem_raw + ((1024u - (dla::smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char *ring = smem;
    unsigned char *scr = smem + (size_t)kStages * kSlot;
    const uint32_t ring_s = dla::smem_u32(ring);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int C = gridDim.x, cta = blockIdx.x;
    const int nph = a.n_gemv == 4 ? PH_N : PH_O + 1;
    unsigned *done = a.sync + SY_DONE;

    auto gemv_of = [&](int ph) -> const SGemv & {
        return a.g[ph == PH_QKV ? 0 : ph == PH_O ? 1 : ph == PH_GU ? 2 : 3];
    };
    // the key counts and positions are caller inputs (no kernel of the library writes them): read
    // them before waiting on the previous kernel, all rows at once
    if (tid < a.nr) {
        s_seq[tid] = a.seqlen[tid];
        s_posr[tid] = a.pos[tid];
    }
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            dla::mbar_init(&full[i], 1);
            dla::mbar_init(&empty[i], kCW);          // every consumer warp's share of a release
            s_iss[i] = 0;
        }
        s_abort = 0;
        s_items_ready = 0;
    }
    __syncthreads();

    auto aborted = [&]() -> bool { return *reinterpret_cast<volatile int *>(&s_abort) != 0; };
    auto set_abort = [&]() {
        *reinterpret_cast<volatile int *>(&s_abort) = 1;
        dl_status_or(a.status, DL_STATUS_SYNC_TIMEOUT);
        atomicOr(a.sync + SY_ABORTED, 1u);
    };
    // this CTA's share of the attention work items
    int it_b, it_e;
    share(P.n_work, cta, C, it_b, it_e);
    const int n_it = min(it_e - it_b, kMaxIt);          // the host refuses plans past kMaxIt per CTA
    // a reader warp is done with stage sq (lane 0, after __syncwarp): its share of the slot's release
    auto release = [&](uint32_t sq, uint32_t cnt) { mbar_arrive_cnt(&empty[sq % kStages], cnt); };

    if (warp >= kCW) {
        // ============================================================ producer warpgroup
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kProdRegs));
        if (warp == kCW && lane == 0) {
            // the whole sequence in order, each stage once its slot's previous fill is released:
            // weights first without waiting on the previous kernel, keys only after it (it may have
            // stored some)
            bool pdl = false, ok = true;
            int k = 0;                                         // stage index in the sequence
            // the slot of stage k is free: its previous fill released by its readers (bounded wait)
            auto slot_free = [&]() -> bool {
                if (k < kStages) return true;
                const uint32_t par = (uint32_t)(((k / kStages) - 1) & 1);
                for (int it = 0; it < (1 << 16); ++it) {
                    if (dla::mbar_try_wait_sleep(&empty[k % kStages], par, 20000u)) return true;
                    if (aborted()) return false;
                }
                return false;
            };
            auto wait_pdl = [&]() {
                if (pdl) return;
                dl_pdl_wait();
                pdl = true;
                dla::prefetch_tmap(&tk);
                dla::prefetch_tmap(&tv);
            };
            for (int ph = 0; ph < nph && ok; ++ph) {
                if (ph == PH_MERGE) continue;
                if (ph == PH_ATTN) {
                    wait_pdl();
                    for (int it = 0; it < (1 << 22) && !*reinterpret_cast<volatile int *>(&s_items_ready); ++it) {
                        if (aborted()) break;
                        __nanosleep(64);
                    }
                    if (!*reinterpret_cast<volatile int *>(&s_items_ready)) {
                        ok = false;
                        break;
                    }
                    for (int j = 0; j < n_it && ok; ++j) {
                        const Item &m = s_items[j];
                        for (int i = 0; i < m.nst; ++i, ++k) {
                            if (aborted() || !slot_free()) {
                                ok = false;
                                break;
                            }
                            const int sl = k % kStages;
                            unsigned char *dst = ring + (size_t)sl * kSlot;
                            const int y = m.h * a.capacity + m.k0 + i * kStKeys;
                            *reinterpret_cast<volatile int *>(&s_iss[sl]) = s_iss[sl] + 1;
                            dla::mbar_expect_tx(&full[sl], 2 * kVOff);
#pragma unroll
                            for (int hf = 0; hf < NH; ++hf) {
                                dla::tma_g2s_3d(dst + hf * kHalfTile, &tk, hf * 64, y, m.reg, &full[sl]);
                                dla::tma_g2s_3d(dst + kVOff + hf * kHalfTile, &tv, hf * 64, y, m.reg, &full[sl]);
                            }
                        }
                    }
                    continue;
                }
                const SGemv &G = gemv_of(ph);
                int ub, ue;
                unit_share(G.RT, G.cs, cta, C, ub, ue);
                int s = ub / G.RT, rt = ub - s * G.RT;
                for (int u = ub; u < ue && ok; ++u) {
                    // unit u: row tile rt over K part s, one slot per kKsl k-tiles
                    const int pt0 = s * kPartKT, pnkt = min(kPartKT, G.KT - pt0);
                    for (int j = 0; j * kKsl < pnkt; ++j, ++k) {
                        if (k >= kStages) wait_pdl();
                        if (aborted() || !slot_free()) {
                            ok = false;
                            break;
                        }
                        const int kt0 = pt0 + j * kKsl, nkt = min(kKsl, pnkt - j * kKsl);
                        const int sl = k % kStages;
                        unsigned char *dst = ring + (size_t)sl * kSlot;
                        *reinterpret_cast<volatile int *>(&s_iss[sl]) = s_iss[sl] + 1;
                        dla::mbar_expect_tx(&full[sl], (uint32_t)nkt * 544u);
                        dla::bulk_g2s(dst, G.qs + ((size_t)rt * G.KT + kt0) * 512, (uint32_t)nkt * 512u, &full[sl]);
                        dla::bulk_g2s(dst + kUnitW, G.d + ((size_t)rt * (G.KT >> 2) + (kt0 >> 2)) * 128,
                                      (uint32_t)nkt * 32u, &full[sl]);
                    }
                    if (++rt == G.RT) {
                        rt = 0;
                        ++s;
                    }
                }
            }
            wait_pdl();
        } else if (warp == kCW + 1) {
            // outputs of projections whose K comes in parts start at zero (the parts are added into
            // them): every CTA zeroes a share, after the previous kernel (it may read them), and
            // counts itself in; a projection's first additions wait for every CTA's count
            dl_pdl_wait();
            bool any_parts = false;
            for (int p = 0; p < a.n_gemv; ++p) {
                const SGemv &G = a.g[p];
                if (G.cs == 1) continue;
                any_parts = true;
                const int64_t n = (int64_t)a.nr * G.n_out;
                int zb, ze;
                share(n, cta, C, zb, ze);
                for (int64_t e = zb + lane; e < ze; e += 32) {
                    const int r = (int)(e / G.n_out), o = (int)(e - (int64_t)r * G.n_out);
                    G.y[(int64_t)r * G.y_stride + o] = 0.f;
                }
            }
            __syncwarp();
            if (any_parts && lane == 0) {
                __threadfence();
                atomicAdd(a.sync + SY_ZEROED, 1u);
            }
        } else if (warp == kCW + 2) {
            // this CTA's work items (the key counts and positions are caller inputs), one lane each
            for (int j = lane; j < n_it; j += 32) item_meta(a, s_seq, s_posr, it_b + j, s_items[j], true);
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                *reinterpret_cast<volatile int *>(&s_items_ready) = 1;
            }
        }
    } else {
        // ============================================================ consumers
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kConsRegs));
        // the work items and the zeroing of the K-part outputs are done by the producer warpgroup's
        // spare warps, off this path
        dl_pdl_wait();
        bool zeroed = true;
        for (int p = 0; p < a.n_gemv; ++p) zeroed = zeroed && a.g[p].cs == 1;
        const int ctid = tid;
        uint32_t seq = 0;
        bool bad = false;

        // wait until done[ph] reaches `target`: one thread polls, every consumer gets its verdict
        // through the barrier (a uniform result, so that all warps take the same barriers after it)
        auto dep_wait = [&](int ph, unsigned target) -> bool {
            bool fail = false;
            if (ctid == 0) {
                bool ok = false;
                for (int it = 0; it < kSpinLimit; ++it) {
                    if (ld_acquire(done + ph) >= target) {
                        ok = true;
                        break;
                    }
                    if (aborted()) break;
                    __nanosleep(it < 64 ? 32 : 256);
                }
                __threadfence();
                if (!ok) set_abort();
                fail = !ok;
            }
            return !csync_or(fail);
        };
        // the same wait on any word of the sync block
        auto dep_wait_word = [&](int word, unsigned target) -> bool {
            bool fail = false;
            if (ctid == 0) {
                bool ok = false;
                for (int it = 0; it < kSpinLimit; ++it) {
                    if (ld_acquire(a.sync + word) >= target) {
                        ok = true;
                        break;
                    }
                    if (aborted()) break;
                    __nanosleep(it < 64 ? 32 : 256);
                }
                __threadfence();
                if (!ok) set_abort();
                fail = !ok;
            }
            return !csync_or(fail);
        };
        // count `n` finished units of phase ph: after the barrier, one thread's fence orders every
        // thread's writes of them (fences are cumulative) before the count
        auto signal = [&](int ph, unsigned n) {
            csync();
            if (ctid == 0 && n) {
                __threadfence();
                atomicAdd(done + ph, n);
            }
        };
        // wait for projection unit sq to land (every lane of the warp): every consumer warp reads every
        // unit, so a warp reaches a slot's fill only after it consumed the fill before it
        auto unit_wait = [&](uint32_t sq) -> bool {
            const bool ok = __all_sync(0xffffffffu, dla::mbar_wait(&full[sq % kStages], (sq / kStages) & 1));
            if (!ok && lane == 0) set_abort();
            return ok;
        };
        // wait for attention stage sq to land.  Warps of different stage groups move through the ring
        // at their own pace, so first wait until the stage has been requested into its slot: its
        // slot's previous fill is then consumed, and the parity wait cannot mistake the fill two back
        // (same parity) for this one
        auto stage_wait = [&](uint32_t sq) -> bool {
            const int sl = sq % kStages, fill = sq / kStages;
            bool ok = true;
            if (lane == 0) {
                for (int it = 0; *reinterpret_cast<volatile int *>(&s_iss[sl]) <= fill; ++it) {
                    if (it > kSpinLimit || aborted()) {
                        ok = false;
                        break;
                    }
                    __nanosleep(32);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0) && __all_sync(0xffffffffu, dla::mbar_wait(&full[sl], fill & 1));
            if (!ok && lane == 0) set_abort();
            return ok;
        };

        for (int ph = 0; ph < nph && !bad; ++ph) {
            if (ph == PH_ATTN) {
                // ================================================= attention
                // the work items described by the spare warp (long since, but bounded); the verdict
                // reaches every consumer through the dependency wait's barrier
                bool items_ok = true;
                if (ctid == 0) {
                    for (int it = 0; !*reinterpret_cast<volatile int *>(&s_items_ready); ++it) {
                        if (it > kSpinLimit || aborted()) {
                            items_ok = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                    __threadfence_block();
                    if (!items_ok) set_abort();
                }
                if (!dep_wait(PH_QKV, (unsigned)(a.g[0].RT * a.g[0].cs)) || !items_ok) {
                    bad = true;
                    break;
                }
                const SGemv &QG = a.g[0];
                const int G = P.n_q / P.n_kv;
                const int ms = P.max_splits;
                const int ib = it_b, ie = it_b + n_it;
                unsigned char *qfrag = scr;                                   // [2][NKS][hi, lo][32] x 16 B
                float *qraw = reinterpret_cast<float *>(scr + 2 * NKS * 1024);   // [kMaxQ][D]
                float *cb = reinterpret_cast<float *>(scr);                   // combine slots (after the stages)
                uint16_t *stash = reinterpret_cast<uint16_t *>(scr + 32 * 1024);  // [row][k, v][D] stored halves
                for (int it = ib; it < ie && !bad; ++it) {
                    const Item &m = s_items[it - ib];
                    if (m.nst == 0) {
                        signal(PH_ATTN, 1u);
                        continue;
                    }
                    const int Q = m.Q;
                    // queries of this KV head (bias first, then the rotation), from the QKV output: every
                    // load of a thread's share issued first, then the rotations (PQ pairs a thread at most)
                    {
                        constexpr int PQ = (kMaxQ * (D / 2) + kCT - 1) / kCT;
                        float x0[PQ], x1[PQ];
                        float2 cs[PQ];
                        bool rt[PQ];
#pragma unroll
                        for (int t = 0; t < PQ; ++t) {
                            const int e = ctid + t * kCT;
                            x0[t] = x1[t] = 0.f;
                            cs[t] = make_float2(1.f, 0.f);
                            rt[t] = false;
                            if (e < Q * (D / 2)) {
                                const int qi = e / (D / 2), jp = e - qi * (D / 2);
                                const int ri = qi / G, head = m.h * G + (qi - ri * G);
                                const int p = m.pos[ri];
                                int i0, i1;
                                const bool rotate = rope_pair(jp, a.rot, a.neox, i0, i1);
                                const float *qv = QG.y + (int64_t)m.row[ri] * QG.y_stride + (int64_t)head * D;
                                x0[t] = __ldcg(qv + i0);
                                x1[t] = __ldcg(qv + i1);
                                rt[t] = rotate && p >= 0 && p < a.max_pos;
                                if (rt[t]) cs[t] = a.cs[(size_t)p * (a.rot >> 1) + jp];
                            }
                        }
#pragma unroll
                        for (int t = 0; t < PQ; ++t) {
                            const int e = ctid + t * kCT;
                            if (e < Q * (D / 2)) {
                                const int qi = e / (D / 2), jp = e - qi * (D / 2);
                                const int head = m.h * G + (qi - (qi / G) * G);
                                int i0, i1;
                                rope_pair(jp, a.rot, a.neox, i0, i1);
                                float v0 = x0[t], v1 = x1[t];
                                if (a.bias) {
                                    v0 += a.bias[(int64_t)head * D + i0];
                                    v1 += a.bias[(int64_t)head * D + i1];
                                }
                                qraw[qi * D + i0] = rt[t] ? fmaf(v0, cs[t].x, -v1 * cs[t].y) : v0;
                                qraw[qi * D + i1] = rt[t] ? fmaf(v0, cs[t].y, v1 * cs[t].x) : v1;
                            }
                        }
                    }
                    // the rows this piece stores: k rotated, k and v clamped into the half range (PS pairs
                    // a thread at most, loads first)
                    if (m.own) {
                        constexpr int PS = (DL_MAX_ROWS * (D / 2) + kCT - 1) / kCT;
                        float k0v[PS], k1v[PS], v0v[PS], v1v[PS];
                        float2 cs[PS];
                        bool rt[PS];
#pragma unroll
                        for (int t = 0; t < PS; ++t) {
                            const int e = ctid + t * kCT;
                            const int i = e / (D / 2), jp = e - i * (D / 2);
                            k0v[t] = k1v[t] = v0v[t] = v1v[t] = 0.f;
                            cs[t] = make_float2(1.f, 0.f);
                            rt[t] = false;
                            if (i < m.nrows && ((m.own >> i) & 1u)) {
                                const int p = m.pos[i], r = m.row[i];
                                const float *kr = QG.y + (int64_t)r * QG.y_stride + (int64_t)(P.n_q + m.h) * D;
                                const float *vr = QG.y + (int64_t)r * QG.y_stride + (int64_t)(P.n_q + P.n_kv + m.h) * D;
                                int i0, i1;
                                const bool rotate = rope_pair(jp, a.rot, a.neox, i0, i1);
                                k0v[t] = __ldcg(kr + i0);
                                k1v[t] = __ldcg(kr + i1);
                                v0v[t] = __ldcg(vr + i0);
                                v1v[t] = __ldcg(vr + i1);
                                rt[t] = rotate;
                                if (rotate) cs[t] = a.cs[(size_t)p * (a.rot >> 1) + jp];
                            }
                        }
#pragma unroll
                        for (int t = 0; t < PS; ++t) {
                            const int e = ctid + t * kCT;
                            const int i = e / (D / 2), jp = e - i * (D / 2);
                            if (i < m.nrows && ((m.own >> i) & 1u)) {
                                const int p = m.pos[i];
                                int i0, i1;
                                rope_pair(jp, a.rot, a.neox, i0, i1);
                                float k0 = k0v[t], k1 = k1v[t], v0 = v0v[t], v1 = v1v[t];
                                if (a.bias) {
                                    const float *bk = a.bias + (int64_t)(P.n_q + m.h) * D;
                                    const float *bv = a.bias + (int64_t)(P.n_q + P.n_kv + m.h) * D;
                                    k0 += bk[i0];
                                    k1 += bk[i1];
                                    v0 += bv[i0];
                                    v1 += bv[i1];
                                }
                                const float y0 = rt[t] ? fmaf(k0, cs[t].x, -k1 * cs[t].y) : k0;
                                const float y1 = rt[t] ? fmaf(k0, cs[t].y, k1 * cs[t].x) : k1;
                                const int64_t base = (int64_t)m.reg * a.region_stride + ((int64_t)m.h * a.capacity + p) * D;
                                const unsigned short hk0 = half_clamped(y0), hk1 = half_clamped(y1);
                                const unsigned short hv0 = half_clamped(v0), hv1 = half_clamped(v1);
                                a.kc[base + i0] = hk0;
                                a.kc[base + i1] = hk1;
                                a.vc[base + i0] = hv0;
                                a.vc[base + i1] = hv1;
                                stash[(i * 2) * D + i0] = hk0;
                                stash[(i * 2) * D + i1] = hk1;
                                stash[(i * 2 + 1) * D + i0] = hv0;
                                stash[(i * 2 + 1) * D + i1] = hv1;
                            }
                        }
                    }
                    // rows whose position lies outside the cache or the table are not stored
                    if (ctid == 0 && m.piece == 0 && m.h == 0)
                        for (int i = 0; i < m.nrows; ++i)
                            if (m.pos[i] < 0 || m.pos[i] >= a.capacity || m.pos[i] >= a.max_pos)
                                dl_status_or(a.status, DL_STATUS_POS_RANGE);
                    csync();                                         // queries and stash in place
                    const int k0 = m.k0, k1 = m.k1, nst = m.nst;
                    // keys past the piece may hold anything (even NaN) in the V rows: zero them
                    auto zero_tail = [&](int sl, int kb0) {
                        unsigned char *vrow = ring + (size_t)sl * kSlot + kVOff;
                        for (int e = lane; e < NH * kStKeys * 8; e += 32) {
                            const int hf = e / (kStKeys * 8), rem = e - hf * kStKeys * 8;
                            if (kb0 + (rem >> 3) >= k1)
                                *reinterpret_cast<uint4 *>(vrow + hf * kHalfTile + rem * 16) = make_uint4(0u, 0u, 0u, 0u);
                        }
                        dla::fence_proxy_async();
                        __syncwarp();
                    };
                    // the rows this piece stored, from the stash into the stage (the copies may have
                    // read the slots before the stores): the same bits a read of the mirror gives
                    auto patch = [&](int sl, int kb0) {
                        bool wrote = false;
                        for (unsigned own = m.own; own; own &= own - 1) {
                            const int i = __ffs(own) - 1;
                            const int key = m.pos[i] - kb0;
                            if (key < 0 || key >= kStKeys) continue;
                            for (int e = lane; e < 2 * (D / 8); e += 32) {
                                const int isv = e / (D / 8), ch = e - isv * (D / 8);
                                const uint4 val = *reinterpret_cast<const uint4 *>(stash + (i * 2 + isv) * D + ch * 8);
                                *reinterpret_cast<uint4 *>(ring + (size_t)sl * kSlot + isv * kVOff + (ch >> 3) * kHalfTile +
                                                           key * 128 + (((ch & 7) ^ (key & 7)) << 4)) = val;
                            }
                            wrote = true;
                        }
                        if (wrote) dla::fence_proxy_async();
                        __syncwarp();
                    };
                    if (Q > kCCMaxQ) {
                        // ---- tensor form: MT query tiles x KS stage groups over the eight warps
                        const int MT = (Q + 15) / 16, KS = kCW / MT;
                        const int mt = warp % MT, grp = warp / MT;
                        for (int fi = ctid; fi < MT * NKS * 32; fi += kCT) {
                            const int t = fi & 31, ks = (fi >> 5) % NKS, qt = (fi >> 5) / NKS;
                            const int gg = t >> 2, cc = t & 3;
                            const int q0i = qt * 16 + gg, q1i = q0i + 8;
                            uint32_t hv[4], lv[4];
#pragma unroll
                            for (int part = 0; part < 4; ++part) {
                                const int qi = (part & 1) ? q1i : q0i;
                                const int col = ks * 16 + 2 * cc + (part >> 1) * 8;
                                float2 v = qi < Q ? *reinterpret_cast<const float2 *>(qraw + qi * D + col)
                                                  : make_float2(0.f, 0.f);
                                v.x *= a.qscale;
                                v.y *= a.qscale;
                                const __half2 hq = __floats2half2_rn(v.x, v.y);
                                const float2 hf = __half22float2(hq);
                                hv[part] = h2_bits(hq);
                                lv[part] = h2_bits(v.x - hf.x, v.y - hf.y);
                            }
                            uint4 *dst = reinterpret_cast<uint4 *>(qfrag + (size_t)(fi >> 5) * 1024 + t * 16);
                            dst[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                            dst[32] = make_uint4(lv[0], lv[1], lv[2], lv[3]);
                        }
                        csync();
                        const unsigned char *myq = qfrag + (size_t)mt * NKS * 1024 + lane * 16;
                        const int r0 = mt * 16 + g, r1 = r0 + 8;
                        const int len0 = r0 < Q ? m.len[r0 / G] : 0;
                        const int len1 = r1 < Q ? m.len[r1 / G] : 0;
                        float o[NDT][4];
#pragma unroll
                        for (int i = 0; i < NDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
                        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
                        for (int i = grp; i < nst; i += KS) {
                            const uint32_t sq = seq + (uint32_t)i;
                            const int sl = sq % kStages;
                            if (!stage_wait(sq)) {
                                bad = true;
                                break;
                            }
                            const uint32_t ksm = ring_s + (uint32_t)sl * kSlot;
                            const uint32_t vsm = ksm + kVOff;
                            const int kb0 = k0 + i * kStKeys;
                            if (kb0 + kStKeys > k1) zero_tail(sl, kb0);
                            if (m.own) patch(sl, kb0);
                            float sc[4][4], slo[4][4];
#pragma unroll
                            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                                for (int e = 0; e < 4; ++e) sc[nt][e] = slo[nt][e] = 0.f;
#pragma unroll
                            for (int ks = 0; ks < NKS; ks += 2) {
                                const uint4 qa = *reinterpret_cast<const uint4 *>(myq + ks * 1024);
                                const uint4 qb = *reinterpret_cast<const uint4 *>(myq + ks * 1024 + 512);
                                const uint4 qc = *reinterpret_cast<const uint4 *>(myq + (ks + 1) * 1024);
                                const uint4 qd = *reinterpret_cast<const uint4 *>(myq + (ks + 1) * 1024 + 512);
                                const uint32_t qh0[4] = {qa.x, qa.y, qa.z, qa.w}, ql0[4] = {qb.x, qb.y, qb.z, qb.w};
                                const uint32_t qh1[4] = {qc.x, qc.y, qc.z, qc.w}, ql1[4] = {qd.x, qd.y, qd.z, qd.w};
                                const int ch = 2 * ks + (lane >> 3);          // 16-byte chunk of the key row
                                const uint32_t half_off = (uint32_t)(ch >> 3) * kHalfTile;
#pragma unroll
                                for (int nt = 0; nt < 4; ++nt) {
                                    const int key = nt * 8 + (lane & 7);
                                    uint32_t b0, b1, b2, b3;
                                    ldsm_x4(b0, b1, b2, b3, ksm + half_off + (uint32_t)(key * 128 + (((ch & 7) ^ (key & 7)) << 4)));
                                    mma_f16(sc[nt], qh0, b0, b1);
                                    mma_f16(slo[nt], ql0, b0, b1);
                                    mma_f16(sc[nt], qh1, b2, b3);
                                    mma_f16(slo[nt], ql1, b2, b3);
                                }
                            }
                            // mask keys past each row's count, online softmax per row (a lane quad = one row)
                            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const int key = kb0 + nt * 8 + 2 * c + e;
                                    const float v0 = sc[nt][e] + slo[nt][e], v1 = sc[nt][2 + e] + slo[nt][2 + e];
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
                            // O += P V over two 16-key steps: two output tiles per transposed 4-matrix load
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const uint32_t pa[4] = {h2_bits(sc[2 * kk][0], sc[2 * kk][1]),
                                                        h2_bits(sc[2 * kk][2], sc[2 * kk][3]),
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
                            // the stage's MT readers release it for all eight consumer warps
                            if (lane == 0) release(sq, mt == 0 ? (uint32_t)(kCW - MT + 1) : 1u);
                        }
                        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
                        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
                        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
                        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
                        // combine the stage groups pairwise: [slot][element][lane]
                        constexpr int SZ = (NDT * 4 + 4) * 32;
                        for (int half = KS >> 1; half >= 1; half >>= 1) {
                            csync();
                            if (grp >= half && grp < 2 * half) {
                                float *b = cb + (size_t)(mt * half + grp - half) * SZ;
#pragma unroll
                                for (int j = 0; j < NDT; ++j)
#pragma unroll
                                    for (int e = 0; e < 4; ++e) b[(j * 4 + e) * 32 + lane] = o[j][e];
                                b[(NDT * 4 + 0) * 32 + lane] = m0;
                                b[(NDT * 4 + 1) * 32 + lane] = m1;
                                b[(NDT * 4 + 2) * 32 + lane] = l0;
                                b[(NDT * 4 + 3) * 32 + lane] = l1;
                            }
                            csync();
                            if (grp < half) {
                                const float *b = cb + (size_t)(mt * half + grp) * SZ;
                                const float pm0 = b[(NDT * 4 + 0) * 32 + lane], pm1 = b[(NDT * 4 + 1) * 32 + lane];
                                const float pl0 = b[(NDT * 4 + 2) * 32 + lane], pl1 = b[(NDT * 4 + 3) * 32 + lane];
                                const float M0 = fmaxf(m0, pm0), M1 = fmaxf(m1, pm1);
                                const float f0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M0);
                                const float g0 = pm0 == -INFINITY ? 0.f : fast_exp2(pm0 - M0);
                                const float f1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M1);
                                const float g1 = pm1 == -INFINITY ? 0.f : fast_exp2(pm1 - M1);
#pragma unroll
                                for (int j = 0; j < NDT; ++j) {
                                    o[j][0] = o[j][0] * f0 + b[(j * 4 + 0) * 32 + lane] * g0;
                                    o[j][1] = o[j][1] * f0 + b[(j * 4 + 1) * 32 + lane] * g0;
                                    o[j][2] = o[j][2] * f1 + b[(j * 4 + 2) * 32 + lane] * g1;
                                    o[j][3] = o[j][3] * f1 + b[(j * 4 + 3) * 32 + lane] * g1;
                                }
                                l0 = l0 * f0 + pl0 * g0;
                                l1 = l1 * f1 + pl1 * g1;
                                m0 = M0;
                                m1 = M1;
                            }
                        }
                        if (grp == 0 && !bad) {
#pragma unroll
                            for (int hr = 0; hr < 2; ++hr) {
                                const int qi = hr ? r1 : r0;
                                if (qi >= Q || m.len[qi / G] <= k0) continue;
                                const float l = hr ? l1 : l0, mm = hr ? m1 : m0;
                                const int ri = qi / G;
                                const int64_t pidx = ((int64_t)m.row[ri] * P.n_q + m.h * G + (qi - ri * G)) * ms + m.piece;
                                const float inv = 1.f / l;
                                float *po = a.part_o + pidx * D;
#pragma unroll
                                for (int j = 0; j < NDT; ++j)
                                    *reinterpret_cast<float2 *>(po + j * 8 + 2 * c) =
                                        make_float2(o[j][2 * hr] * inv, o[j][2 * hr + 1] * inv);
                                if (c == 0) a.part_lse[pidx] = (mm + fast_log2(l)) * 0.69314718055994530942f;
                            }
                        }
                    } else {
                        // ---- CUDA-core form: every warp a stage group, lane = key for the scores,
                        // lanes over the dimensions for P.V
                        constexpr int QM = kCCMaxQ;
                        const int nq = Q;
                        float *pb = reinterpret_cast<float *>(scr) + warp * QM * kStKeys;   // probabilities
                        csync();                                    // the queries are in place
                        float2 o[QM][DPL];
                        float mq[QM], lq[QM];
#pragma unroll
                        for (int q = 0; q < QM; ++q) {
                            mq[q] = -INFINITY;
                            lq[q] = 0.f;
#pragma unroll
                            for (int e = 0; e < DPL; ++e) o[q][e] = make_float2(0.f, 0.f);
                        }
                        int lenq[QM];
#pragma unroll
                        for (int q = 0; q < QM; ++q) lenq[q] = q < nq ? m.len[q / G] : 0;
                        const int d0 = DPL * lane, dch = d0 / 8;
                        for (int i = warp; i < nst; i += kCW) {
                            const uint32_t sq = seq + (uint32_t)i;
                            const int sl = sq % kStages;
                            if (!stage_wait(sq)) {
                                bad = true;
                                break;
                            }
                            const unsigned char *kst = ring + (size_t)sl * kSlot;
                            const unsigned char *vst = kst + kVOff;
                            const int kb0 = k0 + i * kStKeys;
                            if (kb0 + kStKeys > k1) zero_tail(sl, kb0);
                            if (m.own) patch(sl, kb0);
                            float2 s0[QM], s1[QM];
#pragma unroll
                            for (int q = 0; q < QM; ++q) s0[q] = s1[q] = make_float2(0.f, 0.f);
#pragma unroll 2
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
                                        const float4 qa = *reinterpret_cast<const float4 *>(qraw + q * D + ch * 8);
                                        const float4 qc = *reinterpret_cast<const float4 *>(qraw + q * D + ch * 8 + 4);
                                        float2 t = (ch & 1) ? s1[q] : s0[q];
                                        t = __ffma2_rn(make_float2(qa.x, qa.y), k01, t);
                                        t = __ffma2_rn(make_float2(qa.z, qa.w), k23, t);
                                        t = __ffma2_rn(make_float2(qc.x, qc.y), k45, t);
                                        t = __ffma2_rn(make_float2(qc.z, qc.w), k67, t);
                                        if (ch & 1) s1[q] = t; else s0[q] = t;
                                    }
                                }
                            }
                            const int key = kb0 + lane;
                            float ps[QM];
#pragma unroll
                            for (int q = 0; q < QM; ++q) {
                                ps[q] = 0.f;
                                if (q >= nq) continue;
                                const float sv = key < lenq[q] ? ((s0[q].x + s1[q].x) + (s0[q].y + s1[q].y)) * a.qscale
                                                               : -INFINITY;
                                const float mn = fmaxf(mq[q], warp_max(sv));
                                if (mn == -INFINITY) continue;
                                const float al = mq[q] == -INFINITY ? 0.f : fast_exp2(mq[q] - mn);
                                ps[q] = sv == -INFINITY ? 0.f : fast_exp2(sv - mn);
                                lq[q] = lq[q] * al + warp_sum(ps[q]);
                                mq[q] = mn;
#pragma unroll
                                for (int e = 0; e < DPL; ++e) o[q][e] = __fmul2_rn(o[q][e], make_float2(al, al));
                            }
#pragma unroll
                            for (int q = 0; q < QM; ++q)
                                if (q < nq) pb[q * kStKeys + lane] = ps[q];
                            __syncwarp();
                            const unsigned char *vcol = vst + (dch >> 3) * kHalfTile + (d0 & 7) * 2;
#pragma unroll 2
                            for (int j4 = 0; j4 < kStKeys; j4 += 4) {
                                float v[4][DPL];
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const int j = j4 + kk;
                                    const unsigned char *vp = vcol + j * 128 + (((dch & 7) ^ (j & 7)) << 4);
                                    if constexpr (DPL == 4) {
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
                            if (lane == 0) release(sq, (uint32_t)kCW);   // its only reader
                        }
                        // combine the eight warps pairwise: [slot][element][lane]
                        constexpr int SZ = (QM * DPL + 2 * QM) * 32;
                        float ov[QM][DPL];
#pragma unroll
                        for (int q = 0; q < QM; ++q)
#pragma unroll
                            for (int e = 0; e < DPL; ++e) ov[q][e] = o[q][e].x + o[q][e].y;
                        for (int half = kCW >> 1; half >= 1; half >>= 1) {
                            csync();
                            if (warp >= half && warp < 2 * half) {
                                float *b = cb + (size_t)(warp - half) * SZ;
#pragma unroll
                                for (int q = 0; q < QM; ++q) {
#pragma unroll
                                    for (int e = 0; e < DPL; ++e) b[(q * DPL + e) * 32 + lane] = ov[q][e];
                                    b[(QM * DPL + 2 * q) * 32 + lane] = mq[q];
                                    b[(QM * DPL + 2 * q + 1) * 32 + lane] = lq[q];
                                }
                            }
                            csync();
                            if (warp < half) {
                                const float *b = cb + (size_t)warp * SZ;
#pragma unroll
                                for (int q = 0; q < QM; ++q) {
                                    const float pm = b[(QM * DPL + 2 * q) * 32 + lane];
                                    const float pl = b[(QM * DPL + 2 * q + 1) * 32 + lane];
                                    const float M = fmaxf(mq[q], pm);
                                    const float f = mq[q] == -INFINITY ? 0.f : fast_exp2(mq[q] - M);
                                    const float gg = pm == -INFINITY ? 0.f : fast_exp2(pm - M);
#pragma unroll
                                    for (int e = 0; e < DPL; ++e) ov[q][e] = ov[q][e] * f + b[(q * DPL + e) * 32 + lane] * gg;
                                    lq[q] = lq[q] * f + pl * gg;
                                    mq[q] = M;
                                }
                            }
                        }
                        if (warp == 0 && !bad) {
#pragma unroll
                            for (int q = 0; q < QM; ++q) {
                                if (q >= nq || lenq[q] <= k0) continue;
                                const int ri = q / G;
                                const int64_t pidx = ((int64_t)m.row[ri] * P.n_q + m.h * G + (q - ri * G)) * ms + m.piece;
                                const float inv = 1.f / lq[q];
#pragma unroll
                                for (int e = 0; e < DPL; ++e) a.part_o[pidx * D + d0 + e] = ov[q][e] * inv;
                                if (lane == 0) a.part_lse[pidx] = (mq[q] + fast_log2(lq[q])) * 0.69314718055994530942f;
                            }
                        }
                    }
                    bad = csync_or(bad);
                    seq += (uint32_t)nst;
                    signal(PH_ATTN, 1u);
                }
                // every store into the cache of this CTA is done: the next kernel of the stream may
                // launch (the library's kernels read before their own wait only what no kernel
                // still running writes: weights, and cache slots below the rows they store)
                __threadfence();
                dl_pdl_launch_dependents();
                continue;
            }
            if (ph == PH_MERGE) {
                // ================================================= merge
                if (!dep_wait(PH_ATTN, (unsigned)P.n_work)) {
                    bad = true;
                    break;
                }
                constexpr int VPL = D / 32;
                constexpr int kMB = 8;                                         // pieces a warp has in flight
                float *s_acc = reinterpret_cast<float *>(scr);                // [kCW][D]
                float *s_m = s_acc + kCW * D, *s_w = s_m + kCW;
                int mb, me;
                share((int64_t)a.nr * P.n_q, cta, C, mb, me);
                for (int un = mb; un < me; ++un) {
                    const int r = un / P.n_q, hq = un - (un / P.n_q) * P.n_q;
                    const int L = clip_len(s_seq[r], P.row_keys_max[r], a.capacity, nullptr, false);
                    const int np = (L + P.chunk - 1) / P.chunk;
                    float *dst = a.attn + (int64_t)r * a.attn_stride + (int64_t)hq * D;
                    if (np == 0) {
                        for (int d = ctid; d < D; d += kCT) dst[d] = 0.f;
                        if (a.lse && ctid == 0) a.lse[r * P.n_q + hq] = -INFINITY;
                        continue;
                    }
                    const float *pl = a.part_lse + ((int64_t)r * P.n_q + hq) * P.max_splits;
                    const float *po = a.part_o + ((int64_t)r * P.n_q + hq) * P.max_splits * D + lane * VPL;
                    float Mw = -INFINITY, Ww = 0.f, acc[VPL];
#pragma unroll
                    for (int i = 0; i < VPL; ++i) acc[i] = 0.f;
                    for (int p0 = warp; p0 < np; p0 += kCW * kMB) {
                        float lv[kMB], v[kMB][VPL];
#pragma unroll
                        for (int u = 0; u < kMB; ++u) {
                            const int p = p0 + kCW * u;
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
                        float mbx = Mw;
#pragma unroll
                        for (int u = 0; u < kMB; ++u) mbx = fmaxf(mbx, lv[u]);
                        const float sc = Mw == -INFINITY ? 0.f : __expf(Mw - mbx);
                        Ww *= sc;
#pragma unroll
                        for (int i = 0; i < VPL; ++i) acc[i] *= sc;
#pragma unroll
                        for (int u = 0; u < kMB; ++u) {
                            const float w = lv[u] == -INFINITY ? 0.f : __expf(lv[u] - mbx);
                            Ww += w;
#pragma unroll
                            for (int i = 0; i < VPL; ++i) acc[i] = fmaf(w, v[u][i], acc[i]);
                        }
                        Mw = mbx;
                    }
#pragma unroll
                    for (int i = 0; i < VPL; ++i) s_acc[warp * D + lane * VPL + i] = acc[i];
                    if (lane == 0) {
                        s_m[warp] = Mw;
                        s_w[warp] = Ww;
                    }
                    csync();
                    float M = -INFINITY;
#pragma unroll
                    for (int w = 0; w < kCW; ++w) M = fmaxf(M, s_m[w]);
                    float f[kCW], Wt = 0.f;
#pragma unroll
                    for (int w = 0; w < kCW; ++w) {
                        f[w] = s_m[w] == -INFINITY ? 0.f : __expf(s_m[w] - M);
                        Wt += f[w] * s_w[w];
                    }
                    const float inv = 1.f / Wt;
                    for (int d = ctid; d < D; d += kCT) {
                        float t = 0.f;
#pragma unroll
                        for (int w = 0; w < kCW; ++w) t = fmaf(f[w], s_acc[w * D + d], t);
                        dst[d] = t * inv;
                    }
                    if (a.lse && ctid == 0) a.lse[r * P.n_q + hq] = M + logf(Wt);
                    csync();
                }
                signal(PH_MERGE, (unsigned)(me - mb));
                continue;
            }
            // ===================================================== projections
            // a unit is one row tile over one K-part of up to kPartKT k-tiles, streamed as consecutive
            // slots of kKsl k-tiles; warp w multiplies k-tiles [4w, 4w + 4) of every slot, with the
            // activations of its k-tiles in registers (tensor path) or the part's activations in
            // shared memory (CUDA-core path); the warps' sums of a unit meet in shared memory once
            const SGemv &Gv = gemv_of(ph);
            const int dep = ph == PH_QKV ? -1 : ph == PH_O ? PH_MERGE : ph == PH_GU ? PH_O : PH_GU;
            const unsigned target = ph == PH_O ? (unsigned)(a.nr * P.n_q)
                                  : ph == PH_GU ? (unsigned)(a.g[1].RT * a.g[1].cs)
                                  : ph == PH_DOWN ? (unsigned)(a.g[2].RT * a.g[2].cs) : 0u;
            if (dep >= 0 && !dep_wait(dep, target)) {
                bad = true;
                break;
            }
            int ub, ue;
            unit_share(Gv.RT, Gv.cs, cta, C, ub, ue);
            // units per CTA-wide reduction: eight, or four when eight activation rows take the room
            constexpr int RB = NRC > 4 ? kRBMax / 2 : kRBMax;
            constexpr int kRed = RB * kCW * 128 * 4;
            float *red = reinterpret_cast<float *>(scr);                     // [RB][kCW][128]
            float *xs = reinterpret_cast<float *>(scr + kRed);               // CUDA-core path: [NRC][kPartKT * 32]
            float *snc = reinterpret_cast<float *>(scr + kRed);              // tensor path: [kCW][KPW][bias, 1/scale][8]
            static_assert(kRed + NRC * kPartKT * 32 * 4 <= (int)kScratch &&
                          kRed + kCW * kPartSlots * kKWM * 2 * 8 * 4 <= (int)kScratch, "projection scratch fits");
            const int wk0 = warp * kKWM;
            constexpr int KPW = kPartSlots * kKWM;                             // k-tiles of a part per warp
            uint32_t bh[GMMA ? KPW : 1][4], bl[GMMA ? KPW : 1][4];
            // defined here unconditionally: otherwise the compiler keeps the previous projection's
            // values alive across the phases between them (the attention's registers then spill)
#pragma unroll
            for (int jj = 0; jj < (GMMA ? KPW : 1); ++jj)
#pragma unroll
                for (int p = 0; p < 4; ++p) bh[jj][p] = bl[jj][p] = 0u;
            int cur_s = -1;
            unsigned finished = 0;
            for (int u = ub; u < ue && !bad;) {
                const int s = u / Gv.RT;
                const int nb = min(RB, min(ue, (s + 1) * Gv.RT) - u);
                const int kt0 = s * kPartKT, nkt = min(kPartKT, Gv.KT - kt0);
                const int nsl = (nkt + kKsl - 1) / kKsl;                        // slots of a unit of this part
                if (s != cur_s) {
                    cur_s = s;
                    if constexpr (GMMA) {
                        // this warp's k-tiles (slot j, tile i) = kt0 + 32 j + 4 warp + i: each k-tile of an
                        // activation row scaled by a power of two that puts its largest |x| into
                        // [2^14, 2^15), then split into f16 hi + lo (about 22 significant bits); the
                        // k-tile's bias term (-1152 x its column sum) and inverse scale go to shared memory
#pragma unroll
                        for (int jj = 0; jj < KPW; ++jj) {              // every load first (raw bits)
                            const int kl = (jj / kKWM) * kKsl + wk0 + (jj % kKWM);      // part-local k-tile
                            const bool live = kl < nkt && (kt0 + kl) * 32 < Gv.n_in && g < a.nr;
                            const float4 *xr = reinterpret_cast<const float4 *>(Gv.x + (int64_t)g * Gv.x_stride + (kt0 + kl) * 32 + 8 * c);
                            const float4 lo = live ? __ldcg(xr) : make_float4(0.f, 0.f, 0.f, 0.f);
                            const float4 hi = live ? __ldcg(xr + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                            bh[jj][0] = __float_as_uint(lo.x);
                            bl[jj][0] = __float_as_uint(lo.y);
                            bh[jj][1] = __float_as_uint(lo.z);
                            bl[jj][1] = __float_as_uint(lo.w);
                            bh[jj][2] = __float_as_uint(hi.x);
                            bl[jj][2] = __float_as_uint(hi.y);
                            bh[jj][3] = __float_as_uint(hi.z);
                            bl[jj][3] = __float_as_uint(hi.w);
                        }
#pragma unroll
                        for (int jj = 0; jj < KPW; ++jj) {
                            float2 v[4];
#pragma unroll
                            for (int p = 0; p < 4; ++p) v[p] = make_float2(__uint_as_float(bh[jj][p]), __uint_as_float(bl[jj][p]));
                            float mx = 0.f;
#pragma unroll
                            for (int p = 0; p < 4; ++p) mx = fmaxf(mx, fmaxf(fabsf(v[p].x), fabsf(v[p].y)));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                            const int ebits = (int)((__float_as_uint(mx) >> 23) & 0xFFu);
                            const int sexp = mx > 0.f ? min(268 - ebits, 253) : 127;
                            const float sig = __uint_as_float((uint32_t)sexp << 23);
                            float colsum = 0.f;
#pragma unroll
                            for (int p = 0; p < 4; ++p) {
                                const float tx = v[p].x * sig, ty = v[p].y * sig;
                                const __half2 h = __floats2half2_rn(tx, ty);
                                const float2 hf = __half22float2(h);
                                const __half2 l = __floats2half2_rn(tx - hf.x, ty - hf.y);
                                const float2 lf = __half22float2(l);
                                bh[jj][p] = h2_bits(h);
                                bl[jj][p] = h2_bits(l);
                                colsum += (hf.x + lf.x) + (hf.y + lf.y);
                            }
                            colsum += __shfl_xor_sync(0xffffffffu, colsum, 1);
                            colsum += __shfl_xor_sync(0xffffffffu, colsum, 2);
                            if (c == 0) {
                                snc[((warp * KPW + jj) * 2) * 8 + g] = -1152.f * colsum;
                                snc[((warp * KPW + jj) * 2 + 1) * 8 + g] = __uint_as_float((uint32_t)(254 - sexp) << 23);
                            }
                        }
                        __syncwarp();
                    } else {
                        // the part's activation rows in shared memory (zero past n_in)
                        csync();                                 // the previous part's rows are read
                        // every load of the thread first (one round trip), then the stores
                        static_assert(kPartKT * 8 == kCT, "a row of a part is one float4 per thread");
                        float4 v[NRC];
#pragma unroll
                        for (int i = 0; i < NRC; ++i) {
                            const int e = ctid + i * kCT;
                            const int r = e / (nkt * 8), q = e - r * (nkt * 8);       // q: float4 of the part
                            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (e < NRC * nkt * 8 && r < a.nr && (kt0 * 32 + q * 4) < Gv.n_in)
                                v[i] = __ldcg(reinterpret_cast<const float4 *>(Gv.x + (int64_t)r * Gv.x_stride + kt0 * 32) + q);
                        }
#pragma unroll
                        for (int i = 0; i < NRC; ++i) {
                            const int e = ctid + i * kCT;
                            const int r = e / (nkt * 8), q = e - r * (nkt * 8);
                            if (e < NRC * nkt * 8) *reinterpret_cast<float4 *>(xs + r * (kPartKT * 32) + q * 4) = v[i];
                        }
                        csync();
                    }
                }
                csync();                                     // the previous batch's sums are read
#pragma unroll 1
                for (int r = 0; r < nb; ++r) {
                    float2 acc01 = make_float2(0.f, 0.f), acc23 = acc01;   // tensor path: rows g, g+8 x columns 2c, 2c+1
                    float2 accg[NRC], acch[NRC];                         // CUDA-core path: rows g, g+8 x activation rows
#pragma unroll
                    for (int q = 0; q < NRC; ++q) accg[q] = acch[q] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < kPartSlots; ++j) {
                        if (j >= nsl) break;
                        const uint32_t sq = seq + (uint32_t)j;
                        const int sl = sq % kStages;
                        if (!unit_wait(sq)) {
                            bad = true;
                            break;
                        }
                        const unsigned char *sw = ring + (size_t)sl * kSlot;
                        const unsigned char *sd = sw + kUnitW;
                        const int snkt = min(kKsl, nkt - j * kKsl);      // k-tiles of this slot
                        if (wk0 < snkt && GMMA) {
                            // every shared load of the warp's k-tiles first, then the hi and lo products in
                            // independent accumulators, a k-step of all k-tiles at a time (eight chains of
                            // two instead of four chains of four)
                            uint4 w[kKWM];
                            float2 dgh[kKWM];                                // (d[g], d[g+8])
#pragma unroll
                            for (int i = 0; i < kKWM; ++i) {
                                const int kl = wk0 + i;                      // slot-local k-tile
                                w[i] = *reinterpret_cast<const uint4 *>(sw + kl * 512 + lane * 16);
                                dgh[i] = __half22float2(*reinterpret_cast<const __half2 *>(sd + (kl >> 2) * 128 + g * 16 + (kl & 3) * 4));
                            }
                            float th[kKWM][4], tl[kKWM][4];
#pragma unroll
                            for (int i = 0; i < kKWM; ++i)
#pragma unroll
                                for (int p = 0; p < 4; ++p) th[i][p] = tl[i][p] = 0.f;
#pragma unroll
                            for (int i = 0; i < kKWM; ++i) {
                                const int jj = GMMA ? j * kKWM + i : 0;
                                const uint32_t a0 = u8x2_to_h2(w[i].x, 0x4140u), a1 = u8x2_to_h2(w[i].x, 0x4342u);
                                const uint32_t a2 = u8x2_to_h2(w[i].y, 0x4140u), a3 = u8x2_to_h2(w[i].y, 0x4342u);
                                mma16816p(th[i], a0, a1, a2, a3, bh[jj][0], bh[jj][1]);
                                mma16816p(tl[i], a0, a1, a2, a3, bl[jj][0], bl[jj][1]);
                            }
#pragma unroll
                            for (int i = 0; i < kKWM; ++i) {
                                const int jj = GMMA ? j * kKWM + i : 0;
                                const uint32_t a4 = u8x2_to_h2(w[i].z, 0x4140u), a5 = u8x2_to_h2(w[i].z, 0x4342u);
                                const uint32_t a6 = u8x2_to_h2(w[i].w, 0x4140u), a7 = u8x2_to_h2(w[i].w, 0x4342u);
                                mma16816p(th[i], a4, a5, a6, a7, bh[jj][2], bh[jj][3]);
                                mma16816p(tl[i], a4, a5, a6, a7, bl[jj][2], bl[jj][3]);
                            }
#pragma unroll
                            for (int i = 0; i < kKWM; ++i) {
                                // columns 2c, 2c + 1: the k-tile's bias terms and inverse scales
                                const int jj = GMMA ? j * kKWM + i : 0;
                                const float2 nc = *reinterpret_cast<const float2 *>(snc + ((warp * KPW + jj) * 2) * 8 + 2 * c);
                                const float2 us = *reinterpret_cast<const float2 *>(snc + ((warp * KPW + jj) * 2 + 1) * 8 + 2 * c);
                                const float2 t01 = __fadd2_rn(make_float2(th[i][0], th[i][1]), make_float2(tl[i][0], tl[i][1]));
                                const float2 t23 = __fadd2_rn(make_float2(th[i][2], th[i][3]), make_float2(tl[i][2], tl[i][3]));
                                acc01 = __ffma2_rn(make_float2(dgh[i].x * us.x, dgh[i].x * us.y), __fadd2_rn(t01, nc), acc01);
                                acc23 = __ffma2_rn(make_float2(dgh[i].y * us.x, dgh[i].y * us.y), __fadd2_rn(t23, nc), acc23);
                            }
                        } else if (wk0 < snkt) {
#pragma unroll
                            for (int i = 0; i < kKWM; ++i) {
                                const int kl = wk0 + i;                  // slot-local k-tile
                                const uint4 w = *reinterpret_cast<const uint4 *>(sw + kl * 512 + lane * 16);
                                const __half2 sp = *reinterpret_cast<const __half2 *>(sd + (kl >> 2) * 128 + g * 16 + (kl & 3) * 4);
                                const float2 dgh = __half22float2(sp);          // (d[g], d[g+8])
                                const float dg = dgh.x, dh = dgh.y;
                                {
                                    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
                                    float2 wg[4], wh[4];
#pragma unroll
                                    for (int p = 0; p < 4; ++p) {
                                        wg[p] = u8x2_to_f32x2(wd[p], 0);
                                        wh[p] = u8x2_to_f32x2(wd[p], 2);
                                    }
                                    const float *xk = xs + (j * kKsl + kl) * 32 + 8 * c;
#pragma unroll
                                    for (int q = 0; q < NRC; ++q) {
                                        const float *xq = xk + q * (kPartKT * 32);
                                        const float2 x0 = *reinterpret_cast<const float2 *>(xq);
                                        float2 sg = __fmul2_rn(wg[0], x0), sh = __fmul2_rn(wh[0], x0);
#pragma unroll
                                        for (int p = 1; p < 4; ++p) {
                                            const float2 xp = *reinterpret_cast<const float2 *>(xq + 2 * p);
                                            sg = __ffma2_rn(wg[p], xp, sg);
                                            sh = __ffma2_rn(wh[p], xp, sh);
                                        }
                                        accg[q] = __ffma2_rn(make_float2(dg, dg), sg, accg[q]);
                                        acch[q] = __ffma2_rn(make_float2(dh, dh), sh, acch[q]);
                                    }
                                }
                            }
                        }
                        __syncwarp();
                        if (lane == 0) release(sq, 1u);
                    }
                    if (bad) break;
                    seq += (uint32_t)nsl;
                    // this warp's partial of the unit: [unit][warp][row 0..15][column 0..7]
                    float *rw = red + (r * kCW + warp) * 128;
                    if constexpr (GMMA) {
                        *reinterpret_cast<float2 *>(rw + g * 8 + 2 * c) = acc01;
                        *reinterpret_cast<float2 *>(rw + (g + 8) * 8 + 2 * c) = acc23;
                    } else {
#pragma unroll
                        for (int q = 0; q < NRC; ++q) {
                            float vg = accg[q].x + accg[q].y, vh = acch[q].x + acch[q].y;
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
                bad = csync_or(bad);                     // the partials are in place; uniform verdict
                if (Gv.cs > 1 && !zeroed) {
                    if (!dep_wait_word(SY_ZEROED, (unsigned)C)) bad = true;
                    zeroed = true;
                }
                // sum the eight warps' partials in warp order; a unit over the whole K writes its row
                // tile, a unit over a K-slice adds into outputs zeroed at the start (the slices of a
                // row tile arrive in any order, so with more than two of them the last bits of a
                // result may differ from call to call)
                for (int e4 = ctid; e4 < nb * 32; e4 += kCT) {
                    const int r = e4 >> 5, el = (e4 & 31) * 4;
                    const float *rb = red + r * kCW * 128 + el;
                    float4 sum = *reinterpret_cast<const float4 *>(rb);
#pragma unroll
                    for (int w = 1; w < kCW; ++w) {
                        const float4 t = *reinterpret_cast<const float4 *>(rb + w * 128);
                        sum.x += t.x;
                        sum.y += t.y;
                        sum.z += t.z;
                        sum.w += t.w;
                    }
                    const int rt = u + r - s * Gv.RT;
                    const int o = rt * 16 + (el >> 3), col0 = el & 7;
                    if (o < Gv.n_out) {
                        const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if (col0 + q >= a.nr) continue;
                            float *dst = Gv.y + (int64_t)(col0 + q) * Gv.y_stride + o;
                            if (Gv.cs == 1) *dst = sv[q];
                            else atomicAdd(dst, sv[q]);
                        }
                    }
                }
                finished += (unsigned)nb;
                u += nb;
            }
            // row tiles count as finished once every part of them is in: each CTA counts its units,
            // and the next phase waits for RT * cs of them
            signal(ph, finished);
        }
        if (bad) {
            if (ctid == 0) set_abort();
        }
    }

    // =============================================================== finish
    __syncthreads();
    if (tid == 0) {
        // leave no copy in flight (after a failure some stages were never consumed): wait, bounded,
        // for the last stage issued into each slot
        for (int sl = 0; sl < kStages; ++sl)
            if (s_iss[sl] > 0) dla::mbar_wait(&full[sl], (uint32_t)((s_iss[sl] - 1) & 1));
        __threadfence();
        const unsigned prev = atomicAdd(a.sync + SY_FINISH, 1u);
        if (prev == (unsigned)C - 1) {
            // the last CTA: every other CTA is past its last wait; clear the words for the next call
            __threadfence();
            for (int i = 0; i < PH_N; ++i) atomicExch(a.sync + SY_DONE + i, 0u);
            atomicExch(a.sync + SY_ZEROED, 0u);
            atomicExch(a.sync + SY_ABORTED, 0u);
            atomicExch(a.sync + SY_FINISH, 0u);
        }
    }
}

}  // namespace

// ---------------------------------------------------------------- host side

namespace {

using StepKernel = void (*)(StepArgs, CUtensorMap, CUtensorMap);

template <int D>
StepKernel pick_step_d(bool mma, int nrc)
{
    if (mma) return layer_step_kernel<D, true, 1>;
    if constexpr (D == 128) {
        // the CUDA-core projections of wider commands: an option, to compare the two inner products
        if (nrc > 4) return layer_step_kernel<D, false, 8>;
        if (nrc > 2) return layer_step_kernel<D, false, 4>;
    }
    return nrc == 1 ? layer_step_kernel<D, false, 1> : layer_step_kernel<D, false, 2>;
}

StepKernel pick_step(int D, bool mma, int nrc) { return D == 128 ? pick_step_d<128>(mma, nrc) : pick_step_d<64>(mma, nrc); }

size_t round16(size_t x) { return (x + 15) & ~(size_t)15; }

struct StepLayout {
    size_t part_o, part_lse, total;
    int RT[4], KT[4], cs[4];
};

// Workspace: the sync words, then the attention pieces' (o, lse) in dl_decode_attn's layout.
int step_layout(const dl_layer_weights *W, const dl_attn_plan *P, StepLayout *L)
{
    const dl_q8_weight *w[4] = {&W->qkv, &W->o, &W->gu, &W->down};
    const int n = W->gu.qs ? 4 : 2;
    size_t off = SY_WORDS * 4;
    memset(L, 0, sizeof(*L));
    for (int p = 0; p < n; ++p) {
        const int rc = dl_q8_packed_size(w[p]->n_out, w[p]->n_in, nullptr, nullptr);
        if (rc != DL_OK) return rc;
        L->RT[p] = (int)dl::ceil_div(w[p]->n_out, 16);
        L->KT[p] = (int)(dl::ceil_div(w[p]->n_in, 128) * 4);
        L->cs[p] = (int)dl::ceil_div(L->KT[p], kPartKT);
    }
    const size_t po = (size_t)P->rows * P->n_q * P->max_splits * P->head_dim * 4;
    L->part_o = off;
    off += round16(po);
    L->part_lse = off;
    off += round16((size_t)P->rows * P->n_q * P->max_splits * 4);
    L->total = off;
    return DL_OK;
}

bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const char *x = static_cast<const char *>(a), *y = static_cast<const char *>(b);
    return na && nb && x < y + nb && y < x + na;
}

// bytes spanned by `rows` rows of `width` floats at `stride`
size_t span(int rows, int64_t width, int64_t stride) { return ((size_t)(rows - 1) * stride + width) * 4; }

}  // namespace

extern "C" {

int dl_layer_step_workspace_size(const dl_layer_weights *W, const dl_attn_plan *plan, size_t *bytes)
{
    dl::clear_error();
    if (!W || !plan || !bytes) return dl::fail(DL_E_ARG, "dl_layer_step_workspace_size: null pointer");
    if (plan->rows < 1 || plan->rows > DL_MAX_ROWS || plan->max_splits < 1 || plan->n_q < 1)
        return dl::fail(DL_E_ARG, "dl_layer_step_workspace_size: invalid plan");
    StepLayout L;
    const int rc = step_layout(W, plan, &L);
    if (rc != DL_OK) return rc;
    *bytes = L.total;
    return DL_OK;
}

int dl_layer_step(const dl_layer_weights *W, const dl_layer_bufs *B, const float *bias, const int32_t *pos,
                  const dl_rope *rope, const dl_kv_cache *kv, const int32_t *seqlen, const dl_attn_plan *plan,
                  void *workspace, size_t workspace_bytes, int32_t *status, int path, dl_stream_t stream)
{
    dl::clear_error();
    if (!W || !B || !pos || !rope || !kv || !seqlen || !plan || !workspace)
        return dl::fail(DL_E_ARG, "dl_layer_step: null pointer");
    const dl_attn_plan &P = *plan;
    if (P.rows < 1 || P.rows > DL_MAX_ROWS || P.n_sessions < 1 || P.n_sessions > DL_MAX_ROWS || P.chunk < kStKeys ||
        P.chunk % kStKeys != 0 || P.max_splits < 1 || P.n_work < 1 || P.n_kv < 1 || P.n_q % P.n_kv != 0 ||
        P.n_q / P.n_kv > kMaxQ)
        return dl::fail(DL_E_ARG, "dl_layer_step: invalid plan");
    if (P.cluster) return dl::fail(DL_E_ARG, "dl_layer_step: a cluster plan has no pieces in the workspace");
    const int rows = P.rows, D = P.head_dim;
    for (int s = 0; s < P.n_sessions; ++s)
        if ((P.sess_begin[s + 1] - P.sess_begin[s]) * (P.n_q / P.n_kv) > kMaxQ)
            return dl::fail(DL_E_SHAPE, "dl_layer_step: a session's queries exceed %d", kMaxQ);
    if (D != 64 && D != 128) return dl::fail(DL_E_SHAPE, "dl_layer_step: head_dim=%d (64 or 128)", D);
    if (!(kv->elem_bytes == 0 || kv->elem_bytes == 2))
        return dl::fail(DL_E_SHAPE, "dl_layer_step: the f16 mirror only (elem_bytes %d)", kv->elem_bytes);
    if (!kv->k || !kv->v || kv->head_dim != D || kv->n_kv != P.n_kv || kv->capacity < 1 || kv->n_regions < 1 ||
        kv->region_stride < (int64_t)kv->n_kv * kv->capacity * D)
        return dl::fail(DL_E_ARG, "dl_layer_step: cache does not match the plan");
    for (int r = 0; r < rows; ++r)
        if (P.row_region[r] < 0 || P.row_region[r] >= kv->n_regions)
            return dl::fail(DL_E_ARG, "dl_layer_step: row %d region %d outside the cache", r, P.row_region[r]);
    if (!rope->cos_sin || rope->rot_dim < 0 || rope->rot_dim > D || rope->rot_dim % 2 || rope->max_pos < 1 ||
        (reinterpret_cast<uintptr_t>(rope->cos_sin) & 7u))
        return dl::fail(DL_E_ARG, "dl_layer_step: rope table");
    if (path < 0 || path > 2) return dl::fail(DL_E_ARG, "dl_layer_step: path=%d", path);
    const bool mma = path == 2 || (path == 0 && rows > 2);
    if (!mma && rows > 2 && D != 128)
        return dl::fail(DL_E_SHAPE, "dl_layer_step: the CUDA-core projections serve more than 2 rows at head_dim 128 only");
    const bool ffn = W->gu.qs != nullptr;
    const dl_q8_weight *w[4] = {&W->qkv, &W->o, &W->gu, &W->down};
    const int ng = ffn ? 4 : 2;
    const float *xs[4] = {B->x, B->attn, B->x_ffn, B->x_down};
    const int64_t xst[4] = {B->x_stride, B->attn_stride, B->x_ffn_stride, B->x_down_stride};
    float *ys[4] = {B->qkv, B->o, B->gu, B->down};
    const int64_t yst[4] = {B->qkv_stride, B->o_stride, B->gu_stride, B->down_stride};
    for (int p = 0; p < ng; ++p) {
        if (!w[p]->qs || !w[p]->d || !xs[p] || !ys[p]) return dl::fail(DL_E_ARG, "dl_layer_step: projection %d: null pointer", p);
        const int rc = dl_q8_packed_size(w[p]->n_out, w[p]->n_in, nullptr, nullptr);
        if (rc != DL_OK) return rc;
        if (xst[p] < w[p]->n_in || yst[p] < w[p]->n_out)
            return dl::fail(DL_E_ARG, "dl_layer_step: projection %d strides below the row widths", p);
        if (!dl::aligned16(xs[p]) || xst[p] % 4 || !dl::aligned16(w[p]->qs) || !dl::aligned16(w[p]->d))
            return dl::fail(DL_E_ALIGN, "dl_layer_step: projection %d: inputs and planes must be 16-byte aligned", p);
        if (overlap(xs[p], span(rows, w[p]->n_in, xst[p]), ys[p], span(rows, w[p]->n_out, yst[p])))
            return dl::fail(DL_E_ARG, "dl_layer_step: projection %d's output overlaps its input", p);
    }
    if (W->qkv.n_out != (int64_t)(P.n_q + 2 * P.n_kv) * D || W->o.n_in != (int64_t)P.n_q * D)
        return dl::fail(DL_E_SHAPE, "dl_layer_step: QKV must give (n_q + 2 n_kv) head_dim outputs and O take n_q head_dim");
    if (B->attn_stride < (int64_t)P.n_q * D) return dl::fail(DL_E_ARG, "dl_layer_step: attn_stride");
    StepLayout L;
    int rc = step_layout(W, plan, &L);
    if (rc != DL_OK) return rc;
    if (workspace_bytes < L.total)
        return dl::fail(DL_E_WORKSPACE, "dl_layer_step: workspace %zu < %zu bytes", workspace_bytes, L.total);
    if (!dl::aligned16(workspace)) return dl::fail(DL_E_ALIGN, "dl_layer_step: workspace must be 16-byte aligned");
    // outputs: pairwise apart, and apart from the workspace
    const void *outs[6] = {B->qkv, B->attn, B->o, ffn ? B->gu : nullptr, ffn ? B->down : nullptr, B->lse};
    const size_t on[6] = {span(rows, W->qkv.n_out, B->qkv_stride), span(rows, (int64_t)P.n_q * D, B->attn_stride),
                          span(rows, W->o.n_out, B->o_stride), ffn ? span(rows, W->gu.n_out, B->gu_stride) : 0,
                          ffn ? span(rows, W->down.n_out, B->down_stride) : 0, B->lse ? (size_t)rows * P.n_q * 4 : 0};
    for (int i = 0; i < 6; ++i) {
        if (overlap(outs[i], on[i], workspace, L.total))
            return dl::fail(DL_E_ARG, "dl_layer_step: an output overlaps the workspace");
        for (int j = i + 1; j < 6; ++j)
            if (overlap(outs[i], on[i], outs[j], on[j])) return dl::fail(DL_E_ARG, "dl_layer_step: outputs overlap");
    }
    if (B->qkv_stride % 4 || !dl::aligned16(B->qkv)) return dl::fail(DL_E_ALIGN, "dl_layer_step: qkv alignment");

    int sm = 0;
    rc = dl::device_sm_count(&sm);
    if (rc != DL_OK) return rc;
    if (dl::ceil_div(P.n_work, sm) > kMaxIt)
        return dl::fail(DL_E_SHAPE, "dl_layer_step: %d work items exceed %d per SM", P.n_work, kMaxIt);
    const StepKernel kern = pick_step(D, mma, mma ? 1 : rows);   // rows 3, 4 -> 4; 5..8 -> 8
    {
        static std::mutex mu;
        static const void *ready[16][8];
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return dl::cuda_fail(e, "dl_layer_step: cudaGetDevice");
        std::lock_guard<std::mutex> lock(mu);
        bool seen = false;
        int slot = -1;
        for (int i = 0; i < 8 && dev < 16; ++i) {
            if (ready[dev][i] == (const void *)kern) seen = true;
            if (!ready[dev][i] && slot < 0) slot = i;
        }
        if (!seen) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
            if (e != cudaSuccess) return dl::cuda_fail(e, "dl_layer_step: set shared memory");
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return dl::cuda_fail(e, "dl_layer_step: shared-memory carveout");
            int per_sm = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSmemBytes);
            if (e != cudaSuccess) return dl::cuda_fail(e, "dl_layer_step: occupancy");
            if (per_sm < 1) {
                cudaFuncAttributes fa;
                memset(&fa, 0, sizeof(fa));
                cudaFuncGetAttributes(&fa, kern);
                cudaGetLastError();
                return dl::fail(DL_E_SHAPE, "dl_layer_step: the CTA does not fit an SM (%d registers, %zu + %zu bytes "
                                "of shared memory, %d threads)", fa.numRegs, fa.sharedSizeBytes, kSmemBytes, kThreads);
            }
            if (dev < 16 && slot >= 0) ready[dev][slot] = (const void *)kern;
        }
    }
    StepArgs a;
    memset(&a, 0, sizeof(a));
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    for (int p = 0; p < ng; ++p) {
        SGemv &G = a.g[p];
        G.qs = static_cast<const unsigned char *>(w[p]->qs);
        G.d = static_cast<const unsigned char *>(w[p]->d);
        G.x = xs[p];
        G.x_stride = xst[p];
        G.y = ys[p];
        G.y_stride = yst[p];
        G.n_out = (int)w[p]->n_out;
        G.n_in = (int)w[p]->n_in;
        G.KT = L.KT[p];
        G.RT = L.RT[p];
        G.cs = L.cs[p];
    }
    a.n_gemv = ng;
    a.nr = rows;
    a.bias = bias;
    a.pos = pos;
    a.cs = reinterpret_cast<const float2 *>(rope->cos_sin);
    a.rot = rope->rot_dim;
    a.neox = rope->neox;
    a.max_pos = rope->max_pos;
    a.kc = static_cast<uint16_t *>(kv->k);
    a.vc = static_cast<uint16_t *>(kv->v);
    a.region_stride = kv->region_stride;
    a.capacity = kv->capacity;
    a.seqlen = seqlen;
    a.part_o = reinterpret_cast<float *>(ws + L.part_o);
    a.part_lse = reinterpret_cast<float *>(ws + L.part_lse);
    a.attn = B->attn;
    a.attn_stride = B->attn_stride;
    a.lse = B->lse;
    a.qscale = 1.4426950408889634f / sqrtf((float)D);
    a.plan = P;
    a.sync = reinterpret_cast<unsigned *>(ws);
    a.status = status;
    CUtensorMap tk, tv;
    dl_kv_cache kvv = *kv;
    kvv.elem_bytes = 2;
    rc = dl::make_kv_tmap(&tk, kv->k, &kvv);
    if (rc != DL_OK) return rc;
    rc = dl::make_kv_tmap(&tv, kv->v, &kvv);
    if (rc != DL_OK) return rc;
    return dl::launch_pdl(kern, dim3((unsigned)sm), dim3(kThreads), kSmemBytes, static_cast<cudaStream_t>(stream),
                          "dl_layer_step: launch", a, tk, tv);
}

}  // extern "C"
