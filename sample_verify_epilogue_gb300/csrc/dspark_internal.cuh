// Internal definitions shared by the sm_103a kernels of the verify-and-sample epilogue.
//
// Data flow of one call (all on the caller's stream, no host synchronisation):
//   prep_kernel          request checks, segment counts, per-(request, vocab tile) penalty index
//   stream_stats_kernel  the one HBM pass over x and q: per-tile maxima, sums and candidates
//   row_finalize_kernel  per verify row: merge segments, top-k threshold, nucleus, normaliser
//                        (rows needing a whole-vocabulary threshold get it in the same block)
//   accept_kernel        per request: accept scan, eos stop, counters, residual / bonus draw
//                        over the kept list or the whole row, padding of the outputs
//   logprob_kernel       the emitted positions' raw log-softmax and top_logprobs
#pragma once

#include <utility>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/dspark.h"

namespace dspark {

// ---------------------------------------------------------------- sizes
constexpr int kGroups = 2;                                     // independent consumer groups per CTA
constexpr int kGroupWarps = 8;
constexpr int kGroupThreads = kGroupWarps * 32;                // 256
constexpr int kConsumerThreads = kGroups * kGroupThreads;      // 512
constexpr int kStreamThreads = kConsumerThreads + 32;          // + one producer warp
constexpr int kStages = 4;
constexpr int kStageBytes = 48 * 1024;                         // one vocab tile per stage
constexpr int kTileBf16 = kStageBytes / 2;                     // 24576 elements
constexpr int kTileF32 = kStageBytes / 4;                      // 12288 elements
constexpr int kBitmapWordsMax = kTileBf16 / 32;                // 768
constexpr int kPenCap = 256;                                   // penalised tokens per tile held in smem
constexpr int kSegTiles = 4;                                   // vocab tiles per segment
constexpr int kMaxSegTiles = 16;
constexpr int kCandPenGlobal = 1536;                           // per-segment candidates kept in the workspace
constexpr int kMaxCandTopK = 256;                              // top_k above this uses the whole-row path
constexpr int kKeptCap = 1024;                                 // truncated support held as a list
constexpr int kFinalizeThreads = 512;
constexpr int kMergeCap = 8192;                                // merged candidates per row (smem)
constexpr int kMaxB = DSPARK_MAX_B;
constexpr int kLpMaxChunks = 16;                               // chunks per row in the logprob pass
constexpr int kLpMaxGrid = 4 * 1024;                           // CTAs of the logprob pass at most
constexpr int kLpCandPerChunk = 128;                           // unselected keys a chunk may hand on

// ---------------------------------------------------------------- records in the workspace
enum UnitKind : int { kUnitX = 0, kUnitQ = 1 };

struct Plan {
    int n_units;         // unused
    int pad[3];          // pad[0]: error flag set by the streaming pass; pad[1]: bad d2t table;
                         // pad[2]: the logprob pass's item counter
};

enum QLayout : int { kQDense = 0, kQSparse = 1, kQReduced = 2 };

// One segment (consecutive vocab tiles [t0, t1) of one row) with its request's parameters.
struct UnitDesc {
    int slot;            // x: b*(K_max+1)+j ; q: b*K_max+i
    int kind;
    int b;
    int seg;             // segment index within the row
    int t0, t1;
    float temperature;
    int top_k;
    float top_p;
    float presence;
    float frequency;
    int pad;
};

struct TileStats {       // per (row, segment)
    float m_raw;         // x: raw max           | q: max
    float s_raw;         // x: 0                 | q: sum q
    float m_pen;         // x: penalised max
    int   arg_pen;       // x: lowest id attaining m_pen
    float s_temp;        // x: sum exp((x'-m_pen)/T) | q: sum (q/max)^(1/T)
    int   n_pen;         // candidates written (penalised x / q)
    int   pad;
    int   flags;         // kTileOverflow, kTileBad
};
constexpr int kTileOverflowPen = 1;
constexpr int kTileBad = 4;

struct Cand { float v; int id; };

struct PenEntry {        // a token that may carry a penalty in this tile
    int token;
    int base;            // completion-history count
    unsigned mask_lo;    // bit i: d_i == token (i < 32)
    unsigned mask_hi;    // bit i-32
};
struct PenHdr { int n; int overflow; int pad[2]; };

// row modes written by row_finalize
enum RowMode : int {
    kModeInactive = 0,
    kModeGreedy = 1,
    kModeList = 2,       // truncated support held as a list (value-descending)
    kModeFull = 3,       // support = {t : value >= tau}, weights evaluated on the fly
    kModeNeedFull = 4,   // the whole-row path still has to set tau / Z
};

struct XRowOut {
    int    mode;
    int    argmax;       // penalised argmax (lowest id on ties)
    float  m_pen;        // penalised max
    float  tau;          // support threshold on x'
    float  c_l2e;        // log2(e)/T
    float  kth;          // list rows: the k-th largest x' (top-k threshold); -inf when not known
    int    n_kept;
    int    top_k;        // top_k still to apply (whole-row path), 0 = none
    double Z;            // sum of support weights exp2((x'-m_pen)*c_l2e)
    float  top_p;
    int    flags;
};

struct QRowOut {
    int    mode;
    float  qmax;
    float  tau;          // support threshold on q
    float  inv_t;
    double Z;            // sum of support weights (q/qmax)^(1/T) (T=1: q)
    int    top_k;
    float  top_p;
    int    flags;
    int    pad;
};

struct KeptEntry { int id; float w; };
struct TopEntry { int id; float v; };

// One chunk of a row in the logprob pass: its maximum, sum of exp relative to it, top-n list.
struct LpPartial {
    float m;
    float s;
    int n;               // keys of this chunk: in top[], or (listed) in the candidate buffer
    int listed;          // 1: the chunk's gathered keys were written unselected to lp_cand
    TopEntry top[DSPARK_MAX_TOP_LOGPROBS];
};

struct ReqOut {
    int a;               // accepted drafts (up to and including the eos draft when stopped)
    int draw;            // 0 none pending, 1 residual over the whole row, 2 target row over the whole row
    int status;
    int stopped;         // 1: an accepted draft was the eos token; nothing is drawn
};

// Device-side view of the workspace and the call's arguments.
struct Args {
    // shapes
    int B, Km, V, sx, xdtype;
    int tile_x, tiles_x, tile_q, tiles_q, bm_words;
    int nseg_x, nseg_q;    // segments per target / draft row
    int lp_chunks;         // logprob partials the workspace holds (one per logprob CTA)
    int Lq;                // entries of one draft row: V (dense), m (sparse), Vd (reduced)
    int q_layout;          // QLayout
    int lp_pen;            // logprobs over the penalised logits
    int grid_ss;           // CTAs of the streaming pass
    int max_seg;           // segments per (CTA, group) stream, upper bound
    int n_top, want_lp;
    int xslots, qslots;
    // inputs (device)
    const void* x;
    const float* q;
    const int* d;
    const dspark_row_params_t* rows;
    const int* h_off;
    const int* h_ids;
    const int* h_cnt;
    const float* u;
    const int* q_ids;      // sparse: [B * Km * Lq] target ids of the draft entries
    const int* d2t;        // reduced: [Lq] offsets, target id = draft id + d2t[draft id]
    const int* eos;        // [B] end-of-sequence token (< 0: none) or null
    // outputs (device)
    int* out_accept;
    int* out_tokens;
    float* out_lp;
    int* out_top_ids;
    float* out_top_lp;
    int* row_status;
    int* out_stopped;      // [B] or null
    unsigned long long* pos_counts;   // [2 * Km] or null: attempts, then accepts, added to
    // workspace
    Plan* plan;
    UnitDesc* units;       // [grid_ss * kGroups * max_seg] segment streams
    TileStats* ts_x;       // [xslots * nseg_x]
    TileStats* ts_q;       // [qslots * nseg_q]
    Cand* cand_x;          // [xslots * nseg_x * kCandPenGlobal]
    Cand* cand_q;          // [qslots * nseg_q * kCandPenGlobal]
    PenHdr* pen_hdr;       // [B * tiles_x]
    unsigned* pen_bm;      // [B * tiles_x * bm_words]
    PenEntry* pen_ent;     // [B * tiles_x * kPenCap]
    int* draft_base;       // [B * Km]
    int* req_n;            // [2B]: segments of request b (0 if invalid), then its target-row segments
    int* fin_list;         // [1 + xslots + qslots]: count, then the rows left to the block finalize
    XRowOut* xout;         // [xslots]
    KeptEntry* kept;       // [xslots * kKeptCap]
    QRowOut* qout;         // [qslots]
    ReqOut* req;           // [B]
    int* lp_list;          // [1 + xslots]: count, then the rows (b*W + j) the logprob pass reads
    int* lp_done;          // [xslots]: chunks done of each listed row (zeroed by every call)
    LpPartial* lp_part;    // [lp_chunks]: the listed rows' chunk partials, row p's S at [p*S, p*S+S)
    int* t2d;              // reduced: [V] draft id of each target id, -1 for none (built by prep)
    unsigned long long* lp_cand;   // chunk keys left to the row merge, kLpCandPerChunk per chunk (may
                                   // share the target candidate lists' space, unused by then)
};

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float load_x(const void* x, int sx, long long idx) {
    if (sx == 2) {
        unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(x) + idx);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    return __ldg(reinterpret_cast<const float*>(x) + idx);
}

// Order-preserving 32-bit key of a float (-0 folded onto +0, so equal floats share a key).
__device__ __forceinline__ uint32_t fkey(float v) {
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_f(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}
// Composite key: value descending, then id ascending, when sorted descending.
__device__ __forceinline__ unsigned long long ckey(float v, int id) {
    return (static_cast<unsigned long long>(fkey(v)) << 32) | static_cast<unsigned>(0xFFFFFFFFu - static_cast<unsigned>(id));
}
__device__ __forceinline__ int ckey_id(unsigned long long k) {
    return static_cast<int>(0xFFFFFFFFu - static_cast<unsigned>(k & 0xFFFFFFFFull));
}
__device__ __forceinline__ float ckey_v(unsigned long long k) { return key_to_f(static_cast<uint32_t>(k >> 32)); }

// OpenAI penalty in float32 with a fixed operation order: x - ((f*c) + p), no contraction.
__device__ __forceinline__ float penalise(float x, int c, float f, float p) {
    if (c <= 0) return x;
    return __fsub_rn(x, __fadd_rn(__fmul_rn(f, static_cast<float>(c)), p));
}

// Target weight exp((x'-m)/T), computed as 2^((x'-m)*log2(e)/T).
__device__ __forceinline__ float target_weight(float xp, float m, float c_l2e) {
    return exp2f(__fmul_rn(__fsub_rn(xp, m), c_l2e));
}
// Draft weight (q/qmax)^(1/T); at T = 1 the probability itself.
__device__ __forceinline__ float draft_weight(float q, float qmax, float inv_t, bool t_is_one) {
    if (t_is_one) return q;
    if (!(q > 0.f)) return 0.f;
    return exp2f(inv_t * log2f(q / qmax));
}

// Programmatic dependent launch: every kernel after the first waits for its predecessor
// grid to complete (memory included) before touching memory, and lets its own successor
// be launched as soon as all its CTAs are running.  Without the launch attribute both are
// no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
    pdl_wait();
    pdl_trigger();
}

__device__ __forceinline__ unsigned smem_u32(const void* p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier / bulk-copy PTX
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// try_wait that may suspend the thread up to ~hint_ns while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, unsigned parity, unsigned hint_ns) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}
// Non-blocking test of a phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait: returns false when the limit runs out (the caller records an error).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity, long long limit) {
    for (long long i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// One-dimensional bulk copy global -> shared, completing on an mbarrier (TMA engine).
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, unsigned bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// The same copy with an L2 cache policy (from createpolicy) attached.
__device__ __forceinline__ void bulk_g2s_hint(void* dst_smem, const void* src_gmem, unsigned bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        :: "r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

// L2 policy for data read once: its lines are the first to go, so that what the epilogue's
// kernels write and read again (segment statistics, candidate lists, penalty index) stays.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- warp reductions
__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_min(float v) {
    for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
    for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// Sort two values across the 32 lanes of a warp, descending (bitonic network): afterwards
// lane i holds the (i+1)-th largest of each set.
__device__ __forceinline__ void warp_sort2_desc(float& a, float& b) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const float oa = __shfl_xor_sync(0xffffffffu, a, j);
            const float ob = __shfl_xor_sync(0xffffffffu, b, j);
            const bool keep_max = (((lane & j) == 0) == ((lane & k) == 0));
            a = keep_max ? fmaxf(a, oa) : fminf(a, oa);
            b = keep_max ? fmaxf(b, ob) : fminf(b, ob);
        }
    }
}

// c-th largest value across the 32 lanes (with multiplicity), c in [1, 32].
__device__ __forceinline__ float warp_kth_largest(float v, int c) {
    float cur = v, kth = -INFINITY;
    const int lane = threadIdx.x & 31;
    for (int r = 0; r < c; ++r) {
        kth = warp_max(cur);
        unsigned hit = __ballot_sync(0xffffffffu, cur == kth);
        int first = __ffs(hit) - 1;
        if (lane == first) cur = -INFINITY;
    }
    return kth;
}

// ---------------------------------------------------------------- request validity
// Status bits of the parameters alone (the draft ids are checked separately).
__device__ __forceinline__ int params_status(const Args& a, const dspark_row_params_t& r) {
    const bool t_ok = isfinite(r.temperature) && r.temperature >= 0.f;
    const bool p_ok = r.top_p > 0.f && isfinite(r.top_p);
    if (!t_ok || !p_ok || r.top_k < 0 || r.num_drafts < 0 || r.num_drafts > a.Km ||
        !isfinite(r.presence_penalty) || !isfinite(r.frequency_penalty))
        return DSPARK_ROW_BAD_PARAMS;
    if (r.temperature > 0.f && r.num_drafts > 0 && a.q == nullptr) return DSPARK_ROW_BAD_PARAMS;
    return 0;
}

__device__ __forceinline__ bool has_penalty(const dspark_row_params_t& r) {
    return r.presence_penalty != 0.f || r.frequency_penalty != 0.f;
}

// Count of token `tok` at verify position j of request b (history + own draft prefix), from the
// request's penalty index: the tile's sorted history entries by binary search, then its
// draft-only entries; a tile whose list overflowed looks the history up directly.
__device__ __forceinline__ int token_count(const Args& a, int b, int j, int tok) {
    const long long pt = static_cast<long long>(b) * a.tiles_x + tok / a.tile_x;
    const PenHdr h = a.pen_hdr[pt];
    if (!h.overflow) {
        const PenEntry* ent = a.pen_ent + pt * kPenCap;
        const int nh = h.pad[0];
        int l = 0, hi = nh;
        while (l < hi) { const int m = (l + hi) >> 1; if (ent[m].token < tok) l = m + 1; else hi = m; }
        int e = -1;
        if (l < nh && ent[l].token == tok) e = l;
        else for (int k = nh; k < h.n; ++k) if (ent[k].token == tok) { e = k; break; }
        if (e < 0) return 0;
        const PenEntry pe = ent[e];
        const unsigned long long mask = (static_cast<unsigned long long>(pe.mask_hi) << 32) | pe.mask_lo;
        const unsigned long long low = (j >= 64) ? ~0ull : ((1ull << j) - 1ull);
        return pe.base + __popcll(mask & low);
    }
    int base = 0;
    const int hlo = a.h_off ? a.h_off[b] : 0, hhi = a.h_off ? a.h_off[b + 1] : 0;
    int l = hlo, hi = hhi;
    while (l < hi) { const int m = (l + hi) >> 1; if (a.h_ids[m] < tok) l = m + 1; else hi = m; }
    if (l < hhi && a.h_ids[l] == tok) base = a.h_cnt[l];
    for (int q = 0; q < j; ++q) base += (a.d[static_cast<long long>(b) * a.Km + q] == tok);
    return base;
}

// Penalty-index bits of tokens [e0, e0 + n) of request b, n <= 16 (bit q: token e0 + q): one or
// two bitmap words for each vocab tile the range touches.
__device__ __forceinline__ unsigned pen_bits_range(const Args& a, int b, int e0, int n) {
    unsigned bits = 0u;
    for (int e = e0; e < e0 + n;) {
        const int tile = e / a.tile_x, tl = e - tile * a.tile_x;
        const int cnt = min(e0 + n - e, a.tile_x - tl);
        const unsigned* bm = a.pen_bm + (static_cast<long long>(b) * a.tiles_x + tile) * a.bm_words;
        const int w0 = tl >> 5, sh = tl & 31;
        unsigned long long win = bm[w0];
        if (sh + cnt > 32) win |= static_cast<unsigned long long>(bm[w0 + 1]) << 32;
        bits |= (static_cast<unsigned>(win >> sh) & ((1u << cnt) - 1u)) << (e - e0);
        e += cnt;
    }
    return bits;
}

// Draft probability input (before temperature and truncation) of target token t in draft row
// qs = b*Km + i, whatever the layout: the dense entry, the reduced row's entry of the draft id
// standing for t, or the sparse entry with id t (0 where the row has none).
__device__ __forceinline__ float draft_value(const Args& a, long long qs, int t) {
    if (a.q_layout == kQDense) return __ldg(a.q + qs * a.V + t);
    if (a.q_layout == kQReduced) {
        const int e = __ldg(a.t2d + t);
        return e >= 0 ? __ldg(a.q + qs * a.Lq + e) : 0.f;
    }
    const int* ids = a.q_ids + qs * a.Lq;
    for (int e = 0; e < a.Lq; ++e)
        if (__ldg(ids + e) == t) return __ldg(a.q + qs * a.Lq + e);
    return 0.f;
}

// ---------------------------------------------------------------- launchers (one per .cu)
// Launch `kern` on s; pdl: as a programmatic dependent of the previous kernel in s.
template <typename... KArgs, typename... Args2>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                            Args2&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args2>(args)...);
}

cudaError_t launch_prep(const Args& a, cudaStream_t s);
cudaError_t launch_row_finalize_warp(const Args& a, cudaStream_t s, bool pdl);
cudaError_t launch_stream_stats(const Args& a, cudaStream_t s, int grid, bool pdl);
cudaError_t launch_row_finalize(const Args& a, cudaStream_t s);
cudaError_t launch_accept(const Args& a, cudaStream_t s);
cudaError_t launch_logprobs(const Args& a, cudaStream_t s);

}  // namespace dspark
