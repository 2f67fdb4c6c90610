// accept_kernel: one CTA per request.  The acceptance decisions of all drafted positions
// are independent given the rows' truncated distributions, so thread i takes position i:
//   greedy (T = 0): accept iff d_i equals the penalised argmax of target row i (lowest id
//     on ties); the accepted length is the first mismatch (mlx-dspark Changelog, [0.2.0]
//     Changed: cumprod of positionwise matches);
//   T > 0: accept iff u_i < P'_i(d_i) / Q'_i(d_i), always when Q'_i(d_i) = 0 < P'_i(d_i)
//     (v0.0.2 release notes, Highlights: accept with probability min(1, p/q)).
// At the first rejection a the residual max(0, P'_a - Q'_a) is drawn from, or P'_K when all
// K drafts were accepted; greedy emits the argmax.  When the target row's support is a short
// list the draw happens here: weights in double, ids sorted ascending, an exclusive scan, and
// the smallest id whose cumulative mass exceeds u * total.  Whole-vocabulary supports are
// drawn afterwards by the same CTA (finish_request).
//
// A request with an end-of-sequence token stops at the first accepted draft equal to it: its
// accepted length counts that draft, and nothing is drawn (mlx-dspark Changelog, [0.2.0]
// Fixed: stop when an accepted draft is eos mid-block).  Per-position counters record, for
// each draft position, the requests that verified it and those that accepted it (Changelog,
// [0.9.0] Added: per-position acceptance with honest denominators).
//
// The request's emitted positions are listed for the logprob pass (logprob_kernel).
//
// finish_request, at the end of the same CTA: whole-row inverse-CDF draws (every thread sums
// the weights of a contiguous range of ids, a block scan of those sums finds the range holding
// the draw, and its thread walks it), then the logprob outputs past the last emitted position
// (-inf, top ids -1); the emitted positions' values come from logprob_kernel.
#include "block_utils.cuh"

namespace dspark {

namespace {

constexpr int kAcceptThreads = 512;

struct AccSmem {
    int acc[DSPARK_MAX_K + 1];
    unsigned long long sk[kKeptCap];
    double r[kKeptCap];
    double rs[kKeptCap];
    double ex[kKeptCap + 1];
    double dwarp[33];
    int iwarp[32];
    int a;
    int tok;
};

__device__ __forceinline__ int prefix_count(const Args& a, int b, int i, int t) {
    int c = 0;
    for (int q = 0; q < i; ++q) c += (a.d[static_cast<long long>(b) * a.Km + q] == t);
    return c;
}

// Target probability P'_j(d_j) of the drafted token at position j (0 outside the support).
// Its count is the history count recorded by the penalty index plus the draft prefix.
__device__ __forceinline__ double target_prob_of_draft(const Args& a, const XRowOut& xo, int b, int j, int t,
                                                       const dspark_row_params_t& r) {
    const long long slot = static_cast<long long>(b) * (a.Km + 1) + j;
    const float xv = load_x(a.x, a.sx, slot * a.V + t);
    int c = 0;
    if (has_penalty(r)) c = a.draft_base[static_cast<long long>(b) * a.Km + j] + prefix_count(a, b, j, t);
    const float xp = penalise(xv, c, r.frequency_penalty, r.presence_penalty);
    if (!(xp >= xo.tau)) return 0.0;
    return static_cast<double>(target_weight(xp, xo.m_pen, xo.c_l2e)) / xo.Z;
}

__device__ __forceinline__ double draft_prob(const Args& a, const QRowOut& qo, int b, int i, int t, bool t_one) {
    const long long qs = static_cast<long long>(b) * a.Km + i;
    const float qv = draft_value(a, qs, t);
    if (!(qv >= qo.tau)) return 0.0;
    return static_cast<double>(draft_weight(qv, qo.qmax, qo.inv_t, t_one)) / qo.Z;
}

__device__ void write_error(const Args& a, int b, int st) {
    const int tid = threadIdx.x;
    const int W = a.Km + 1;
    for (int j = tid; j < W; j += blockDim.x) {
        a.out_tokens[static_cast<long long>(b) * W + j] = -1;
        if (a.out_lp) a.out_lp[static_cast<long long>(b) * W + j] = -INFINITY;
    }
    for (int e = tid; e < W * a.n_top; e += blockDim.x) {
        if (a.out_top_ids) a.out_top_ids[static_cast<long long>(b) * W * a.n_top + e] = -1;
        if (a.out_top_lp) a.out_top_lp[static_cast<long long>(b) * W * a.n_top + e] = -INFINITY;
    }
    if (tid == 0) {
        a.out_accept[b] = -1;
        a.row_status[b] = st;
        if (a.out_stopped) a.out_stopped[b] = 0;
        a.req[b] = ReqOut{-1, 0, st, 0};
    }
}

// ============================================================================ finish
constexpr int kFinishThreads = 512;
static_assert(kFinishThreads == kAcceptThreads, "the whole-row draw runs in the acceptance CTA");

struct FinishSmem {
    double dwarp[33];
    double th_ex[kFinishThreads + 1];
    double th_sum[kFinishThreads];
    int sp_ids[DSPARK_MAX_SPARSE_M];      // a sparse draft row, ids ascending
    float sp_val[DSPARK_MAX_SPARSE_M];
    int found_chunk;
    int tok;
};

struct DrawCtx {
    const Args* a;
    int b, row_j;
    long long xslot, qslot;
    XRowOut xo;
    QRowOut qo;
    bool residual, t_one, pen, use_p_only;
    float f, p;
    float inv_zp, inv_zq;      // 1/Z of the target and draft supports (Z lies in [1, V])
    const int* sp_ids;         // sparse draft row (shared memory), ids ascending
    const float* sp_val;
    int sp_m;
};

// Draft input of token t at the draw row: a binary search of the staged sparse row, else the
// dense or reduced row.
__device__ __forceinline__ float draw_q(const DrawCtx& c, int t) {
    if (c.a->q_layout != kQSparse) return draft_value(*c.a, c.qslot, t);
    int l = 0, h = c.sp_m;
    while (l < h) { const int m = (l + h) >> 1; if (c.sp_ids[m] < t) l = m + 1; else h = m; }
    return (l < c.sp_m && c.sp_ids[l] == t) ? c.sp_val[l] : 0.f;
}

// Residual (or target) weight of token t of the draw row.  Per element in float (FP64 is
// slow on this part); sums over elements are compensated or taken in double.
__device__ __forceinline__ float draw_weight_of(const DrawCtx& c, int t, float xv, float qv, bool penalised) {
    if (penalised) xv = penalise(xv, token_count(*c.a, c.b, c.row_j, t), c.f, c.p);
    float P = 0.f;
    if (xv >= c.xo.tau) P = target_weight(xv, c.xo.m_pen, c.xo.c_l2e) * c.inv_zp;
    if (!c.residual || c.use_p_only) return P;
    float Q = 0.f;
    if (qv >= c.qo.tau) Q = draft_weight(qv, c.qo.qmax, c.qo.inv_t, c.t_one) * c.inv_zq;
    return fmaxf(0.f, P - Q);
}

// Sum of the weights of [r0, r1) (Kahan-compensated float), sixteen loads at a time.
__device__ double range_sum(const DrawCtx& c, int r0, int r1) {
    const Args& a = *c.a;
    const bool need_q = c.residual && !c.use_p_only;
    float sum = 0.f, comp = 0.f;
    for (int e0 = r0; e0 < r1; e0 += 16) {
        float xv[16], qv[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const int e = e0 + q;
            xv[q] = e < r1 ? load_x(a.x, a.sx, c.xslot * a.V + e) : -INFINITY;
            qv[q] = (need_q && e < r1) ? draw_q(c, e) : 0.f;
        }
        const unsigned pb = c.pen ? pen_bits_range(a, c.b, e0, min(16, r1 - e0)) : 0u;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float w = e0 + q < r1 ? draw_weight_of(c, e0 + q, xv[q], qv[q], (pb >> q) & 1u) : 0.f;
            const float y = w - comp;
            const float t = sum + y;
            comp = (t - sum) - y;
            sum = t;
        }
    }
    return static_cast<double>(sum) - static_cast<double>(comp);
}

// Inverse-CDF draw over the whole row: the smallest token whose cumulative weight exceeds
// u * total (ascending ids).  Each thread sums a contiguous range; a block scan of the range
// sums finds the range holding the draw, whose thread walks it in double.  An all-zero
// residual draws from the target row instead.
__device__ int whole_row_draw(FinishSmem& s, DrawCtx& c, float u) {
    const Args& a = *c.a;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int span = (a.V + nt - 1) / nt;
    const int r0 = min(a.V, tid * span), r1 = min(a.V, r0 + span);
    for (int attempt = 0; attempt < 2; ++attempt) {
        const double mine = range_sum(c, r0, r1);
        s.th_sum[tid] = mine;
        __syncthreads();
        block_scan_excl_d(s.th_sum, s.th_ex, nt, s.dwarp);
        const double total = s.th_ex[nt];
        if (!(total > 0.0) && c.residual && !c.use_p_only) {
            c.use_p_only = true;
            __syncthreads();
            continue;
        }
        const double target = static_cast<double>(u) * total;
        if (tid == 0) { s.found_chunk = nt; s.tok = -1; }
        __syncthreads();
        const double ex = s.th_ex[tid];
        if (mine > 0.0 && ex + mine > target) atomicMin(&s.found_chunk, tid);
        __syncthreads();
        int owner = s.found_chunk;
        __syncthreads();                                // every thread has read it before it changes
        if (owner == nt) {                              // rounding: the last range with mass
            if (tid == 0) {
                int last = -1;
                for (int t = nt - 1; t >= 0; --t) if (s.th_sum[t] > 0.0) { last = t; break; }
                s.found_chunk = last;
            }
            __syncthreads();
            owner = s.found_chunk;
        }
        if (owner < 0) return -1;
        // the owner's range, one element per thread (span <= blockDim whenever V <= blockDim^2;
        // otherwise in rounds), scanned in double in id order
        const double before = s.th_ex[owner];
        const int o0 = min(a.V, owner * span), o1 = min(a.V, o0 + span);
        __syncthreads();                                // found_chunk and th_ex[owner] read by all
        if (tid == 0) { s.found_chunk = a.V; s.tok = -1; }
        double run = before;
        for (int base = o0; base < o1; base += nt) {
            const int e = base + tid;
            float w = 0.f;
            if (e < o1) {
                const float qv = (c.residual && !c.use_p_only) ? draw_q(c, e) : 0.f;
                w = draw_weight_of(c, e, load_x(a.x, a.sx, c.xslot * a.V + e), qv,
                                   c.pen && (pen_bits_range(a, c.b, e, 1) & 1u));
            }
            __syncthreads();
            s.th_sum[tid] = static_cast<double>(w);
            __syncthreads();
            block_scan_excl_d(s.th_sum, s.th_ex, nt, s.dwarp);
            const double ex = run + s.th_ex[tid];
            if (w > 0.f && ex + static_cast<double>(w) > target) atomicMin(&s.found_chunk, e);
            if (w > 0.f) atomicMax(&s.tok, e);                 // last element with mass so far
            run += s.th_ex[nt];
            __syncthreads();
            if (s.found_chunk < a.V) break;
        }
        const int tok = s.found_chunk < a.V ? s.found_chunk : s.tok;
        __syncthreads();
        return tok;
    }
    return -1;
}

// The request's whole-row draw (when one is pending) and the logprob outputs past its last
// emitted position; the same CTA, after the acceptance decisions.
__device__ void finish_request(const Args& a, FinishSmem& s, int b, const ReqOut ro) {
    const int tid = threadIdx.x;
    const int W = a.Km + 1;
    const long long xs0 = static_cast<long long>(b) * W;
    const int acc_len = ro.a;
    if (ro.draw) {
        const dspark_row_params_t r = a.rows[b];
        DrawCtx c;
        c.a = &a;
        c.b = b;
        c.row_j = acc_len;
        c.xslot = xs0 + acc_len;
        c.qslot = static_cast<long long>(b) * a.Km + acc_len;
        c.xo = a.xout[c.xslot];
        c.residual = ro.draw == 1;
        if (c.residual) c.qo = a.qout[c.qslot];
        c.t_one = r.temperature == 1.f;
        c.pen = has_penalty(r);
        c.use_p_only = false;
        c.f = r.frequency_penalty;
        c.p = r.presence_penalty;
        c.inv_zp = c.xo.Z > 0.0 ? static_cast<float>(1.0 / c.xo.Z) : 0.f;
        c.inv_zq = (c.residual && c.qo.Z > 0.0) ? static_cast<float>(1.0 / c.qo.Z) : 0.f;
        c.sp_ids = s.sp_ids;
        c.sp_val = s.sp_val;
        c.sp_m = 0;
        if (c.residual && a.q_layout == kQSparse) {
            // stage the sparse row sorted by id (ids of a valid row are distinct): rank = ids below
            const int m = a.Lq;
            const int* ids = a.q_ids + c.qslot * m;
            for (int e = tid; e < m; e += blockDim.x) {
                const int id = ids[e];
                int rank = 0;
                for (int k = 0; k < m; ++k) rank += ids[k] < id;
                s.sp_ids[rank] = id;
                s.sp_val[rank] = a.q[c.qslot * m + e];
            }
            c.sp_m = m;
            __syncthreads();
        }
        const int tok = whole_row_draw(s, c, a.u[(xs0 + acc_len) * 2 + 1]);
        if (tid == 0) a.out_tokens[xs0 + acc_len] = tok;
        __syncthreads();
    }
    // ---- logprob outputs past the last emitted token (the emitted positions: logprob_kernel)
    const int n_em = ro.stopped ? acc_len : acc_len + 1;
    if (a.out_lp)
        for (int j = n_em + tid; j < W; j += blockDim.x) a.out_lp[xs0 + j] = -INFINITY;
    for (int e = n_em * a.n_top + tid; e < W * a.n_top; e += blockDim.x) {
        if (a.out_top_ids) a.out_top_ids[xs0 * a.n_top + e] = -1;
        if (a.out_top_lp) a.out_top_lp[xs0 * a.n_top + e] = -INFINITY;
    }
}

// The acceptance kernel's shared memory: the list draw's arrays, then (reused) the whole-row
// draw's.
union AcceptSmem {
    AccSmem acc;
    FinishSmem fin;
};

__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(Args a) {
    pdl_enter();
    extern __shared__ __align__(16) unsigned char acc_raw[];
    AcceptSmem& su = *reinterpret_cast<AcceptSmem*>(acc_raw);
    AccSmem& s = su.acc;
    const int b = blockIdx.x, tid = threadIdx.x;
    int st = a.row_status[b];
    const dspark_row_params_t r = a.rows[b];
    // a d2t table that does not invert makes every sampled request with drafts invalid
    if (a.q_layout == kQReduced && a.plan->pad[1] && !(st & DSPARK_ROW_BAD_PARAMS) && r.temperature > 0.f &&
        r.num_drafts > 0)
        st |= DSPARK_ROW_BAD_DRAFT;
    // an invalid request reports what is wrong with its inputs, not what its rows then gave
    if (st & (DSPARK_ROW_BAD_PARAMS | DSPARK_ROW_BAD_HISTORY | DSPARK_ROW_BAD_DRAFT)) st &= ~DSPARK_ROW_NONFINITE;
    if (a.plan->pad[0]) st |= DSPARK_ROW_INTERNAL;
    if (st) { write_error(a, b, st); return; }
    const int K = r.num_drafts;
    const bool greedy = !(r.temperature > 0.f);
    const bool t_one = r.temperature == 1.f;
    const int W = a.Km + 1;
    const long long xs0 = static_cast<long long>(b) * W;
    const long long qs0 = static_cast<long long>(b) * a.Km;
    // ---- acceptance decisions, one thread per drafted position
    if (tid < K) {
        const int t = a.d[qs0 + tid];
        bool ok;
        if (greedy) {
            ok = (t == a.xout[xs0 + tid].argmax);
        } else {
            const XRowOut xo = a.xout[xs0 + tid];
            const QRowOut qo = a.qout[qs0 + tid];
            const double P = target_prob_of_draft(a, xo, b, tid, t, r);
            const double Q = draft_prob(a, qo, b, tid, t, t_one);
            const double u = static_cast<double>(a.u[(xs0 + tid) * 2 + 0]);
            ok = (Q == 0.0) ? (P > 0.0) : (u < P / Q);
        }
        s.acc[tid] = ok ? 1 : 0;
    }
    __syncthreads();
    int first = K;
    if (tid < K && !s.acc[tid]) first = tid;
    const int verified = block_min_i(first, s.iwarp);     // accepted drafts before any stop
    // ---- end-of-sequence stop: the first accepted draft equal to the request's eos token
    const int eos = a.eos ? a.eos[b] : -1;
    int stop_at = W;
    if (eos >= 0 && tid < verified && a.d[qs0 + tid] == eos) stop_at = tid;
    stop_at = block_min_i(stop_at, s.iwarp);
    const bool stopped = stop_at < verified;
    const int acc_len = stopped ? stop_at + 1 : verified;
    // ---- per-position counters: verified positions (the first rejected one included), accepted ones
    if (a.pos_counts && tid < K) {
        const bool attempted = stopped ? tid < acc_len : tid <= verified;
        if (attempted) atomicAdd(a.pos_counts + tid, 1ull);
        if (tid < acc_len) atomicAdd(a.pos_counts + a.Km + tid, 1ull);
    }
    // ---- the emitted token at position acc_len (none after a stop)
    int draw = 0;
    int tok = -1;
    const XRowOut xa = a.xout[xs0 + acc_len];
    if (stopped) {
        // nothing to draw
    } else if (greedy) {
        tok = xa.argmax;
    } else if (xa.mode == kModeList && xa.n_kept <= 64) {
        // a short kept list: one warp, two entries per lane, sorted by id in registers, scanned
        // with shuffles (the block-wide sort and scans below cost a barrier per step)
        if (tid < 32) {
            const int lane = tid;
            const int n = xa.n_kept;
            const bool residual = acc_len < K;
            QRowOut qa{};
            if (residual) qa = a.qout[qs0 + acc_len];
            const KeptEntry* kl = a.kept + (xs0 + acc_len) * kKeptCap;
            unsigned long long key[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int e = lane + 32 * h;
                key[h] = 0ull;
                if (e < n) {
                    const KeptEntry ke = kl[e];
                    const double P = static_cast<double>(ke.w) / xa.Z;
                    double rv = P;
                    if (residual) rv = fmax(0.0, P - draft_prob(a, qa, b, acc_len, ke.id, t_one));
                    s.r[e] = rv;
                    key[h] = (static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<unsigned>(ke.id)) << 32) |
                             static_cast<unsigned>(e);
                }
            }
            __syncwarp();
            // bitonic sort of the 64 keys, descending (= ids ascending); key h of lane l sits at l + 32h
            for (int size = 2; size <= 64; size <<= 1)
                for (int stride = size >> 1; stride > 0; stride >>= 1) {
                    if (stride == 32) {
                        const unsigned long long hi = key[0] > key[1] ? key[0] : key[1];
                        const unsigned long long lo = key[0] > key[1] ? key[1] : key[0];
                        key[0] = hi;
                        key[1] = lo;
                    } else {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int pos = lane + 32 * h;
                            const unsigned long long o = __shfl_xor_sync(0xffffffffu, key[h], stride);
                            const bool keep_max = ((pos & stride) == 0) == ((pos & size) == 0);
                            key[h] = keep_max ? (key[h] > o ? key[h] : o) : (key[h] < o ? key[h] : o);
                        }
                    }
                }
            // weights in id order (position p = lane + 32h), inclusive scans of each half
            auto scan = [&](bool from_p, double (&w)[2], double (&inc)[2]) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int pos = lane + 32 * h;
                    const int idx = static_cast<int>(key[h] & 0xFFFFFFFFull);
                    w[h] = pos < n ? (from_p ? static_cast<double>(kl[idx].w) / xa.Z : s.r[idx]) : 0.0;
                    double v = w[h];
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const double y = __shfl_up_sync(0xffffffffu, v, o);
                        if (lane >= o) v += y;
                    }
                    inc[h] = v;
                }
                inc[1] += __shfl_sync(0xffffffffu, inc[0], 31);
                return __shfl_sync(0xffffffffu, inc[1], 31);
            };
            double w[2], inc[2];
            double total = scan(false, w, inc);
            if (!(total > 0.0)) total = scan(true, w, inc);      // empty residual: draw from P'
            const double target = static_cast<double>(a.u[(xs0 + acc_len) * 2 + 1]) * total;
            // exclusive prefix = the inclusive prefix one position down, so the intervals tile [0, total)
            double ex0 = __shfl_up_sync(0xffffffffu, inc[0], 1), ex1 = __shfl_up_sync(0xffffffffu, inc[1], 1);
            const double top0 = __shfl_sync(0xffffffffu, inc[0], 31);
            if (lane == 0) { ex0 = 0.0; ex1 = top0; }
            const unsigned h0 = __ballot_sync(0xffffffffu, inc[0] > target && ex0 <= target && lane < n);
            const unsigned h1 = __ballot_sync(0xffffffffu, inc[1] > target && ex1 <= target && lane + 32 < n);
            int pos = h0 ? __ffs(h0) - 1 : (h1 ? 32 + __ffs(h1) - 1 : -1);
            if (pos < 0) {                                    // rounding put u*total at the very top
                const unsigned m0 = __ballot_sync(0xffffffffu, w[0] > 0.0), m1 = __ballot_sync(0xffffffffu, w[1] > 0.0);
                pos = m1 ? 32 + 31 - __clz(m1) : (m0 ? 31 - __clz(m0) : -1);
            }
            const unsigned long long kp0 = __shfl_sync(0xffffffffu, key[0], pos & 31);
            const unsigned long long kp1 = __shfl_sync(0xffffffffu, key[1], pos & 31);
            const unsigned long long kp = pos >= 32 ? kp1 : kp0;
            if (lane == 0) s.tok = pos >= 0 ? static_cast<int>(0xFFFFFFFFu - static_cast<unsigned>(kp >> 32)) : -1;
        }
        __syncthreads();
        tok = s.tok;
    } else if (xa.mode == kModeList) {
        const int n = xa.n_kept;
        const bool residual = acc_len < K;
        QRowOut qa{};
        if (residual) qa = a.qout[qs0 + acc_len];
        const KeptEntry* kl = a.kept + (xs0 + acc_len) * kKeptCap;
        for (int e = tid; e < n; e += blockDim.x) {
            const KeptEntry ke = kl[e];
            const double P = static_cast<double>(ke.w) / xa.Z;
            double rv = P;
            if (residual) rv = fmax(0.0, P - draft_prob(a, qa, b, acc_len, ke.id, t_one));
            s.r[e] = rv;
            s.sk[e] = (static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<unsigned>(ke.id)) << 32) |
                      static_cast<unsigned>(e);
        }
        const int P2 = next_pow2(max(n, 2));
        for (int e = n + tid; e < P2; e += blockDim.x) s.sk[e] = 0ull;
        block_bitonic_desc(s.sk, P2);                   // ascending token id
        for (int e = tid; e < n; e += blockDim.x) s.rs[e] = s.r[s.sk[e] & 0xFFFFFFFFull];
        __syncthreads();
        block_scan_excl_d(s.rs, s.ex, n, s.dwarp);
        if (!(s.ex[n] > 0.0)) {                          // empty residual: draw from P'
            for (int e = tid; e < n; e += blockDim.x)
                s.rs[e] = static_cast<double>(kl[s.sk[e] & 0xFFFFFFFFull].w) / xa.Z;
            __syncthreads();
            block_scan_excl_d(s.rs, s.ex, n, s.dwarp);
        }
        const double target = static_cast<double>(a.u[(xs0 + acc_len) * 2 + 1]) * s.ex[n];
        if (tid == 0) s.tok = -1;
        __syncthreads();
        for (int e = tid; e < n; e += blockDim.x)
            if (s.ex[e + 1] > target && s.ex[e] <= target) s.tok = e;
        __syncthreads();
        int pos = s.tok;
        if (pos < 0) {                                    // rounding put u*total at the very top
            int last = -1;
            for (int e = tid; e < n; e += blockDim.x) if (s.rs[e] > 0.0) last = max(last, e);
            pos = -block_min_i(-last, s.iwarp);
        }
        tok = pos >= 0 ? static_cast<int>(0xFFFFFFFFu - static_cast<unsigned>(s.sk[pos] >> 32)) : -1;
    } else {
        draw = (acc_len < K) ? 1 : 2;                     // whole-row draw in finish_request
    }
    for (int j = tid; j < W; j += blockDim.x) {
        int v = -1;
        if (j < acc_len) v = a.d[qs0 + j];
        else if (j == acc_len) v = tok;
        a.out_tokens[xs0 + j] = v;
    }
    if (tid == 0) {
        a.out_accept[b] = acc_len;
        if (a.out_stopped) a.out_stopped[b] = stopped ? 1 : 0;
        a.req[b] = ReqOut{acc_len, draw, 0, stopped ? 1 : 0};
        if (a.want_lp || a.n_top > 0) {                     // rows of the logprob pass
            const int n_em = stopped ? acc_len : acc_len + 1;
            const int base = atomicAdd(&a.lp_list[0], n_em);
            for (int j = 0; j < n_em; ++j) a.lp_list[1 + base + j] = static_cast<int>(xs0) + j;
        }
    }
    __syncthreads();                                      // the list draw's shared memory is free
    finish_request(a, su.fin, b, ReqOut{acc_len, draw, 0, stopped ? 1 : 0});
}

}  // namespace

cudaError_t launch_accept(const Args& a, cudaStream_t s) {
    const size_t smem = sizeof(AcceptSmem);
    cudaError_t e = cudaFuncSetAttribute(accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_k(accept_kernel, dim3(a.B), dim3(kAcceptThreads), smem, s, true, a);
}

}  // namespace dspark
