// stream_stats_kernel: the single HBM pass over the target logits x and the draft
// probabilities q.  Everything else in the epilogue works on what this pass leaves behind.
//
// Persistent: one CTA per SM walks the flat list of work units (one vocab tile of one row
// each).  A producer warp moves each tile into a 3-stage shared-memory ring with the TMA
// bulk-copy engine (cp.async.bulk, completion counted on an mbarrier), together with the
// tile's penalty bitmap and penalised-token list; 16 consumer warps read the tile from
// shared memory twice:
//   pass 1: per-thread maxima of the raw logits and of the penalised logits
//           (x' = x - ((f*c) + p), mlx-dspark Changelog [0.2.0] Added, penalties);
//   then    a lower bound theta on the tile's k-th largest value: every warp finds the
//           c-th largest of its lanes' maxima (c = ceil(k / 16)), theta = the least of
//           them, so at least 16*c >= k distinct logits of the tile are >= theta;
//   pass 2: raw sum of exp (for the log-softmax of logprobs), the tempered sum when the row
//           has no top-k, the lowest index attaining the penalised max (greedy), and the
//           candidates >= theta (for the top-k threshold of the row, mlx-dspark Changelog
//           [0.20.2] Changed: the threshold comes from small selections, not a full sort).
// Draft tiles get the same treatment with q as the key (top-k of q^(1/T) is top-k of q).
#include "dspark_internal.cuh"

namespace dspark {

namespace {

constexpr long long kWaitLimit = 1ll << 22;
constexpr float kL2E = 1.4426950408889634f;

struct StageMeta {
    int kind, slot, b, j;
    int tile, e0, e1, nvec;
    int vec_e0, pen, pen_n, pen_nh;
    int pen_over, top_k, pad0, pad1;
    float temperature, top_p, presence, frequency;
};

struct Smem {
    alignas(128) unsigned char data[kStages][kStageBytes];
    alignas(16) unsigned bm[kStages][kBitmapWordsMax];
    alignas(16) PenEntry ent[kStages][kPenCap];
    StageMeta meta[kStages];
    Cand cpen[2][kSmemCandPen];
    Cand craw[2][kSmemCandRaw];
    float red1[2][kConsumerWarps][4];
    float red2[2][kConsumerWarps][4];
    int cnt_pen[2];
    int cnt_raw[2];
    alignas(8) uint64_t full[kStages];
    alignas(8) uint64_t empty[kStages];
    int error;
};

__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Count of token `tok` at verify position j: history base + draft prefix occurrences.
__device__ __forceinline__ int pen_count(const Smem& sm, int stage, const StageMeta& m, const Args& a, int tok) {
    if (!m.pen_over) {
        const PenEntry* ent = sm.ent[stage];
        int l = 0, h = m.pen_nh;
        while (l < h) { const int md = (l + h) >> 1; if (ent[md].token < tok) l = md + 1; else h = md; }
        int e = -1;
        if (l < m.pen_nh && ent[l].token == tok) e = l;
        else for (int k = m.pen_nh; k < m.pen_n; ++k) if (ent[k].token == tok) { e = k; break; }
        if (e < 0) return 0;
        const unsigned long long mask = (static_cast<unsigned long long>(ent[e].mask_hi) << 32) | ent[e].mask_lo;
        const unsigned long long low = (m.j >= 64) ? ~0ull : ((1ull << m.j) - 1ull);
        return ent[e].base + __popcll(mask & low);
    }
    // overflowed tile: look the token up in the caller's history and the draft prefix
    int base = 0;
    const int hlo = a.h_off ? a.h_off[m.b] : 0, hhi = a.h_off ? a.h_off[m.b + 1] : 0;
    int l = hlo, h = hhi;
    while (l < h) { const int md = (l + h) >> 1; if (a.h_ids[md] < tok) l = md + 1; else h = md; }
    if (l < hhi && a.h_ids[l] == tok) base = a.h_cnt[l];
    for (int i = 0; i < m.j; ++i) base += (a.d[static_cast<long long>(m.b) * a.Km + i] == tok);
    return base;
}

__device__ __forceinline__ unsigned bitmap_bits(const unsigned* bm, int off, int n) {
    // n (<= 8) bits of the tile bitmap starting at bit `off`
    const int w = off >> 5, s = off & 31;
    unsigned long long two = bm[w];
    if (s + n > 32) two |= static_cast<unsigned long long>(bm[w + 1]) << 32;
    return static_cast<unsigned>(two >> s) & ((1u << n) - 1u);
}

template <int SX>
__device__ __forceinline__ float elem(const uint4& w, int k) {
    if (SX == 2) {
        const uint32_t word = (k < 2) ? w.x : (k < 4) ? w.y : (k < 6) ? w.z : w.w;
        return (k & 1) ? bf16_hi(word) : bf16_lo(word);
    } else {
        const uint32_t word = (k == 0) ? w.x : (k == 1) ? w.y : (k == 2) ? w.z : w.w;
        return __uint_as_float(word);
    }
}

// Maximum (NaN-propagating) of the elements of one 16-byte vector.
template <int SX>
__device__ __forceinline__ float vec_max(const uint4& w) {
    if (SX == 2) {
        __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w.x);
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w.y);
        __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&w.z);
        __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&w.w);
        __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
        const uint32_t mw = *reinterpret_cast<const uint32_t*>(&m);
        return max_nan(bf16_lo(mw), bf16_hi(mw));
    } else {
        return max_nan(max_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                       max_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
}

__device__ __forceinline__ void push(Cand* buf, int* cnt, int cap, float v, int id) {
    const int p = atomicAdd(cnt, 1);
    if (p < cap) buf[p] = Cand{v, id};
}

// ------------------------------------------------------------------ one target-logit tile
template <int SX>
__device__ void process_x(const Args& a, Smem& sm, int stage, const StageMeta& m, int cb) {
    constexpr int EPV = 16 / SX;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned char* data = sm.data[stage];
    const unsigned* bm = sm.bm[stage];
    const bool greedy = !(m.temperature > 0.f);
    const int k = m.top_k;
    const bool need_lp = a.want_lp || a.n_top > 0;
    const bool need_raw = a.n_top > 0;
    const bool need_cand = !greedy && k > 0 && k < a.V && k <= kMaxCandTopK;
    const bool need_temp = !greedy && (k == 0 || k >= a.V);
    const float f = m.frequency, p = m.presence;
    const long long xrow = static_cast<long long>(m.slot) * a.V;
    const int e_tail = m.vec_e0 + m.nvec * EPV;

    // ---- pass 1: maxima
    float mu = -INFINITY;          // unpenalised elements (raw == penalised)
    float mpen = -INFINITY;        // penalised elements, penalised value
    float mrawp = -INFINITY;       // penalised elements, raw value
    for (int v = tid; v < m.nvec; v += kConsumerThreads) {
        const uint4 w = *reinterpret_cast<const uint4*>(data + v * 16);
        const int e = m.vec_e0 + v * EPV;
        const unsigned bits = m.pen ? bitmap_bits(bm, e - m.e0, EPV) : 0u;
        if (bits == 0u) {
            mu = max_nan(mu, vec_max<SX>(w));
        } else {
#pragma unroll
            for (int q = 0; q < EPV; ++q) {
                const float xv = elem<SX>(w, q);
                if (bits & (1u << q)) {
                    const float xp = penalise(xv, pen_count(sm, stage, m, a, e + q), f, p);
                    mpen = max_nan(mpen, xp);
                    mrawp = max_nan(mrawp, xv);
                } else {
                    mu = max_nan(mu, xv);
                }
            }
        }
    }
    // head / tail elements outside the 16-byte-aligned interior: plain loads
    if (tid < 2) {
        const int lo = tid == 0 ? m.e0 : e_tail;
        const int hi = tid == 0 ? m.vec_e0 : m.e1;
        for (int e = lo; e < hi; ++e) {
            const float xv = load_x(a.x, SX, xrow + e);
            if (m.pen && ((bm[(e - m.e0) >> 5] >> ((e - m.e0) & 31)) & 1u)) {
                mpen = max_nan(mpen, penalise(xv, pen_count(sm, stage, m, a, e), f, p));
                mrawp = max_nan(mrawp, xv);
            } else {
                mu = max_nan(mu, xv);
            }
        }
    }
    const float lane_raw = max_nan(mu, mrawp);
    const float lane_pen = max_nan(mu, mpen);
    {
        float wr = lane_raw, wp = lane_pen;
        for (int o = 16; o; o >>= 1) {
            wr = max_nan(wr, __shfl_xor_sync(0xffffffffu, wr, o));
            wp = max_nan(wp, __shfl_xor_sync(0xffffffffu, wp, o));
        }
        const float thp = need_cand ? warp_kth_largest(lane_pen, (k + kConsumerWarps - 1) / kConsumerWarps) : 0.f;
        const float thr = need_raw ? warp_kth_largest(lane_raw, (a.n_top + kConsumerWarps - 1) / kConsumerWarps) : 0.f;
        if (lane == 0) {
            sm.red1[cb][warp][0] = wr; sm.red1[cb][warp][1] = wp;
            sm.red1[cb][warp][2] = thp; sm.red1[cb][warp][3] = thr;
        }
    }
    named_barrier_sync(1, kConsumerThreads);
    if (tid == 0) { sm.cnt_pen[cb ^ 1] = 0; sm.cnt_raw[cb ^ 1] = 0; }
    float m_raw = -INFINITY, m_pen = -INFINITY, th_p = INFINITY, th_r = INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
        m_raw = max_nan(m_raw, sm.red1[cb][w][0]);
        m_pen = max_nan(m_pen, sm.red1[cb][w][1]);
        th_p = fminf(th_p, sm.red1[cb][w][2]);
        th_r = fminf(th_r, sm.red1[cb][w][3]);
    }
    if (!need_cand) th_p = INFINITY;
    if (!need_raw) th_r = INFINITY;
    const float th_lo = fminf(th_p, th_r);
    const float mr_l2e = m_raw * kL2E;
    const float c_l2e = need_temp ? kL2E / m.temperature : 0.f;
    const bool raw_ok = isfinite(m_raw);

    // ---- pass 2: sums, greedy argmax, candidates
    float s_raw = 0.f, s_temp = 0.f;
    int arg = 0x7FFFFFFF;
    for (int v = tid; v < m.nvec; v += kConsumerThreads) {
        const uint4 w = *reinterpret_cast<const uint4*>(data + v * 16);
        const int e = m.vec_e0 + v * EPV;
        const unsigned bits = m.pen ? bitmap_bits(bm, e - m.e0, EPV) : 0u;
        if (need_lp && raw_ok) {
#pragma unroll
            for (int q = 0; q < EPV; ++q) s_raw += ex2_approx(fmaf(elem<SX>(w, q), kL2E, -mr_l2e));
        }
        if (bits == 0u) {
            if (need_temp) {
#pragma unroll
                for (int q = 0; q < EPV; ++q) s_temp += ex2_approx(__fsub_rn(elem<SX>(w, q), m_pen) * c_l2e);
            }
            const float vm = (greedy || th_lo < INFINITY) ? vec_max<SX>(w) : -INFINITY;
            if (greedy && vm >= m_pen && arg == 0x7FFFFFFF) {
#pragma unroll
                for (int q = 0; q < EPV; ++q)
                    if (elem<SX>(w, q) == m_pen) { arg = min(arg, e + q); }
            }
            if (vm >= th_lo) {
#pragma unroll
                for (int q = 0; q < EPV; ++q) {
                    const float xv = elem<SX>(w, q);
                    if (xv >= th_p) push(sm.cpen[cb], &sm.cnt_pen[cb], kSmemCandPen, xv, e + q);
                    if (xv >= th_r) push(sm.craw[cb], &sm.cnt_raw[cb], kSmemCandRaw, xv, e + q);
                }
            }
        } else {
#pragma unroll
            for (int q = 0; q < EPV; ++q) {
                const float xv = elem<SX>(w, q);
                const float xp = (bits & (1u << q)) ? penalise(xv, pen_count(sm, stage, m, a, e + q), f, p) : xv;
                if (need_temp) s_temp += ex2_approx(__fsub_rn(xp, m_pen) * c_l2e);
                if (greedy && xp == m_pen && arg == 0x7FFFFFFF) arg = e + q;
                if (xp >= th_p) push(sm.cpen[cb], &sm.cnt_pen[cb], kSmemCandPen, xp, e + q);
                if (xv >= th_r) push(sm.craw[cb], &sm.cnt_raw[cb], kSmemCandRaw, xv, e + q);
            }
        }
    }
    if (tid < 2) {
        const int lo = tid == 0 ? m.e0 : e_tail;
        const int hi = tid == 0 ? m.vec_e0 : m.e1;
        for (int e = lo; e < hi; ++e) {
            const float xv = load_x(a.x, SX, xrow + e);
            int c = 0;
            if (m.pen && ((bm[(e - m.e0) >> 5] >> ((e - m.e0) & 31)) & 1u)) c = pen_count(sm, stage, m, a, e);
            const float xp = penalise(xv, c, f, p);
            if (need_lp && raw_ok) s_raw += ex2_approx(fmaf(xv, kL2E, -mr_l2e));
            if (need_temp) s_temp += ex2_approx(__fsub_rn(xp, m_pen) * c_l2e);
            if (greedy && xp == m_pen) arg = min(arg, e);
            if (xp >= th_p) push(sm.cpen[cb], &sm.cnt_pen[cb], kSmemCandPen, xp, e);
            if (xv >= th_r) push(sm.craw[cb], &sm.cnt_raw[cb], kSmemCandRaw, xv, e);
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);    // the stage's shared memory is no longer read
    s_raw = warp_sum(s_raw);
    s_temp = warp_sum(s_temp);
    arg = warp_min_i(arg);
    if (lane == 0) {
        sm.red2[cb][warp][0] = s_raw; sm.red2[cb][warp][1] = s_temp;
        sm.red2[cb][warp][2] = __int_as_float(arg);
    }
    named_barrier_sync(1, kConsumerThreads);
    const int n_pen = sm.cnt_pen[cb], n_raw = sm.cnt_raw[cb];
    const long long ti = static_cast<long long>(m.slot) * a.tiles_x + m.tile;
    if (tid == 0) {
        float sr = 0.f, st = 0.f;
        int ag = 0x7FFFFFFF;
        for (int w = 0; w < kConsumerWarps; ++w) {
            sr += sm.red2[cb][w][0];
            st += sm.red2[cb][w][1];
            ag = min(ag, __float_as_int(sm.red2[cb][w][2]));
        }
        TileStats ts;
        ts.m_raw = m_raw; ts.s_raw = sr; ts.m_pen = m_pen; ts.arg_pen = ag; ts.s_temp = st;
        ts.flags = 0;
        ts.n_pen = need_cand ? n_pen : 0;
        ts.n_raw = need_raw ? n_raw : 0;
        if (need_cand && n_pen > kCandPenGlobal) { ts.flags |= kTileOverflowPen; ts.n_pen = 0; }
        if (need_raw && n_raw > kCandRawGlobal) { ts.flags |= kTileOverflowRaw; ts.n_raw = 0; }
        if (!isfinite(m_raw) || !isfinite(m_pen)) ts.flags |= kTileBad;
        a.ts_x[ti] = ts;
    }
    if (need_cand && n_pen <= kCandPenGlobal) {
        Cand* dst = a.cand_x + ti * kCandPenGlobal;
        for (int i = tid; i < n_pen; i += kConsumerThreads) dst[i] = sm.cpen[cb][i];
    }
    if (need_raw && n_raw <= kCandRawGlobal) {
        Cand* dst = a.cand_raw + ti * kCandRawGlobal;
        for (int i = tid; i < n_raw; i += kConsumerThreads) dst[i] = sm.craw[cb][i];
    }
}

// ------------------------------------------------------------------ one draft-probability tile
__device__ void process_q(const Args& a, Smem& sm, int stage, const StageMeta& m, int cb) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned char* data = sm.data[stage];
    const int k = m.top_k;
    const bool need_cand = k > 0 && k < a.V && k <= kMaxCandTopK;
    const bool need_sum = !need_cand && (k == 0 || k >= a.V);
    const bool t_one = m.temperature == 1.f;
    const long long qrow = static_cast<long long>(m.slot) * a.V;
    const int e_tail = m.vec_e0 + m.nvec * 4;
    float mx = -INFINITY, mn = INFINITY, sum = 0.f;
    for (int v = tid; v < m.nvec; v += kConsumerThreads) {
        const float4 w = *reinterpret_cast<const float4*>(data + v * 16);
        mx = max_nan(max_nan(mx, w.x), max_nan(w.y, max_nan(w.z, w.w)));
        mn = fminf(fminf(mn, w.x), fminf(w.y, fminf(w.z, w.w)));
        if (need_sum && t_one) sum += (w.x + w.y) + (w.z + w.w);
    }
    if (tid < 2) {
        const int lo = tid == 0 ? m.e0 : e_tail;
        const int hi = tid == 0 ? m.vec_e0 : m.e1;
        for (int e = lo; e < hi; ++e) {
            const float v = __ldg(a.q + qrow + e);
            mx = max_nan(mx, v); mn = fminf(mn, v);
            if (need_sum && t_one) sum += v;
        }
    }
    {
        float wm = mx, wn = mn;
        for (int o = 16; o; o >>= 1) {
            wm = max_nan(wm, __shfl_xor_sync(0xffffffffu, wm, o));
            wn = fminf(wn, __shfl_xor_sync(0xffffffffu, wn, o));
        }
        const float th = need_cand ? warp_kth_largest(mx, (k + kConsumerWarps - 1) / kConsumerWarps) : 0.f;
        if (lane == 0) {
            sm.red1[cb][warp][0] = wm; sm.red1[cb][warp][1] = wn;
            sm.red1[cb][warp][2] = th; sm.red1[cb][warp][3] = 0.f;
        }
    }
    named_barrier_sync(1, kConsumerThreads);
    if (tid == 0) { sm.cnt_pen[cb ^ 1] = 0; sm.cnt_raw[cb ^ 1] = 0; }
    float qmax = -INFINITY, qmin = INFINITY, th = INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
        qmax = max_nan(qmax, sm.red1[cb][w][0]);
        qmin = fminf(qmin, sm.red1[cb][w][1]);
        th = fminf(th, sm.red1[cb][w][2]);
    }
    if (!need_cand) th = INFINITY;
    const float inv_t = 1.f / m.temperature;
    float s_temp = 0.f;
    if (need_cand || (need_sum && !t_one)) {
        for (int v = tid; v < m.nvec; v += kConsumerThreads) {
            const float4 w = *reinterpret_cast<const float4*>(data + v * 16);
            const int e = m.vec_e0 + v * 4;
            if (need_sum && !t_one) {
                s_temp += draft_weight(w.x, qmax, inv_t, false) + draft_weight(w.y, qmax, inv_t, false) +
                          draft_weight(w.z, qmax, inv_t, false) + draft_weight(w.w, qmax, inv_t, false);
            }
            if (need_cand && max_nan(max_nan(w.x, w.y), max_nan(w.z, w.w)) >= th) {
                if (w.x >= th) push(sm.cpen[cb], &sm.cnt_pen[cb], kSmemCandPen, w.x, e);
                if (w.y >= th) push(sm.cpen[cb], &sm.cnt_pen[cb], kSmemCandPen, w.y, e + 1);
                if (w.z >= th) push(sm.cpen[cb], &sm.cnt_pen[cb], kSmemCandPen, w.z, e + 2);
                if (w.w >= th) push(sm.cpen[cb], &sm.cnt_pen[cb], kSmemCandPen, w.w, e + 3);
            }
        }
    }
    if (tid < 2 && (need_cand || (need_sum && !t_one))) {
        const int lo = tid == 0 ? m.e0 : e_tail;
        const int hi = tid == 0 ? m.vec_e0 : m.e1;
        for (int e = lo; e < hi; ++e) {
            const float v = __ldg(a.q + qrow + e);
            if (need_sum && !t_one) s_temp += draft_weight(v, qmax, inv_t, false);
            if (need_cand && v >= th) push(sm.cpen[cb], &sm.cnt_pen[cb], kSmemCandPen, v, e);
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);
    sum = warp_sum(sum);
    s_temp = warp_sum(s_temp);
    if (lane == 0) { sm.red2[cb][warp][0] = sum; sm.red2[cb][warp][1] = s_temp; }
    named_barrier_sync(1, kConsumerThreads);
    const int n = sm.cnt_pen[cb];
    const long long ti = static_cast<long long>(m.slot) * a.tiles_q + m.tile;
    if (tid == 0) {
        float s1 = 0.f, s2 = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) { s1 += sm.red2[cb][w][0]; s2 += sm.red2[cb][w][1]; }
        TileStats ts;
        ts.m_raw = qmax; ts.s_raw = s1; ts.m_pen = qmin; ts.arg_pen = 0; ts.s_temp = s2;
        ts.n_pen = need_cand ? n : 0; ts.n_raw = 0; ts.flags = 0;
        if (need_cand && n > kCandPenGlobal) { ts.flags |= kTileOverflowPen; ts.n_pen = 0; }
        if (!(qmin >= 0.f) || !(qmax <= 3.0e38f)) ts.flags |= kTileBad;
        a.ts_q[ti] = ts;
    }
    if (need_cand && n <= kCandPenGlobal) {
        Cand* dst = a.cand_q + ti * kCandPenGlobal;
        for (int i = tid; i < n; i += kConsumerThreads) dst[i] = sm.cpen[cb][i];
    }
}

// ------------------------------------------------------------------ the kernel
template <int SX>
__global__ void __launch_bounds__(kStreamThreads, 1) stream_stats_kernel(Args a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x;
    const int n_units = a.plan->n_units;
    const int G = gridDim.x;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.empty[s], kConsumerWarps); }
        sm.cnt_pen[0] = sm.cnt_pen[1] = 0;
        sm.cnt_raw[0] = sm.cnt_raw[1] = 0;
        sm.error = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (tid >= kConsumerThreads) {
        // ---------------- producer warp
        const int lane = tid & 31;
        int it = 0;
        bool failed = false;
        for (int base = blockIdx.x; base < n_units && !failed; base += 32 * G) {
            const int ul = base + lane * G;
            UnitDesc ud{0, 0, 0, 0};
            dspark_row_params_t rp{};
            PenHdr ph{0, 0, {0, 0}};
            if (ul < n_units) {
                ud = a.units[ul];
                rp = a.rows[ud.b];
                if (ud.kind == kUnitX && has_penalty(rp)) ph = a.pen_hdr[static_cast<long long>(ud.b) * a.tiles_x + ud.tile];
            }
            for (int l = 0; l < 32; ++l) {
                const int u = base + l * G;
                if (u >= n_units) break;
                const int slot = __shfl_sync(0xffffffffu, ud.slot, l);
                const int kind = __shfl_sync(0xffffffffu, ud.kind, l);
                const int tile = __shfl_sync(0xffffffffu, ud.tile, l);
                const int b = __shfl_sync(0xffffffffu, ud.b, l);
                const float T = __shfl_sync(0xffffffffu, rp.temperature, l);
                const int topk = __shfl_sync(0xffffffffu, rp.top_k, l);
                const float topp = __shfl_sync(0xffffffffu, rp.top_p, l);
                const float pres = __shfl_sync(0xffffffffu, rp.presence_penalty, l);
                const float freq = __shfl_sync(0xffffffffu, rp.frequency_penalty, l);
                const int pn = __shfl_sync(0xffffffffu, ph.n, l);
                const int pover = __shfl_sync(0xffffffffu, ph.overflow, l);
                const int pnh = __shfl_sync(0xffffffffu, ph.pad[0], l);
                const int stage = it % kStages;
                const unsigned parity = ((it / kStages) & 1) ^ 1;
                if (lane == 0) {
                    if (!mbar_wait_bounded(&sm.empty[stage], parity, kWaitLimit)) {
                        sm.error = 1;
                        failed = true;
                    } else {
                        StageMeta& m = sm.meta[stage];
                        const bool isx = kind == kUnitX;
                        const int es = isx ? SX : 4;
                        const int tile_n = isx ? a.tile_x : a.tile_q;
                        const int e0 = tile * tile_n, e1 = min(a.V, e0 + tile_n);
                        const unsigned char* row = isx
                            ? static_cast<const unsigned char*>(a.x) + static_cast<long long>(slot) * a.V * es
                            : reinterpret_cast<const unsigned char*>(a.q) + static_cast<long long>(slot) * a.V * 4;
                        const uintptr_t A0 = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(e0) * es;
                        const uintptr_t A1 = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(e1) * es;
                        uintptr_t c0 = (A0 + 15) & ~static_cast<uintptr_t>(15);
                        uintptr_t c1 = A1 & ~static_cast<uintptr_t>(15);
                        if (c1 < c0) c1 = c0;
                        const unsigned bytes = static_cast<unsigned>(c1 - c0);
                        m.kind = kind; m.slot = slot; m.b = b;
                        m.j = isx ? slot - b * (a.Km + 1) : slot - b * a.Km;
                        m.tile = tile; m.e0 = e0; m.e1 = e1;
                        m.nvec = static_cast<int>(bytes / 16);
                        m.vec_e0 = e0 + static_cast<int>((c0 - A0) / es);
                        if (bytes == 0) m.vec_e0 = e1;
                        m.pen = isx && (pres != 0.f || freq != 0.f);
                        m.pen_n = pn; m.pen_nh = pnh; m.pen_over = pover;
                        m.top_k = topk; m.temperature = T; m.top_p = topp;
                        m.presence = pres; m.frequency = freq;
                        unsigned tx = bytes;
                        const unsigned bm_bytes = static_cast<unsigned>(a.bm_words) * 4u;
                        const unsigned ent_bytes = m.pen && !pover ? static_cast<unsigned>(pn) * 16u : 0u;
                        if (m.pen) tx += bm_bytes + ent_bytes;
                        mbar_arrive_expect_tx(&sm.full[stage], tx);
                        if (bytes) bulk_g2s(sm.data[stage], reinterpret_cast<const void*>(c0), bytes, &sm.full[stage]);
                        if (m.pen) {
                            const long long pt = static_cast<long long>(b) * a.tiles_x + tile;
                            bulk_g2s(sm.bm[stage], a.pen_bm + pt * a.bm_words, bm_bytes, &sm.full[stage]);
                            if (ent_bytes) bulk_g2s(sm.ent[stage], a.pen_ent + pt * kPenCap, ent_bytes, &sm.full[stage]);
                        }
                    }
                }
                failed = __shfl_sync(0xffffffffu, failed, 0);
                if (failed) break;
                ++it;
            }
        }
        // drain: wait (bounded) for the copies of the last stages to land before exiting
        if (lane == 0) {
            for (int r = max(0, it - kStages); r < it; ++r)
                mbar_wait_bounded(&sm.full[r % kStages], (r / kStages) & 1, kWaitLimit);
        }
        return;
    }

    // ---------------- consumer warps
    int it = 0;
    for (int u = blockIdx.x; u < n_units; u += G, ++it) {
        const int stage = it % kStages;
        const unsigned parity = (it / kStages) & 1;
        if (!mbar_wait_bounded(&sm.full[stage], parity, kWaitLimit)) { sm.error = 1; }
        named_barrier_sync(2, kConsumerThreads);
        if (sm.error) break;
        const StageMeta m = sm.meta[stage];
        const int cb = it & 1;
        if (m.kind == kUnitX) process_x<SX>(a, sm, stage, m, cb);
        else process_q(a, sm, stage, m, cb);
    }
    if (threadIdx.x == 0 && sm.error) atomicOr(&a.plan->pad[0], 1);
}

}  // namespace

size_t stream_stats_smem_bytes() { return sizeof(Smem); }

cudaError_t launch_stream_stats(const Args& a, cudaStream_t s, int grid) {
    const size_t smem = sizeof(Smem);
    cudaError_t e;
    if (a.sx == 2) {
        e = cudaFuncSetAttribute(stream_stats_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        stream_stats_kernel<2><<<grid, kStreamThreads, smem, s>>>(a);
    } else {
        e = cudaFuncSetAttribute(stream_stats_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        stream_stats_kernel<4><<<grid, kStreamThreads, smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace dspark
