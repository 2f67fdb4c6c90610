// stream_stats_kernel: the single HBM pass over the target logits x and the draft
// probabilities q.  Everything else in the epilogue works on what this pass leaves behind.
//
// Work unit = a segment: a few consecutive vocab tiles of one row.  Persistent CTAs, one per
// SM; each CTA has two independent consumer groups of 8 warps and a producer warp.  The
// producer moves tiles into a 4-stage shared-memory ring (two stages per group) with the TMA
// bulk-copy engine (cp.async.bulk, completion counted on an mbarrier; the tiles with an
// evict-first L2 policy), together with each tile's penalty bitmap and penalised-token list,
// serving both groups' segment streams.
//
// A group processes a segment in one sweep:
//   first tile: pass 1 gives per-thread maxima of the penalised logits
//     (x' = x - ((f*c) + p), mlx-dspark Changelog [0.2.0] Added, penalties); every warp sorts
//     its lanes' maxima and takes the c-th largest (c = ceil(k/8)); theta = the least of the
//     8 warps' values, so at least 8*c >= k distinct logits of the first tile are >= theta,
//     hence every member of the segment's top-k is >= theta.  Pass 2 then accumulates and
//     filters as below;
//   later tiles: one pass each: the raw maximum (a non-finite logit shows there), the
//     penalised maximum with a rescaled sum of exp (the normaliser when there is no
//     top-k), the lowest index attaining the penalised max (greedy), and the candidates
//     >= theta (the top-k threshold of the row comes from these, mlx-dspark Changelog
//     [0.20.2] Changed: small selections instead of a full vocabulary sort);
//   end of segment: one reduction and one write of the statistics (the candidates went
//     straight to the segment's lists in global memory as they were found, positions taken
//     from counters in shared memory).
// Draft tiles get the same treatment with q as the key (top-k of q^(1/T) is top-k of q).  A
// draft row given sparsely or over a reduced vocabulary is streamed as it is stored (its m or
// Vd entries): the truncated draft distribution depends on the multiset of values alone, and
// the tokens the row leaves out have probability 0.
// The raw log-softmax and the raw top-n of logprobs are not taken here: they are needed at
// the emitted positions only, which logprob_kernel reads after the draws.
#include "dspark_internal.cuh"

namespace dspark {

namespace {

constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s: no healthy wait comes close
#ifdef DSPARK_TEST_EXPIRED_WAITS
// Test build only: every consumer wait for a tile counts as expired at once, and the producer
// gives up after 100 us without progress, so each call ends with DSPARK_ROW_INTERNAL on every
// valid request.  The producer's final wait for its own copies in flight keeps the 2 s bound.
constexpr bool kExpireAtOnce = true;
constexpr unsigned long long kIdleNs = 100000ull;
#else
constexpr bool kExpireAtOnce = false;
constexpr unsigned long long kIdleNs = kWaitNs;
#endif

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for a phase with a time bound; false when the bound expires.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kWaitNs) return false;
    return true;
}

// The same, giving up at once when *err is set (another thread of the group already gave up).
__device__ __forceinline__ bool wait_phase_or_err(uint64_t* bar, unsigned parity, const volatile int* err) {
    if (kExpireAtOnce) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (*err || globaltimer() - t0 > kWaitNs) return false;
    return true;
}
constexpr float kL2E = 1.4426950408889634f;
constexpr int kVecPerThread = kStageBytes / 16 / kGroupThreads;     // 12 vectors per thread and tile
static_assert(kVecPerThread % 2 == 0, "vectors are scanned in pairs");

struct StageMeta {
    int kind, slot, b, j;
    int seg, tile, e0, e1;
    int nvec, vec_e0, pen, pen_n;
    int pen_nh, pen_over, top_k, first;
    int last, pad0, pad1, pad2;
    float temperature, top_p, presence, frequency;
};

struct GroupSmem {
    float4 red1[kGroupWarps];    // first-tile maxima and thresholds
    float4 red[kGroupWarps];     // end-of-segment partials
    float4 red2[kGroupWarps];
    int n_pen;                   // entries appended to the segment's global candidate list
    int error;
    unsigned short flist[kGroupWarps][64];   // per warp: the tile's flagged vectors, (slot << 5) | lane
};

struct Smem {
    alignas(128) unsigned char data[kStages][kStageBytes];
    alignas(16) unsigned bm[kStages][kBitmapWordsMax];
    alignas(16) PenEntry ent[kStages][kPenCap];
    StageMeta meta[kStages];
    GroupSmem grp[kGroups];
    alignas(8) uint64_t full[kStages];
    alignas(8) uint64_t empty[kStages];
};

__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void group_sync(int g) { named_barrier_sync(1 + g, kGroupThreads); }

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

__device__ __forceinline__ bool bitmap_bit(const unsigned* bm, int off) {
    return (bm[off >> 5] >> (off & 31)) & 1u;
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

// Two elements of a vector as a float2 (pair q: elements 2q and 2q+1).
template <int SX>
__device__ __forceinline__ float2 elem_pair(const uint4& w, int q) {
    if (SX == 2) {
        const uint32_t word = (q == 0) ? w.x : (q == 1) ? w.y : (q == 2) ? w.z : w.w;
        return make_float2(bf16_lo(word), bf16_hi(word));
    } else {
        return q == 0 ? make_float2(__uint_as_float(w.x), __uint_as_float(w.y))
                      : make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
    }
}

// acc += 2^(x*scale - off) over the vector's elements, pairwise in f32x2.
template <int SX>
__device__ __forceinline__ float2 vec_exp_sum(const uint4& w, float2 acc, float scale, float off) {
    const float2 sc = make_float2(scale, scale);
    const float2 no = make_float2(-off, -off);
#pragma unroll
    for (int q = 0; q < 8 / SX; ++q) {
        const float2 t = __ffma2_rn(elem_pair<SX>(w, q), sc, no);
        acc = __fadd2_rn(acc, make_float2(ex2_approx(t.x), ex2_approx(t.y)));
    }
    return acc;
}

__device__ __forceinline__ void push(Cand* buf, int* cnt, int cap, float v, int id) {
    const int p = atomicAdd(cnt, 1);
    if (p < cap) buf[p] = Cand{v, id};
}

// Group-wide reduction of (max, max, min, min) from per-warp float4 slots; every thread gets it.
__device__ __forceinline__ float4 group_reduce_mmnn(const float4* red) {
    const int lane = threadIdx.x & 31;
    float4 v = lane < kGroupWarps ? red[lane] : make_float4(-INFINITY, -INFINITY, INFINITY, INFINITY);
#pragma unroll
    for (int o = kGroupWarps / 2; o; o >>= 1) {
        v.x = max_nan(v.x, __shfl_xor_sync(0xffffffffu, v.x, o));
        v.y = max_nan(v.y, __shfl_xor_sync(0xffffffffu, v.y, o));
        v.z = fminf(v.z, __shfl_xor_sync(0xffffffffu, v.z, o));
        v.w = fminf(v.w, __shfl_xor_sync(0xffffffffu, v.w, o));
    }
    v.x = __shfl_sync(0xffffffffu, v.x, 0);
    v.y = __shfl_sync(0xffffffffu, v.y, 0);
    v.z = __shfl_sync(0xffffffffu, v.z, 0);
    v.w = __shfl_sync(0xffffffffu, v.w, 0);
    return v;
}

// Combine (max, sum relative to max) pairs over a warp; scale converts value gaps to log2.
__device__ __forceinline__ void warp_merge_ms(float& m, float& s, float scale) {
    const float M = [&] {
        float t = m;
        for (int o = 16; o; o >>= 1) t = max_nan(t, __shfl_xor_sync(0xffffffffu, t, o));
        return t;
    }();
    float r = (s > 0.f && m > -INFINITY && M > -INFINITY) ? s * ex2_approx((m - M) * scale) : 0.f;
    for (int o = 16; o; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    m = M;
    s = r;
}

// ------------------------------------------------------------------ warp-cooperative appends
// Append the elements of one 16-byte vector flagged in `mask` (bit q = element q) to one of
// the segment's candidate lists in global memory: each lane with candidates takes its
// positions with one shared atomic on the list's counter (a lane-wide prefix and a single
// atomic per warp was a longer dependency chain in this per-tile step).
template <int SX>
__device__ __forceinline__ void warp_append(Cand* buf, int* cnt, int cap, unsigned mask, const uint4& w, int e,
                                            int tag) {
    if (!mask) return;
    int base = atomicAdd(cnt, __popc(mask));
    while (mask) {
        const int q = __ffs(mask) - 1;
        mask &= mask - 1u;
        if (base < cap) buf[base] = Cand{elem<SX>(w, q), (e + q) | tag};
        ++base;
    }
}

// Append every element flagged in this thread's (f0, f1) bit set (bit EPV*i+q: element q of
// the thread's i-th vector of the tile in shared memory), warp-cooperatively: one prefix and
// one shared atomic per warp and tile.  All lanes of the warp call it.
template <int SX>
__device__ __forceinline__ void flush_flags(Cand* buf, int* cnt, int cap, unsigned long long f0, unsigned long long f1,
                                            const unsigned char* data, int vec_e0, int gt, int tag) {
    constexpr int EPV = 16 / SX;
    const int n = __popcll(f0) + __popcll(f1);
    if (!__ballot_sync(0xffffffffu, n != 0)) return;
    const int lane = threadIdx.x & 31;
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int base = 0;
    if (lane == 31) base = atomicAdd(cnt, incl);
    base = __shfl_sync(0xffffffffu, base, 31) + incl - n;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        unsigned long long f = h ? f1 : f0;
        while (f) {
            const int bit = __ffsll(f) - 1 + 64 * h;
            f &= f - 1ull;
            const int i = bit / EPV, q = bit % EPV;
            const int v = gt + i * kGroupThreads;
            const uint4 w = *reinterpret_cast<const uint4*>(data + v * 16);
            if (base < cap) buf[base] = Cand{elem<SX>(w, q), (vec_e0 + v * EPV + q) | tag};
            ++base;
        }
    }
}

// Bit q set where element q of the vector is >= th.
template <int SX>
__device__ __forceinline__ unsigned ge_mask(const uint4& w, float th) {
    unsigned m = 0u;
#pragma unroll
    for (int q = 0; q < 16 / SX; ++q) m |= (elem<SX>(w, q) >= th ? 1u : 0u) << q;
    return m;
}

// The same for the flush of a bf16 tile, on bf16 pairs against th2 = th rounded down to bf16:
// bit q set where element q >= th2 (every element >= th, and those equal to th2 < th besides,
// which only adds candidates below the threshold).
__device__ __forceinline__ unsigned ge_mask_bf16(const uint4& w, __nv_bfloat162 th2) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&w);
    unsigned m = 0u;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const unsigned mk = __hge2_mask(p[h], th2);       // 0xFFFF per half that holds
        m |= ((mk & 1u) | ((mk >> 15) & 2u)) << (2 * h);
    }
    return m;
}

// Position of the r-th (0-based) set bit of b; requires r < popc(b).
__device__ __forceinline__ int nth_set_bit(unsigned b, int r) {
    int pos = 0;
#pragma unroll
    for (int s = 16; s; s >>= 1) {
        const int c = __popc(b & ((1u << s) - 1u));
        if (r >= c) { r -= c; b >>= s; pos += s; }
    }
    return pos;
}

// Item t of the warp's flagged vectors in slot order, dealt by slot-wise ballots (-1 past
// the end).  Out of line: it only runs when a warp flags more vectors than its list holds,
// and keeping it out of the flush keeps the hot loop small in the instruction cache.
__device__ __noinline__ int deal_by_ballots(unsigned vflags, int t, int wv) {
    int run = 0, v = -1;
    for (int i = 0; i < kVecPerThread; ++i) {
        const unsigned b = __ballot_sync(0xffffffffu, (vflags >> i) & 1u);
        const int n = __popc(b);
        const int r = t - run;
        if (r >= 0 && r < n) v = wv + nth_set_bit(b, r) + i * kGroupThreads;
        run += n;
    }
    return v;
}

// Candidate extraction from the vectors the threads flagged during a scan (bit i of
// `vflags`: the thread's i-th vector of the tile has an element at or above the
// threshold).  The warp's flagged vectors are dealt out to its lanes 32 at a time, so a lane
// with many flags does not hold up the others: a prefix over the lanes' flag counts places
// them in a per-warp list (more than 64 fall back to slot-wise ballots).  For each vector,
// the elements >= th_p (bf16: >= th_p rounded down to bf16) without a penalty bit are
// appended to the candidate list `lp` (CAND) and folded into the running penalised maximum
// and the lowest index attaining it (TRACK).
// Every lane of the warp calls it.
template <int SX, bool PEN, bool CAND, bool TRACK>
__device__ __forceinline__ void flush_vectors(GroupSmem& gs, Cand* lp, unsigned vflags, const unsigned char* data,
                                              const unsigned* bm, int vec_e0, int bit0, int gt,
                                              float th_p, float& m_p, int& arg) {
    constexpr int EPV = 16 / SX;
    const int lane = threadIdx.x & 31;
    const int wv = gt - lane;                             // vector index of lane 0, slot 0
    const __nv_bfloat162 th2 = __bfloat162bfloat162(__float2bfloat16_rd(th_p));
    // the warp's flagged vectors in (lane, slot) order: a prefix over the lanes' counts, each
    // lane writing its own into the warp's list
    const int nf = __popc(vflags);
    int incl = nf;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total == 0) return;
    unsigned short* list = gs.flist[gt >> 5];
    const bool listed = total <= 64;
    if (listed) {
        int pos = incl - nf;
        for (unsigned f = vflags; f; f &= f - 1u) list[pos++] = static_cast<unsigned short>(((__ffs(f) - 1) << 5) | lane);
        __syncwarp();
    }
    for (int base = 0; base < total; base += 32) {
        const int t = base + lane;                        // this lane's item of the round
        int v = -1;
        if (listed) {
            if (t < total) { const unsigned it = list[t]; v = wv + static_cast<int>(it & 31u) + static_cast<int>(it >> 5) * kGroupThreads; }
        } else {
            v = deal_by_ballots(vflags, t, wv);           // more flags than the list holds
        }
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        unsigned mp = 0u;
        int e = 0;
        if (v >= 0) {
            w = *reinterpret_cast<const uint4*>(data + v * 16);
            e = vec_e0 + v * EPV;
            const unsigned bits = PEN ? bitmap_bits(bm, bit0 + v * EPV, EPV) : 0u;
            if constexpr (SX == 2) mp = ge_mask_bf16(w, th2) & ~bits;
            else mp = ge_mask<SX>(w, th_p) & ~bits;
        }
        if (CAND) warp_append<SX>(lp, &gs.n_pen, kCandPenGlobal, mp, w, e, 0);
        if (TRACK) {
            while (mp) {
                const int q = __ffs(mp) - 1;
                mp &= mp - 1u;
                const float x = elem<SX>(w, q);
                if (x > m_p) { m_p = x; arg = e + q; }
                else if (x == m_p && e + q < arg) arg = e + q;
            }
        }
    }
    if (listed) __syncwarp();                             // the list is rewritten by the next flush
}

// ------------------------------------------------------------------ target-logit segments
struct XState {
    float m_r;           // raw running max (NaN-propagating: shows a non-finite logit)
    float m_p, s_t;      // penalised running max, sum of 2^((x' - m_p)*c_l2e)
    int arg;             // lowest index attaining m_p seen by this thread
    float th_p;          // candidate threshold (segment-wide)
};

template <int SX>
struct XCtx {
    const Args& a;
    Smem& sm;
    GroupSmem& gs;
    int g, stage;
    const StageMeta& m;
    bool greedy, need_cand, need_temp;
    float f, p, c_l2e;
    Cand* lp;            // the segment's penalised-candidate list (global)
};

// Raw value of element e of the current tile: shared memory for the aligned interior,
// a plain load for the head / tail.
template <int SX>
__device__ __forceinline__ float x_at(const XCtx<SX>& c, int e) {
    const StageMeta& m = c.m;
    if (e >= m.vec_e0 && e < m.vec_e0 + m.nvec * (16 / SX)) {
        const unsigned char* p = c.sm.data[c.stage] + static_cast<long long>(e - m.vec_e0) * SX;
        return SX == 2 ? __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p)) << 16)
                       : *reinterpret_cast<const float*>(p);
    }
    return load_x(c.a.x, SX, static_cast<long long>(m.slot) * c.a.V + e);
}

// Fold a penalised value xp (element e) into the penalised statistics; `xr` is its raw
// value whose term was already added to the tempered sum by the vector pass (undone here).
template <int SX>
__device__ __forceinline__ void pen_fold(const XCtx<SX>& c, XState& st, float xp, float xr, int e, bool undo_raw) {
    if (xp > st.m_p) {
        if (c.need_temp) st.s_t = (st.m_p > -INFINITY) ? st.s_t * ex2_approx((st.m_p - xp) * c.c_l2e) : 0.f;
        st.m_p = xp;
        st.arg = e;
    } else if (xp == st.m_p && e < st.arg) {
        st.arg = e;
    } else if (xp != xp) {
        st.m_p = xp;
    }
    if (c.need_temp) {
        st.s_t += ex2_approx((xp - st.m_p) * c.c_l2e);
        if (undo_raw) st.s_t -= ex2_approx((xr - st.m_p) * c.c_l2e);
    }
    if (xp >= st.th_p) push(c.lp, &c.gs.n_pen, kCandPenGlobal, xp, e);
}

// One 16-byte vector: the raw maximum over all its elements, penalised statistics over the
// elements without a penalty bit (the penalised ones are folded in by x_entries).
template <int SX>
__device__ __forceinline__ void x_vec(const XCtx<SX>& c, XState& st, const uint4& w, int e, unsigned bits,
                                      unsigned& mask_p) {
    constexpr int EPV = 16 / SX;
    const float vm = vec_max<SX>(w);
    st.m_r = max_nan(st.m_r, vm);
    // penalised max over unpenalised elements
    float vp = vm;
    if (bits != 0u) {
        vp = -INFINITY;
#pragma unroll
        for (int q = 0; q < EPV; ++q)
            if (!((bits >> q) & 1u)) vp = max_nan(vp, elem<SX>(w, q));
    }
    if (!(vp <= st.m_p)) {
        const float nm = max_nan(st.m_p, vp);
        if (c.need_temp) st.s_t = (st.m_p > -INFINITY && nm == nm) ? st.s_t * ex2_approx((st.m_p - nm) * c.c_l2e) : 0.f;
        st.m_p = nm;
        st.arg = 0x7FFFFFFF;
#pragma unroll
        for (int q = 0; q < EPV; ++q)
            if (!((bits >> q) & 1u) && elem<SX>(w, q) == nm) st.arg = min(st.arg, e + q);
    } else if (c.greedy && vp == st.m_p && st.arg == 0x7FFFFFFF) {
#pragma unroll
        for (int q = 0; q < EPV; ++q)
            if (!((bits >> q) & 1u) && elem<SX>(w, q) == vp) st.arg = min(st.arg, e + q);
    }
    if (c.need_temp) {
        // all elements; the penalised ones are corrected by x_entries
        const float2 t = vec_exp_sum<SX>(w, make_float2(0.f, 0.f), c.c_l2e, st.m_p * c.c_l2e);
        st.s_t += t.x + t.y;
    }
    // candidates: unpenalised values for top-k (penalised: x_entries); the caller appends
    // them warp-cooperatively
    mask_p = (c.need_cand && vp >= st.th_p) ? (ge_mask<SX>(w, st.th_p) & ~bits) : 0u;
}

// A penalised value on the fast path: values >= th_p update the running maximum / lowest
// index attaining it, and are top-k candidates when the row needs them.
template <int SX>
__device__ __forceinline__ void fold_fast(const XCtx<SX>& c, XState& st, float xp, int e) {
    if (xp >= st.th_p) {
        if (xp > st.m_p) { st.m_p = xp; st.arg = e; }
        else if (xp == st.m_p && e < st.arg) st.arg = e;
        if (c.need_cand) push(c.lp, &c.gs.n_pen, kCandPenGlobal, xp, e);
    }
}

// The tile's possibly-penalised tokens (history and draft tokens, from the penalty index):
// each thread takes some, computes x' = x - ((f*c) + p) with c = history + own draft prefix,
// and folds it into the penalised statistics.  pass1: only the maximum.
template <int SX>
__device__ __forceinline__ void x_entries(const XCtx<SX>& c, XState& st, bool pass1, bool fast, float& lane_pen) {
    const StageMeta& m = c.m;
    const int gt = threadIdx.x - c.g * kGroupThreads;
    const PenEntry* ent = c.sm.ent[c.stage];
    const unsigned long long low = (m.j >= 64) ? ~0ull : ((1ull << m.j) - 1ull);
    for (int i = gt; i < m.pen_n; i += kGroupThreads) {
        const PenEntry pe = ent[i];
        const int t = pe.token;
        if (t < m.e0 || t >= m.e1) continue;
        const unsigned long long mask = (static_cast<unsigned long long>(pe.mask_hi) << 32) | pe.mask_lo;
        const int cnt = pe.base + __popcll(mask & low);
        const float xr = x_at(c, t);
        const float xp = penalise(xr, cnt, c.f, c.p);
        if (pass1) lane_pen = max_nan(lane_pen, xp);
        else if (fast) fold_fast(c, st, xp, t);
        else pen_fold(c, st, xp, xr, t, true);
    }
}

// Overflowed penalty index (more penalised tokens in the tile than fit): element-by-element
// over the vectors carrying penalty bits, counts looked up in the caller's history.
template <int SX>
__device__ __forceinline__ void x_vec_overflow(const XCtx<SX>& c, XState& st, const uint4& w, int e, unsigned bits,
                                               bool pass1, float& lane_pen) {
    constexpr int EPV = 16 / SX;
#pragma unroll
    for (int q = 0; q < EPV; ++q) {
        if (!((bits >> q) & 1u)) continue;
        const float xr = elem<SX>(w, q);
        const float xp = penalise(xr, pen_count(c.sm, c.stage, c.m, c.a, e + q), c.f, c.p);
        if (pass1) lane_pen = max_nan(lane_pen, xp);
        else pen_fold(c, st, xp, xr, e + q, true);
    }
}

// Fast path over a tile whose penalty index overflowed: each thread folds the penalised
// tokens of its own vectors, their counts looked up in the caller's history.
template <int SX>
__device__ void x_overflow_fast(const XCtx<SX>& c, XState& st, const unsigned char* data, const unsigned* bm,
                                int gt) {
    constexpr int EPV = 16 / SX;
    const StageMeta& m = c.m;
    for (int i = 0; i < kVecPerThread; ++i) {
        const int v = gt + i * kGroupThreads;
        if (v >= m.nvec) break;
        const int e = m.vec_e0 + v * EPV;
        unsigned bits = bitmap_bits(bm, e - m.e0, EPV);
        if (!bits) continue;
        const uint4 w = *reinterpret_cast<const uint4*>(data + v * 16);
        while (bits) {
            const int q = __ffs(bits) - 1;
            bits &= bits - 1u;
            fold_fast(c, st, penalise(elem<SX>(w, q), pen_count(c.sm, c.stage, m, c.a, e + q), c.f, c.p), e + q);
        }
    }
}

template <int SX>
__device__ __forceinline__ uint4 neg_inf_vec() {
    const uint32_t ni = SX == 2 ? 0xFF80FF80u : 0xFF800000u;
    return make_uint4(ni, ni, ni, ni);
}

// The scan of one tile for every row that does not need the tempered sum: raw maximum, and
// one flag bit per vector whose maximum is >= th.  All per-element work on candidates is
// left to flush_vectors.
// bf16 pairs throughout: the vector maximum and the running maximum stay packed, and the
// threshold is rounded down to bf16 (a vector is flagged at least whenever its float maximum
// reaches th; the flush compares each element in float).  FULL: the tile fills the stage.
template <bool FULL>
__device__ __forceinline__ unsigned x_scan_flags_bf16(XState& st, const unsigned char* data, int gt, int nvec,
                                                      float th) {
    unsigned fl = 0u;
    const __nv_bfloat162 th2 = __bfloat162bfloat162(__float2bfloat16_rd(th));
    const __nv_bfloat162 ninf = __bfloat162bfloat162(__float2bfloat16(-INFINITY));
    __nv_bfloat162 r0 = ninf, r1 = ninf;
#pragma unroll
    for (int i = 0; i < kVecPerThread; i += 2) {
        const int v0 = gt + i * kGroupThreads, v1 = v0 + kGroupThreads;
        if (!FULL && v0 >= nvec) break;
        const bool ok1 = FULL || v1 < nvec;
        const uint4 w0 = *reinterpret_cast<const uint4*>(data + v0 * 16);
        const uint4 w1 = ok1 ? *reinterpret_cast<const uint4*>(data + v1 * 16) : neg_inf_vec<2>();
        const __nv_bfloat162* p0 = reinterpret_cast<const __nv_bfloat162*>(&w0);
        const __nv_bfloat162* p1 = reinterpret_cast<const __nv_bfloat162*>(&w1);
        const __nv_bfloat162 m0 = __hmax2_nan(__hmax2_nan(p0[0], p0[1]), __hmax2_nan(p0[2], p0[3]));
        const __nv_bfloat162 m1 = __hmax2_nan(__hmax2_nan(p1[0], p1[1]), __hmax2_nan(p1[2], p1[3]));
        r0 = __hmax2_nan(r0, m0);
        r1 = __hmax2_nan(r1, m1);
        fl |= (__hge2_mask(m0, th2) ? 1u : 0u) << i;
        fl |= ((ok1 && __hge2_mask(m1, th2)) ? 1u : 0u) << (i + 1);
    }
    const __nv_bfloat162 r = __hmax2_nan(r0, r1);
    const uint32_t rw = *reinterpret_cast<const uint32_t*>(&r);
    st.m_r = max_nan(st.m_r, max_nan(bf16_lo(rw), bf16_hi(rw)));
    return fl;
}

template <int SX>
__device__ __forceinline__ unsigned x_scan_flags(XState& st, const unsigned char* data, int gt, int nvec, float th) {
    if constexpr (SX == 2)
        return nvec == kVecPerThread * kGroupThreads ? x_scan_flags_bf16<true>(st, data, gt, nvec, th)
                                                     : x_scan_flags_bf16<false>(st, data, gt, nvec, th);
    unsigned fl = 0u;
    float m0 = st.m_r, m1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < kVecPerThread; i += 2) {
        const int v0 = gt + i * kGroupThreads, v1 = v0 + kGroupThreads;
        if (v0 >= nvec) break;
        const bool ok1 = v1 < nvec;
        const uint4 w0 = *reinterpret_cast<const uint4*>(data + v0 * 16);
        const uint4 w1 = ok1 ? *reinterpret_cast<const uint4*>(data + v1 * 16) : neg_inf_vec<SX>();
        const float vm0 = vec_max<SX>(w0), vm1 = vec_max<SX>(w1);
        m0 = max_nan(m0, vm0);
        m1 = max_nan(m1, vm1);
        // the filler past the end of the tile is never flagged
        fl |= (vm0 >= th ? 1u : 0u) << i;
        fl |= ((ok1 && vm1 >= th) ? 1u : 0u) << (i + 1);
    }
    st.m_r = max_nan(m0, m1);
    return fl;
}

template <int SX, bool PEN>
__device__ __forceinline__ void x_flush_cand(bool cand, GroupSmem& gs, Cand* lp, unsigned fl, const unsigned char* data,
                                             const unsigned* bm, int vec_e0, int bit0, int gt, XState& st) {
    if (cand) flush_vectors<SX, PEN, true, true>(gs, lp, fl, data, bm, vec_e0, bit0, gt, st.th_p, st.m_p, st.arg);
    else flush_vectors<SX, PEN, false, true>(gs, lp, fl, data, bm, vec_e0, bit0, gt, st.th_p, st.m_p, st.arg);
}

// Scan and candidate flush of one tile on the fast path.
template <int SX>
__device__ __forceinline__ void x_fast_pass(const XCtx<SX>& c, XState& st, const unsigned char* data,
                                            const unsigned* bm, int gt) {
    const StageMeta& m = c.m;
    const unsigned fl = x_scan_flags<SX>(st, data, gt, m.nvec, st.th_p);
    const int bit0 = m.vec_e0 - m.e0;
    if (m.pen) x_flush_cand<SX, true>(c.need_cand, c.gs, c.lp, fl, data, bm, m.vec_e0, bit0, gt, st);
    else x_flush_cand<SX, false>(c.need_cand, c.gs, c.lp, fl, data, bm, m.vec_e0, bit0, gt, st);
}

template <int SX>
__device__ void x_tile(const XCtx<SX>& c, XState& st) {
    constexpr int EPV = 16 / SX;
    const StageMeta& m = c.m;
    const int gt = threadIdx.x - c.g * kGroupThreads;
    const int lane = threadIdx.x & 31, warp = gt >> 5;
    const unsigned char* data = c.sm.data[c.stage];
    const unsigned* bm = c.sm.bm[c.stage];
    const long long xrow = static_cast<long long>(m.slot) * c.a.V;
    const int e_tail = m.vec_e0 + m.nvec * EPV;
    const bool use_entries = m.pen && !m.pen_over;
    const bool overflow = m.pen && m.pen_over;
    // fast path: every row but those needing the tempered sum (a property of the row, so
    // the same for all tiles of a segment)
    const bool fast = !c.need_temp;

    if (m.first) {
        // ---- pass 1 over the first tile: maxima, then the segment's candidate thresholds
        float mu0 = -INFINITY, mu1 = -INFINITY, mrw = -INFINITY, mpen = -INFINITY;
        int v = gt;
        for (; v + kGroupThreads < m.nvec; v += 2 * kGroupThreads) {
            const uint4 w0 = *reinterpret_cast<const uint4*>(data + v * 16);
            const uint4 w1 = *reinterpret_cast<const uint4*>(data + (v + kGroupThreads) * 16);
            const int e0 = m.vec_e0 + v * EPV, e1 = e0 + kGroupThreads * EPV;
            const unsigned b0 = m.pen ? bitmap_bits(bm, e0 - m.e0, EPV) : 0u;
            const unsigned b1 = m.pen ? bitmap_bits(bm, e1 - m.e0, EPV) : 0u;
            const float v0 = vec_max<SX>(w0), v1 = vec_max<SX>(w1);
            mrw = max_nan(mrw, max_nan(v0, v1));
            // vectors holding a penalised token are left out of the penalised lane maxima
            mu0 = max_nan(mu0, b0 ? -INFINITY : v0);
            mu1 = max_nan(mu1, b1 ? -INFINITY : v1);
            if (overflow && (b0 | b1)) {
                XState dummy{};
                x_vec_overflow<SX>(c, dummy, w0, e0, b0, true, mpen);
                x_vec_overflow<SX>(c, dummy, w1, e1, b1, true, mpen);
            }
        }
        for (; v < m.nvec; v += kGroupThreads) {
            const uint4 w = *reinterpret_cast<const uint4*>(data + v * 16);
            const int e = m.vec_e0 + v * EPV;
            const unsigned bits = m.pen ? bitmap_bits(bm, e - m.e0, EPV) : 0u;
            const float vv = vec_max<SX>(w);
            mrw = max_nan(mrw, vv);
            mu0 = max_nan(mu0, bits ? -INFINITY : vv);
            if (overflow && bits) { XState dummy{}; x_vec_overflow<SX>(c, dummy, w, e, bits, true, mpen); }
        }
        if (gt < 2) {
            const int lo = gt == 0 ? m.e0 : e_tail, hi = gt == 0 ? m.vec_e0 : m.e1;
            for (int e = lo; e < hi; ++e) {
                const float xv = load_x(c.a.x, SX, xrow + e);
                mrw = max_nan(mrw, xv);
                if (m.pen && bitmap_bit(bm, e - m.e0)) {
                    if (overflow) mpen = max_nan(mpen, penalise(xv, pen_count(c.sm, c.stage, m, c.a, e), c.f, c.p));
                } else {
                    mu0 = max_nan(mu0, xv);
                }
            }
        }
        if (use_entries) { XState dummy{}; x_entries<SX>(c, dummy, true, false, mpen); }
        const float lane_raw = mrw, lane_pen = max_nan(max_nan(mu0, mu1), mpen);
        float wr = lane_raw, wp = lane_pen;
        for (int o = 16; o; o >>= 1) {
            wr = max_nan(wr, __shfl_xor_sync(0xffffffffu, wr, o));
            wp = max_nan(wp, __shfl_xor_sync(0xffffffffu, wp, o));
        }
        float thp = 0.f;
        if (c.need_cand) {
            float sp = lane_pen, unused = 0.f;
            warp_sort2_desc(sp, unused);
            thp = __shfl_sync(0xffffffffu, sp, (m.top_k + kGroupWarps - 1) / kGroupWarps - 1);
        }
        if (lane == 0) c.gs.red1[warp] = make_float4(wr, wp, thp, INFINITY);
        group_sync(c.g);
        const float4 r = group_reduce_mmnn(c.gs.red1);
        // The segment starts from the first tile's maxima.  Each lane value above is the
        // penalised value of a distinct element, so every warp has at least cp elements >= its
        // cp-th largest lane value and the tile at least top_k elements >= the minimum over
        // warps: nothing of the row's top-k lies below th_p.  On the fast path th_p of a row
        // without a top-k list is the tile's penalised maximum (over the same elements), so the
        // segment's penalised maximum and argmax are found among the values >= th_p.
        st.m_r = r.x;
        st.m_p = fast ? -INFINITY : r.y;
        st.s_t = 0.f;
        st.arg = 0x7FFFFFFF;
        st.th_p = c.need_cand ? r.z : (fast ? r.y : INFINITY);
    }

    // ---- the accumulation / filter pass over this tile.  General path: candidate flags
    // are kept per thread (bit EPV*i+q: element q of the thread's i-th vector) and appended
    // once at the end.
    float unused = 0.f;
    unsigned long long fp0 = 0ull, fp1 = 0ull;
    if (fast) {
        x_fast_pass<SX>(c, st, data, bm, gt);
        if (overflow) x_overflow_fast<SX>(c, st, data, bm, gt);
    }
#pragma unroll 2
    for (int i = 0; i < (fast ? 0 : kVecPerThread); ++i) {
        const int v = gt + i * kGroupThreads;
        if (v >= m.nvec) break;
        const uint4 w = *reinterpret_cast<const uint4*>(data + v * 16);
        const int e = m.vec_e0 + v * EPV;
        const unsigned bits = m.pen ? bitmap_bits(bm, e - m.e0, EPV) : 0u;
        unsigned mp = 0u;
        x_vec<SX>(c, st, w, e, bits, mp);
        if (overflow && bits) x_vec_overflow<SX>(c, st, w, e, bits, false, unused);
        const int sh = i * EPV;
        if (sh < 64) fp0 |= static_cast<unsigned long long>(mp) << sh;
        else fp1 |= static_cast<unsigned long long>(mp) << (sh - 64);
    }
    if (!fast && c.need_cand) flush_flags<SX>(c.lp, &c.gs.n_pen, kCandPenGlobal, fp0, fp1, data, m.vec_e0, gt, 0);
    if (gt < 2) {
        const int lo = gt == 0 ? m.e0 : e_tail, hi = gt == 0 ? m.vec_e0 : m.e1;
        for (int e = lo; e < hi; ++e) {
            const float xv = load_x(c.a.x, SX, xrow + e);
            st.m_r = max_nan(st.m_r, xv);
            const bool bit = m.pen && bitmap_bit(bm, e - m.e0);
            if (fast) {
                if (!bit) fold_fast(c, st, xv, e);
                else if (overflow) fold_fast(c, st, penalise(xv, pen_count(c.sm, c.stage, m, c.a, e), c.f, c.p), e);
            }
            else if (!bit) pen_fold(c, st, xv, xv, e, false);
            else if (overflow) pen_fold(c, st, penalise(xv, pen_count(c.sm, c.stage, m, c.a, e), c.f, c.p), xv, e, false);
            else if (c.need_temp) st.s_t += ex2_approx((xv - st.m_p) * c.c_l2e);   // undone by x_entries
        }
    }
    if (use_entries) x_entries<SX>(c, st, false, fast, unused);
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.sm.empty[c.stage]);     // this stage is no longer read
}

template <int SX>
__device__ void x_finish(const XCtx<SX>& c, XState& st) {
    const StageMeta& m = c.m;
    const int gt = threadIdx.x - c.g * kGroupThreads;
    const int lane = threadIdx.x & 31, warp = gt >> 5;
    float mr = st.m_r, mp = st.m_p, stt = st.s_t;
    // argmax: lowest index among lanes whose running max equals the warp max
    float wp = mp;
    for (int o = 16; o; o >>= 1) wp = max_nan(wp, __shfl_xor_sync(0xffffffffu, wp, o));
    int arg = (mp == wp) ? st.arg : 0x7FFFFFFF;
    arg = warp_min_i(arg);
    for (int o = 16; o; o >>= 1) mr = max_nan(mr, __shfl_xor_sync(0xffffffffu, mr, o));
    warp_merge_ms(mp, stt, c.c_l2e);
    if (lane == 0) {
        c.gs.red[warp] = make_float4(mr, 0.f, mp, stt);
        c.gs.red2[warp] = make_float4(__int_as_float(arg), 0.f, 0.f, 0.f);
    }
    group_sync(c.g);                                      // partials written, every append done
    const long long ti = static_cast<long long>(m.slot) * c.a.nseg_x + m.seg;
    if (warp == 0) {
        float4 r = lane < kGroupWarps ? c.gs.red[lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        int ag = lane < kGroupWarps ? __float_as_int(c.gs.red2[lane].x) : 0x7FFFFFFF;
        float Mr = r.x, Mp = r.z, St = r.w;
        float Mp_all = Mp;
        for (int o = 16; o; o >>= 1) Mp_all = max_nan(Mp_all, __shfl_xor_sync(0xffffffffu, Mp_all, o));
        ag = (Mp == Mp_all) ? ag : 0x7FFFFFFF;
        ag = warp_min_i(ag);
        for (int o = 16; o; o >>= 1) Mr = max_nan(Mr, __shfl_xor_sync(0xffffffffu, Mr, o));
        warp_merge_ms(Mp, St, c.c_l2e);
        if (lane == 0) {
            const int n_pen = c.gs.n_pen;
            TileStats ts;
            ts.m_raw = Mr; ts.s_raw = 0.f; ts.m_pen = Mp; ts.arg_pen = ag; ts.s_temp = St;
            ts.flags = 0;
            ts.n_pen = c.need_cand ? n_pen : 0;
            if (c.need_cand && n_pen > kCandPenGlobal) { ts.flags |= kTileOverflowPen; ts.n_pen = 0; }
            // NaN or +inf anywhere shows in the maxima; -inf logits are allowed (zero probability)
            if (Mr != Mr || Mr == INFINITY || Mp != Mp || Mp == INFINITY) ts.flags |= kTileBad;
            c.a.ts_x[ti] = ts;
            // counters for the next segment: its first append follows its first-tile barrier,
            // which this warp reaches only after this write
            c.gs.n_pen = 0;
        }
    }
}

// ------------------------------------------------------------------ draft-probability segments
struct QState {
    float mx, mn, sum;   // running max / min; sum of q (T = 1) or of (q/mx)^(1/T)
    float th;
};

__device__ __forceinline__ void q_elem(QState& st, float v, bool need_sum, bool t_one, float inv_t, bool filt,
                                       GroupSmem& gs, Cand* lp, int e) {
    if (need_sum && !t_one && v > st.mx) {
        st.sum = (st.mx > 0.f) ? st.sum * exp2f(inv_t * log2f(st.mx / v)) : 0.f;
    }
    st.mx = max_nan(st.mx, v);
    st.mn = fminf(st.mn, v);
    if (need_sum) st.sum += t_one ? v : draft_weight(v, st.mx, inv_t, false);
    if (filt && v >= st.th) push(lp, &gs.n_pen, kCandPenGlobal, v, e);
}

// The scan of one draft tile of a top-k row.  Raw bit patterns: for values with a clear sign
// bit the unsigned order is the float order (NaNs above +inf), so one integer max per element
// gives both the vector flags and the running maximum.  A set sign bit (a negative value, -0.0
// or a negative NaN) puts its vector above every threshold (ge_mask then decides in float) and
// sends this thread's part of the tile through the float maximum and minimum.  FULL: the tile
// fills the stage, so every thread has all its vectors and nothing is bounds-checked.
template <bool FULL>
__device__ __forceinline__ unsigned q_scan_flags(QState& st, const unsigned char* data, int gt, int nvec) {
    unsigned vfl = 0u, u0 = 0u, u1 = 0u;
    const float th = st.th;
    const unsigned thb = th > 0.f ? __float_as_uint(th) : 0u;
#pragma unroll
    for (int i = 0; i < kVecPerThread; i += 2) {
        const int v0 = gt + i * kGroupThreads, v1 = v0 + kGroupThreads;
        if (!FULL && v0 >= nvec) break;
        const bool ok1 = FULL || v1 < nvec;
        const uint4 w0 = *reinterpret_cast<const uint4*>(data + v0 * 16);
        const uint4 w1 = ok1 ? *reinterpret_cast<const uint4*>(data + v1 * 16) : make_uint4(0u, 0u, 0u, 0u);
        const unsigned vm0 = max(__vimax3_u32(w0.x, w0.y, w0.z), w0.w);
        const unsigned vm1 = max(__vimax3_u32(w1.x, w1.y, w1.z), w1.w);
        u0 = max(u0, vm0);
        u1 = max(u1, vm1);
        vfl |= (vm0 >= thb ? 1u : 0u) << i;
        vfl |= ((ok1 && vm1 >= thb) ? 1u : 0u) << (i + 1);
    }
    const unsigned ut = max(u0, u1);
    if (ut < 0x80000000u) {
        if (FULL || gt < nvec) st.mx = max_nan(st.mx, __uint_as_float(ut));
    } else {
        float mx = st.mx, mn = st.mn;
        for (int i = 0; i < kVecPerThread; ++i) {
            const int v = gt + i * kGroupThreads;
            if (v >= nvec) break;
            const float4 w = *reinterpret_cast<const float4*>(data + v * 16);
            mx = max_nan(mx, max_nan(max_nan(w.x, w.y), max_nan(w.z, w.w)));
            mn = fminf(mn, fminf(fminf(w.x, w.y), fminf(w.z, w.w)));
        }
        st.mx = mx;
        st.mn = mn;
    }
    return vfl;
}

__device__ void q_tile(const Args& a, Smem& sm, GroupSmem& gs, int g, int stage, const StageMeta& m, QState& st) {
    const int gt = threadIdx.x - g * kGroupThreads;
    const int lane = threadIdx.x & 31, warp = gt >> 5;
    const unsigned char* data = sm.data[stage];
    const int k = m.top_k;
    const bool need_cand = k > 0 && k < a.Lq && k <= kMaxCandTopK;
    const bool need_sum = !need_cand && (k == 0 || k >= a.Lq);
    const bool t_one = m.temperature == 1.f;
    const float inv_t = 1.f / m.temperature;
    const long long qrow = static_cast<long long>(m.slot) * a.Lq;
    const int e_tail = m.vec_e0 + m.nvec * 4;
    Cand* const lp = a.cand_q + (static_cast<long long>(m.slot) * a.nseg_q + m.seg) * kCandPenGlobal;
    if (m.first) {
        float mx0 = -INFINITY, mx1 = -INFINITY;
        int v = gt;
        for (; v + kGroupThreads < m.nvec; v += 2 * kGroupThreads) {
            const float4 w0 = *reinterpret_cast<const float4*>(data + v * 16);
            const float4 w1 = *reinterpret_cast<const float4*>(data + (v + kGroupThreads) * 16);
            mx0 = max_nan(max_nan(mx0, w0.x), max_nan(w0.y, max_nan(w0.z, w0.w)));
            mx1 = max_nan(max_nan(mx1, w1.x), max_nan(w1.y, max_nan(w1.z, w1.w)));
        }
        for (; v < m.nvec; v += kGroupThreads) {
            const float4 w = *reinterpret_cast<const float4*>(data + v * 16);
            mx0 = max_nan(max_nan(mx0, w.x), max_nan(w.y, max_nan(w.z, w.w)));
        }
        if (gt < 2) {
            const int lo = gt == 0 ? m.e0 : e_tail, hi = gt == 0 ? m.vec_e0 : m.e1;
            for (int e = lo; e < hi; ++e) mx0 = max_nan(mx0, __ldg(a.q + qrow + e));
        }
        const float mx = max_nan(mx0, mx1);
        float wm = mx;
        for (int o = 16; o; o >>= 1) wm = max_nan(wm, __shfl_xor_sync(0xffffffffu, wm, o));
        float th = 0.f;
        if (need_cand) {
            float s0 = mx, s1 = 0.f;
            warp_sort2_desc(s0, s1);
            th = __shfl_sync(0xffffffffu, s0, (k + kGroupWarps - 1) / kGroupWarps - 1);
        }
        if (lane == 0) gs.red1[warp] = make_float4(wm, -INFINITY, th, INFINITY);
        group_sync(g);
        const float4 r = group_reduce_mmnn(gs.red1);
        st.mx = need_sum && !t_one ? r.x : -INFINITY;     // the tempered sum starts from the tile max
        st.mn = INFINITY;
        st.sum = 0.f;
        st.th = need_cand ? r.z : INFINITY;
    }
    if (need_cand) {
        // common case: vectors in pairs, one flag per vector whose maximum reaches the
        // threshold; the flagged vectors' candidates are extracted afterwards
        const unsigned vfl = m.nvec == kVecPerThread * kGroupThreads ? q_scan_flags<true>(st, data, gt, m.nvec)
                                                                     : q_scan_flags<false>(st, data, gt, m.nvec);
        float m_unused = 0.f;
        int a_unused = 0;
        flush_vectors<4, false, true, false>(gs, lp, vfl, data, nullptr, m.vec_e0, 0, gt, st.th, m_unused, a_unused);
    }
#pragma unroll 2
    for (int i = 0; i < (need_cand ? 0 : kVecPerThread); ++i) {
        const int v = gt + i * kGroupThreads;
        if (v >= m.nvec) break;
        const int e = m.vec_e0 + v * 4;
        const uint4 wu = *reinterpret_cast<const uint4*>(data + v * 16);
        const float4 w = *reinterpret_cast<const float4*>(&wu);
        const float vm = max_nan(max_nan(w.x, w.y), max_nan(w.z, w.w));
        const float vn = fminf(fminf(w.x, w.y), fminf(w.z, w.w));
        if (need_sum && !t_one) {
            if (!(vm <= st.mx)) {
                q_elem(st, w.x, true, false, inv_t, false, gs, lp, e);
                q_elem(st, w.y, true, false, inv_t, false, gs, lp, e + 1);
                q_elem(st, w.z, true, false, inv_t, false, gs, lp, e + 2);
                q_elem(st, w.w, true, false, inv_t, false, gs, lp, e + 3);
            } else {
                st.sum += draft_weight(w.x, st.mx, inv_t, false) + draft_weight(w.y, st.mx, inv_t, false) +
                          draft_weight(w.z, st.mx, inv_t, false) + draft_weight(w.w, st.mx, inv_t, false);
            }
        } else if (need_sum) {
            st.sum += (w.x + w.y) + (w.z + w.w);
        }
        st.mx = max_nan(st.mx, vm);
        st.mn = fminf(st.mn, vn);
    }
    if (gt < 2) {
        const int lo = gt == 0 ? m.e0 : e_tail, hi = gt == 0 ? m.vec_e0 : m.e1;
        for (int e = lo; e < hi; ++e) q_elem(st, __ldg(a.q + qrow + e), need_sum, t_one, inv_t, need_cand, gs, lp, e);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);
}

__device__ void q_finish(const Args& a, GroupSmem& gs, int g, const StageMeta& m, QState& st) {
    const int gt = threadIdx.x - g * kGroupThreads;
    const int lane = threadIdx.x & 31, warp = gt >> 5;
    const int k = m.top_k;
    const bool need_cand = k > 0 && k < a.Lq && k <= kMaxCandTopK;
    const bool need_sum = !need_cand && (k == 0 || k >= a.Lq);
    const bool t_one = m.temperature == 1.f;
    const float inv_t = 1.f / m.temperature;
    float mx = st.mx, mn = st.mn, sum = st.sum;
    float M = mx;
    for (int o = 16; o; o >>= 1) M = max_nan(M, __shfl_xor_sync(0xffffffffu, M, o));
    float mnw = mn;
    for (int o = 16; o; o >>= 1) mnw = fminf(mnw, __shfl_xor_sync(0xffffffffu, mnw, o));
    // sums of (q/mx)^(1/T) are rescaled to the warp max; plain sums of q are not
    float r = sum;
    if (need_sum && !t_one) r = (sum > 0.f && mx > 0.f) ? sum * exp2f(inv_t * log2f(mx / M)) : 0.f;
    r = warp_sum(r);
    if (lane == 0) gs.red[warp] = make_float4(M, r, mnw, 0.f);
    group_sync(g);                                        // partials written, every append done
    const long long ti = static_cast<long long>(m.slot) * a.nseg_q + m.seg;
    if (warp == 0) {
        const float4 v = lane < kGroupWarps ? gs.red[lane] : make_float4(-INFINITY, 0.f, INFINITY, 0.f);
        float Mg = v.x;
        for (int o = 16; o; o >>= 1) Mg = max_nan(Mg, __shfl_xor_sync(0xffffffffu, Mg, o));
        float s = v.y;
        if (need_sum && !t_one) s = (s > 0.f && v.x > 0.f) ? s * exp2f(inv_t * log2f(v.x / Mg)) : 0.f;
        s = warp_sum(s);
        float mnn = v.z;
        for (int o = 16; o; o >>= 1) mnn = fminf(mnn, __shfl_xor_sync(0xffffffffu, mnn, o));
        if (lane == 0) {
            const int n = gs.n_pen;                       // draft segments append no raw entries
            TileStats ts;
            ts.m_raw = Mg; ts.s_raw = t_one ? s : 0.f; ts.m_pen = mnn; ts.arg_pen = 0; ts.s_temp = t_one ? 0.f : s;
            ts.n_pen = need_cand ? n : 0; ts.pad = 0; ts.flags = 0;
            if (need_cand && n > kCandPenGlobal) { ts.flags |= kTileOverflowPen; ts.n_pen = 0; }
            if (!(mnn >= 0.f) || !(Mg <= 3.0e38f)) ts.flags |= kTileBad;
            a.ts_q[ti] = ts;
            // counters for the next segment: its first append follows its first-tile barrier,
            // which this warp reaches only after this write
            gs.n_pen = 0;
        }
    }
}

// Segments in the stream of (CTA c, group g): positions m with c + G*(g + 2m) < S.
__device__ __forceinline__ int stream_len(int S, int G, int c, int g) {
    const int first = c + G * g;
    return first >= S ? 0 : (S - 1 - first) / (2 * G) + 1;
}

// The plan, derived by every CTA from the per-request segment counts: the call's target
// segments come first (request b's at [bx_b, bx_b + nx_b), its rows' in order), then its draft
// segments (request b's at Sx + [bq_b, bq_b + nq_b)), so that the two consumer groups of a
// CTA mostly run the same kind of tile, and one code path, at a time.  Segment s goes to CTA
// s mod G, consumer group (s div G) mod 2, position s div 2G of that group's stream.  The CTA
// writes the descriptors of its own two streams to its slice of the unit array and returns
// the number of segments S.  The exclusive prefixes of the counts are built in the first
// data stage, which no copy has touched yet.  Every thread of the CTA calls it.
__device__ int build_streams(const Args& a, Smem& sm, int c, int G) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int B = a.B;
    int* bx = reinterpret_cast<int*>(sm.data[0]);            // [B + 1]
    int* bq = bx + B + 1;                                     // [B + 1]
    static_assert(sizeof(int) * 2 * (kMaxB + 1) <= kStageBytes, "plan scratch must fit one stage");
    if (tid < 32) {
        // lane l scans its own chunk of requests, then the chunk totals are scanned across lanes
        const int chunk = (B + 31) / 32;
        const int lo = min(B, lane * chunk), hi = min(B, lo + chunk);
        int sx = 0, sq = 0;
        for (int b = lo; b < hi; ++b) { const int nx = a.req_n[B + b]; sx += nx; sq += a.req_n[b] - nx; }
        int ix = sx, iq = sq;
        for (int o = 1; o < 32; o <<= 1) {
            const int yx = __shfl_up_sync(0xffffffffu, ix, o);
            const int yq = __shfl_up_sync(0xffffffffu, iq, o);
            if (lane >= o) { ix += yx; iq += yq; }
        }
        int rx = ix - sx, rq = iq - sq;
        for (int b = lo; b < hi; ++b) {
            const int nx = a.req_n[B + b];
            bx[b] = rx; rx += nx;
            bq[b] = rq; rq += a.req_n[b] - nx;
        }
        if (lane == 31) { bx[B] = ix; bq[B] = iq; }
    }
    __syncthreads();
    const int Sx = bx[B];
    const int S = Sx + bq[B];
    for (int idx = tid; idx < kGroups * a.max_seg; idx += blockDim.x) {
        const int g = idx / a.max_seg, m = idx - g * a.max_seg;
        const long long s = c + static_cast<long long>(G) * (g + 2 * m);
        if (s >= S) continue;
        const bool is_x = s < Sx;
        const int* base = is_x ? bx : bq;
        const int key = static_cast<int>(is_x ? s : s - Sx);
        int l = 0, h = B;                                     // last b with base[b] <= key (and segments)
        while (h - l > 1) {
            const int mid = (l + h) >> 1;
            if (base[mid] <= key) l = mid; else h = mid;
        }
        const int b = l;
        const int local = key - base[b];
        const dspark_row_params_t r = a.rows[b];
        UnitDesc ud;
        ud.b = b;
        int tiles, nseg;
        if (is_x) {
            ud.kind = kUnitX;
            ud.slot = b * (a.Km + 1) + local / a.nseg_x;
            ud.seg = local % a.nseg_x;
            tiles = a.tiles_x; nseg = a.nseg_x;
        } else {
            ud.kind = kUnitQ;
            ud.slot = b * a.Km + local / a.nseg_q;
            ud.seg = local % a.nseg_q;
            tiles = a.tiles_q; nseg = a.nseg_q;
        }
        ud.t0 = static_cast<int>(static_cast<long long>(ud.seg) * tiles / nseg);
        ud.t1 = static_cast<int>(static_cast<long long>(ud.seg + 1) * tiles / nseg);
        ud.temperature = r.temperature;
        ud.top_k = r.top_k;
        ud.top_p = r.top_p;
        ud.presence = r.presence_penalty;
        ud.frequency = r.frequency_penalty;
        ud.pad = 0;
        a.units[(static_cast<long long>(c) * kGroups + g) * a.max_seg + m] = ud;
    }
    __syncthreads();                                          // descriptors written, scratch free
    return S;
}

// ------------------------------------------------------------------ the kernel
template <int SX>
__global__ void __launch_bounds__(kStreamThreads, 1) stream_stats_kernel(Args a) {
    pdl_enter();
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x;
    const int G = gridDim.x;
    const int c = blockIdx.x;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.empty[s], kGroupWarps); }
        for (int g = 0; g < kGroups; ++g) {
            sm.grp[g].n_pen = 0; sm.grp[g].error = 0;
        }
        fence_mbar_init();
    }
    const int S = build_streams(a, sm, c, G);

    if (tid >= kConsumerThreads) {
        // ---------------- producer warp.  Lane 16g+f holds field f of group g's current,
        // next and next-but-one segment descriptors, and the penalty header of tile t0+f of
        // the group's current and next segment; lane 0 issues the copies.
        const int lane = tid & 31;
        const int mg = lane >> 4, ml = lane & 15;
        // the tiles are read once per call: evict-first in L2, so that the 0.8 GB streamed
        // through it do not push out the statistics, candidate lists and penalty index that
        // this and the following kernels write and read
        const uint64_t stream_policy = l2_evict_first_policy();
        constexpr int kFields = sizeof(UnitDesc) / sizeof(int);
        static_assert(kFields <= 16, "descriptor fields must fit a half warp");
        const int* streams = reinterpret_cast<const int*>(a.units + static_cast<long long>(c) * kGroups * a.max_seg);
        const int my_len = stream_len(S, G, c, mg);
        auto load_field = [&](int p) { return (p < my_len && ml < kFields) ? streams[(mg * a.max_seg + p) * kFields + ml] : 0; };
        // field f of group g's descriptor held in register r
        auto fld = [&](int r, int g, int f) { return __shfl_sync(0xffffffffu, r, g * 16 + f); };
        constexpr int F_SLOT = 0, F_KIND = 1, F_B = 2, F_SEG = 3, F_T0 = 4, F_T1 = 5, F_T = 6, F_TOPK = 7,
                      F_TOPP = 8, F_PRES = 9, F_FREQ = 10;
        auto load_hdr = [&](int r) {          // headers of the segment described by register r (own group)
            PenHdr h{0, 0, {0, 0}};
            const int kind = __shfl_sync(0xffffffffu, r, mg * 16 + F_KIND);
            const int b = __shfl_sync(0xffffffffu, r, mg * 16 + F_B);
            const int t0 = __shfl_sync(0xffffffffu, r, mg * 16 + F_T0);
            const int t1 = __shfl_sync(0xffffffffu, r, mg * 16 + F_T1);
            const float pres = __int_as_float(__shfl_sync(0xffffffffu, r, mg * 16 + F_PRES));
            const float freq = __int_as_float(__shfl_sync(0xffffffffu, r, mg * 16 + F_FREQ));
            if (kind == kUnitX && (pres != 0.f || freq != 0.f) && t0 + ml < t1)
                h = a.pen_hdr[static_cast<long long>(b) * a.tiles_x + t0 + ml];
            return h;
        };
        int dcur = load_field(0), dnxt = load_field(1), dnxt2 = load_field(2);
        PenHdr hcur = load_hdr(dcur);
        PenHdr hnxt = load_hdr(dnxt);
        int len0 = stream_len(S, G, c, 0), len1 = stream_len(S, G, c, 1);
        int pos0 = 0, pos1 = 0, iss0 = 0, iss1 = 0;
        int tc0 = fld(dcur, 0, F_T0), tc1 = fld(dcur, 1, F_T0);
        bool failed = false;
        unsigned long long idle = 0;
        while (!failed && (pos0 < len0 || pos1 < len1)) {
            bool progressed = false;
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
                const int pos = g ? pos1 : pos0, len = g ? len1 : len0, iss = g ? iss1 : iss0;
                const int tile = g ? tc1 : tc0;
                if (pos >= len) continue;
                const int stage = g + 2 * (iss & 1);
                const unsigned parity = ((iss >> 1) & 1) ^ 1;
                int ready = 0;
                if (lane == 0) ready = mbar_test_wait(&sm.empty[stage], parity) ? 1 : 0;
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (!ready) continue;
                const int slot = fld(dcur, g, F_SLOT), kind = fld(dcur, g, F_KIND), b = fld(dcur, g, F_B);
                const int seg = fld(dcur, g, F_SEG), t0 = fld(dcur, g, F_T0), t1 = fld(dcur, g, F_T1);
                const float T = __int_as_float(fld(dcur, g, F_T));
                const int topk = fld(dcur, g, F_TOPK);
                const float topp = __int_as_float(fld(dcur, g, F_TOPP));
                const float pres = __int_as_float(fld(dcur, g, F_PRES));
                const float freq = __int_as_float(fld(dcur, g, F_FREQ));
                const int src = g * 16 + (tile - t0);
                const int pn = __shfl_sync(0xffffffffu, hcur.n, src);
                const int pover = __shfl_sync(0xffffffffu, hcur.overflow, src);
                const int pnh = __shfl_sync(0xffffffffu, hcur.pad[0], src);
                if (lane == 0) {
                    StageMeta& m = sm.meta[stage];
                    const bool isx = kind == kUnitX;
                    const int es = isx ? SX : 4;
                    const int tile_n = isx ? a.tile_x : a.tile_q;
                    const int row_n = isx ? a.V : a.Lq;
                    const int e0 = tile * tile_n, e1 = min(row_n, e0 + tile_n);
                    const unsigned char* row = isx
                        ? static_cast<const unsigned char*>(a.x) + static_cast<long long>(slot) * a.V * es
                        : reinterpret_cast<const unsigned char*>(a.q) + static_cast<long long>(slot) * a.Lq * 4;
                    const uintptr_t A0 = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(e0) * es;
                    const uintptr_t A1 = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(e1) * es;
                    uintptr_t c0 = (A0 + 15) & ~static_cast<uintptr_t>(15);
                    uintptr_t c1 = A1 & ~static_cast<uintptr_t>(15);
                    if (c1 < c0) c1 = c0;
                    const unsigned bytes = static_cast<unsigned>(c1 - c0);
                    m.kind = kind; m.slot = slot; m.b = b;
                    m.j = isx ? slot - b * (a.Km + 1) : slot - b * a.Km;
                    m.seg = seg; m.tile = tile; m.e0 = e0; m.e1 = e1;
                    m.nvec = static_cast<int>(bytes / 16);
                    m.vec_e0 = (bytes == 0) ? e1 : e0 + static_cast<int>((c0 - A0) / es);
                    m.pen = isx && (pres != 0.f || freq != 0.f);
                    m.pen_n = pn; m.pen_nh = pnh; m.pen_over = pover;
                    m.top_k = topk; m.first = tile == t0; m.last = tile == t1 - 1;
                    m.temperature = T; m.top_p = topp; m.presence = pres; m.frequency = freq;
                    unsigned tx = bytes;
                    const unsigned bm_bytes = static_cast<unsigned>(a.bm_words) * 4u;
                    const unsigned ent_bytes = m.pen && !pover ? static_cast<unsigned>(pn) * 16u : 0u;
                    if (m.pen) tx += bm_bytes + ent_bytes;
                    mbar_arrive_expect_tx(&sm.full[stage], tx);
                    if (bytes) bulk_g2s_hint(sm.data[stage], reinterpret_cast<const void*>(c0), bytes, &sm.full[stage],
                                             stream_policy);
                    if (m.pen) {
                        const long long pt = static_cast<long long>(b) * a.tiles_x + tile;
                        bulk_g2s(sm.bm[stage], a.pen_bm + pt * a.bm_words, bm_bytes, &sm.full[stage]);
                        if (ent_bytes) bulk_g2s(sm.ent[stage], a.pen_ent + pt * kPenCap, ent_bytes, &sm.full[stage]);
                    }
                }
                progressed = true;
                if (g) { ++iss1; ++tc1; } else { ++iss0; ++tc0; }
                if (tile + 1 >= t1) {
                    // next segment of group g: its descriptor and headers were prefetched
                    const int npos = pos + 1;
                    if (g) pos1 = npos; else pos0 = npos;
                    if (mg == g) {
                        dcur = dnxt;
                        dnxt = dnxt2;
                        hcur = hnxt;
                        dnxt2 = load_field(npos + 2);
                    }
                    if (g) tc1 = fld(dcur, 1, F_T0); else tc0 = fld(dcur, 0, F_T0);
                    // headers of the new next segment (its descriptor is already in registers)
                    const PenHdr h = load_hdr(dnxt);
                    if (mg == g) hnxt = h;
                }
            }
            if (!progressed) {
                if (idle == 0) idle = globaltimer();
                else if (globaltimer() - idle > kIdleNs) failed = true;
                __nanosleep(128);
            } else {
                idle = 0;
            }
        }
        if (failed && lane == 0) atomicOr(&a.plan->pad[0], 1);
        // drain: wait (bounded) for the last copies of each group to land before exiting
        if (lane == 0) {
            for (int r = max(0, iss0 - 2); r < iss0; ++r) wait_phase(&sm.full[0 + 2 * (r & 1)], (r >> 1) & 1);
            for (int r = max(0, iss1 - 2); r < iss1; ++r) wait_phase(&sm.full[1 + 2 * (r & 1)], (r >> 1) & 1);
        }
        return;
    }

    // ---------------- consumer group g: its segments, tile by tile
    const int g = tid / kGroupThreads;
    const int gt = tid - g * kGroupThreads;
    GroupSmem& gs = sm.grp[g];
    const int nseg = stream_len(S, G, c, g);
    // The tile counts come from this group's segment descriptors, so every warp of the group
    // walks the same tiles and meets the same group barriers (one in the first tile's pass,
    // one in a segment's finish) whatever happens to the data; warps are not synchronised
    // tile by tile.  A tile whose wait gave up is skipped with only its barriers, so a warp
    // that gave up and one whose tile arrived still pass the same barriers.
    const UnitDesc* my = a.units + (static_cast<long long>(c) * kGroups + g) * a.max_seg;
    int nt_next = nseg > 0 ? my[0].t1 - my[0].t0 : 0;
    int cnt = 0;                                           // tiles consumed by this group
    XState xs{};
    QState qs{};
    for (int sgi = 0; sgi < nseg; ++sgi) {
        const int ntile = min(nt_next, kMaxSegTiles);
        if (sgi + 1 < nseg) nt_next = my[sgi + 1].t1 - my[sgi + 1].t0;
        for (int ti = 0; ti < ntile; ++ti, ++cnt) {
            const int stage = g + 2 * (cnt & 1);
            const unsigned parity = (cnt >> 1) & 1;
            if (!wait_phase_or_err(&sm.full[stage], parity, &gs.error)) {
                gs.error = 1;
                if (ti == 0) group_sync(g);
                if (ti == ntile - 1) group_sync(g);
                continue;
            }
            StageMeta m = sm.meta[stage];
            const bool last = ti == ntile - 1;
            m.first = ti == 0;                             // barrier decisions follow the descriptor
            m.last = last;
            if (m.kind == kUnitX) {
                const bool greedy = !(m.temperature > 0.f);
                const int k = m.top_k;
                const long long ti = static_cast<long long>(m.slot) * a.nseg_x + m.seg;
                XCtx<SX> ctx{a, sm, gs, g, stage, m, greedy,
                             !greedy && k > 0 && k < a.V && k <= kMaxCandTopK, !greedy && (k == 0 || k >= a.V),
                             m.frequency, m.presence, (!greedy && (k == 0 || k >= a.V)) ? kL2E / m.temperature : 0.f,
                             a.cand_x + ti * kCandPenGlobal};
                x_tile<SX>(ctx, xs);
                if (last) x_finish<SX>(ctx, xs);
            } else {
                q_tile(a, sm, gs, g, stage, m, qs);
                if (last) q_finish(a, gs, g, m, qs);
            }
        }
    }
    if (gt == 0 && gs.error) atomicOr(&a.plan->pad[0], 1);
}

}  // namespace

size_t stream_stats_smem_bytes() { return sizeof(Smem); }

cudaError_t launch_stream_stats(const Args& a, cudaStream_t s, int grid, bool pdl) {
    const size_t smem = sizeof(Smem);
    cudaError_t e;
    if (a.sx == 2) {
        e = cudaFuncSetAttribute(stream_stats_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        e = launch_k(stream_stats_kernel<2>, dim3(grid), dim3(kStreamThreads), smem, s, pdl, a);
    } else {
        e = cudaFuncSetAttribute(stream_stats_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        e = launch_k(stream_stats_kernel<4>, dim3(grid), dim3(kStreamThreads), smem, s, pdl, a);
    }
    return e;
}

}  // namespace dspark
