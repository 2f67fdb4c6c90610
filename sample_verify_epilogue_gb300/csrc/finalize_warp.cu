// row_finalize_warp_kernel: one WARP per verify row, for the rows whose truncated support
// settles from the streaming pass's candidates alone (the common case).  It computes the same
// records as the block-per-row finalize (segment merge, top-k threshold, sorted survivors,
// weights, nucleus; mlx-dspark Changelog, [0.1.0] Added, top-p / top-k sampling;
// [0.20.2] Changed, selection instead of a full vocabulary sort) with warp shuffles and
// per-warp shared memory instead of block barriers: the candidates' order-preserving keys
// are staged (long lists after a first read that bounds the k-th largest key from below, so
// only keys that can be in the top-k are kept), the threshold is selected on them, and the
// survivors are sorted.
// Rows it cannot settle here (more candidates, segments or survivors than a warp holds,
// overflowed candidate lists, rows that need a whole-row pass) are appended to a list that
// row_finalize_kernel then works through.
#include "block_utils.cuh"

namespace dspark {

namespace {

constexpr float kL2E = 1.4426950408889634f;
constexpr int kRowsPerBlockMax = 8;    // warps (rows) per block: 8 when one block per SM covers all rows, else 4
constexpr int kWKeyCap = 2048;         // candidate keys one warp stages
constexpr int kWSegCap = 64;           // segments per row
constexpr int kWSurvCap = 256;         // survivors one warp sorts

struct WarpSmem {
    uint32_t keys[kWKeyCap];
    int ids[kWKeyCap];
    unsigned long long sk[kWSurvCap];  // survivors: (key << 32) | (0xFFFFFFFF - id)
    int off[kWSegCap + 1];             // flat position of each segment's first candidate pair
    int cnt[kWSegCap];                 // candidates of each segment
};

// The row's candidate lists: segment t holds its candidates at base + t*cap.
struct WCands {
    const Cand* base;
    int cap;
    int nseg;
};

__device__ __forceinline__ float nan_max(float a, float b) {
    return (a != a || b != b) ? __int_as_float(0x7fc00000) : fmaxf(a, b);
}

// Walks the row's flat index of candidate pairs (segment l holds pair positions
// [off[l], off[l+1]); pair j of a segment is its candidates 2j and 2j+1, one 16-byte load) in
// increasing order, one position at a time per lane.
struct PairCursor {
    int l, lo, hi;
    __device__ __forceinline__ explicit PairCursor(const WarpSmem& w) : l(0), lo(0), hi(w.off[1]) {}
    // The pair's address; *second = whether its second candidate exists.
    __device__ __forceinline__ const uint4* at(const WarpSmem& w, const WCands& cs, int p, bool* second) {
        while (p >= hi) { ++l; lo = hi; hi = w.off[l + 1]; }
        const int j = p - lo;
        *second = 2 * j + 1 < w.cnt[l];
        return reinterpret_cast<const uint4*>(cs.base + static_cast<long long>(l) * cs.cap) + j;
    }
};

// Stage the keys of the row's candidates (segment t: n_t entries) in shared memory in one read
// of the lists (eight 16-byte loads, sixteen candidates, in flight per lane).  With k > 0
// only keys reaching a lower bound of the k-th largest key are staged: every lane keeps the
// C >= c = ceil(k/32) largest keys it has read, and at least 32c >= k keys reach the least of
// the lanes' c-th largest, so that bound, raised after every batch, never passes a member of
// the top-k (ties included).  Returns the number staged, or -1 when it exceeds kWKeyCap or
// there are more than kWSegCap segments.
constexpr int kWMaxC = 8;                                 // ceil(k / 32) for k <= kMaxCandTopK
static_assert(32 * kWMaxC >= kMaxCandTopK, "per-lane depth must cover k");

template <int C>
__device__ int warp_stage_t(WarpSmem& w, const WCands& cs, int npairs, int c) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    uint32_t top[C];                                      // descending; 0 = nothing yet
#pragma unroll
    for (int q = 0; q < C; ++q) top[q] = 0u;
    uint32_t lb = 0u;
    int m = 0;
    PairCursor cur(w);
    for (int p0 = 0; p0 < npairs; p0 += 32 * 8) {
        uint4 v[8];
        unsigned two = 0u;                                // bit u: pair u has its second candidate
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int p = p0 + lane + 32 * u;
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (p < npairs) {
                bool sec;
                v[u] = *cur.at(w, cs, p, &sec);
                two |= (sec ? 1u : 0u) << u;
            }
        }
        uint32_t key[16];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const bool one = p0 + lane + 32 * u < npairs;
            key[2 * u] = one ? fkey(__uint_as_float(v[u].x)) : 0u;
            key[2 * u + 1] = (one && ((two >> u) & 1u)) ? fkey(__uint_as_float(v[u].z)) : 0u;
        }
        if (c > 0) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                uint32_t x = key[e];
#pragma unroll
                for (int q = 0; q < C; ++q) {             // insertion into the lane's top list
                    const uint32_t t = top[q];
                    const bool sw = x > t;
                    top[q] = sw ? x : t;
                    x = sw ? t : x;
                }
            }
            uint32_t mine = 0u;
#pragma unroll
            for (int q = 0; q < C; ++q) if (q == c - 1) mine = top[q];
            lb = max(lb, __reduce_min_sync(0xffffffffu, mine));
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const bool f = key[e] != 0u && key[e] >= lb;
            const unsigned b = __ballot_sync(0xffffffffu, f);
            const int pos = m + __popc(b & lt);
            if (f && pos < kWKeyCap) {
                w.keys[pos] = key[e];
                w.ids[pos] = static_cast<int>((e & 1) ? v[e >> 1].w : v[e >> 1].y);
            }
            m += __popc(b);
        }
    }
    __syncwarp();
    return m > kWKeyCap ? -1 : m;
}

// lane_n: this lane's segment's candidate count when the caller holds it (rows of at most 32
// segments), else -1.
__device__ int warp_stage(WarpSmem& w, const TileStats* ts, const WCands& cs, int k, int lane_n) {
    const int lane = threadIdx.x & 31;
    if (cs.nseg > kWSegCap) return -1;
    int total = 0, npairs = 0;
    for (int t0 = 0; t0 < cs.nseg; t0 += 32) {
        const int t = t0 + lane;
        const int n = t < cs.nseg ? (lane_n >= 0 ? lane_n : ts[t].n_pen) : 0;
        const int np = (n + 1) >> 1;
        int incl = np;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (t < cs.nseg) { w.off[t] = npairs + incl - np; w.cnt[t] = n; }
        npairs += __shfl_sync(0xffffffffu, incl, 31);
        total += __reduce_add_sync(0xffffffffu, static_cast<unsigned>(n));
    }
    if (lane == 0) w.off[cs.nseg] = npairs;
    __syncwarp();
    if (total == 0) return 0;
    const int c = (k > 0 && k <= 32 * kWMaxC && total > 64) ? (k + 31) / 32 : 0;
    if (c == 0 && total > kWKeyCap) return -1;
    return c <= 1 ? warp_stage_t<1>(w, cs, npairs, c)
         : c == 2 ? warp_stage_t<2>(w, cs, npairs, c)
         : c <= 4 ? warp_stage_t<4>(w, cs, npairs, c)
                  : warp_stage_t<kWMaxC>(w, cs, npairs, c);
}

// k-th largest (1-based, with multiplicity) of the keys keys[0..n), 1 <= k <= n, by a bitwise
// search from the top: the bits above the highest one where the largest and smallest key
// differ are common; below it each bit is set iff at least k keys reach the value with it.
__device__ uint32_t kth_key_bits(const uint32_t* keys, int n, int k) {
    const int lane = threadIdx.x & 31;
    uint32_t mx = 0u, mn = 0xFFFFFFFFu;
    for (int i = lane; i < n; i += 32) { const uint32_t v = keys[i]; mx = max(mx, v); mn = min(mn, v); }
    mx = __reduce_max_sync(0xffffffffu, mx);
    mn = __reduce_min_sync(0xffffffffu, mn);
    if (mx == mn) return mx;
    const int hb = 31 - __clz(mx ^ mn);
    uint32_t prefix = hb == 31 ? 0u : (mx & ~((2u << hb) - 1u));
    for (int b = hb; b >= 0; --b) {
        const uint32_t cand = prefix | (1u << b);
        unsigned c = 0u;
        for (int i = lane; i < n; i += 32) c += keys[i] >= cand ? 1u : 0u;
        if (static_cast<int>(__reduce_add_sync(0xffffffffu, c)) >= k) prefix = cand;
    }
    return prefix;
}

// The same with each lane's keys held in registers (n <= 32 * E).
template <int E>
__device__ uint32_t kth_key_regs(const uint32_t* keys, int n, int k) {
    const int lane = threadIdx.x & 31;
    uint32_t kr[E];
    uint32_t mx = 0u, mn = 0xFFFFFFFFu;
#pragma unroll
    for (int h = 0; h < E; ++h) {
        const int i = lane + 32 * h;
        kr[h] = i < n ? keys[i] : 0u;
        if (i < n) { mx = max(mx, kr[h]); mn = min(mn, kr[h]); }
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    mn = __reduce_min_sync(0xffffffffu, mn);
    if (mx == mn) return mx;
    const int hb = 31 - __clz(mx ^ mn);
    uint32_t prefix = hb == 31 ? 0u : (mx & ~((2u << hb) - 1u));
    for (int b = hb; b >= 0; --b) {
        const uint32_t cand = prefix | (1u << b);
        unsigned c = 0u;
#pragma unroll
        for (int h = 0; h < E; ++h) c += kr[h] >= cand ? 1u : 0u;     // padding keys (0) never count
        if (static_cast<int>(__reduce_add_sync(0xffffffffu, c)) >= k) prefix = cand;
    }
    return prefix;
}

__device__ __forceinline__ uint32_t warp_kth(WarpSmem& w, int n, int k) {
    if (n <= 128) return kth_key_regs<4>(w.keys, n, k);
    if (n <= 512) return kth_key_regs<16>(w.keys, n, k);
    return kth_key_bits(w.keys, n, k);
}

// Staged candidates with key >= kth, sorted by (value desc, id asc) into w.sk[0..count);
// returns the count, or -1 when there are more than kWSurvCap.
__device__ int warp_survivors(WarpSmem& w, int n, uint32_t kth) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    int cnt = 0;
    for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < n ? w.keys[i] : 0u;
        const bool f = i < n && key >= kth;
        const unsigned b = __ballot_sync(0xffffffffu, f);
        const int pos = cnt + __popc(b & lt);
        if (f && pos < kWSurvCap)
            w.sk[pos] = (static_cast<unsigned long long>(key) << 32) |
                        static_cast<unsigned>(0xFFFFFFFFu - static_cast<unsigned>(w.ids[i]));
        cnt += __popc(b);
    }
    if (cnt > kWSurvCap) return -1;
    __syncwarp();
    // sort by rank (keys are distinct): key i goes to the number of keys above it, through the
    // staged-key area, which is free now
    unsigned long long* tmp = reinterpret_cast<unsigned long long*>(w.keys);
    static_assert(sizeof(w.keys) >= kWSurvCap * sizeof(unsigned long long), "rank sort buffer");
    for (int i = lane; i < cnt; i += 32) {
        const unsigned long long x = w.sk[i];
        int r = 0;
        for (int j = 0; j < cnt; ++j) r += w.sk[j] > x;
        tmp[r] = x;
    }
    __syncwarp();
    for (int i = lane; i < cnt; i += 32) w.sk[i] = tmp[i];
    __syncwarp();
    return cnt;
}

// Survivors of the staged keys for a top-k (1 <= k <= n): the k-th largest key, then the keys
// reaching it, sorted.
__device__ int warp_topk_survivors(WarpSmem& w, int n, int k, uint32_t* kth_out = nullptr) {
    const uint32_t kth = warp_kth(w, n, k);
    if (kth_out) *kth_out = kth;
    return warp_survivors(w, n, kth);
}

// Nucleus over the sorted survivors w.sk[0..cnt) with weights wfn(value) (fixed order: up to
// 64 survivors, two interleaved 32-wide scans; more, lane l sums its consecutive chunk, then
// the chunk sums are scanned across lanes).  Kept = the
// tie groups whose exclusive mass is < top_p * Z.  Returns the number kept; *zk = kept mass.
// With `dst`, the kept entries (id, weight) are written there.
template <typename WFn>
__device__ int warp_nucleus(const WarpSmem& w, int cnt, float top_p, WFn wfn, double* zk, KeptEntry* dst) {
    const int lane = threadIdx.x & 31;
    if (cnt <= 64) {
        // up to 64 survivors: element i at lane i % 32, half i / 32; the prefix is two 32-wide
        // shuffle scans side by side (fixed order), not a chain of eight additions per lane
        double wv[2], inc[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = lane + 32 * h;
            wv[h] = i < cnt ? static_cast<double>(wfn(ckey_v(w.sk[i]))) : 0.0;
            inc[h] = wv[h];
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y0 = __shfl_up_sync(0xffffffffu, inc[0], o);
            const double y1 = __shfl_up_sync(0xffffffffu, inc[1], o);
            if (lane >= o) { inc[0] += y0; inc[1] += y1; }
        }
        const double tot0 = __shfl_sync(0xffffffffu, inc[0], 31);
        inc[1] += tot0;
        const double Z = __shfl_sync(0xffffffffu, inc[1], 31);
        // exclusive prefix of element i = the inclusive prefix of element i - 1
        double ex[2];
        ex[0] = __shfl_up_sync(0xffffffffu, inc[0], 1);
        ex[1] = __shfl_up_sync(0xffffffffu, inc[1], 1);
        if (lane == 0) { ex[0] = 0.0; ex[1] = tot0; }
        int kept = cnt;
        if (top_p < 1.f) {
            const double lim = static_cast<double>(top_p) * Z;
            int first_drop = cnt;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h;
                if (i > 0 && i < cnt && (w.sk[i] >> 32) != (w.sk[i - 1] >> 32) && !(ex[h] < lim))
                    first_drop = min(first_drop, i);
            }
            kept = __reduce_min_sync(0xffffffffu, first_drop);
        }
        const double e0 = __shfl_sync(0xffffffffu, ex[0], kept & 31);
        const double e1 = __shfl_sync(0xffffffffu, ex[1], kept & 31);
        *zk = kept == cnt ? Z : (kept >= 32 ? e1 : e0);
        if (dst) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h;
                if (i < kept) dst[i] = KeptEntry{ckey_id(w.sk[i]), static_cast<float>(wv[h])};
            }
        }
        return kept;
    }
    constexpr int kPer = kWSurvCap / 32;
    const int lo = lane * kPer;
    double wv[kPer];
    double sum = 0.0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        wv[q] = lo + q < cnt ? static_cast<double>(wfn(ckey_v(w.sk[lo + q]))) : 0.0;
        sum += wv[q];
    }
    double incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const double Z = __shfl_sync(0xffffffffu, incl, 31);
    double ex = incl - sum;                    // mass strictly before this lane's chunk
    int kept = cnt;
    if (top_p < 1.f) {
        const double lim = static_cast<double>(top_p) * Z;
        int first_drop = cnt;
        double run = ex;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = lo + q;
            if (i > 0 && i < cnt && (w.sk[i] >> 32) != (w.sk[i - 1] >> 32) && !(run < lim) && first_drop == cnt)
                first_drop = i;
            run += wv[q];
        }
        for (int o = 16; o; o >>= 1) first_drop = min(first_drop, __shfl_xor_sync(0xffffffffu, first_drop, o));
        kept = first_drop;
    }
    // kept mass: exclusive prefix at index `kept`, held by the lane whose chunk contains it
    double at = ex;
#pragma unroll
    for (int q = 0; q < kPer; ++q) if (lo + q < kept) at += wv[q];
    const int owner = min(31, kept / kPer);
    double zkept = __shfl_sync(0xffffffffu, at, owner);
    if (kept == cnt) zkept = Z;
    *zk = zkept;
    if (dst) {
#pragma unroll
        for (int q = 0; q < kPer; ++q)
            if (lo + q < kept) dst[lo + q] = KeptEntry{ckey_id(w.sk[lo + q]), static_cast<float>(wv[q])};
    }
    return kept;
}

// Target row (b, j).  Returns false when the row needs the block path (nothing final written).
__device__ bool warp_finalize_x(WarpSmem& w, const Args& a, int slot, int b) {
    const int lane = threadIdx.x & 31;
    const dspark_row_params_t r = a.rows[b];
    const int nseg = a.nseg_x;
    const TileStats* ts = a.ts_x + static_cast<long long>(slot) * nseg;
    // each lane's segment statistics, read once when the row has at most 32 segments
    const bool cached = nseg <= 32;
    TileStats mine{};
    if (cached && lane < nseg) mine = ts[lane];
    float mr = -INFINITY, mp = -INFINITY;
    int fl = 0;
    for (int t = lane; t < nseg; t += 32) {
        const TileStats x = cached ? mine : ts[t];
        mr = nan_max(mr, x.m_raw);
        mp = nan_max(mp, x.m_pen);
        fl |= x.flags;
    }
    for (int o = 16; o; o >>= 1) {
        mr = nan_max(mr, __shfl_xor_sync(0xffffffffu, mr, o));
        mp = nan_max(mp, __shfl_xor_sync(0xffffffffu, mp, o));
        fl |= __shfl_xor_sync(0xffffffffu, fl, o);
    }
    XRowOut o{};
    o.mode = kModeInactive;
    o.kth = -INFINITY;
    if ((fl & kTileBad) || !isfinite(mr) || !isfinite(mp)) {
        if (lane == 0) {
            atomicOr(&a.row_status[b], DSPARK_ROW_NONFINITE);
            a.xout[slot] = o;
        }
        return true;
    }
    const bool greedy = !(r.temperature > 0.f);
    const float c_l2e = greedy ? 0.f : kL2E / r.temperature;
    const int k = r.top_k;
    const bool list = !greedy && k > 0 && k < a.V;
    // rows that need a whole-row pass go to the block path straight away
    if (!greedy && !list && r.top_p < 1.f) return false;
    if (list && (k > kMaxCandTopK || (fl & kTileOverflowPen))) return false;
    int arg = 0x7FFFFFFF;
    double stemp = 0.0;
    for (int t = lane; t < nseg; t += 32) {
        const TileStats x = cached ? mine : ts[t];
        if (x.m_pen == mp) arg = min(arg, x.arg_pen);
        // the tempered sum is the normaliser of a row without a top-k list only
        if (!greedy && !list) stemp += static_cast<double>(x.s_temp) * static_cast<double>(exp2f((x.m_pen - mp) * c_l2e));
    }
    for (int off = 16; off; off >>= 1) {
        arg = min(arg, __shfl_xor_sync(0xffffffffu, arg, off));
        stemp += __shfl_xor_sync(0xffffffffu, stemp, off);
    }
    o.argmax = arg;
    o.m_pen = mp;
    o.c_l2e = c_l2e;
    o.top_p = r.top_p;
    o.tau = -INFINITY;
    o.top_k = 0;
    o.n_kept = 0;
    o.flags = fl;
    if (greedy) {
        o.mode = kModeGreedy;
    } else if (list) {
        const WCands cs{a.cand_x + static_cast<long long>(slot) * nseg * kCandPenGlobal, kCandPenGlobal, nseg};
        const int n = warp_stage(w, ts, cs, k, cached ? mine.n_pen : -1);
        if (n < k) return false;               // too many candidates to stage, or fewer than k
        uint32_t kth = 0u;
        const int cnt = warp_topk_survivors(w, n, k, &kth);
        if (cnt <= 0) return false;
        o.kth = key_to_f(kth);
        double zk;
        const int kept = warp_nucleus(w, cnt, r.top_p, [&](float v) { return target_weight(v, mp, c_l2e); }, &zk,
                                      a.kept + static_cast<long long>(slot) * kKeptCap);
        o.mode = kModeList;
        o.n_kept = kept;
        o.Z = zk;
        o.tau = ckey_v(w.sk[kept - 1]);
        __syncwarp();
    } else {
        o.Z = stemp;
        o.mode = kModeFull;                    // top_p >= 1 here
    }
    if (lane == 0) a.xout[slot] = o;
    return true;
}

// Draft row (b, i).  Returns false when the row needs the block path.
__device__ bool warp_finalize_q(WarpSmem& w, const Args& a, int qslot, int b) {
    const int lane = threadIdx.x & 31;
    const dspark_row_params_t r = a.rows[b];
    const int nseg = a.nseg_q;
    const TileStats* ts = a.ts_q + static_cast<long long>(qslot) * nseg;
    const bool cached = nseg <= 32;
    TileStats mine{};
    if (cached && lane < nseg) mine = ts[lane];
    float qmax = -INFINITY;
    int fl = 0;
    for (int t = lane; t < nseg; t += 32) {
        const TileStats x = cached ? mine : ts[t];
        qmax = nan_max(qmax, x.m_raw);
        fl |= x.flags;
    }
    for (int o = 16; o; o >>= 1) {
        qmax = nan_max(qmax, __shfl_xor_sync(0xffffffffu, qmax, o));
        fl |= __shfl_xor_sync(0xffffffffu, fl, o);
    }
    const bool t_one = r.temperature == 1.f;
    const float inv_t = 1.f / r.temperature;
    double z = 0.0;
    for (int t = lane; t < nseg; t += 32) {
        const TileStats x = cached ? mine : ts[t];
        if (t_one) z += static_cast<double>(x.s_raw);
        else if (x.m_raw > 0.f)
            z += static_cast<double>(x.s_temp) * static_cast<double>(exp2f(inv_t * log2f(x.m_raw / qmax)));
    }
    for (int off = 16; off; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    QRowOut o{};
    o.mode = kModeInactive;
    if ((fl & kTileBad) || !(qmax > 0.f) || !isfinite(qmax)) {
        if (lane == 0) { atomicOr(&a.row_status[b], DSPARK_ROW_NONFINITE); a.qout[qslot] = o; }
        return true;
    }
    if (a.Lq <= kWSurvCap) {
        // a short draft row (sparse pairs, a small draft vocabulary): settled from its values
        const long long base = static_cast<long long>(qslot) * a.Lq;
        for (int e = lane; e < a.Lq; e += 32) {
            w.keys[e] = fkey(__ldg(a.q + base + e));
            w.ids[e] = e;
        }
        __syncwarp();
        const int kk = r.top_k;
        const int cnt = warp_topk_survivors(w, a.Lq, (kk > 0 && kk < a.Lq) ? kk : a.Lq);
        double zk;
        const int kept = warp_nucleus(w, cnt, r.top_p,
                                      [&](float v) { return draft_weight(v, qmax, inv_t, t_one); }, &zk, nullptr);
        o.qmax = qmax;
        o.inv_t = inv_t;
        o.top_k = 0;
        o.top_p = r.top_p;
        o.flags = fl;
        o.mode = kModeList;
        o.Z = zk;
        o.tau = ckey_v(w.sk[kept - 1]);
        __syncwarp();
        if (lane == 0) a.qout[qslot] = o;
        return true;
    }
    const int k = r.top_k;
    const bool list = k > 0 && k < a.Lq;
    if (!list && r.top_p < 1.f) return false;
    if (list && (k > kMaxCandTopK || (fl & kTileOverflowPen))) return false;
    o.qmax = qmax;
    o.inv_t = inv_t;
    o.tau = -INFINITY;
    o.top_k = 0;
    o.top_p = r.top_p;
    o.flags = fl;
    if (list) {
        const WCands cs{a.cand_q + static_cast<long long>(qslot) * nseg * kCandPenGlobal, kCandPenGlobal, nseg};
        const int n = warp_stage(w, ts, cs, k, cached ? mine.n_pen : -1);
        if (n < k) return false;
        const int cnt = warp_topk_survivors(w, n, k);
        if (cnt <= 0) return false;
        double zk;
        const int kept = warp_nucleus(w, cnt, r.top_p,
                                      [&](float v) { return draft_weight(v, qmax, inv_t, t_one); }, &zk, nullptr);
        o.mode = kModeList;
        o.Z = zk;
        o.tau = ckey_v(w.sk[kept - 1]);
        __syncwarp();
    } else {
        o.Z = z;
        o.mode = kModeFull;
        if (!(z > 0.0)) {
            if (lane == 0) atomicOr(&a.row_status[b], DSPARK_ROW_NONFINITE);
        }
    }
    if (lane == 0) a.qout[qslot] = o;
    return true;
}

// Blocks of up to 32 * kRowsPerBlockMax threads; the register cap keeps the kernel free of spills
// (the compiler's default for 256-thread blocks spilled).
__global__ void __maxnreg__(96) row_finalize_warp_kernel(Args a) {
    pdl_enter();
    // a bounded wait of the streaming pass gave up: its statistics are incomplete and every
    // request reports DSPARK_ROW_INTERNAL, so nothing here may read them
    if (a.plan->pad[0]) return;
    extern __shared__ __align__(16) unsigned char wfin_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WarpSmem& w = reinterpret_cast<WarpSmem*>(wfin_raw)[warp];
    const int row = blockIdx.x * static_cast<int>(blockDim.x >> 5) + warp;
    if (row >= a.xslots + a.qslots) return;
    bool done = true;
    if (row < a.xslots) {
        const int b = row / (a.Km + 1), j = row % (a.Km + 1);
        if ((a.row_status[b] & (DSPARK_ROW_BAD_PARAMS | DSPARK_ROW_BAD_DRAFT)) || j > a.rows[b].num_drafts) {
            if (lane == 0) { XRowOut o{}; o.mode = kModeInactive; o.kth = -INFINITY; a.xout[row] = o; }
        } else {
            done = warp_finalize_x(w, a, row, b);
        }
    } else {
        const int qs = row - a.xslots;
        const int b = qs / a.Km, i = qs % a.Km;
        const dspark_row_params_t r = a.rows[b];
        if ((a.row_status[b] & (DSPARK_ROW_BAD_PARAMS | DSPARK_ROW_BAD_DRAFT)) || i >= r.num_drafts ||
            !(r.temperature > 0.f)) {
            if (lane == 0) { QRowOut o{}; o.mode = kModeInactive; a.qout[qs] = o; }
        } else {
            done = warp_finalize_q(w, a, qs, b);
        }
    }
    if (!done && lane == 0) {
        const int p = atomicAdd(&a.fin_list[0], 1);
        a.fin_list[1 + p] = row;
    }
}

}  // namespace

cudaError_t launch_row_finalize_warp(const Args& a, cudaStream_t s, bool pdl) {
    const int rows = a.xslots + a.qslots;
    // all rows in one wave of one 8-warp block per SM when they fit (measured 1-1.5 us shorter
    // than 4-warp blocks at B=64); more rows: 4-warp blocks, three per SM
    const int rpb = rows <= kRowsPerBlockMax * a.grid_ss ? kRowsPerBlockMax : 4;
    const int grid = (rows + rpb - 1) / rpb;
    const size_t smem = sizeof(WarpSmem) * rpb;
    cudaError_t e = cudaFuncSetAttribute(row_finalize_warp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_k(row_finalize_warp_kernel, dim3(grid), dim3(32 * rpb), smem, s, pdl, a);
}

}  // namespace dspark
