// row_finalize_warp_kernel: one WARP per verify row, for the rows whose truncated support
// settles from the streaming pass's candidates alone (the common case).  It computes the same
// records as the block-per-row finalize (segment merge, top-k threshold, sorted survivors,
// weights, nucleus, raw top-n; mlx-dspark Changelog, [0.1.0] Added, top-p / top-k sampling;
// [0.20.2] Changed, selection instead of a full vocabulary sort) with warp shuffles and
// per-warp shared memory instead of block barriers: the candidates' order-preserving keys
// are staged, the threshold is selected on them, and only the survivors' ids are fetched.
// Rows it cannot settle here (more candidates, segments or survivors than a warp holds,
// overflowed candidate lists, rows that need a whole-row pass) are appended to a list that
// row_finalize_kernel then works through.
#include "block_utils.cuh"

namespace dspark {

namespace {

constexpr float kL2E = 1.4426950408889634f;
constexpr int kRowsPerBlock = 4;       // warps (rows) per block
constexpr int kWKeyCap = 2048;         // candidate keys one warp stages
constexpr int kWSegCap = 64;           // segments per row
constexpr int kWSurvCap = 256;         // survivors one warp sorts

struct WarpSmem {
    uint32_t keys[kWKeyCap];
    int ids[kWKeyCap];
    unsigned long long sk[kWSurvCap];  // survivors: (key << 32) | (0xFFFFFFFF - id)
    int off[kWSegCap + 1];             // staged position of each segment's first candidate
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

// Stage the keys of the row's candidates (segment t: n_t entries) in shared memory, with the
// segment offsets; all segments' loads are issued together (flat index -> segment from the
// offsets).  Returns the total, or -1 when it exceeds kWKeyCap or there are more than
// kWSegCap segments.
__device__ int warp_stage(WarpSmem& w, const TileStats* ts, const WCands& cs, bool raw) {
    const int lane = threadIdx.x & 31;
    if (cs.nseg > kWSegCap) return -1;
    int total = 0;
    for (int t0 = 0; t0 < cs.nseg; t0 += 32) {
        const int t = t0 + lane;
        const int n = t < cs.nseg ? (raw ? ts[t].n_raw : ts[t].n_pen) : 0;
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (t < cs.nseg) w.off[t] = total + incl - n;
        total += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (total > kWKeyCap) return -1;
    if (lane == 0) w.off[cs.nseg] = total;
    __syncwarp();
    for (int i0 = lane; i0 < total; i0 += 512) {             // sixteen loads in flight per lane
        Cand v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int i = i0 + 32 * u;
            if (i < total) {
                int l = 0, h = cs.nseg;                       // segment with off[l] <= i < off[l+1]
                while (h - l > 1) {
                    const int mid = (l + h) >> 1;
                    if (w.off[mid] <= i) l = mid; else h = mid;
                }
                v[u] = cs.base[static_cast<long long>(l) * cs.cap + (i - w.off[l])];
            }
        }
#pragma unroll
        for (int u = 0; u < 16; ++u)
            if (i0 + 32 * u < total) { w.keys[i0 + 32 * u] = fkey(v[u].v); w.ids[i0 + 32 * u] = v[u].id; }
    }
    __syncwarp();
    return total;
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

__device__ __forceinline__ uint32_t warp_kth(WarpSmem& w, int n, int k) { return kth_key_bits(w.keys, n, k); }

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
    const int P = next_pow2(max(cnt, 2));
    for (int i = cnt + lane; i < P; i += 32) w.sk[i] = 0ull;
    __syncwarp();
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = lane; i < P / 2; i += 32) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const unsigned long long x = w.sk[lo], y = w.sk[hi];
                if ((x < y) == desc) { w.sk[lo] = y; w.sk[hi] = x; }
            }
            __syncwarp();
        }
    }
    return cnt;
}

// Nucleus over the sorted survivors w.sk[0..cnt) with weights wfn(value) (fixed order: lane
// l sums its consecutive chunk, then the chunk sums are scanned across lanes).  Kept = the
// tie groups whose exclusive mass is < top_p * Z.  Returns the number kept; *zk = kept mass.
// With `dst`, the kept entries (id, weight) are written there.
template <typename WFn>
__device__ int warp_nucleus(const WarpSmem& w, int cnt, float top_p, WFn wfn, double* zk, KeptEntry* dst) {
    const int lane = threadIdx.x & 31;
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

// Raw top-n list of a target row from its raw candidates; false when it needs the block path.
__device__ bool warp_topn(WarpSmem& w, const Args& a, const TileStats* ts, int slot) {
    const int lane = threadIdx.x & 31;
    const int nseg = a.nseg_x;
    const WCands cs{a.cand_raw + static_cast<long long>(slot) * nseg * kCandRawGlobal, kCandRawGlobal, nseg};
    const int n = warp_stage(w, ts, cs, true);
    const int nt = min(a.n_top, a.V);
    if (n < nt) return false;                  // also n = -1
    const uint32_t kth = warp_kth(w, n, nt);
    const int cnt = warp_survivors(w, n, kth);
    if (cnt < nt) return false;
    TopEntry* dst = a.topn + static_cast<long long>(slot) * DSPARK_MAX_TOP_LOGPROBS;
    for (int i = lane; i < nt; i += 32) dst[i] = TopEntry{ckey_id(w.sk[i]), ckey_v(w.sk[i])};
    __syncwarp();
    return true;
}

// Target row (b, j).  Returns false when the row needs the block path (nothing final written).
__device__ bool warp_finalize_x(WarpSmem& w, const Args& a, int slot, int b) {
    const int lane = threadIdx.x & 31;
    const dspark_row_params_t r = a.rows[b];
    const int nseg = a.nseg_x;
    const TileStats* ts = a.ts_x + static_cast<long long>(slot) * nseg;
    float mr = -INFINITY, mp = -INFINITY;
    int fl = 0;
    for (int t = lane; t < nseg; t += 32) {
        const TileStats x = ts[t];
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
    if (a.n_top > 0 && (fl & kTileOverflowRaw)) return false;
    int arg = 0x7FFFFFFF;
    double sraw = 0.0, stemp = 0.0;
    for (int t = lane; t < nseg; t += 32) {
        const TileStats x = ts[t];
        if (x.m_pen == mp) arg = min(arg, x.arg_pen);
        sraw += static_cast<double>(x.s_raw) * exp2(static_cast<double>(x.m_raw - mr) * kL2E);
        if (!greedy) stemp += static_cast<double>(x.s_temp) * exp2(static_cast<double>(x.m_pen - mp) * c_l2e);
    }
    for (int off = 16; off; off >>= 1) {
        arg = min(arg, __shfl_xor_sync(0xffffffffu, arg, off));
        sraw += __shfl_xor_sync(0xffffffffu, sraw, off);
        stemp += __shfl_xor_sync(0xffffffffu, stemp, off);
    }
    o.argmax = arg;
    o.m_pen = mp;
    o.lse = mr + static_cast<float>(log(sraw));
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
        const int n = warp_stage(w, ts, cs, false);
        if (n < k) return false;               // too many candidates to stage, or fewer than k
        const uint32_t kth = warp_kth(w, n, k);
        const int cnt = warp_survivors(w, n, kth);
        if (cnt <= 0) return false;
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
    if (a.n_top > 0 && !warp_topn(w, a, ts, slot)) return false;
    if (lane == 0) a.xout[slot] = o;
    return true;
}

// Draft row (b, i).  Returns false when the row needs the block path.
__device__ bool warp_finalize_q(WarpSmem& w, const Args& a, int qslot, int b) {
    const int lane = threadIdx.x & 31;
    const dspark_row_params_t r = a.rows[b];
    const int nseg = a.nseg_q;
    const TileStats* ts = a.ts_q + static_cast<long long>(qslot) * nseg;
    float qmax = -INFINITY;
    int fl = 0;
    for (int t = lane; t < nseg; t += 32) {
        const TileStats x = ts[t];
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
        const TileStats x = ts[t];
        if (t_one) z += static_cast<double>(x.s_raw);
        else if (x.m_raw > 0.f)
            z += static_cast<double>(x.s_temp) * exp2(static_cast<double>(inv_t) * log2(static_cast<double>(x.m_raw) / qmax));
    }
    for (int off = 16; off; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    QRowOut o{};
    o.mode = kModeInactive;
    if ((fl & kTileBad) || !(qmax > 0.f) || !isfinite(qmax)) {
        if (lane == 0) { atomicOr(&a.row_status[b], DSPARK_ROW_NONFINITE); a.qout[qslot] = o; }
        return true;
    }
    const int k = r.top_k;
    const bool list = k > 0 && k < a.V;
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
        const int n = warp_stage(w, ts, cs, false);
        if (n < k) return false;
        const uint32_t kth = warp_kth(w, n, k);
        const int cnt = warp_survivors(w, n, kth);
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

// ------------------------------------------------------------------ segment trimming
// Every member of a row's top-k (ties included) that lies in segment s is also among s's
// own top-k (with ties): s holds fewer than k values above the row's k-th largest.  So each
// segment's candidate list can be cut to its own top-k before the row-level selection, one
// warp per list, all lists at once.
constexpr int kTrimCap = 1536;         // longest list (the global caps)
constexpr int kTrimStage = 512;        // survivors of the first stage kept for the exact second
constexpr int kTrimMaxC = 8;           // ceil(k / 32) for k <= kMaxCandTopK

struct TrimSmem {
    uint32_t keys[kTrimStage];
    int ids[kTrimStage];
};
static_assert(kTrimCap >= kCandPenGlobal && kTrimCap >= kCandRawGlobal, "a whole list must fit");
static_assert(32 * kTrimMaxC >= kMaxCandTopK, "per-lane depth must cover k");

// Cut the list c[0..*n) down towards its own top-k (ties kept), in place, *n updated.
//   1. Each lane keeps the c = ceil(k/32) largest keys of its share; the least of the
//      lanes' c-th largest is a lower bound of the list's k-th largest (32c >= k keys reach it).
//   2. The entries at or above that bound are compacted over the list's front; when at most
//      kTrimStage remain they are also staged, the exact k-th largest is found among them
//      and only the entries reaching it are kept.
__device__ void trim_list(TrimSmem& w, Cand* c, int* n_io, int k) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    const int n = *n_io;
    if (n <= k || n > kTrimCap) return;
    const int cdepth = (k + 31) / 32;
    uint32_t top[kTrimMaxC];                              // descending; 0 = nothing yet
#pragma unroll
    for (int q = 0; q < kTrimMaxC; ++q) top[q] = 0u;
    for (int i0 = lane; i0 < n; i0 += 512) {              // sixteen loads in flight per lane
        float v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) if (i0 + 32 * u < n) v[u] = c[i0 + 32 * u].v;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            uint32_t x = i0 + 32 * u < n ? fkey(v[u]) : 0u;
#pragma unroll
            for (int q = 0; q < kTrimMaxC; ++q) {         // insertion into the lane's top list
                const bool sw = q < cdepth && x > top[q];
                const uint32_t t = top[q];
                top[q] = sw ? x : t;
                x = sw ? t : x;
            }
        }
    }
    uint32_t lb = 0u;
#pragma unroll
    for (int q = 0; q < kTrimMaxC; ++q) if (q == cdepth - 1) lb = top[q];
    lb = __reduce_min_sync(0xffffffffu, lb);
    // stage 1: keep key >= lb (each batch is read before any of it is written; writes land at
    // or below the batch being read)
    int m = 0;
    for (int i0 = 0; i0 < n; i0 += 512) {
        Cand e[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) { const int i = i0 + lane + 32 * u; if (i < n) e[u] = c[i]; }
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int i = i0 + lane + 32 * u;
            const uint32_t key = i < n ? fkey(e[u].v) : 0u;
            const bool f = i < n && key >= lb;
            const unsigned b = __ballot_sync(0xffffffffu, f);
            const int pos = m + __popc(b & lt);
            if (f) {
                c[pos] = e[u];
                if (pos < kTrimStage) { w.keys[pos] = key; w.ids[pos] = e[u].id; }
            }
            m += __popc(b);
        }
        __syncwarp();
    }
    if (m > kTrimStage) {                                 // keep the stage-1 result
        if (lane == 0) *n_io = m;
        __syncwarp();
        return;
    }
    // stage 2: exact k-th largest among the m staged entries
    const uint32_t kth = kth_key_bits(w.keys, m, k);
    int r = 0;
    for (int base = 0; base < m; base += 32) {
        const int i = base + lane;
        const bool f = i < m && w.keys[i] >= kth;
        const unsigned b = __ballot_sync(0xffffffffu, f);
        if (f) c[r + __popc(b & lt)] = Cand{key_to_f(w.keys[i]), w.ids[i]};
        r += __popc(b);
    }
    if (lane == 0) *n_io = r;
    __syncwarp();
}

__global__ void __launch_bounds__(32 * kRowsPerBlock) cand_trim_kernel(Args a) {
    pdl_enter();
    extern __shared__ __align__(16) unsigned char trim_raw[];
    const int warp = threadIdx.x >> 5;
    TrimSmem& w = reinterpret_cast<TrimSmem*>(trim_raw)[warp];
    const long long gw = static_cast<long long>(blockIdx.x) * kRowsPerBlock + warp;
    const long long nx = static_cast<long long>(a.xslots) * a.nseg_x;
    if (gw < nx) {
        const int slot = static_cast<int>(gw / a.nseg_x), t = static_cast<int>(gw % a.nseg_x);
        const int b = slot / (a.Km + 1), j = slot % (a.Km + 1);
        const dspark_row_params_t r = a.rows[b];
        if ((a.row_status[b] & (DSPARK_ROW_BAD_PARAMS | DSPARK_ROW_BAD_DRAFT)) || j > r.num_drafts) return;
        TileStats* ts = a.ts_x + static_cast<long long>(slot) * a.nseg_x + t;
        const long long ti = static_cast<long long>(slot) * a.nseg_x + t;
        const int fl = ts->flags;
        const int k = r.top_k;
        if (r.temperature > 0.f && k > 0 && k < a.V && k <= kMaxCandTopK && !(fl & kTileOverflowPen))
            trim_list(w, a.cand_x + ti * kCandPenGlobal, &ts->n_pen, k);
        if (a.n_top > 0 && !(fl & kTileOverflowRaw))
            trim_list(w, a.cand_raw + ti * kCandRawGlobal, &ts->n_raw, min(a.n_top, a.V));
    } else {
        const long long gq = gw - nx;
        if (gq >= static_cast<long long>(a.qslots) * a.nseg_q) return;
        const int qs = static_cast<int>(gq / a.nseg_q), t = static_cast<int>(gq % a.nseg_q);
        const int b = qs / a.Km, i = qs % a.Km;
        const dspark_row_params_t r = a.rows[b];
        if ((a.row_status[b] & (DSPARK_ROW_BAD_PARAMS | DSPARK_ROW_BAD_DRAFT)) || i >= r.num_drafts ||
            !(r.temperature > 0.f)) return;
        TileStats* ts = a.ts_q + static_cast<long long>(qs) * a.nseg_q + t;
        const int k = r.top_k;
        if (k > 0 && k < a.V && k <= kMaxCandTopK && !(ts->flags & kTileOverflowPen))
            trim_list(w, a.cand_q + gq * kCandPenGlobal, &ts->n_pen, k);
    }
}

__global__ void __launch_bounds__(32 * kRowsPerBlock) row_finalize_warp_kernel(Args a) {
    pdl_enter();
    extern __shared__ __align__(16) unsigned char wfin_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WarpSmem& w = reinterpret_cast<WarpSmem*>(wfin_raw)[warp];
    const int row = blockIdx.x * kRowsPerBlock + warp;
    if (row >= a.xslots + a.qslots) return;
    bool done = true;
    if (row < a.xslots) {
        const int b = row / (a.Km + 1), j = row % (a.Km + 1);
        if ((a.row_status[b] & (DSPARK_ROW_BAD_PARAMS | DSPARK_ROW_BAD_DRAFT)) || j > a.rows[b].num_drafts) {
            if (lane == 0) { XRowOut o{}; o.mode = kModeInactive; a.xout[row] = o; }
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

cudaError_t launch_row_finalize_warp(const Args& a, cudaStream_t s, bool pdl_first) {
    {
        const long long lists = static_cast<long long>(a.xslots) * a.nseg_x + static_cast<long long>(a.qslots) * a.nseg_q;
        const int grid = static_cast<int>((lists + kRowsPerBlock - 1) / kRowsPerBlock);
        const size_t smem = sizeof(TrimSmem) * kRowsPerBlock;
        cudaError_t e = cudaFuncSetAttribute(cand_trim_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        e = launch_k(cand_trim_kernel, dim3(grid), dim3(32 * kRowsPerBlock), smem, s, pdl_first, a);
        if (e != cudaSuccess) return e;
    }
    const int rows = a.xslots + a.qslots;
    const int grid = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    const size_t smem = sizeof(WarpSmem) * kRowsPerBlock;
    cudaError_t e = cudaFuncSetAttribute(row_finalize_warp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_k(row_finalize_warp_kernel, dim3(grid), dim3(32 * kRowsPerBlock), smem, s, true, a);
}

}  // namespace dspark
