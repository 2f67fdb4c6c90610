// row_finalize_kernel: one CTA per verify row left by the warp finalize (target position (b, j)
// or draft position (b, i)).  Merges the per-segment statistics of the streaming pass and settles the row's
// truncated distribution:
//   - target rows: penalised max and argmax (greedy), the top-k
//     threshold tau_k = k-th largest penalised logit among the merged segment candidates (exact:
//     every member of the row's top-k is a candidate of its own segment), the survivors
//     {x' >= tau_k} sorted by (value desc, id asc), their weights exp((x'-max)/T), and the
//     nucleus: a survivor is kept iff the renormalised mass strictly above its value is
//     < top_p (mlx-dspark Changelog, [0.1.0] Added, top-p / top-k on draft and target;
//     [0.20.2] Changed, selection instead of a full vocabulary sort);
//   - draft rows: the same with q as the key and (q/qmax)^(1/T) as the weight.
// Rows whose support is not a short list (no top-k, or more survivors than fit) keep a
// threshold and a normaliser instead; those that still need a whole-row threshold get it in
// the same block from the whole-row path below.
#include "block_utils.cuh"

namespace dspark {

namespace {

constexpr float kL2E = 1.4426950408889634f;
constexpr int kFinThreads = 256;
constexpr int kKeyCap = 4096;          // candidate keys staged in shared memory
constexpr int kMaxSegs = 1024;         // segments per row (V <= 2^24 with 12,288-element tiles: 228)

struct FinSmem {
    union {
        uint32_t keys[kKeyCap];        // candidate keys (selection)
        double ex[kKeptCap + 1];       // exclusive prefix of survivor weights (nucleus)
    } u;
    unsigned long long sk[kKeptCap];   // survivors: (key << 32) | (0xFFFFFFFF - id)
    double w[kKeptCap];
    int off[kMaxSegs + 1];             // candidate offsets per segment
    int whist[kFinThreads / 32][256];  // per-warp radix histograms
    int hist[256];
    int bcast[4];
    double dwarp[33];
    float fwarp[32];
    int iwarp[32];
    int n;
    int staged;
};

// The candidate lists of one row: segment s holds n_s (value, id) pairs at base + s*cap.
struct CandSet {
    const Cand* base;
    int cap;
    int nseg;
    int total;
};

// Offsets of the row's candidate lists (from the segment statistics) and, when they fit, the
// keys staged in shared memory.  Returns the set, total = -1 when any list overflowed.
__device__ CandSet stage_candidates(FinSmem& s, const TileStats* ts, const Cand* base, int cap, int nseg) {
    const int tid = threadIdx.x;
    CandSet cs{base, cap, nseg, 0};
    if (nseg > kMaxSegs) { cs.total = -1; return cs; }
    for (int t = tid; t < nseg; t += blockDim.x) s.off[t + 1] = ts[t].n_pen;
    __syncthreads();
    if (tid == 0) {
        s.off[0] = 0;
        for (int t = 1; t <= nseg; ++t) s.off[t] += s.off[t - 1];
        s.staged = s.off[nseg] <= kKeyCap;
    }
    __syncthreads();
    cs.total = s.off[nseg];
    if (s.staged) {
        const int warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
        for (int t = warp; t < nseg; t += nw) {
            const int o = s.off[t], n = s.off[t + 1] - o;
            const Cand* src = base + static_cast<long long>(t) * cap;
            for (int i = lane; i < n; i += 32) s.u.keys[o + i] = fkey(src[i].v);
        }
    }
    __syncthreads();
    return cs;
}

// Call fn(key) for every candidate (each thread a share), from shared memory when staged.
template <typename Fn>
__device__ __forceinline__ void for_each_key(const FinSmem& s, const CandSet& cs, Fn fn) {
    const int tid = threadIdx.x;
    if (s.staged) {
        for (int i = tid; i < cs.total; i += blockDim.x) fn(s.u.keys[i]);
    } else {
        for (int t = 0; t < cs.nseg; ++t) {
            const int n = s.off[t + 1] - s.off[t];
            const Cand* src = cs.base + static_cast<long long>(t) * cs.cap;
            for (int i = tid; i < n; i += blockDim.x) fn(fkey(src[i].v));
        }
    }
}

// k-th largest key (1-based, with multiplicity) of the candidate set: four 8-bit radix passes.
__device__ uint32_t kth_largest(FinSmem& s, const CandSet& cs, int k) {
    const int tid = threadIdx.x;
    uint32_t prefix = 0, pmask = 0;
    int kk = k;
    const int warp = tid >> 5, lane = tid & 31;
    int* wh = s.whist[warp];
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < (kFinThreads / 32) * 256; i += blockDim.x) (&s.whist[0][0])[i] = 0;
        __syncthreads();
        // keys of one row share their top bits, so lanes are grouped by bin before the atomic
        for_each_key(s, cs, [&](uint32_t key) {
            const unsigned bin = ((key & pmask) == prefix) ? ((key >> shift) & 255u) : 0xFFFFFFFFu;
            const unsigned grp = __match_any_sync(__activemask(), bin);
            if (bin != 0xFFFFFFFFu && lane == __ffs(grp) - 1) atomicAdd(&wh[bin], __popc(grp));
        });
        __syncthreads();
        for (int i = tid; i < 256; i += blockDim.x) {
            int t = 0;
#pragma unroll
            for (int w = 0; w < kFinThreads / 32; ++w) t += s.whist[w][i];
            s.hist[i] = t;
        }
        __syncthreads();
        if (tid < 32) {
            int c[8], sum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) { c[q] = s.hist[255 - 8 * tid - q]; sum += c[q]; }
            int incl = sum;
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += y;
            }
            const int excl = incl - sum;
            if (excl < kk && incl >= kk) {
                int run = excl;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (run + c[q] >= kk) { s.bcast[0] = 255 - 8 * tid - q; s.bcast[1] = kk - run; break; }
                    run += c[q];
                }
            }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(s.bcast[0]) << shift;
        pmask |= 255u << shift;
        kk = s.bcast[1];
        __syncthreads();
    }
    return prefix;
}

// Candidates with key >= kth, sorted by (value desc, id asc) into s.sk[0..count); returns the
// count, or -1 when there are more than kKeptCap.
__device__ int sorted_survivors(FinSmem& s, const CandSet& cs, uint32_t kth) {
    const int tid = threadIdx.x;
    if (tid == 0) s.n = 0;
    __syncthreads();
    for (int t = 0; t < cs.nseg; ++t) {
        const int n = s.off[t + 1] - s.off[t];
        const Cand* src = cs.base + static_cast<long long>(t) * cs.cap;
        for (int i = tid; i < n; i += blockDim.x) {
            const Cand c = src[i];
            const uint32_t key = fkey(c.v);
            if (key >= kth) {
                const int p = atomicAdd(&s.n, 1);
                if (p < kKeptCap) s.sk[p] = (static_cast<unsigned long long>(key) << 32) |
                                            static_cast<unsigned>(0xFFFFFFFFu - static_cast<unsigned>(c.id));
            }
        }
    }
    __syncthreads();
    const int cnt = s.n;
    if (cnt > kKeptCap) return -1;
    const int P = next_pow2(max(cnt, 2));
    for (int i = cnt + tid; i < P; i += blockDim.x) s.sk[i] = 0ull;
    block_bitonic_desc(s.sk, P);
    return cnt;
}

// Nucleus over s.sk[0..cnt) with weights s.w[0..cnt); returns the number kept (>= 1) and the
// kept mass.  Kept = tie groups whose exclusive mass is < top_p * Z.
__device__ int nucleus(FinSmem& s, int cnt, float top_p, double* zkept) {
    const int tid = threadIdx.x;
    block_scan_excl_d(s.w, s.u.ex, cnt, s.dwarp);
    const double Z = s.u.ex[cnt];
    int kept = cnt;
    if (top_p < 1.f) {
        const double lim = static_cast<double>(top_p) * Z;
        int first_drop = cnt;
        for (int i = tid; i < cnt; i += blockDim.x) {
            const bool start = (i == 0) || ((s.sk[i] >> 32) != (s.sk[i - 1] >> 32));
            if (start && i > 0 && !(s.u.ex[i] < lim)) first_drop = min(first_drop, i);
        }
        kept = block_min_i(first_drop, s.iwarp);
    }
    *zkept = s.u.ex[kept];
    __syncthreads();
    return kept;
}

// ============================================================================ whole-row path
// Whole-row path: rows whose top-k threshold or nucleus cannot come from candidates
// (top_k = 0 with top_p < 1, top_k above the candidate limit, tie-heavy rows that overflow
// the candidate buffers) get an exact whole-row selection here, re-reading the row once per
// pass: radix passes over the order-preserving key with count histograms (top-k, top-n);
// for the nucleus a fixed-point mass histogram over weight buckets, the boundary bucket and
// an exact settlement among its elements (full_nucleus), with radix passes over mass
// histograms as its fallback.  Fixed-point masses make the sums independent of the order of
// the atomic additions.

constexpr double kFix = 274877906944.0;         // 2^38

struct FullSmem {
    unsigned long long mass[2048];
    unsigned cnt[2048];
    unsigned bm[kBitmapWordsMax];
    PenEntry ent[kPenCap];
    int bcast[32];
    unsigned long long ubcast[4];
    int tl_n, tl_over;
    int n_gt;
    double dwarp_plim;
    uint4 tb[2][kStageBytes / 32];     // double-buffered half vocab tile (cp.async)
};

// Value of element e of the row: penalised target logit or draft probability.
struct RowSource {
    const Args* a;
    bool is_x;
    long long base;      // row offset in elements
    int b, j;
    float f, p;
    bool pen;
};

__device__ int full_pen_count(const FullSmem& s, const RowSource& src, int tok, int nh, int n, int over) {
    const Args& a = *src.a;
    if (!over) {
        int l = 0, h = nh;
        while (l < h) { const int md = (l + h) >> 1; if (s.ent[md].token < tok) l = md + 1; else h = md; }
        int e = -1;
        if (l < nh && s.ent[l].token == tok) e = l;
        else for (int k = nh; k < n; ++k) if (s.ent[k].token == tok) { e = k; break; }
        if (e < 0) return 0;
        const unsigned long long mask = (static_cast<unsigned long long>(s.ent[e].mask_hi) << 32) | s.ent[e].mask_lo;
        const unsigned long long low = (src.j >= 64) ? ~0ull : ((1ull << src.j) - 1ull);
        return s.ent[e].base + __popcll(mask & low);
    }
    int base = 0;
    const int hlo = a.h_off ? a.h_off[src.b] : 0, hhi = a.h_off ? a.h_off[src.b + 1] : 0;
    int l = hlo, h = hhi;
    while (l < h) { const int md = (l + h) >> 1; if (a.h_ids[md] < tok) l = md + 1; else h = md; }
    if (l < hhi && a.h_ids[l] == tok) base = a.h_cnt[l];
    for (int i = 0; i < src.j; ++i) base += (a.d[static_cast<long long>(src.b) * a.Km + i] == tok);
    return base;
}

// Element k of a 16-byte vector of SX-byte values (k may be a run-time index).
template <int SX>
__device__ __forceinline__ float vec_elem(const uint4& w, int k) {
    if (SX == 2) {
        const uint32_t word = (k < 2) ? w.x : (k < 4) ? w.y : (k < 6) ? w.z : w.w;
        return __uint_as_float((k & 1) ? (word & 0xFFFF0000u) : (word << 16));
    }
    return __uint_as_float((k == 0) ? w.x : (k == 1) ? w.y : (k == 2) ? w.z : w.w);
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// One pass over the row calling fn(e, value, raw) for every element, in chunks of half a
// vocab tile (two chunks per penalty tile of a target row).  The 16-byte-aligned interior of
// each chunk is copied into shared memory with cp.async, the next chunk's copy in flight while
// this one is visited; the unaligned edges are read element by element.  The penalty index of
// each target tile is staged in shared memory before its first chunk.
template <int SX, typename Fn>
__device__ void for_each_elem_t(FullSmem& s, const RowSource& src, Fn fn) {
    const Args& a = *src.a;
    constexpr int EPV = 16 / SX;
    const int tid = threadIdx.x, nt = blockDim.x;
    const unsigned char* rowp = src.is_x ? static_cast<const unsigned char*>(a.x) + src.base * SX
                                         : reinterpret_cast<const unsigned char*>(a.q + src.base);
    const int head = static_cast<int>(((16u - static_cast<unsigned>(reinterpret_cast<uintptr_t>(rowp) & 15u)) & 15u) / SX);
    const int tile_n = (src.is_x ? a.tile_x : kStageBytes / 4) / 2;   // chunk: half a tile
    const int row_n = src.is_x ? a.V : a.Lq;              // a draft row holds Lq entries
    const int ntiles = (row_n + tile_n - 1) / tile_n;
    // aligned interior [va, vb) of tile t: element e starts a vector iff (e - head) % EPV == 0
    auto interior = [&](int t, int& va, int& vb) {
        const int e0 = t * tile_n, e1 = min(row_n, e0 + tile_n);
        const int lo = max(e0, head);
        va = min(e1, head + ((lo - head + EPV - 1) / EPV) * EPV);
        vb = (e1 >= va + EPV) ? head + ((e1 - head) / EPV) * EPV : va;
    };
    auto issue = [&](int t) {
        if (t < ntiles) {
            int va, vb;
            interior(t, va, vb);
            const uint4* g = reinterpret_cast<const uint4*>(rowp + static_cast<long long>(va) * SX);
            uint4* d = s.tb[t & 1];
            for (int i = tid; i < (vb - va) / EPV; i += nt) cp_async16(d + i, g + i);
        }
        cp_async_commit();
    };
    __syncthreads();                                      // the buffers are free
    issue(0);
    for (int t = 0; t < ntiles; ++t) {
        const int e0 = t * tile_n, e1 = min(row_n, e0 + tile_n);
        __syncthreads();                                  // tile t-1 visited: its buffer is free
        issue(t + 1);
        int nh = 0, n = 0, over = 0;
        const int p0 = (t >> 1) * a.tile_x;               // start of the penalty tile
        if (src.pen) {
            const long long pt = static_cast<long long>(src.b) * a.tiles_x + (t >> 1);
            const PenHdr h = a.pen_hdr[pt];
            n = h.n; nh = h.pad[0]; over = h.overflow;
            if (!(t & 1)) {                               // first chunk of the tile: stage its index
                for (int w = tid; w < a.bm_words; w += nt) s.bm[w] = a.pen_bm[pt * a.bm_words + w];
                if (!over) for (int k = tid; k < n; k += nt) s.ent[k] = a.pen_ent[pt * kPenCap + k];
            }
        }
        cp_async_wait_one();                              // this thread's copies of tile t landed
        __syncthreads();                                  // everyone's, and the penalty index
        auto visit = [&](int e, float raw) {
            float v = raw;
            if (src.is_x && src.pen && ((s.bm[(e - p0) >> 5] >> ((e - p0) & 31)) & 1u))
                v = penalise(raw, full_pen_count(s, src, e, nh, n, over), src.f, src.p);
            fn(e, v, raw);
        };
        int va, vb;
        interior(t, va, vb);
        for (int e = e0 + tid; e < va; e += nt)
            visit(e, SX == 2 ? load_x(a.x, 2, src.base + e) : __uint_as_float(reinterpret_cast<const uint32_t*>(rowp)[e]));
        for (int e = vb + tid; e < e1; e += nt)
            visit(e, SX == 2 ? load_x(a.x, 2, src.base + e) : __uint_as_float(reinterpret_cast<const uint32_t*>(rowp)[e]));
        const uint4* buf = s.tb[t & 1];
        for (int vi = tid; vi < (vb - va) / EPV; vi += nt) {
            const uint4 w = buf[vi];
#pragma unroll
            for (int q = 0; q < EPV; ++q) visit(va + vi * EPV + q, vec_elem<SX>(w, q));
        }
    }
    __syncthreads();
}

template <typename Fn>
__device__ __forceinline__ void for_each_elem(FullSmem& s, const RowSource& src, Fn fn) {
    if (src.is_x && src.a->sx == 2) for_each_elem_t<2>(s, src, fn);
    else for_each_elem_t<4>(s, src, fn);
}

// Exact k-th largest key (1-based) over the row; use_raw selects the raw value.
__device__ uint32_t full_kth(FullSmem& s, const RowSource& src, int k, bool use_raw) {
    const int tid = threadIdx.x;
    uint32_t prefix = 0, pmask = 0;
    int kk = k;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = shifts[pass];
        const unsigned wm = (1u << widths[pass]) - 1u;
        for (int i = tid; i < 2048; i += blockDim.x) s.cnt[i] = 0u;
        __syncthreads();
        for_each_elem(s, src, [&](int, float v, float raw) {
            const uint32_t key = fkey(use_raw ? raw : v);
            if ((key & pmask) == prefix) atomicAdd(&s.cnt[(key >> sh) & wm], 1u);
        });
        if (tid == 0) {
            int run = 0;
            for (int d = static_cast<int>(wm); d >= 0; --d) {
                const int c = static_cast<int>(s.cnt[d]);
                if (run + c >= kk) { s.bcast[0] = d; s.bcast[1] = kk - run; break; }
                run += c;
            }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(s.bcast[0]) << sh;
        pmask |= wm << sh;
        kk = s.bcast[1];
        __syncthreads();
    }
    return prefix;
}

// Nucleus over {value key >= floor_key} by three radix passes over the key: returns the
// smallest kept key and the kept mass.  The fallback of full_nucleus below.
template <typename WFn>
__device__ uint32_t full_nucleus_radix(FullSmem& s, const RowSource& src, uint32_t floor_key, float top_p, WFn wfn,
                                       double* zkept) {
    const int tid = threadIdx.x;
    uint32_t prefix = 0, pmask = 0;
    unsigned long long above = 0;     // fixed-point mass strictly above the current prefix range
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = shifts[pass];
        const unsigned wm = (1u << widths[pass]) - 1u;
        for (int i = tid; i < 2048; i += blockDim.x) s.mass[i] = 0ull;
        __syncthreads();
        for_each_elem(s, src, [&](int, float v, float) {
            const uint32_t key = fkey(v);
            if (key >= floor_key && (key & pmask) == prefix) {
                const float w = wfn(v);
                const unsigned long long fx = __float2ull_rn(w * 274877906944.0f);
                atomicAdd(&s.mass[(key >> sh) & wm], fx);
            }
        });
        if (tid == 0 && pass == 0) {
            unsigned long long z = 0;
            for (int d = 0; d <= static_cast<int>(wm); ++d) z += s.mass[d];
            s.ubcast[1] = z;
        }
        __syncthreads();
        if (!(top_p < 1.f)) {                 // no nucleus: only the normaliser is needed
            *zkept = static_cast<double>(s.ubcast[1]) / kFix;
            __syncthreads();
            return floor_key;
        }
        if (tid == 0) {
            const double zt = static_cast<double>(s.ubcast[1]);
            const double plim = static_cast<double>(top_p) * zt;
            // last bin (descending) whose mass-above is < top_p * Z
            unsigned long long run = above;
            int pick = -1;
            unsigned long long pick_above = above;
            for (int d = static_cast<int>(wm); d >= 0; --d) {
                const unsigned long long m = s.mass[d];
                if (m == 0ull) continue;
                if (static_cast<double>(run) < plim) { pick = d; pick_above = run; }
                else break;
                run += m;
            }
            if (pick < 0) pick = 0;
            s.bcast[0] = pick;
            s.ubcast[0] = pick_above;
            s.ubcast[2] = s.mass[pick];
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(s.bcast[0]) << sh;
        pmask |= wm << sh;
        above = s.ubcast[0];
        __syncthreads();
    }
    *zkept = static_cast<double>(above + s.ubcast[2]) / kFix;
    return prefix;
}

// Nucleus over {value key >= floor_key} by a mass histogram over weight buckets:
//   pass 1: every element's fixed-point weight goes to bucket(v), a monotone (non-increasing)
//           function of the value that spreads the row over kNucBuckets buckets of 1/32 of a
//           binary order of magnitude of the weight each; elements whose weight is certainly
//           below the nucleus boundary (w < w_lo, from the bound w_cross > (1-top_p) Z / (V+1)
//           on the crossing element's weight) are only summed, per thread, into the total;
//   descent: the boundary bucket beta is the last bucket whose mass above is < top_p * Z;
//           every element of an earlier bucket is kept and none of a later one;
//   pass 2: the elements of beta are gathered into shared memory and the kept tie groups are
//           settled exactly among them (exclusive mass of a group = mass above beta + mass of
//           the larger keys of beta).
// The masses are the same 2^-38 fixed-point weights as the radix path, so the threshold and the
// kept mass are identical to it; a boundary bucket that is the last one, meets the summed-only
// elements, or holds more than the gather capacity falls back to the radix path.
// wfn(v) is the weight (<= 1), bfn(v) the bucket, z_est an estimate of the total weight in
// wfn's units (0 when unknown: no element is summed-only).
constexpr int kNucBuckets = 2048;
static_assert(kTileBf16 % 2 == 0 && kTileF32 % 2 == 0, "whole-row chunks are half tiles");
constexpr int kNucGather = 2048;

template <typename WFn, typename BFn>
__device__ uint32_t full_nucleus(FullSmem& s, const RowSource& src, uint32_t floor_key, float top_p, WFn wfn,
                                 BFn bfn, double z_est, double* zkept) {
    const int tid = threadIdx.x;
    const bool nuc = top_p < 1.f;
    const float w_lo = (nuc && z_est > 0.0)
        ? static_cast<float>(0.5 * (1.0 - static_cast<double>(top_p)) * z_est / (static_cast<double>(src.a->V) + 1.0))
        : 0.f;
    if (tid == 0) { s.n_gt = kNucBuckets; s.ubcast[3] = 0ull; }
    for (int i = tid; i < kNucBuckets; i += blockDim.x) s.mass[i] = 0ull;
    __syncthreads();
    unsigned long long tail = 0ull;
    int tmin = kNucBuckets;
    for_each_elem(s, src, [&](int, float v, float) {
        if (fkey(v) < floor_key) return;
        const float w = wfn(v);
        const unsigned long long fx = __float2ull_rn(w * 274877906944.0f);
        if (!nuc) { tail += fx; return; }
        const int bk = bfn(v);
        if (w < w_lo) { tail += fx; tmin = min(tmin, bk); }
        else if (fx != 0ull) atomicAdd(&s.mass[bk], fx);
    });
    // total of the summed-only weights (integer sums: independent of the order)
    for (int o = 16; o > 0; o >>= 1) {
        tail += __shfl_xor_sync(0xffffffffu, tail, o);
        tmin = min(tmin, __shfl_xor_sync(0xffffffffu, tmin, o));
    }
    if ((tid & 31) == 0) {
        if (tail) atomicAdd(&s.ubcast[3], tail);
        if (tmin < kNucBuckets) atomicMin(&s.n_gt, tmin);
    }
    __syncthreads();
    if (!nuc) {
        *zkept = static_cast<double>(s.ubcast[3]) / kFix;
        __syncthreads();
        return floor_key;
    }
    // descent: total, then the boundary bucket (one warp: per-lane contiguous chunks of buckets)
    if (tid < 32) {
        constexpr int kPer = kNucBuckets / 32;
        unsigned long long part = 0ull;
        for (int d = 0; d < kPer; ++d) part += s.mass[tid * kPer + d];
        unsigned long long incl = part;
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
            if (tid >= o) incl += y;
        }
        const unsigned long long total_b = __shfl_sync(0xffffffffu, incl, 31);
        const double zt = static_cast<double>(total_b + s.ubcast[3]);
        const double plim = static_cast<double>(top_p) * zt;
        // the lane whose chunk holds the last bucket with mass-above < plim: the last lane whose
        // exclusive prefix is < plim and whose chunk is not empty
        const unsigned long long excl = incl - part;
        const unsigned cand = __ballot_sync(0xffffffffu, part != 0ull && static_cast<double>(excl) < plim);
        if (tid == 0) { s.bcast[0] = -1; }
        __syncwarp();
        if (cand) {
            const int L = 31 - __clz(cand);
            if (tid == L) {
                unsigned long long run = excl;
                int pick = -1;
                unsigned long long pick_above = 0ull, pick_mass = 0ull;
                for (int d = 0; d < kPer; ++d) {
                    const unsigned long long m = s.mass[tid * kPer + d];
                    if (m == 0ull) continue;
                    if (static_cast<double>(run) < plim) { pick = tid * kPer + d; pick_above = run; pick_mass = m; }
                    else break;
                    run += m;
                }
                s.bcast[0] = pick;
                s.ubcast[0] = pick_above;
                s.ubcast[2] = pick_mass;
                s.dwarp_plim = plim;
            }
        }
    }
    __syncthreads();
    const int beta = s.bcast[0];
    const unsigned long long above = s.ubcast[0];
    const double plim = s.dwarp_plim;
    const bool ok = beta >= 0 && beta < kNucBuckets - 1 && beta < s.n_gt &&
                    static_cast<double>(above + s.ubcast[2]) >= plim;
    __syncthreads();
    if (!ok) return full_nucleus_radix(s, src, floor_key, top_p, wfn, zkept);
    // pass 2: gather the boundary bucket (keys in cnt[], weights in mass[])
    if (tid == 0) s.tl_n = 0;
    __syncthreads();
    for_each_elem(s, src, [&](int, float v, float) {
        const uint32_t key = fkey(v);
        if (key < floor_key || bfn(v) != beta) return;
        const int p = atomicAdd(&s.tl_n, 1);
        if (p < kNucGather) { s.cnt[p] = key; s.mass[p] = __float2ull_rn(wfn(v) * 274877906944.0f); }
    });
    const int n = s.tl_n;
    if (n > kNucGather) { __syncthreads(); return full_nucleus_radix(s, src, floor_key, top_p, wfn, zkept); }
    // exact settlement: a key is kept iff above + (mass of larger keys of beta) < plim
    if (tid == 0) { s.bcast[1] = static_cast<int>(0xFFFFFFFFu); }
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
        const uint32_t ki = s.cnt[i];
        unsigned long long ex = above;
        for (int jj = 0; jj < n; ++jj) ex += (s.cnt[jj] > ki) ? s.mass[jj] : 0ull;
        if (static_cast<double>(ex) < plim) atomicMin(reinterpret_cast<unsigned*>(&s.bcast[1]), ki);
    }
    __syncthreads();
    const uint32_t tau = static_cast<uint32_t>(s.bcast[1]);
    unsigned long long kept = 0ull;
    for (int i = tid; i < n; i += blockDim.x) kept += (s.cnt[i] >= tau) ? s.mass[i] : 0ull;
    for (int o = 16; o > 0; o >>= 1) kept += __shfl_xor_sync(0xffffffffu, kept, o);
    if (tid == 0) s.ubcast[1] = 0ull;
    __syncthreads();
    if ((tid & 31) == 0 && kept) atomicAdd(&s.ubcast[1], kept);
    __syncthreads();
    *zkept = static_cast<double>(above + s.ubcast[1]) / kFix;
    __syncthreads();
    return tau;
}

// Whole-row selection for a target row whose support could not come from candidates;
// updates o (threshold, normaliser, mode).
__device__ void whole_row_x(const Args& a, FullSmem& s, int slot, int b, int j, XRowOut& o) {
    const dspark_row_params_t r = a.rows[b];
    RowSource src{&a, true, static_cast<long long>(slot) * a.V, b, j, r.frequency_penalty, r.presence_penalty,
                  has_penalty(r)};
    if (o.mode == kModeNeedFull) {
        uint32_t floor_key = fkey(o.tau);
        if (o.top_k > 0) floor_key = full_kth(s, src, o.top_k, false);
        const float mp = o.m_pen, c = o.c_l2e;
        const float cs = c * 32.f;                       // 32 buckets per binary order of the weight
        const double z_est = (floor_key == fkey(-INFINITY)) ? o.Z : 0.0;
        double z;
        const uint32_t kk = full_nucleus(s, src, floor_key, o.top_p < 1.f ? o.top_p : 2.f,
                                         [&](float v) { return target_weight(v, mp, c); },
                                         [&](float v) {
                                             const float d = __fmul_rn(__fsub_rn(mp, v), cs);
                                             return d < static_cast<float>(kNucBuckets - 1) ? max(0, static_cast<int>(d)) : kNucBuckets - 1;
                                         }, z_est, &z);
        o.tau = (o.top_p < 1.f) ? key_to_f(kk) : key_to_f(floor_key);
        o.Z = z;
        o.top_k = 0;
        o.mode = kModeFull;
    }
}

__device__ void whole_row_q(const Args& a, FullSmem& s, int qs, int b, int i, QRowOut& o) {
    RowSource src{&a, false, static_cast<long long>(qs) * a.Lq, b, i, 0.f, 0.f, false};
    uint32_t floor_key = fkey(o.tau);
    if (o.top_k > 0) floor_key = full_kth(s, src, o.top_k, false);
    const float qmax = o.qmax, inv_t = o.inv_t;
    const bool t_one = inv_t == 1.f;
    // bucket from the order of magnitude of q/qmax read off the float bits (monotone in q)
    const int qmax_bits = __float_as_int(qmax);
    const float sq = inv_t * (32.f / 8388608.f);
    const double z_est = (floor_key == fkey(-INFINITY)) ? (t_one ? o.Z / qmax : o.Z) : 0.0;
    double z;
    const uint32_t kk = full_nucleus(s, src, floor_key, o.top_p < 1.f ? o.top_p : 2.f,
                                     [&](float v) { return draft_weight(v, qmax, inv_t, t_one) / (t_one ? qmax : 1.f); },
                                     [&](float v) {
                                         const int vb = __float_as_int(v);    // q <= qmax: no overflow for q >= 0
                                         const float d = vb < 0 ? 3.0e38f : static_cast<float>(qmax_bits - vb) * sq;
                                         return d < static_cast<float>(kNucBuckets - 1) ? max(0, static_cast<int>(d)) : kNucBuckets - 1;
                                     }, z_est, &z);
    o.tau = (o.top_p < 1.f) ? key_to_f(kk) : key_to_f(floor_key);
    if (t_one) z *= qmax;
    o.Z = z;
    o.top_k = 0;
    o.mode = kModeFull;
    if (!(z > 0.0) && threadIdx.x == 0) atomicOr(&a.row_status[b], DSPARK_ROW_NONFINITE);
}

__device__ void finalize_x(const Args& a, FinSmem& s, int slot, int b, int j) {
    const int tid = threadIdx.x;
    const dspark_row_params_t r = a.rows[b];
    const int nseg = a.nseg_x;
    const TileStats* ts = a.ts_x + static_cast<long long>(slot) * nseg;
    XRowOut o{};
    o.kth = -INFINITY;                                    // not kept by the block path
    o.mode = kModeInactive;
    float mr = -INFINITY, mp = -INFINITY;
    int fl = 0;
    for (int t = tid; t < nseg; t += blockDim.x) {
        const TileStats x = ts[t];
        mr = (mr != mr || x.m_raw != x.m_raw) ? __int_as_float(0x7fc00000) : fmaxf(mr, x.m_raw);
        mp = (mp != mp || x.m_pen != x.m_pen) ? __int_as_float(0x7fc00000) : fmaxf(mp, x.m_pen);
        fl |= x.flags;
    }
    mr = block_max_nan(mr, s.fwarp);
    mp = block_max_nan(mp, s.fwarp);
    fl = block_or_i(fl, s.iwarp);
    if ((fl & kTileBad) || !isfinite(mr) || !isfinite(mp)) {
        if (tid == 0) {
            atomicOr(&a.row_status[b], DSPARK_ROW_NONFINITE);
            a.xout[slot] = o;
        }
        return;
    }
    int arg = 0x7FFFFFFF;
    double stemp = 0.0;
    const bool greedy = !(r.temperature > 0.f);
    const float c_l2e = greedy ? 0.f : kL2E / r.temperature;
    for (int t = tid; t < nseg; t += blockDim.x) {
        const TileStats x = ts[t];
        if (x.m_pen == mp) arg = min(arg, x.arg_pen);
        if (!greedy) stemp += static_cast<double>(x.s_temp) * static_cast<double>(exp2f((x.m_pen - mp) * c_l2e));
    }
    arg = block_min_i(arg, s.iwarp);
    stemp = block_sum_d(stemp, s.dwarp);
    o.argmax = arg;
    o.m_pen = mp;
    o.c_l2e = c_l2e;
    o.top_p = r.top_p;
    o.tau = -INFINITY;
    o.top_k = 0;
    o.n_kept = 0;
    o.flags = fl;
    const int k = r.top_k;
    if (greedy) {
        o.mode = kModeGreedy;
    } else if (k > 0 && k < a.V) {
        CandSet cs{nullptr, 0, 0, -1};
        if (k <= kMaxCandTopK && !(fl & kTileOverflowPen))
            cs = stage_candidates(s, ts, a.cand_x + static_cast<long long>(slot) * nseg * kCandPenGlobal,
                                  kCandPenGlobal, nseg);
        if (cs.total >= k) {
            const uint32_t kth = kth_largest(s, cs, k);
            const int cnt = sorted_survivors(s, cs, kth);
            if (cnt > 0) {
                for (int i = tid; i < cnt; i += blockDim.x)
                    s.w[i] = static_cast<double>(target_weight(ckey_v(s.sk[i]), mp, c_l2e));
                __syncthreads();
                double zk;
                const int kept = nucleus(s, cnt, r.top_p, &zk);
                KeptEntry* dst = a.kept + static_cast<long long>(slot) * kKeptCap;
                for (int i = tid; i < kept; i += blockDim.x) dst[i] = KeptEntry{ckey_id(s.sk[i]), static_cast<float>(s.w[i])};
                o.mode = kModeList;
                o.n_kept = kept;
                o.Z = zk;
                o.tau = ckey_v(s.sk[kept - 1]);
            } else {
                o.mode = kModeNeedFull;                       // too many survivors: threshold known
                o.tau = key_to_f(kth);
            }
        } else {
            o.mode = kModeNeedFull;                           // select over the whole row
            o.top_k = k;
        }
        __syncthreads();
    } else {
        o.Z = stemp;
        o.mode = (r.top_p < 1.f) ? kModeNeedFull : kModeFull;
    }
    __syncthreads();
    if (o.mode == kModeNeedFull) whole_row_x(a, *reinterpret_cast<FullSmem*>(&s), slot, b, j, o);
    if (tid == 0) a.xout[slot] = o;
}

__device__ void finalize_q(const Args& a, FinSmem& s, int qslot, int b, int i) {
    const int tid = threadIdx.x;
    const dspark_row_params_t r = a.rows[b];
    const int nseg = a.nseg_q;
    const TileStats* ts = a.ts_q + static_cast<long long>(qslot) * nseg;
    QRowOut o{};
    o.mode = kModeInactive;
    float qmax = -INFINITY;
    int fl = 0;
    for (int t = tid; t < nseg; t += blockDim.x) {
        const TileStats x = ts[t];
        qmax = (qmax != qmax || x.m_raw != x.m_raw) ? __int_as_float(0x7fc00000) : fmaxf(qmax, x.m_raw);
        fl |= x.flags;
    }
    qmax = block_max_nan(qmax, s.fwarp);
    fl = block_or_i(fl, s.iwarp);
    const bool t_one = r.temperature == 1.f;
    const float inv_t = 1.f / r.temperature;
    double z = 0.0;
    for (int t = tid; t < nseg; t += blockDim.x) {
        const TileStats x = ts[t];
        if (t_one) z += static_cast<double>(x.s_raw);
        else if (x.m_raw > 0.f) z += static_cast<double>(x.s_temp) * static_cast<double>(exp2f(inv_t * log2f(x.m_raw / qmax)));
    }
    z = block_sum_d(z, s.dwarp);
    if ((fl & kTileBad) || !(qmax > 0.f) || !isfinite(qmax)) {
        if (tid == 0) { atomicOr(&a.row_status[b], DSPARK_ROW_NONFINITE); a.qout[qslot] = o; }
        return;
    }
    o.qmax = qmax;
    o.inv_t = inv_t;
    o.tau = -INFINITY;
    o.top_k = 0;
    o.top_p = r.top_p;
    o.flags = fl;
    const int k = r.top_k;
    if (k > 0 && k < a.Lq) {
        CandSet cs{nullptr, 0, 0, -1};
        if (k <= kMaxCandTopK && !(fl & kTileOverflowPen))
            cs = stage_candidates(s, ts, a.cand_q + static_cast<long long>(qslot) * nseg * kCandPenGlobal,
                                  kCandPenGlobal, nseg);
        if (cs.total >= k) {
            const uint32_t kth = kth_largest(s, cs, k);
            const int cnt = sorted_survivors(s, cs, kth);
            if (cnt > 0) {
                for (int e = tid; e < cnt; e += blockDim.x)
                    s.w[e] = static_cast<double>(draft_weight(ckey_v(s.sk[e]), qmax, inv_t, t_one));
                __syncthreads();
                double zk;
                const int kept = nucleus(s, cnt, r.top_p, &zk);
                o.mode = kModeList;
                o.Z = zk;
                o.tau = ckey_v(s.sk[kept - 1]);
            } else {
                o.mode = kModeNeedFull;
                o.tau = key_to_f(kth);
            }
        } else {
            o.mode = kModeNeedFull;
            o.top_k = k;
        }
    } else {
        o.Z = z;
        o.mode = (r.top_p < 1.f) ? kModeNeedFull : kModeFull;
        if (o.mode == kModeFull && !(z > 0.0)) {
            if (tid == 0) atomicOr(&a.row_status[b], DSPARK_ROW_NONFINITE);
        }
    }
    __syncthreads();
    if (o.mode == kModeNeedFull) whole_row_q(a, *reinterpret_cast<FullSmem*>(&s), qslot, b, i, o);
    if (tid == 0) a.qout[qslot] = o;
}

__device__ void finalize_row(const Args& a, FinSmem& s, int slot) {
    if (slot < a.xslots) {
        const int b = slot / (a.Km + 1), j = slot % (a.Km + 1);
        if ((a.row_status[b] & (DSPARK_ROW_BAD_PARAMS | DSPARK_ROW_BAD_DRAFT)) || j > a.rows[b].num_drafts) {
            if (threadIdx.x == 0) { XRowOut o{}; o.mode = kModeInactive; o.kth = -INFINITY; a.xout[slot] = o; }
            return;
        }
        finalize_x(a, s, slot, b, j);
    } else {
        const int qs = slot - a.xslots;
        const int b = qs / a.Km, i = qs % a.Km;
        const dspark_row_params_t r = a.rows[b];
        if ((a.row_status[b] & (DSPARK_ROW_BAD_PARAMS | DSPARK_ROW_BAD_DRAFT)) || i >= r.num_drafts ||
            !(r.temperature > 0.f)) {
            if (threadIdx.x == 0) { QRowOut o{}; o.mode = kModeInactive; a.qout[qs] = o; }
            return;
        }
        finalize_q(a, s, qs, b, i);
    }
}

// The rows the warp finalize left (fin_list), each by a whole block.
__global__ void __launch_bounds__(kFinThreads, 2) row_finalize_kernel(Args a) {
    pdl_enter();
    if (a.plan->pad[0]) return;                           // streaming statistics incomplete
    extern __shared__ __align__(16) unsigned char fin_raw[];
    FinSmem& s = *reinterpret_cast<FinSmem*>(fin_raw);
    const int n = a.fin_list[0];
    for (int i = blockIdx.x; i < n; i += gridDim.x) {
        finalize_row(a, s, a.fin_list[1 + i]);
        __syncthreads();                                  // shared memory reused by the next row
    }
}

}  // namespace

cudaError_t launch_row_finalize(const Args& a, cudaStream_t s) {
    const size_t smem = sizeof(FinSmem) > sizeof(FullSmem) ? sizeof(FinSmem) : sizeof(FullSmem);
    cudaError_t e = cudaFuncSetAttribute(row_finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int rows = a.xslots + a.qslots;
    const int grid = rows < 4 * a.grid_ss ? rows : 4 * a.grid_ss;
    return launch_k(row_finalize_kernel, dim3(grid), dim3(kFinThreads), smem, s, true, a);
}


}  // namespace dspark
