// logprob_kernel: the raw log-softmax of each emitted token and the top_logprobs list at its
// position (mlx-dspark Changelog, [0.2.0] Added, "logprobs / top_logprobs": the raw target
// log-softmax of each committed token plus the top candidates, gathered on the GPU only when
// requested).  Only the positions a request emits from (j <= accept length) need them, so
// they are taken after the draws, from those rows alone: accept_kernel lists the rows.
//
// The R listed rows are cut into S chunks each, S = min(16, grid / R, V / 8192) at least 1, so
// that the R * S chunks fill the persistent grid (four 256-thread CTAs per SM) in one wave and
// the emitted rows of a call are read by every SM, not by one SM per row; each CTA takes chunks
// from a counter.  A chunk streams from HBM in batches of kLpVec 16-byte vectors per thread,
// the next batch's loads in flight while the current one is reduced, for
//   - the chunk's maximum m and its sum of exp(x - m) (per thread a running maximum, the sum
//     rescaled at most once per batch; then a fixed reduction order);
//   - the chunk's n largest logits by (value descending, id ascending).  For a row settled by
//     a top-k list (k >= n) theta is the row's k-th largest penalised logit: at least k logits
//     of the row reach it (their raw values are no smaller when the penalties are not
//     negative), so every one of the row's top n does.  Otherwise, after the first batch,
//     theta = the n-th largest of the 256 threads' maxima (a bitwise search over block counts):
//     at least n distinct logits of that batch reach it, so every one of the chunk's top n does,
//     and the logits >= theta of every batch are gathered as they stream by; the chunk's top n
//     are then found among the gathered logits: the n-th largest value by a bitwise search,
//     and the logits at or above it ranked.  When ties put more logits >= theta
//     than fit, the chunk is settled exactly from L2: the n-th largest value v by a bitwise
//     search over counts, the logits above v, then the lowest ids equal to v.
// The CTA that completes a row's last chunk (a counter per row) merges the S partials in a
// fixed order: LSE = M + log(sum_c s_c exp(m_c - M)) and the row's top n among the chunks'
// sorted lists.
// It then writes logprob = x[token] - LSE and the top list.  Results do not depend on
// scheduling.
//
// Penalised mode (the other reading of "raw target log-softmax"): the same over the penalised
// logits x' of the position.  Tokens the penalty index flags for the request (history and
// drafts) are set to -inf in the streamed vectors; after the stream, each thread takes the
// flagged tokens of its share of the chunk's bitmap words one by one, as x' = x less the
// penalty of its count at that position, into its maximum and sum and, at or above theta,
// its warp's candidates.  Every other logit is its own x'.
#include "block_utils.cuh"

namespace dspark {

namespace {

constexpr int kLpThreads = 256;
constexpr int kLpBlocksPerSm = 4;
constexpr int kLpWarps = kLpThreads / 32;
constexpr int kLpCandCap = 2048;
constexpr int kLpVec = 4;                    // 16-byte vectors per thread and batch
constexpr int kLpStages = 2;                 // batches of a chunk in flight
constexpr int kLpWarpCap = kLpCandCap / kLpWarps;
constexpr int kLpMergeLists = kLpMaxChunks;  // chunk partials the merge copies to shared memory
constexpr int kLpMinChunk = 8192;            // logits per chunk at least
constexpr int kLpSelCap = 256;               // keys at the n-th largest value and above, ranked directly
constexpr float kL2E = 1.4426950408889634f;

struct LpSmem {
    uint4 stage[kLpStages][kLpVec * kLpThreads];   // batches of the chunk, filled by bulk copies
    unsigned long long full[kLpStages];    // their mbarriers
    unsigned long long keys[kLpCandCap];   // (fkey(value) << 32) | (0xFFFFFFFF - id); warp w: [w*kLpWarpCap, ...)
    float tmax[kLpThreads];
    float wm[kLpWarps];
    float wsum[kLpWarps];
    int wcnt[kLpWarps + 1];
    int scnt[2][kLpWarps];                 // top_select's per-warp counts (two alternating sets)
    unsigned long long sel[kLpSelCap];     // top_select's keys reaching the threshold
    int wn[kLpWarps];                      // keys each warp gathered
    double dwarp[33];
    int n;
    int last;
    int item;
    float theta;
    float xt;                              // the merge: the emitted token's (penalised) logit
    unsigned long long top[2 * DSPARK_MAX_TOP_LOGPROBS];
    float mm[kLpMergeLists];               // the merge's copies of the chunk partials
    float ms[kLpMergeLists];
    int mn[kLpMergeLists];
    int ml[kLpMergeLists];
};

// Sort s.keys[0..cnt) descending (cnt <= kLpCandCap): one warp with shuffles when cnt <= 64,
// else a block bitonic network.
__device__ void sort_keys_desc(LpSmem& s, int cnt) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (cnt <= 64) {
        if (tid < 32) {
            // bitonic sort of 64 keys held two per lane: key h of lane l sits at position l + 32h
            unsigned long long k[2];
            k[0] = lane < cnt ? s.keys[lane] : 0ull;
            k[1] = lane + 32 < cnt ? s.keys[lane + 32] : 0ull;
            for (int size = 2; size <= 64; size <<= 1) {
                for (int stride = size >> 1; stride > 0; stride >>= 1) {
                    if (stride == 32) {                  // partners in the same lane (size 64)
                        const unsigned long long hi = k[0] > k[1] ? k[0] : k[1];
                        const unsigned long long lo = k[0] > k[1] ? k[1] : k[0];
                        k[0] = hi;
                        k[1] = lo;
                    } else {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int pos = lane + 32 * h;
                            const unsigned long long o = __shfl_xor_sync(0xffffffffu, k[h], stride);
                            const bool lower = (pos & stride) == 0;
                            const bool desc = (pos & size) == 0;
                            // the lower position of a descending pair keeps the larger key
                            const bool keep_max = lower == desc;
                            k[h] = keep_max ? (k[h] > o ? k[h] : o) : (k[h] < o ? k[h] : o);
                        }
                    }
                }
            }
            if (lane < cnt) s.keys[lane] = k[0];
            if (lane + 32 < cnt) s.keys[lane + 32] = k[1];
        }
        __syncthreads();
        return;
    }
    const int P = next_pow2(cnt);
    for (int i = cnt + tid; i < P; i += blockDim.x) s.keys[i] = 0ull;
    block_bitonic_desc(s.keys, P);
}

// Exclusive prefix over the block of per-thread counts (thread order); returns the thread's
// offset and sets *total.  Two barriers.
__device__ int block_excl_count(LpSmem& s, int c, int* total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s.wcnt[warp] = incl;
    __syncthreads();
    int off = 0, tot = 0;
    for (int w = 0; w < kLpThreads / 32; ++w) {
        if (w < warp) off += s.wcnt[w];
        tot += s.wcnt[w];
    }
    __syncthreads();
    *total = tot;
    return off + incl - c;
}

__device__ __forceinline__ unsigned long long lp_gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for a batch's copy with a 2 s bound; false when the bound expires.
__device__ __forceinline__ bool lp_wait(unsigned long long* bar, unsigned parity) {
    uint64_t* b = reinterpret_cast<uint64_t*>(bar);
    if (mbar_try_wait(b, parity)) return true;
    const unsigned long long t0 = lp_gtimer();
    while (!mbar_try_wait(b, parity))
        if (lp_gtimer() - t0 > 2000000000ull) return false;
    return true;
}

template <int SX>
__device__ __forceinline__ float lp_elem(const uint4& w, int q) {
    if (SX == 2) {
        const uint32_t word = (q < 2) ? w.x : (q < 4) ? w.y : (q < 6) ? w.z : w.w;
        return __uint_as_float((q & 1) ? (word & 0xFFFF0000u) : (word << 16));
    }
    return __uint_as_float((q == 0) ? w.x : (q == 1) ? w.y : (q == 2) ? w.z : w.w);
}

// Maximum of a 16-byte vector (no NaN here: rows with a NaN never reach this pass), packed:
// bf16 pairs with bf16x2 max, fp32 with a float max chain.  vmax2 keeps a bf16x2 pair.
template <int SX>
__device__ __forceinline__ uint32_t vmax_word(const uint4& w) {
    if (SX == 2) {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w.y);
        const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&w.z);
        const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&w.w);
        const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
        return *reinterpret_cast<const uint32_t*>(&m);
    }
    return __float_as_uint(fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                                 fmaxf(__uint_as_float(w.z), __uint_as_float(w.w))));
}
template <int SX>
__device__ __forceinline__ uint32_t vmax_combine(uint32_t a, uint32_t b) {
    if (SX == 2) {
        const __nv_bfloat162 m = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
        return *reinterpret_cast<const uint32_t*>(&m);
    }
    return __float_as_uint(fmaxf(__uint_as_float(a), __uint_as_float(b)));
}
template <int SX>
__device__ __forceinline__ float vmax_float(uint32_t m) {
    if (SX == 2) return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
    return __uint_as_float(m);
}


// Exact top-n of a chunk whose logits >= theta did not fit the key buffer (ties): the n-th
// largest value v (with multiplicity) by a bitwise search over counts, the logits above v (fewer
// than n), then the lowest ids equal to v in id order.  Reads the chunk from L2 again.
// The logit of position j of request b at token e as the pass sees it: x, or x' in penalised mode.
struct LpRow {
    int b, j;
    float f, p;
};
template <bool PEN>
__device__ __forceinline__ float lp_value(const Args& a, const LpRow& r, int e, float x) {
    if (!PEN || !(pen_bits_range(a, r.b, e, 1) & 1u)) return x;
    return penalise(x, token_count(a, r.b, r.j, e), r.f, r.p);
}

template <int SX, bool PEN>
__device__ int lp_exact_top(const Args& a, LpSmem& s, long long slot, int c0, int c1, int va, int vb, int n_top,
                            const LpRow& pr) {
    constexpr int EPV = 16 / SX;
    const int tid = threadIdx.x;
    auto val = [&](int e) { return lp_value<PEN>(a, pr, e, load_x(a.x, SX, slot * a.V + e)); };
    auto vload = [&](int v, float (&xs)[EPV]) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(a.x) +
                                                             (slot * a.V + va) * SX) + v);
#pragma unroll
        for (int q = 0; q < EPV; ++q) xs[q] = lp_elem<SX>(w, q);
        if (PEN) {
            const unsigned bits = pen_bits_range(a, pr.b, va + v * EPV, EPV);
            if (bits)
#pragma unroll
                for (int q = 0; q < EPV; ++q)
                    if ((bits >> q) & 1u) xs[q] = penalise(xs[q], token_count(a, pr.b, pr.j, va + v * EPV + q), pr.f, pr.p);
        }
    };
    const int nv = (vb - va) / EPV;
    auto count_ge = [&](uint32_t key) {
        int c = 0;
        for (int e = c0 + tid; e < va; e += kLpThreads) c += fkey(val(e)) >= key;
        for (int e = vb + tid; e < c1; e += kLpThreads) c += fkey(val(e)) >= key;
        for (int v = tid; v < nv; v += kLpThreads) {
            float xs[EPV];
            vload(v, xs);
#pragma unroll
            for (int q = 0; q < EPV; ++q) c += fkey(xs[q]) >= key;
        }
        int tot = 0;
        block_excl_count(s, c, &tot);
        return tot;
    };
    uint32_t kth = 0u;
    for (int bit = 31; bit >= 0; --bit)
        if (count_ge(kth | (1u << bit)) >= n_top) kth |= 1u << bit;
    // the logits above kth (fewer than n_top), then the lowest ids equal to it, in id order
    if (tid == 0) s.n = 0;
    __syncthreads();
    for (int e = c0 + tid; e < va; e += kLpThreads) {
        const float x = val(e);
        if (fkey(x) > kth) { const int p = atomicAdd(&s.n, 1); s.keys[p] = ckey(x, e); }
    }
    for (int e = vb + tid; e < c1; e += kLpThreads) {
        const float x = val(e);
        if (fkey(x) > kth) { const int p = atomicAdd(&s.n, 1); s.keys[p] = ckey(x, e); }
    }
    for (int v = tid; v < nv; v += kLpThreads) {
        float xs[EPV];
        vload(v, xs);
#pragma unroll
        for (int q = 0; q < EPV; ++q) {
            const float x = xs[q];
            if (fkey(x) > kth) { const int p = atomicAdd(&s.n, 1); s.keys[p] = ckey(x, va + v * EPV + q); }
        }
    }
    __syncthreads();
    const int n_gt = s.n;
    const int need = n_top - n_gt;
    int got = 0;
    // id order: [c0, va) one element per thread per round, the vectors 256 per round, [vb, c1)
    const int rounds_h = (va - c0 + kLpThreads - 1) / kLpThreads, rounds_v = (nv + kLpThreads - 1) / kLpThreads;
    const int rounds_t = (c1 - vb + kLpThreads - 1) / kLpThreads;
    for (int r = 0; r < rounds_h + rounds_v + rounds_t && got < need; ++r) {
        int mine = 0, base_id = 0;
        float xs[EPV];
        int ne = 0;
        if (r < rounds_h) {
            const int e = c0 + r * kLpThreads + tid;
            if (e < va) { xs[0] = val(e); ne = 1; base_id = e; }
        } else if (r < rounds_h + rounds_v) {
            const int v = (r - rounds_h) * kLpThreads + tid;
            if (v < nv) {
                vload(v, xs);
                ne = EPV;
                base_id = va + v * EPV;
            }
        } else {
            const int e = vb + (r - rounds_h - rounds_v) * kLpThreads + tid;
            if (e < c1) { xs[0] = val(e); ne = 1; base_id = e; }
        }
#pragma unroll
        for (int q = 0; q < EPV; ++q) mine += (q < ne && fkey(xs[q]) == kth) ? 1 : 0;
        int tot = 0;
        int pos = got + block_excl_count(s, mine, &tot);
#pragma unroll
        for (int q = 0; q < EPV; ++q)
            if (q < ne && fkey(xs[q]) == kth) {
                if (pos < need) s.keys[n_gt + pos] = ckey(xs[q], base_id + q);
                ++pos;
            }
        got += tot;
    }
    __syncthreads();
    const int cnt = n_gt + min(got, need);
    sort_keys_desc(s, cnt);
    return cnt;
}

// The n largest of the keys held in `lists` shared-memory lists (list l: n_l keys at
// keys + l * stride), by rank: every key counts the keys above it (keys are distinct), and a
// key of rank r < n lands in top[r].  All threads take part; returns min(n, total).
__device__ int rank_select(const unsigned long long* keys, const int* nl, int lists, int stride, int n,
                           unsigned long long* top) {
    int total = 0;
    for (int l = 0; l < lists; ++l) total += nl[l];
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        int l = 0, r = i;
        while (r >= nl[l]) { r -= nl[l]; ++l; }
        const unsigned long long key = keys[l * stride + r];
        int rank = 0;
        for (int m = 0; m < lists && rank < n; ++m) {
            const unsigned long long* km = keys + m * stride;
            for (int q = 0; q < nl[m]; ++q) rank += km[q] > key;
        }
        if (rank < n) top[rank] = key;
    }
    __syncthreads();
    return min(n, total);
}

// The n largest of the keys held in the lists (as rank_select), for many keys: the n-th largest
// value v (32-bit value key, with multiplicity) by a bitwise search over counts, then only the
// keys of value >= v (n and their ties) ranked.  Falls back to rank_select over everything when
// ties put more than kLpSelCap keys at v or above.
__device__ int top_select(LpSmem& s, const unsigned long long* keys, const int* nl, int lists, int stride, int n,
                          unsigned long long* top) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int total = 0;
    for (int l = 0; l < lists; ++l) total += nl[l];
    // up to one key per thread, ranking every key against all (no barrier per step) is shorter
    if (total <= kLpThreads || total > kLpThreads * 8) return rank_select(keys, nl, lists, stride, n, top);
    uint32_t mine[8];                                     // this thread's keys' value parts (0: none)
    unsigned long long full[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int i = tid + r * kLpThreads;
        full[r] = 0ull;
        if (i < total) {
            int l = 0, q = i;
            while (q >= nl[l]) { q -= nl[l]; ++l; }
            full[r] = keys[l * stride + q];
        }
        mine[r] = static_cast<uint32_t>(full[r] >> 32);
    }
    // block count of value keys >= cand: warp sums, alternating shared sets (one barrier a step)
    auto count_ge = [&](uint32_t cand, int set) {
        int c = 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) c += (full[r] != 0ull && mine[r] >= cand) ? 1 : 0;
        c = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c)));
        if (lane == 0) s.scnt[set][warp] = c;
        __syncthreads();
        int t = 0;
        for (int w = 0; w < kLpWarps; ++w) t += s.scnt[set][w];
        return t;
    };
    uint32_t v = 0u;
    int set = 0;
    for (int bit = 31; bit >= 0; --bit, set ^= 1)
        if (count_ge(v | (1u << bit), set) >= n) v |= 1u << bit;
    // the keys of value >= v, compacted, then ranked
    if (tid == 0) s.n = 0;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 8; ++r)
        if (full[r] != 0ull && mine[r] >= v) {
            const int p = atomicAdd(&s.n, 1);
            if (p < kLpSelCap) s.sel[p] = full[r];
        }
    __syncthreads();
    const int m = s.n;
    if (m > kLpSelCap) return rank_select(keys, nl, lists, stride, n, top);
    for (int i = tid; i < m; i += blockDim.x) {
        const unsigned long long key = s.sel[i];
        int rank = 0;
        for (int q = 0; q < m; ++q) rank += s.sel[q] > key;
        if (rank < n) top[rank] = key;
    }
    __syncthreads();
    return min(n, total);
}

// One chunk [c0, c1) of target row `slot`: its maximum, its sum of exp relative to it and its
// top-n list, written to *out.
// cand: when non-null, a chunk whose gathered keys all fit (at most kLpCandPerChunk) writes them
// there unselected and leaves the selection to the row merge.
// The 16-byte-aligned interior [va, vb) of chunk [c0, c1) of target row `slot`: nv vectors
// from g (element e starts a vector iff (e - head) % EPV == 0).
template <int SX>
struct LpGeom {
    int va, vb, nv;
    const uint4* g;
    __device__ LpGeom(const Args& a, long long slot, int c0, int c1) {
        constexpr int EPV = 16 / SX;
        const unsigned char* rowp = static_cast<const unsigned char*>(a.x) + slot * a.V * SX;
        const int head = static_cast<int>(((16u - static_cast<unsigned>(reinterpret_cast<uintptr_t>(rowp) & 15u)) & 15u) / SX);
        const int lo = max(c0, head);
        va = min(c1, head + ((lo - head + EPV - 1) / EPV) * EPV);
        vb = (c1 >= va + EPV) ? head + ((c1 - head) / EPV) * EPV : va;
        nv = (vb - va) / EPV;
        g = reinterpret_cast<const uint4*>(rowp + static_cast<long long>(va) * SX);
    }
};

constexpr int kLpStep = kLpVec * kLpThreads;             // vectors per batch

// Thread 0: bulk copy of batch q of a chunk into stage (nbat + q) % kLpStages.  The logits are read
// for the last time in the call: evict-first in L2.
__device__ __forceinline__ void lp_issue(LpSmem& s, const uint4* g, int nv, int nbat, int q) {
    const int st = (nbat + q) % kLpStages;
    const unsigned bytes = 16u * static_cast<unsigned>(min(kLpStep, nv - q * kLpStep));
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(reinterpret_cast<uint64_t*>(&s.full[st]), bytes);
    bulk_g2s_hint(s.stage[st], g + static_cast<long long>(q) * kLpStep, bytes, reinterpret_cast<uint64_t*>(&s.full[st]),
                  l2_evict_first_policy());
}

// Thread 0, as soon as the chunk is known: its first kLpStages batches (lp_chunk issues the rest).
template <int SX>
__device__ __forceinline__ void lp_issue_first(const Args& a, LpSmem& s, long long slot, int c0, int c1, int nbat) {
    const LpGeom<SX> gm(a, slot, c0, c1);
    const int nb = (gm.nv + kLpStep - 1) / kLpStep;
    for (int q = 0; q < kLpStages && q < nb; ++q) lp_issue(s, gm.g, gm.nv, nbat, q);
}

template <int SX, bool PEN>
// theta_known: a lower bound of the row's n-th largest logit known before the pass (the row's
// top-k threshold, below), else -inf with known == false.  The first kLpStages batches were issued by
// lp_issue_first.
__device__ void lp_chunk(const Args& a, LpSmem& s, long long slot, int c0, int c1, LpPartial* out, const LpRow& pr,
                         int& nbat, unsigned long long* cand, bool known, float theta_known) {
    constexpr int EPV = 16 / SX;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const LpGeom<SX> gm(a, slot, c0, c1);
    const int va = gm.va, vb = gm.vb, nv = gm.nv;
    const uint32_t ninf = SX == 2 ? 0xFF80FF80u : 0xFF800000u;     // -inf filler past the interior
    const int n_top = min(a.n_top, c1 - c0);
    // edges: thread 0 takes [c0, va), thread 1 takes [vb, c1) (fewer than EPV each)
    const int eh0 = tid == 0 ? c0 : (tid == 1 ? vb : 0);
    const int eh1 = tid == 0 ? va : (tid == 1 ? c1 : 0);
    float edge[EPV];
#pragma unroll
    for (int q = 0; q < EPV; ++q)
        edge[q] = (eh0 + q < eh1 && !(PEN && (pen_bits_range(a, pr.b, eh0 + q, 1) & 1u)))
                      ? load_x(a.x, SX, slot * a.V + eh0 + q) : -INFINITY;
    float tm = -INFINITY, ts = 0.f;
#pragma unroll
    for (int q = 0; q < EPV; ++q) tm = fmaxf(tm, edge[q]);
    if (tm > -INFINITY)
#pragma unroll
        for (int q = 0; q < EPV; ++q) ts += ex2_approx((edge[q] - tm) * kL2E);
    if (lane == 0) s.wn[warp] = 0;                        // keys this warp gathered
    __syncwarp();
    float theta = INFINITY;
    // the interior streams through two shared-memory stages, one batch (kLpVec vectors per
    // thread) each, copied by the bulk-copy engine: CTA batch counter nbat picks the stage
    // (nbat % kLpStages) and the phase ((nbat / kLpStages) & 1) of its barrier
    constexpr int kStep = kLpStep;
    const int nb = (nv + kStep - 1) / kStep;
    bool dead = false;                                    // a wait of this thread gave up
    auto load = [&](uint4 (&w)[kLpVec], int q) {
        const int st = (nbat + q) % kLpStages;
        if (!dead && !lp_wait(&s.full[st], ((nbat + q) / kLpStages) & 1)) {
            dead = true;
            atomicOr(&a.row_status[pr.b], DSPARK_ROW_INTERNAL);
        }
#pragma unroll
        for (int i = 0; i < kLpVec; ++i) {
            const int v = q * kStep + tid + i * kLpThreads;
            w[i] = v < nv ? s.stage[st][tid + i * kLpThreads] : make_uint4(ninf, ninf, ninf, ninf);
        }
    };
    // the logits >= theta of a batch, appended to the warp's list by the lanes holding them
    // (a shared-memory counter per warp; a hit is rare for a lane, so no warp-wide step per slot)
    auto gather = [&](const uint4 (&w)[kLpVec], int v0) {
        unsigned long long* k = s.keys + warp * kLpWarpCap;
#pragma unroll
        for (int i = 0; i < kLpVec; ++i) {
            const int v = v0 + tid + i * kLpThreads;
            if (v < nv && vmax_float<SX>(vmax_word<SX>(w[i])) >= theta) {
#pragma unroll
                for (int q = 0; q < EPV; ++q) {
                    const float x = lp_elem<SX>(w[i], q);
                    if (x >= theta) {
                        const int pos = atomicAdd(&s.wn[warp], 1);
                        if (pos < kLpWarpCap) k[pos] = ckey(x, va + v * EPV + q);
                    }
                }
            }
        }
    };
    auto reduce = [&](const uint4 (&w)[kLpVec]) {
        uint32_t bw = vmax_word<SX>(w[0]);
#pragma unroll
        for (int i = 1; i < kLpVec; ++i) bw = vmax_combine<SX>(bw, vmax_word<SX>(w[i]));
        const float bm = vmax_float<SX>(bw);
        if (bm > tm) {
            ts = (tm > -INFINITY) ? ts * ex2_approx((tm - bm) * kL2E) : 0.f;
            tm = bm;
        }
        if (tm > -INFINITY) {
            const float off = tm * kL2E;
            float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kLpVec; ++i)
#pragma unroll
                for (int q = 0; q < EPV; q += 2) {
                    const float2 t = __ffma2_rn(make_float2(lp_elem<SX>(w[i], q), lp_elem<SX>(w[i], q + 1)),
                                                make_float2(kL2E, kL2E), make_float2(-off, -off));
                    if (i & 1) acc1 = __fadd2_rn(acc1, make_float2(ex2_approx(t.x), ex2_approx(t.y)));
                    else acc0 = __fadd2_rn(acc0, make_float2(ex2_approx(t.x), ex2_approx(t.y)));
                }
            ts += (acc0.x + acc0.y) + (acc1.x + acc1.y);
        }
    };
    // penalised mode: the tokens the penalty index flags leave the streamed words (-inf); after
    // the stream they are taken one by one as x' (pen_tail)
    auto pen_mask = [&](uint4 (&w)[kLpVec], int v0) {
#pragma unroll
        for (int i = 0; i < kLpVec; ++i) {
            const int v = v0 + tid + i * kLpThreads;
            if (v >= nv) continue;
            const unsigned bits = pen_bits_range(a, pr.b, va + v * EPV, EPV);
            uint32_t* wd[4] = {&w[i].x, &w[i].y, &w[i].z, &w[i].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                if (SX == 2) {
                    const unsigned two = (bits >> (2 * h)) & 3u;
                    const uint32_t keep = ((two & 1u) ? 0u : 0x0000FFFFu) | ((two & 2u) ? 0u : 0xFFFF0000u);
                    const uint32_t set = ((two & 1u) ? 0x0000FF80u : 0u) | ((two & 2u) ? 0xFF800000u : 0u);
                    *wd[h] = (*wd[h] & keep) | set;
                } else if ((bits >> h) & 1u) {
                    *wd[h] = 0xFF800000u;
                }
            }
        }
    };
    // the flagged tokens of [c0, c1), 32 per bitmap word: x' into the thread's maximum and sum,
    // and gathered when >= theta
    auto pen_tail = [&]() {
        unsigned long long* k = s.keys + warp * kLpWarpCap;
        const int w0 = c0 >> 5, w1 = (c1 + 31) >> 5;
        for (int w = w0 + tid; w < w1; w += kLpThreads) {
            const int t0 = w << 5;
            const int tile = t0 / a.tile_x;
            unsigned bits = a.pen_bm[(static_cast<long long>(pr.b) * a.tiles_x + tile) * a.bm_words +
                                     ((t0 - tile * a.tile_x) >> 5)];
            if (t0 < c0) bits &= ~0u << (c0 - t0);
            if (t0 + 32 > c1) bits &= (c1 - t0 >= 32) ? ~0u : ((1u << (c1 - t0)) - 1u);
            while (bits) {
                const int t = t0 + __ffs(bits) - 1;
                bits &= bits - 1;
                const float xp = penalise(load_x(a.x, SX, slot * a.V + t), token_count(a, pr.b, pr.j, t), pr.f, pr.p);
                if (xp > tm) {
                    ts = (tm > -INFINITY) ? ts * ex2_approx((tm - xp) * kL2E) : 0.f;
                    tm = xp;
                }
                if (tm > -INFINITY) ts += ex2_approx((xp - tm) * kL2E);
                if (n_top > 0 && xp >= theta) {
                    const int pos = atomicAdd(&s.wn[warp], 1);
                    if (pos < kLpWarpCap) k[pos] = ckey(xp, t);
                }
            }
        }
    };
    for (int q = 0; q < max(nb, 1); ++q) {
        const int v0 = q * kStep;
        uint4 w[kLpVec];
        if (q < nb) {
            load(w, q);
        } else {
#pragma unroll
            for (int i = 0; i < kLpVec; ++i) w[i] = make_uint4(ninf, ninf, ninf, ninf);
        }
        __syncthreads();                                  // the stage is read: refill it
        if (tid == 0 && q + kLpStages < nb) lp_issue(s, gm.g, nv, nbat, q + kLpStages);
        if (PEN) pen_mask(w, v0);
        reduce(w);
        if (q == 0 && n_top > 0) {
            if (known) {
                theta = theta_known;
            } else {
                // theta from the first batch and the edges: the n-th largest of the threads'
                // maxima (a bitwise search over block counts), so at least n logits reach it
                const uint32_t mykey = fkey(tm);
                uint32_t th = 0u;
                for (int bit = 31; bit >= 0; --bit)
                    if (__syncthreads_count(mykey >= (th | (1u << bit))) >= n_top) th |= 1u << bit;
                theta = key_to_f(th);
            }
            // the edges' logits >= theta
            unsigned long long* k = s.keys + warp * kLpWarpCap;
#pragma unroll
            for (int e = 0; e < EPV; ++e)
                if (eh0 + e < eh1 && edge[e] >= theta) {
                    const int pos = atomicAdd(&s.wn[warp], 1);
                    if (pos < kLpWarpCap) k[pos] = ckey(edge[e], eh0 + e);
                }
        }
        if (n_top > 0) gather(w, v0);
    }
    nbat += nb;
    if (PEN) pen_tail();
    // block (max, sum): warp trees, then the warps in order
    {
        float m = tm, sm = ts;
        for (int o = 16; o; o >>= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, m, o);
            const float os = __shfl_xor_sync(0xffffffffu, sm, o);
            const float nm = fmaxf(m, om);
            sm = (nm > -INFINITY) ? sm * ex2_approx((m - nm) * kL2E) + os * ex2_approx((om - nm) * kL2E) : 0.f;
            m = nm;
        }
        if (lane == 0) { s.wm[warp] = m; s.wsum[warp] = sm; }
    }
    __syncthreads();
    int cnt = 0;
    int listed = 0;
    if (n_top > 0) {
        bool fits = true;
        int total = 0, before = 0;
        for (int q = 0; q < kLpWarps; ++q) {
            fits = fits && s.wn[q] <= kLpWarpCap;
            total += s.wn[q];
            if (q < warp) before += s.wn[q];
        }
        if (fits && cand && total <= kLpCandPerChunk) {
            // hand the gathered keys on unselected: each warp writes its list at its offset
            for (int i = lane; i < s.wn[warp]; i += 32) cand[before + i] = s.keys[warp * kLpWarpCap + i];
            cnt = total;
            listed = 1;
        } else if (fits) {
            // the chunk's n largest among the warps' gathered keys, by rank
            cnt = top_select(s, s.keys, s.wn, kLpWarps, kLpWarpCap, n_top, s.top);
            for (int i = tid; i < cnt; i += blockDim.x) out->top[i] = TopEntry{ckey_id(s.top[i]), ckey_v(s.top[i])};
        } else {
            cnt = min(lp_exact_top<SX, PEN>(a, s, slot, c0, c1, va, vb, n_top, pr), n_top);
            for (int i = tid; i < cnt; i += blockDim.x) out->top[i] = TopEntry{ckey_id(s.keys[i]), ckey_v(s.keys[i])};
        }
    }
    if (tid == 0) {
        float m = s.wm[0], sm = s.wsum[0];
        for (int q = 1; q < kLpWarps; ++q) {
            const float nm = fmaxf(m, s.wm[q]);
            sm = (nm > -INFINITY) ? sm * ex2_approx((m - nm) * kL2E) + s.wsum[q] * ex2_approx((s.wm[q] - nm) * kL2E) : 0.f;
            m = nm;
        }
        out->m = m;
        out->s = sm;
        out->n = cnt;
        out->listed = listed;
    }
}

// The CTA that completed row `slot` (request b, position j): merge the S chunk partials and
// write logprob and top_logprobs.  The whole CTA first copies the partials into shared memory
// in one parallel read; then one warp forms LSE = M + log(sum_c s_c exp(m_c - M)) with the
// chunks in a fixed order (lane l takes chunks l, l + 32, ... in order, then a fixed shuffle
// tree), and all threads select the row's top n among the chunks' lists by rank.
__device__ void lp_merge(const Args& a, LpSmem& s, long long slot, int b, int j, const LpPartial* part,
                         const unsigned long long* cands, int S, const LpRow& pr, bool pen) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int W = a.Km + 1;
    const int n_top = a.n_top;
    // the partials were written by other CTAs of this launch: read them from L2 (__ldcg).  Each
    // chunk's keys (its top list, or its unselected candidates) are staged one after another;
    // S <= kLpMergeLists chunks of at most kLpCandPerChunk keys fit the key buffer
    static_assert(kLpMergeLists * kLpCandPerChunk <= kLpCandCap, "merge staging");
    // the emitted token's logit, fetched by the last warp (which stages no keys: every chunk
    // holds fewer keys than the threads before it) while the others copy the partials
    constexpr int kTokThread = kLpThreads - 32;
    static_assert(kLpCandPerChunk <= kTokThread && DSPARK_MAX_TOP_LOGPROBS <= kTokThread, "token thread");
    int tok = -1;
    if (tid == kTokThread && a.out_lp) tok = a.out_tokens[static_cast<long long>(b) * W + j];
    for (int c = tid; c < S; c += blockDim.x) {
        s.mm[c] = __ldcg(&part[c].m);
        s.ms[c] = __ldcg(&part[c].s);
        s.mn[c] = __ldcg(&part[c].n);
        s.ml[c] = __ldcg(&part[c].listed);
    }
    __syncthreads();
    // A chunk holds at most kLpCandPerChunk unselected keys or n_top listed ones, so a thread
    // copies at most one key per chunk; four chunks' loads are in flight before their stores.
    static_assert(kLpCandPerChunk <= kLpThreads && DSPARK_MAX_TOP_LOGPROBS <= kLpThreads, "one key per thread");
    static_assert(kLpMergeLists % 4 == 0, "chunks in fours");
    int off = 0;
    for (int c0 = 0; c0 < S; c0 += 4) {
        unsigned long long kv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + u;
            kv[u] = 0ull;
            if (c < S && tid < s.mn[c])
                kv[u] = s.ml[c] ? __ldcg(cands + static_cast<long long>(c) * kLpCandPerChunk + tid)
                                : ckey(__ldcg(&part[c].top[tid].v), __ldcg(&part[c].top[tid].id));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + u;
            if (c < S) {
                if (tid < s.mn[c]) s.keys[off + tid] = kv[u];
                off += s.mn[c];
            }
        }
    }
    if (tid == 0) s.wcnt[0] = off;
    if (tid == kTokThread && a.out_lp) {                  // -inf: no token (its logprob is -inf too)
        const float xt = tok >= 0 ? load_x(a.x, a.sx, slot * a.V + tok) : -INFINITY;
        s.xt = tok < 0 ? -INFINITY : (pen ? lp_value<true>(a, pr, tok, xt) : xt);
    }
    __syncthreads();
    if (tid < 32) {
        float mm = -INFINITY;
        for (int c = lane; c < S; c += 32) mm = fmaxf(mm, s.mm[c]);
        mm = warp_max(mm);
        float sum = 0.f;
        if (mm > -INFINITY)
            for (int c = lane; c < S; c += 32)
                if (s.mm[c] > -INFINITY) sum += s.ms[c] * ex2_approx((s.mm[c] - mm) * kL2E);
        sum = warp_sum(sum);
        const float lse = mm + logf(sum);
        if (lane == 0) {
            s.theta = lse;
            if (a.out_lp) a.out_lp[static_cast<long long>(b) * W + j] = s.xt - lse;
        }
    }
    if (n_top <= 0) return;
    // the row's n largest among the chunks' lists, by rank (the lse is in s.theta after the barrier)
    const int cnt = top_select(s, s.keys, s.wcnt, 1, 0, n_top, s.top);
    const float lse = s.theta;
    const long long o = (static_cast<long long>(b) * W + j) * n_top;
    for (int q = tid; q < n_top; q += blockDim.x) {
        const bool ok = q < cnt;
        if (a.out_top_ids) a.out_top_ids[o + q] = ok ? ckey_id(s.top[q]) : -1;
        if (a.out_top_lp) a.out_top_lp[o + q] = ok ? ckey_v(s.top[q]) - lse : -INFINITY;
    }
}

// PEN_MODE: the call asked for penalised logprobs (rows of requests without a penalty still
// take the raw path: their x' is x and they have no penalty index).
template <int SX, bool PEN_MODE>
__global__ void __launch_bounds__(kLpThreads, kLpBlocksPerSm) logprob_kernel(Args a) {
    pdl_enter();
    extern __shared__ __align__(16) unsigned char lp_raw[];
    LpSmem& s = *reinterpret_cast<LpSmem*>(lp_raw);
    const int R = a.lp_list[0];
    if (R == 0) return;
    if (threadIdx.x == 0) {
        for (int st = 0; st < kLpStages; ++st) mbar_init(reinterpret_cast<uint64_t*>(&s.full[st]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    int nbat = 0;                                         // batches this CTA has streamed
    const int W = a.Km + 1;
    // chunks per row: all R * S chunks in one wave of this grid
    const int S = max(1, min(min(kLpMaxChunks, static_cast<int>(gridDim.x) / R), a.V / kLpMinChunk));
    const int chunk = ((a.V + S - 1) / S + 7) / 8 * 8;
    const int items = R * S;
    // item blockIdx.x first (S is chosen so that all R * S items fit the grid when R does);
    // past the grid, the next items come from a counter
    for (int it = blockIdx.x; it < items;) {
        const int p = it / S, c = it - p * S;                 // listed row p, its chunk c
        const int row = a.lp_list[1 + p];                    // b * W + j
        const int b = row / W, j = row % W;
        const int c0 = c * chunk, c1 = min(a.V, c0 + chunk);
        if (threadIdx.x == 0) lp_issue_first<SX>(a, s, row, c0, c1, nbat);   // before the row's parameters arrive
        LpPartial* part = a.lp_part + static_cast<long long>(p) * S;   // the row's S partials
        const dspark_row_params_t r = a.rows[b];
        const LpRow pr{b, j, r.frequency_penalty, r.presence_penalty};
        const bool pen = PEN_MODE && has_penalty(r);
        // a target row settled by a top-k list with k >= n: its k-th largest x' bounds the n-th
        // largest logit from below (x' itself in penalised mode; the raw x >= x' when the
        // penalties are not negative), so the pass gathers from there without a search
        const XRowOut xo = a.xout[row];
        const bool known = a.n_top > 0 && xo.mode == kModeList && r.top_k >= a.n_top && xo.kth > -INFINITY &&
                           (pen || (r.presence_penalty >= 0.f && r.frequency_penalty >= 0.f));
        unsigned long long* cands = a.lp_cand + static_cast<long long>(p) * S * kLpCandPerChunk;
        unsigned long long* cand = S > 1 ? cands + static_cast<long long>(c) * kLpCandPerChunk : nullptr;
        if (PEN_MODE && pen) lp_chunk<SX, PEN_MODE>(a, s, row, c0, c1, part + c, pr, nbat, cand, known, xo.kth);
        else lp_chunk<SX, false>(a, s, row, c0, c1, part + c, pr, nbat, cand, known, xo.kth);
        // the CTA finishing the row's last chunk merges them: partial written, then counted
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            s.last = atomicAdd(&a.lp_done[p], 1) == S - 1;
        }
        __syncthreads();
        if (s.last) {
            __threadfence();
            lp_merge(a, s, row, b, j, part, cands, S, pr, pen);
        }
        if (items <= static_cast<int>(gridDim.x)) break;
        __syncthreads();                                     // shared memory reused by the next item
        if (threadIdx.x == 0) s.item = static_cast<int>(gridDim.x) + atomicAdd(&a.plan->pad[2], 1);
        __syncthreads();
        it = s.item;
    }
}

}  // namespace

template <int SX, bool PEN>
cudaError_t launch_lp(const Args& a, cudaStream_t s) {
    const size_t smem = sizeof(LpSmem);
    const int grid = kLpBlocksPerSm * a.grid_ss;           // persistent: four CTAs per SM
    cudaError_t e = cudaFuncSetAttribute(logprob_kernel<SX, PEN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_k(logprob_kernel<SX, PEN>, dim3(grid), dim3(kLpThreads), smem, s, true, a);
}

cudaError_t launch_logprobs(const Args& a, cudaStream_t s) {
    if (a.sx == 2) return a.lp_pen ? launch_lp<2, true>(a, s) : launch_lp<2, false>(a, s);
    return a.lp_pen ? launch_lp<4, true>(a, s) : launch_lp<4, false>(a, s);
}

}  // namespace dspark
