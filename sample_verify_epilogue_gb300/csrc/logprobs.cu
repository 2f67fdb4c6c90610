// logprob_kernel: the raw log-softmax of each emitted token and the top_logprobs list at its
// position (mlx-dspark Changelog, [0.2.0] Added, "logprobs / top_logprobs": the raw target
// log-softmax of each committed token plus the top candidates, gathered on the GPU only when
// requested).  Only the positions a request emits from (j <= accept length) need them, so
// they are taken after the draws, from those rows alone: accept_kernel lists the rows.
//
// One CTA of 1024 threads per listed row (the launch has one CTA per possible row; the rest
// return at once).  It streams the row from HBM in batches of kLpVec 16-byte vectors per
// thread, the next batch's loads in flight while the current one is reduced, for
//   - the row's maximum m and its sum of exp(x - m) (per thread a running maximum, the sum
//     rescaled at most once per batch; then a fixed reduction order);
//   - the row's n largest logits by (value descending, id ascending).  After the first batch,
//     theta = the least over the 32 warps of each warp's ceil(n/32)-th largest thread maximum:
//     at least n distinct logits of that batch reach it, so every one of the row's top n does,
//     and the logits >= theta of every batch are gathered as they stream by; each warp sorts
//     its share and one warp merges the 32 sorted lists.  When ties put more logits >= theta
//     than fit, the row is settled exactly from L2: the n-th largest value v by a bitwise
//     search over counts, the logits above v, then the lowest ids equal to v.
// It then writes logprob = x[token] - (m + log s) and the top list.  Results do not depend on
// scheduling.
//
// Penalised mode (the other reading of "raw target log-softmax"): the same over the penalised
// logits x' of the position.  Tokens the penalty index flags for the request (history and
// drafts) have their logit replaced by x' as each batch arrives: the vector's lane is set to
// -inf for the packed reduction and x' is folded into the thread's maximum and sum, and
// gathered, on its own.  Every other logit is its own x'.
#include "block_utils.cuh"

namespace dspark {

namespace {

constexpr int kLpThreads = 1024;
constexpr int kLpWarps = kLpThreads / 32;
constexpr int kLpCandCap = 4096;
constexpr int kLpVec = 4;                    // 16-byte vectors per thread and batch
constexpr int kLpWarpCap = kLpCandCap / kLpWarps;
constexpr int kLpMergeLists = 256;           // chunk partials the merge copies to shared memory
constexpr float kL2E = 1.4426950408889634f;

struct LpSmem {
    unsigned long long keys[kLpCandCap];   // (fkey(value) << 32) | (0xFFFFFFFF - id); warp w: [w*kLpWarpCap, ...)
    float tmax[kLpThreads];
    float wth[kLpWarps];
    float wm[kLpWarps];
    float wsum[kLpWarps];
    int wcnt[kLpWarps + 1];
    int wn[kLpWarps];                      // keys each warp gathered
    double dwarp[33];
    int n;
    int last;
    int item;
    float theta;
    unsigned long long top[2 * DSPARK_MAX_TOP_LOGPROBS];
    int mcur[kLpMergeLists];               // the merge's list cursors
    float mm[kLpMergeLists];               // the merge's copies of the chunk partials
    float ms[kLpMergeLists];
    int mn[kLpMergeLists];
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

// Append element (v, id) to the gathered keys when there is room.
__device__ __forceinline__ void lp_push(LpSmem& s, float v, int id) {
    const int p = atomicAdd(&s.n, 1);
    if (p < kLpCandCap) s.keys[p] = ckey(v, id);
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

// Each warp sorts its gathered keys (descending) in place; warp w's keys sit at
// s.keys[w * kLpWarpCap, + s.wn[w]).  Lists longer than 64 are sorted by the warp with a
// bitonic network over shared memory.
__device__ void lp_sort_warp_lists(LpSmem& s) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long* k = s.keys + warp * kLpWarpCap;
    const int cnt = min(s.wn[warp], kLpWarpCap);
    if (cnt <= 64) {
        unsigned long long r[2];
        r[0] = lane < cnt ? k[lane] : 0ull;
        r[1] = lane + 32 < cnt ? k[lane + 32] : 0ull;
        for (int size = 2; size <= 64; size <<= 1)
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                if (stride == 32) {
                    const unsigned long long hi = r[0] > r[1] ? r[0] : r[1];
                    const unsigned long long lo = r[0] > r[1] ? r[1] : r[0];
                    r[0] = hi;
                    r[1] = lo;
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int pos = lane + 32 * h;
                        const unsigned long long o = __shfl_xor_sync(0xffffffffu, r[h], stride);
                        const bool keep_max = ((pos & stride) == 0) == ((pos & size) == 0);
                        r[h] = keep_max ? (r[h] > o ? r[h] : o) : (r[h] < o ? r[h] : o);
                    }
                }
            }
        if (lane < cnt) k[lane] = r[0];
        if (lane + 32 < cnt) k[lane + 32] = r[1];
        __syncwarp();
        return;
    }
    const int P = next_pow2(cnt);
    for (int i = cnt + lane; i < P; i += 32) k[i] = 0ull;
    __syncwarp();
    for (int size = 2; size <= P; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = lane; i < P / 2; i += 32) {
                const int lo = 2 * i - (i & (stride - 1)), hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const unsigned long long x = k[lo], y = k[hi];
                if ((x < y) == desc) { k[lo] = y; k[hi] = x; }
            }
            __syncwarp();
        }
}

// One chunk [c0, c1) of target row `slot`: its maximum, its sum of exp relative to it and its
// top-n list, written to *out.
template <int SX, bool PEN>
__device__ void lp_chunk(const Args& a, LpSmem& s, long long slot, int c0, int c1, LpPartial* out, const LpRow& pr) {
    constexpr int EPV = 16 / SX;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned char* rowp = static_cast<const unsigned char*>(a.x) + slot * a.V * SX;
    const int head = static_cast<int>(((16u - static_cast<unsigned>(reinterpret_cast<uintptr_t>(rowp) & 15u)) & 15u) / SX);
    // aligned interior [va, vb): element e starts a vector iff (e - head) % EPV == 0
    const int lo = max(c0, head);
    const int va = min(c1, head + ((lo - head + EPV - 1) / EPV) * EPV);
    const int vb = (c1 >= va + EPV) ? head + ((c1 - head) / EPV) * EPV : va;
    const int nv = (vb - va) / EPV;
    const uint4* g = reinterpret_cast<const uint4*>(rowp + static_cast<long long>(va) * SX);
    const uint32_t ninf = SX == 2 ? 0xFF80FF80u : 0xFF800000u;     // -inf filler past the interior
    const int n_top = min(a.n_top, c1 - c0);
    // edges: thread 0 takes [c0, va), thread 1 takes [vb, c1) (fewer than EPV each)
    const int eh0 = tid == 0 ? c0 : (tid == 1 ? vb : 0);
    const int eh1 = tid == 0 ? va : (tid == 1 ? c1 : 0);
    float edge[EPV];
#pragma unroll
    for (int q = 0; q < EPV; ++q)
        edge[q] = eh0 + q < eh1 ? lp_value<PEN>(a, pr, eh0 + q, load_x(a.x, SX, slot * a.V + eh0 + q)) : -INFINITY;
    float tm = -INFINITY, ts = 0.f;
#pragma unroll
    for (int q = 0; q < EPV; ++q) tm = fmaxf(tm, edge[q]);
    if (tm > -INFINITY)
#pragma unroll
        for (int q = 0; q < EPV; ++q) ts += ex2_approx((edge[q] - tm) * kL2E);
    if (lane == 0) s.wn[warp] = 0;                        // keys this warp gathered
    __syncwarp();
    float theta = INFINITY;
    uint4 wa[kLpVec], wb[kLpVec];
    auto load = [&](uint4 (&w)[kLpVec], int v0) {
#pragma unroll
        for (int i = 0; i < kLpVec; ++i) {
            const int v = v0 + tid + i * kLpThreads;
            w[i] = v < nv ? __ldg(g + v) : make_uint4(ninf, ninf, ninf, ninf);
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
    // penalised mode: the flagged tokens of a batch leave the packed words (-inf) and enter the
    // thread's maximum and sum as x', gathered at once when theta is known (later, for batch 0)
    auto fold = [&](float xp) {
        if (xp > tm) {
            ts = (tm > -INFINITY) ? ts * ex2_approx((tm - xp) * kL2E) : 0.f;
            tm = xp;
        }
        if (tm > -INFINITY) ts += ex2_approx((xp - tm) * kL2E);
    };
    auto pen_fix = [&](uint4 (&w)[kLpVec], int v0, bool gather_now) {
        unsigned long long* k = s.keys + warp * kLpWarpCap;
#pragma unroll
        for (int i = 0; i < kLpVec; ++i) {
            const int v = v0 + tid + i * kLpThreads;
            if (v >= nv) continue;
            const int e0 = va + v * EPV;
            const unsigned bits = pen_bits_range(a, pr.b, e0, EPV);
            if (!bits) continue;
#pragma unroll
            for (int q = 0; q < EPV; ++q) {
                if (!((bits >> q) & 1u)) continue;
                const float xp = penalise(lp_elem<SX>(w[i], q), token_count(a, pr.b, pr.j, e0 + q), pr.f, pr.p);
                fold(xp);
                if (gather_now && xp >= theta && n_top > 0) {
                    const int pos = atomicAdd(&s.wn[warp], 1);
                    if (pos < kLpWarpCap) k[pos] = ckey(xp, e0 + q);
                }
            }
            // the flagged lanes leave the packed words: -inf in their halves (bf16) or words (fp32)
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
    // batch 0's flagged tokens once theta is known (their logits re-read; the words were masked)
    auto pen_gather0 = [&]() {
        unsigned long long* k = s.keys + warp * kLpWarpCap;
        for (int i = 0; i < kLpVec; ++i) {
            const int v = tid + i * kLpThreads;
            if (v >= nv) continue;
            const int e0 = va + v * EPV;
            unsigned bits = pen_bits_range(a, pr.b, e0, EPV);
            while (bits) {
                const int q = __ffs(bits) - 1;
                bits &= bits - 1;
                const float xp = penalise(load_x(a.x, SX, slot * a.V + e0 + q), token_count(a, pr.b, pr.j, e0 + q),
                                          pr.f, pr.p);
                if (xp >= theta) {
                    const int pos = atomicAdd(&s.wn[warp], 1);
                    if (pos < kLpWarpCap) k[pos] = ckey(xp, e0 + q);
                }
            }
        }
    };
    constexpr int kStep = kLpVec * kLpThreads;
    load(wa, 0);
    for (int v0 = 0; v0 < max(nv, 1); v0 += 2 * kStep) {
        // batch v0 in wa (loaded), batch v0 + kStep into wb while wa is reduced
        if (v0 + kStep < nv) load(wb, v0 + kStep);
        if (PEN) pen_fix(wa, v0, v0 > 0);
        reduce(wa);
        if (v0 == 0 && n_top > 0) {
            // theta from the first batch and the edges
            const float wk = warp_kth_largest(tm, (n_top + kLpWarps - 1) / kLpWarps);
            if (lane == 0) s.wth[warp] = wk;
            __syncthreads();
            theta = s.wth[0];
            for (int q = 1; q < kLpWarps; ++q) theta = fminf(theta, s.wth[q]);
            // the edges' logits >= theta
            unsigned long long* k = s.keys + warp * kLpWarpCap;
#pragma unroll
            for (int q = 0; q < EPV; ++q)
                if (eh0 + q < eh1 && edge[q] >= theta) {
                    const int pos = atomicAdd(&s.wn[warp], 1);
                    if (pos < kLpWarpCap) k[pos] = ckey(edge[q], eh0 + q);
                }
            if (PEN) pen_gather0();
        }
        if (n_top > 0) gather(wa, v0);
        if (v0 + kStep >= nv) break;
        if (v0 + 2 * kStep < nv) load(wa, v0 + 2 * kStep);
        if (PEN) pen_fix(wb, v0 + kStep, true);
        reduce(wb);
        if (n_top > 0) gather(wb, v0 + kStep);
    }
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
    if (n_top > 0) {
        bool fits = true;
        for (int q = 0; q < kLpWarps; ++q) fits = fits && s.wn[q] <= kLpWarpCap;
        if (fits) {
            lp_sort_warp_lists(s);
            __syncthreads();
            // warp 0 merges the eight sorted lists: n rounds, lane q < 8 offers list q's head
            if (tid < 32) {
                int cur = 0;
                const int mine_n = lane < kLpWarps ? s.wn[lane] : 0;
                for (int r = 0; r < n_top; ++r) {
                    const unsigned long long h = cur < mine_n ? s.keys[lane * kLpWarpCap + cur] : 0ull;
                    unsigned long long best = h;
                    for (int off = 16; off; off >>= 1) {
                        const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, off);
                        best = y > best ? y : best;
                    }
                    if (best == 0ull) break;
                    if (h == best) ++cur;                  // keys are unique: one lane holds it
                    if (lane == 0) s.top[r] = best;
                    cnt = r + 1;
                }
                cnt = __shfl_sync(0xffffffffu, cnt, 0);
                for (int i = lane; i < cnt; i += 32) out->top[i] = TopEntry{ckey_id(s.top[i]), ckey_v(s.top[i])};
                if (lane == 0) s.n = cnt;
            }
            __syncthreads();
            cnt = s.n;
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
    }
}

// Rows of more than kLpMergeLists chunks (vocabularies above 4M): the row's top-n by sorting
// the chunk lists in batches that fit the key buffer, keeping the best n after each batch.
__device__ void lp_merge_large(const Args& a, LpSmem& s, long long slot, int b, int j, const LpPartial* part, int S,
                               const LpRow& pr, bool pen) {
    const int tid = threadIdx.x;
    const int W = a.Km + 1;
    const int n_top = a.n_top;
    float mm = -INFINITY;
    for (int c = tid; c < S; c += blockDim.x) mm = fmaxf(mm, __ldcg(&part[c].m));
    mm = block_max_nan(mm, s.tmax);
    float sum = 0.f;
    if (mm > -INFINITY)
        for (int c = tid; c < S; c += blockDim.x) {
            const float mc = __ldcg(&part[c].m);
            if (mc > -INFINITY) sum += __ldcg(&part[c].s) * ex2_approx((mc - mm) * kL2E);
        }
    sum = static_cast<float>(block_sum_d(static_cast<double>(sum), s.dwarp));
    const float lse = mm + logf(sum);
    if (tid == 0 && a.out_lp) {
        const int t = a.out_tokens[static_cast<long long>(b) * W + j];
        const float xt = t >= 0 ? load_x(a.x, a.sx, slot * a.V + t) : 0.f;
        a.out_lp[static_cast<long long>(b) * W + j] = t >= 0 ? (pen ? lp_value<true>(a, pr, t, xt) : xt) - lse : -INFINITY;
    }
    int have = 0;
    for (int c0 = 0; c0 < S;) {
        int c1 = c0, room = kLpCandCap - have;
        while (c1 < S && __ldcg(&part[c1].n) <= room) { room -= __ldcg(&part[c1].n); ++c1; }
        int base = have;
        for (int c = c0; c < c1; ++c) {
            const int nc = __ldcg(&part[c].n);
            for (int i = tid; i < nc; i += blockDim.x)
                s.keys[base + i] = ckey(__ldcg(&part[c].top[i].v), __ldcg(&part[c].top[i].id));
            base += nc;
        }
        __syncthreads();
        sort_keys_desc(s, base);
        have = min(base, n_top);
        c0 = c1;
    }
    const long long o = (static_cast<long long>(b) * W + j) * n_top;
    for (int q = tid; q < n_top; q += blockDim.x) {
        const bool ok = q < have;
        if (a.out_top_ids) a.out_top_ids[o + q] = ok ? ckey_id(s.keys[q]) : -1;
        if (a.out_top_lp) a.out_top_lp[o + q] = ok ? ckey_v(s.keys[q]) - lse : -INFINITY;
    }
}

// The CTA that completed row `slot` (request b, position j): merge the S chunk partials and
// write logprob and top_logprobs.  The whole CTA first copies the partials into shared memory
// in one parallel read (the merge would otherwise wait on L2 once per step), then one warp:
// LSE = M + log(sum_s S_s exp(m_s - M)) with the chunks in a fixed order (lane l takes chunks
// l, l + 32, ... in order, then a fixed shuffle tree), and the row's top-n by an n-round merge
// of the chunks' sorted lists (every round the lanes offer the largest head among their lists
// and the winner's list advances).
__device__ void lp_merge(const Args& a, LpSmem& s, long long slot, int b, int j, const LpPartial* part, int S,
                         const LpRow& pr, bool pen) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int W = a.Km + 1;
    const int n_top = a.n_top;
    // the partials were written by other CTAs of this launch: read them from L2 (__ldcg)
    const bool staged = S <= kLpMergeLists && S * n_top <= kLpCandCap;
    if (S > kLpMergeLists && n_top > 0) {
        lp_merge_large(a, s, slot, b, j, part, S, pr, pen);
        return;
    }
    for (int c = tid; c < S && c < kLpMergeLists; c += blockDim.x) {   // (more are read from L2)
        s.mm[c] = __ldcg(&part[c].m);
        s.ms[c] = __ldcg(&part[c].s);
        s.mn[c] = __ldcg(&part[c].n);
    }
    if (staged)
        for (int e = tid; e < S * n_top; e += blockDim.x) {
            const int c = e / n_top, k = e - c * n_top;
            s.keys[e] = ckey(__ldcg(&part[c].top[k].v), __ldcg(&part[c].top[k].id));
        }
    __syncthreads();
    if (tid >= 32) return;
    auto pm = [&](int c) { return c < kLpMergeLists ? s.mm[c] : __ldcg(&part[c].m); };
    auto ps = [&](int c) { return c < kLpMergeLists ? s.ms[c] : __ldcg(&part[c].s); };
    auto pn = [&](int c) { return c < kLpMergeLists ? s.mn[c] : __ldcg(&part[c].n); };
    float mm = -INFINITY;
    for (int c = lane; c < S; c += 32) mm = fmaxf(mm, pm(c));
    mm = warp_max(mm);
    float sum = 0.f;
    if (mm > -INFINITY)
        for (int c = lane; c < S; c += 32)
            if (pm(c) > -INFINITY) sum += ps(c) * ex2_approx((pm(c) - mm) * kL2E);
    sum = warp_sum(sum);
    const float lse = mm + logf(sum);
    if (lane == 0 && a.out_lp) {
        const int t = a.out_tokens[static_cast<long long>(b) * W + j];
        const float xt = t >= 0 ? load_x(a.x, a.sx, slot * a.V + t) : 0.f;
        a.out_lp[static_cast<long long>(b) * W + j] = t >= 0 ? (pen ? lp_value<true>(a, pr, t, xt) : xt) - lse : -INFINITY;
    }
    if (n_top <= 0) return;
    // cursor of every chunk list: a chunk list c is read at position cur[c / 32] of lane c % 32's
    // slot c / 32 (kept in shared memory for up to kLpMergeLists lists, else in registers' reach)
    int* cur = s.mcur;
    for (int c = lane; c < S && c < kLpMergeLists; c += 32) cur[c] = 0;
    __syncwarp();
    const long long o = (static_cast<long long>(b) * W + j) * n_top;
    for (int q = 0; q < n_top; ++q) {
        unsigned long long best = 0ull;
        int bc = -1;
        for (int c = lane; c < S && c < kLpMergeLists; c += 32) {
            const int k = cur[c];
            if (k < pn(c)) {
                const unsigned long long key = staged ? s.keys[c * n_top + k]
                                                      : ckey(__ldcg(&part[c].top[k].v), __ldcg(&part[c].top[k].id));
                if (bc < 0 || key > best) { best = key; bc = c; }
            }
        }
        unsigned long long wbest = best;
        for (int off = 16; off; off >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, wbest, off);
            wbest = y > wbest ? y : wbest;
        }
        const unsigned who = __ballot_sync(0xffffffffu, bc >= 0 && best == wbest);
        if (who == 0u) {                                   // fewer logits than n_top in the row
            if (lane == 0) {
                if (a.out_top_ids) a.out_top_ids[o + q] = -1;
                if (a.out_top_lp) a.out_top_lp[o + q] = -INFINITY;
            }
            continue;
        }
        if (lane == __ffs(who) - 1) cur[bc] += 1;
        if (lane == 0) {
            if (a.out_top_ids) a.out_top_ids[o + q] = ckey_id(wbest);
            if (a.out_top_lp) a.out_top_lp[o + q] = ckey_v(wbest) - lse;
        }
        __syncwarp();
    }
}

// PEN_MODE: the call asked for penalised logprobs (rows of requests without a penalty still
// take the raw path: their x' is x and they have no penalty index).
template <int SX, bool PEN_MODE>
__global__ void __launch_bounds__(kLpThreads, 1) logprob_kernel(Args a) {
    pdl_enter();
    extern __shared__ __align__(16) unsigned char lp_raw[];
    LpSmem& s = *reinterpret_cast<LpSmem*>(lp_raw);
    if (static_cast<int>(blockIdx.x) >= a.lp_list[0]) return;
    const int W = a.Km + 1;
    const int row = a.lp_list[1 + blockIdx.x];            // b * W + j
    const int b = row / W, j = row % W;
    LpPartial* part = a.lp_part + row;
    const dspark_row_params_t r = a.rows[b];
    const LpRow pr{b, j, r.frequency_penalty, r.presence_penalty};
    const bool pen = PEN_MODE && has_penalty(r);
    if (PEN_MODE && pen) lp_chunk<SX, PEN_MODE>(a, s, row, 0, a.V, part, pr);
    else lp_chunk<SX, false>(a, s, row, 0, a.V, part, pr);
    __syncthreads();                                      // the partial (global) is visible to the CTA
    lp_merge(a, s, row, b, j, part, 1, pr, pen);
}

}  // namespace

template <int SX, bool PEN>
cudaError_t launch_lp(const Args& a, cudaStream_t s) {
    const size_t smem = sizeof(LpSmem);
    const int grid = a.xslots;                             // one CTA per row that may be listed
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
