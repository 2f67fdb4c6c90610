// prep_kernel: request checks, the segment counts of the streaming pass and the
// per-(request, vocab tile) penalty index, in one launch.
//
// Block b*tiles_x + t checks request b's parameters and draft ids; block t = 0 also writes
// the row_status bits and the number of segments the request needs (K_b+1 target rows and,
// when T > 0, K_b draft rows; none for an invalid request), from which every streaming CTA
// derives the plan.  For a request with a non-zero penalty, the block then builds, for the
// vocab tile
// t, the tokens of that tile which may carry a penalty: the request's completion-history
// tokens in the tile (with their counts) and its draft tokens in the tile, each with a
// bit mask of the draft positions holding it.  Verify position j then counts
// c = base + popcount(mask & ((1 << j) - 1)), i.e. the history plus its own draft prefix
// (mlx-dspark Changelog, [0.2.0] Added, "presence_penalty / frequency_penalty").  A bitmap
// over the tile marks those tokens so the streaming pass tests eight logits per byte.
//
// Draft layouts other than dense: block t = 0 of a sampled request checks its sparse draft rows
// (ids in [0, V), no id twice in a row).  For a reduced draft vocabulary, blocks past the
// B * tiles_x request blocks invert the d2t table into t2d (target id -> draft id, -1 for none),
// flagging a target id outside [0, V) or reached twice (mlx-dspark Changelog, [0.8.0] Added:
// a draft id d stands for target id d + d2t[d]; a mismatched table is refused, never decoded).
#include "dspark_internal.cuh"

namespace dspark {

namespace {

constexpr int kPrepThreads = 256;

// First indices in ids[lo, hi) with ids[idx] >= key0 and >= key1 (key0 <= key1), by a
// block-wide 256-way narrowing of both ranges at once.
__device__ void block_lower_bound2(const int* ids, int lo, int hi, int key0, int key1, int& r0, int& r1) {
    const int tid = threadIdx.x;
    int lo0 = lo, hi0 = hi, lo1 = lo, hi1 = hi;
    // each range is narrowed until it is empty; the answer is then its lo
    while (hi0 > lo0 || hi1 > lo1) {
        const int len0 = hi0 - lo0, len1 = hi1 - lo1;
        const int st0 = max(1, (len0 + kPrepThreads - 1) / kPrepThreads);
        const int st1 = max(1, (len1 + kPrepThreads - 1) / kPrepThreads);
        const int p0 = lo0 + tid * st0, p1 = lo1 + tid * st1;
        const int v0 = (len0 > 0 && p0 < hi0) ? __ldg(ids + p0) : 0;
        const int v1 = (len1 > 0 && p1 < hi1) ? __ldg(ids + p1) : 0;
        const int c0 = __syncthreads_count(len0 > 0 && p0 < hi0 && v0 < key0);
        const int c1 = __syncthreads_count(len1 > 0 && p1 < hi1 && v1 < key1);
        // predicates form a prefix (ids ascending): ids[lo + (c-1)*st] < key <= ids[lo + c*st]
        if (len0 > 0) {
            if (c0 == 0) hi0 = lo0;
            else { const int nl = lo0 + (c0 - 1) * st0 + 1; hi0 = min(hi0, lo0 + c0 * st0); lo0 = nl; }
        }
        if (len1 > 0) {
            if (c1 == 0) hi1 = lo1;
            else { const int nl = lo1 + (c1 - 1) * st1 + 1; hi1 = min(hi1, lo1 + c1 * st1); lo1 = nl; }
        }
    }
    r0 = lo0;
    r1 = lo1;
}

__device__ void penalty_index_block(const Args& a, int b, int t) {
    __shared__ unsigned s_bm[kBitmapWordsMax];
    __shared__ PenEntry s_ent[kPenCap];
    __shared__ int s_d[DSPARK_MAX_K];
    __shared__ dspark_row_params_t s_r;
    __shared__ int s_hlo, s_hhi, s_n, s_nh, s_over, s_bad;
    const int tid = threadIdx.x;
    // one round trip for the parameters, the drafts and the history bounds
    if (tid == 0) s_r = a.rows[b];
    if (tid == 32) { s_hlo = a.h_off ? a.h_off[b] : 0; s_hhi = a.h_off ? a.h_off[b + 1] : 0; }
    if (tid >= 64 && tid < 64 + a.Km) s_d[tid - 64] = a.d[static_cast<long long>(b) * a.Km + (tid - 64)];
    if (tid == 0) s_bad = 0;
    if (b == 0 && t == 0 && tid == 0) a.fin_list[0] = 0;    // rows left to the block finalize
    __syncthreads();
    const dspark_row_params_t r = s_r;
    const int K = r.num_drafts;
    const int pst = params_status(a, r);
    if (pst == 0)
        for (int i = tid; i < K; i += kPrepThreads) if (s_d[i] < 0 || s_d[i] >= a.V) s_bad = 1;
    if (t == 0 && pst == 0 && a.q_layout == kQSparse && r.temperature > 0.f && a.q != nullptr) {
        const int m = a.Lq;
        int bad = 0;
        for (int e = tid; e < K * m; e += kPrepThreads) {
            const int i = e / m, k = e - i * m;
            const int* ids = a.q_ids + (static_cast<long long>(b) * a.Km + i) * m;
            const int id = __ldg(ids + k);
            if (id < 0 || id >= a.V) bad = 1;
            for (int k2 = 0; k2 < k; ++k2) bad |= (__ldg(ids + k2) == id);
        }
        if (__syncthreads_or(bad) && tid == 0) s_bad = 1;
    }
    __syncthreads();
    if (t == 0 && tid == 0) {
        const int st = pst ? pst : (s_bad ? DSPARK_ROW_BAD_DRAFT : 0);
        if (st) atomicOr(&a.row_status[b], st);
        const int nx = st ? 0 : (K + 1) * a.nseg_x;
        a.req_n[b] = st ? 0 : nx + (r.temperature > 0.f ? K * a.nseg_q : 0);
        a.req_n[a.B + b] = nx;
    }
    if (pst || s_bad) return;
    const int e0 = t * a.tile_x, e1 = min(a.V, e0 + a.tile_x);
    const int hlo = s_hlo, hhi = s_hhi;
    // history validation (once per request): ascending ids in range, positive counts
    if (t == 0 && hhi > hlo) {
        int bad = 0;
        for (int k0 = hlo + tid; k0 < hhi; k0 += 4 * kPrepThreads) {
            int id[4], pv[4], cn[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {            // four independent loads in flight
                const int k = k0 + u * kPrepThreads;
                id[u] = k < hhi ? a.h_ids[k] : 0;
                pv[u] = (k < hhi && k > hlo) ? a.h_ids[k - 1] : -1;
                cn[u] = k < hhi ? a.h_cnt[k] : 1;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = k0 + u * kPrepThreads;
                if (k < hhi && (id[u] < 0 || id[u] >= a.V || cn[u] <= 0 || pv[u] >= id[u])) bad = 1;
            }
        }
        if (__syncthreads_or(bad) && tid == 0) atomicOr(&a.row_status[b], DSPARK_ROW_BAD_HISTORY);
    }
    if (!has_penalty(r)) return;
    for (int w = tid; w < a.bm_words; w += kPrepThreads) s_bm[w] = 0u;
    int h0 = hlo, h1 = hlo;
    if (hhi > hlo) block_lower_bound2(a.h_ids, hlo, hhi, e0, e1, h0, h1);
    const int nh = h1 - h0;
    if (tid == 0) { s_nh = min(nh, kPenCap); s_over = nh > kPenCap; }
    __syncthreads();
    for (int k = tid; k < nh; k += kPrepThreads) {
        const int id = a.h_ids[h0 + k];
        if (k < kPenCap) s_ent[k] = PenEntry{id, a.h_cnt[h0 + k], 0u, 0u};
        if (id >= e0 && id < e1) atomicOr(&s_bm[(id - e0) >> 5], 1u << ((id - e0) & 31));
    }
    __syncthreads();
    // draft tokens in this tile: serial over positions (K <= 64), in order, all in shared memory
    if (tid == 0) {
        int n = s_nh;
        for (int i = 0; i < K; ++i) {
            const int tok = s_d[i];
            if (tok < e0 || tok >= e1) continue;
            int base = 0, slot = -1;
            if (!s_over) {
                int l = 0, h = s_nh;
                while (l < h) { const int m = (l + h) >> 1; if (s_ent[m].token < tok) l = m + 1; else h = m; }
                if (l < s_nh && s_ent[l].token == tok) { slot = l; base = s_ent[l].base; }
            } else {
                int l = h0, h = h1;
                while (l < h) { const int m = (l + h) >> 1; if (a.h_ids[m] < tok) l = m + 1; else h = m; }
                if (l < h1 && a.h_ids[l] == tok) { base = a.h_cnt[l]; slot = (l - h0 < kPenCap) ? l - h0 : -2; }
            }
            if (slot == -1) {
                for (int e = s_nh; e < n; ++e) if (s_ent[e].token == tok) { slot = e; break; }
                if (slot == -1) {
                    if (n < kPenCap) { s_ent[n] = PenEntry{tok, 0, 0u, 0u}; slot = n++; }
                    else { s_over = 1; slot = -2; }
                }
            }
            if (slot >= 0) {
                if (i < 32) s_ent[slot].mask_lo |= 1u << i; else s_ent[slot].mask_hi |= 1u << (i - 32);
            }
            a.draft_base[static_cast<long long>(b) * a.Km + i] = base;
            s_bm[(tok - e0) >> 5] |= 1u << ((tok - e0) & 31);
        }
        s_n = n;
    }
    __syncthreads();
    const long long pt = static_cast<long long>(b) * a.tiles_x + t;
    for (int w = tid; w < a.bm_words; w += kPrepThreads) a.pen_bm[pt * a.bm_words + w] = s_bm[w];
    for (int k = tid; k < s_n; k += kPrepThreads) a.pen_ent[pt * kPenCap + k] = s_ent[k];
    if (tid == 0) {
        PenHdr h;
        h.n = s_n; h.overflow = s_over; h.pad[0] = s_nh; h.pad[1] = 0;
        a.pen_hdr[pt] = h;
    }
}

// Blocks past the request blocks: the inverse of the d2t table, four draft ids per thread.
__device__ void d2t_block(const Args& a, int blk) {
    int bad = 0;
    for (int k = 0; k < 4; ++k) {
        const long long e = (static_cast<long long>(blk) * 4 + k) * kPrepThreads + threadIdx.x;
        if (e >= a.Lq) break;
        const long long t = e + static_cast<long long>(__ldg(a.d2t + e));
        if (t < 0 || t >= a.V) { bad = 1; continue; }
        if (atomicCAS(a.t2d + t, -1, static_cast<int>(e)) != -1) bad = 1;
    }
    if (bad) atomicOr(&a.plan->pad[1], 1);
}

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(Args a) {
    pdl_trigger();
    const int nreq = a.B * a.tiles_x;
    if (static_cast<int>(blockIdx.x) >= nreq) {
        d2t_block(a, blockIdx.x - nreq);
        return;
    }
    penalty_index_block(a, blockIdx.x / a.tiles_x, blockIdx.x % a.tiles_x);
}

}  // namespace

cudaError_t launch_prep(const Args& a, cudaStream_t s) {
    const int nd2t = (a.q_layout == kQReduced && a.q) ? (a.Lq + 4 * kPrepThreads - 1) / (4 * kPrepThreads) : 0;
    const int grid = a.B * a.tiles_x + nd2t;
    return launch_k(prep_kernel, dim3(grid), dim3(kPrepThreads), 0, s, false, a);
}

}  // namespace dspark
