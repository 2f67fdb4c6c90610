// Host side of the C ABI: argument checks, workspace layout, the launch sequence.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "dspark_internal.cuh"

namespace dspark {

size_t stream_stats_smem_bytes();

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

constexpr int kMaxGrid = 1024;           // streaming CTAs on any device (an SM count bound)

// The draft layout of a call (dense unless params->extras says otherwise).
struct QOpts {
    int layout;          // QLayout
    int Lq;              // entries of one draft row
};

QOpts q_opts(const dspark_params_t* p) {
    const dspark_extras_t* x = p->extras;
    if (!x || x->q_layout == DSPARK_Q_DENSE) return QOpts{kQDense, p->V};
    return QOpts{x->q_layout == DSPARK_Q_SPARSE ? kQSparse : kQReduced, x->q_row_len};
}

struct Layout {
    int tile_x, tiles_x, tile_q, tiles_q, bm_words, xslots, qslots, nseg_x, nseg_q, lp_chunks, Lq;
    long long seg_max;
    size_t off_plan, off_req_n, off_fin_list, off_units, off_ts_x, off_ts_q, off_cand_x, off_cand_q;
    size_t off_pen_hdr, off_pen_bm, off_pen_ent, off_draft_base, off_xout, off_kept, off_qout, off_req;
    size_t off_lp_part, off_t2d, off_lp_cand;
    bool lp_cand_alias;
    size_t zero_bytes;   // the call record cleared by every call: plan, logprob row counters, list count
    size_t total;
};

bool shapes_ok(const dspark_params_t* p) {
    if (!p) return false;
    if (p->B < 1 || p->B > kMaxB) return false;
    if (p->K_max < 0 || p->K_max > DSPARK_MAX_K) return false;
    if (p->V < 1 || p->V > DSPARK_MAX_V) return false;
    if (p->logits_dtype != DSPARK_BF16 && p->logits_dtype != DSPARK_FP32) return false;
    if (p->n_top_logprobs < 0 || p->n_top_logprobs > DSPARK_MAX_TOP_LOGPROBS) return false;
    if (const dspark_extras_t* x = p->extras) {
        if (x->logprob_mode != DSPARK_LOGPROBS_RAW && x->logprob_mode != DSPARK_LOGPROBS_PENALISED) return false;
        if (x->q_layout == DSPARK_Q_SPARSE) {
            if (x->q_row_len < 1 || x->q_row_len > DSPARK_MAX_SPARSE_M) return false;
        } else if (x->q_layout == DSPARK_Q_REDUCED) {
            if (x->q_row_len < 1 || x->q_row_len > p->V) return false;
        } else if (x->q_layout != DSPARK_Q_DENSE) {
            return false;
        }
    }
    return true;
}

Layout make_layout(const dspark_params_t* p) {
    Layout L{};
    const long long B = p->B, Km = p->K_max, V = p->V;
    const int sx = p->logits_dtype == DSPARK_BF16 ? 2 : 4;
    L.tile_x = sx == 2 ? kTileBf16 : kTileF32;
    L.tile_q = kTileF32;
    L.tiles_x = static_cast<int>((V + L.tile_x - 1) / L.tile_x);
    const QOpts qo = q_opts(p);
    L.Lq = qo.Lq;
    L.tiles_q = static_cast<int>((static_cast<long long>(L.Lq) + L.tile_q - 1) / L.tile_q);
    L.bm_words = ((L.tile_x + 31) / 32 + 3) / 4 * 4;
    L.xslots = static_cast<int>(B * (Km + 1));
    L.qslots = static_cast<int>(B * Km);
    L.nseg_x = (L.tiles_x + kSegTiles - 1) / kSegTiles;
    L.nseg_q = (L.tiles_q + kSegTiles - 1) / kSegTiles;
    // the logprob pass: R listed rows of S chunks, R * S <= its grid when S > 1, else R <= xslots
    L.lp_chunks = L.xslots > kLpMaxGrid ? L.xslots : kLpMaxGrid;
    const size_t xt = static_cast<size_t>(L.xslots) * L.nseg_x;
    const size_t qt = static_cast<size_t>(L.qslots) * L.nseg_q;
    const size_t pt = static_cast<size_t>(B) * L.tiles_x;
    L.seg_max = static_cast<long long>(xt + qt);
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
    // call record: Plan, then lp_done [xslots], then lp_list [1 + xslots] (its count cleared too)
    L.zero_bytes = sizeof(Plan) + static_cast<size_t>(L.xslots + 1) * sizeof(int);
    L.off_plan = take(L.zero_bytes + static_cast<size_t>(L.xslots) * sizeof(int));
    L.off_req_n = take(static_cast<size_t>(2 * B) * sizeof(int));
    L.off_fin_list = take(static_cast<size_t>(1 + L.xslots + L.qslots) * sizeof(int));
    // segment streams: grid x groups x ceil(S / (groups*grid)) entries <= S + groups*grid
    L.off_units = take((xt + qt + static_cast<size_t>(kGroups) * kMaxGrid) * sizeof(UnitDesc));
    L.off_ts_x = take(xt * sizeof(TileStats));
    L.off_ts_q = take(qt * sizeof(TileStats));
    L.off_cand_x = take(xt * kCandPenGlobal * sizeof(Cand));
    L.off_cand_q = take(qt * kCandPenGlobal * sizeof(Cand));
    L.off_pen_hdr = take(pt * sizeof(PenHdr));
    L.off_pen_bm = take(pt * L.bm_words * sizeof(unsigned));
    L.off_pen_ent = take(pt * kPenCap * sizeof(PenEntry));
    L.off_draft_base = take(static_cast<size_t>(B * Km) * sizeof(int) + 4);
    L.off_xout = take(static_cast<size_t>(L.xslots) * sizeof(XRowOut));
    L.off_kept = take(static_cast<size_t>(L.xslots) * kKeptCap * sizeof(KeptEntry));
    L.off_qout = take(static_cast<size_t>(L.qslots) * sizeof(QRowOut) + 16);
    L.off_req = take(static_cast<size_t>(B) * sizeof(ReqOut));
    L.off_lp_part = take(static_cast<size_t>(L.lp_chunks) * sizeof(LpPartial));
    L.off_t2d = take(qo.layout == kQReduced ? static_cast<size_t>(V) * sizeof(int) : 0);
    // the logprob pass's chunk candidates (R * S <= its grid and <= xslots * kLpMaxChunks chunks)
    // live in the streaming pass's target candidate lists, dead by then, when those are large
    // enough, else in a region of their own
    const size_t lp_cand_bytes = static_cast<size_t>(std::min<long long>(kLpMaxGrid, static_cast<long long>(L.xslots) *
                                                                                      kLpMaxChunks)) *
                                 kLpCandPerChunk * sizeof(unsigned long long);
    L.lp_cand_alias = xt * kCandPenGlobal * sizeof(Cand) >= lp_cand_bytes;
    L.off_lp_cand = L.lp_cand_alias ? L.off_cand_x : take(lp_cand_bytes);
    L.total = o;
    return L;
}

template <typename T>
T* at(void* base, size_t off) { return reinterpret_cast<T*>(static_cast<unsigned char*>(base) + off); }

dspark_status_t run(const void* logits, const float* q, const int32_t* draft_ids, const dspark_counts_t* counts,
                    const dspark_params_t* p, const float* uniforms, int32_t* out_accept_len, int32_t* out_tokens,
                    float* out_logprobs, int32_t* out_top_ids, float* out_top_logprobs) {
    if (!shapes_ok(p)) return DSPARK_ERR_INVALID_ARG;
    if (!logits || !uniforms || !out_accept_len || !out_tokens || !p->rows || !p->row_status)
        return DSPARK_ERR_INVALID_ARG;
    if (p->K_max > 0 && !draft_ids) return DSPARK_ERR_INVALID_ARG;
    if (p->want_logprobs && !out_logprobs) return DSPARK_ERR_INVALID_ARG;
    if (p->n_top_logprobs > 0 && (!out_top_ids || !out_top_logprobs)) return DSPARK_ERR_INVALID_ARG;
    const int sx = p->logits_dtype == DSPARK_BF16 ? 2 : 4;
    if (reinterpret_cast<uintptr_t>(logits) % sx || (q && reinterpret_cast<uintptr_t>(q) % 4))
        return DSPARK_ERR_INVALID_ARG;
    const bool has_hist = counts && counts->row_offsets;
    if (has_hist && (!counts->token_ids || !counts->counts)) return DSPARK_ERR_INVALID_ARG;
    const dspark_extras_t* ex = p->extras;
    const QOpts qo = q_opts(p);
    if (qo.layout == kQSparse && q && (!ex->q_ids || reinterpret_cast<uintptr_t>(ex->q_ids) % 4))
        return DSPARK_ERR_INVALID_ARG;
    if (qo.layout == kQReduced && q && !ex->d2t) return DSPARK_ERR_INVALID_ARG;
    const Layout L = make_layout(p);
    if (!p->workspace || p->workspace_bytes < L.total) return DSPARK_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(p->workspace) % kAlign) return DSPARK_ERR_WORKSPACE;

    cudaStream_t s = static_cast<cudaStream_t>(p->stream);
    void* ws = p->workspace;
    Args a{};
    a.B = p->B; a.Km = p->K_max; a.V = p->V; a.sx = sx; a.xdtype = p->logits_dtype;
    a.tile_x = L.tile_x; a.tiles_x = L.tiles_x; a.tile_q = L.tile_q; a.tiles_q = L.tiles_q; a.bm_words = L.bm_words;
    a.nseg_x = L.nseg_x; a.nseg_q = L.nseg_q; a.lp_chunks = L.lp_chunks;
    a.Lq = L.Lq; a.q_layout = qo.layout;
    a.lp_pen = (ex && ex->logprob_mode == DSPARK_LOGPROBS_PENALISED) ? 1 : 0;
    a.q_ids = ex ? ex->q_ids : nullptr;
    a.d2t = ex ? ex->d2t : nullptr;
    a.eos = ex ? ex->eos_ids : nullptr;
    a.out_stopped = ex ? ex->out_stopped : nullptr;
    a.pos_counts = (ex && p->K_max > 0) ? ex->pos_counts : nullptr;
    a.n_top = p->n_top_logprobs; a.want_lp = p->want_logprobs ? 1 : 0;
    a.xslots = L.xslots; a.qslots = L.qslots;
    a.x = logits; a.q = q; a.d = draft_ids; a.rows = p->rows;
    a.h_off = has_hist ? counts->row_offsets : nullptr;
    a.h_ids = has_hist ? counts->token_ids : nullptr;
    a.h_cnt = has_hist ? counts->counts : nullptr;
    a.u = uniforms;
    a.out_accept = out_accept_len; a.out_tokens = out_tokens; a.out_lp = out_logprobs;
    a.out_top_ids = out_top_ids; a.out_top_lp = out_top_logprobs; a.row_status = p->row_status;
    a.plan = at<Plan>(ws, L.off_plan);
    a.req_n = at<int>(ws, L.off_req_n);
    a.fin_list = at<int>(ws, L.off_fin_list);
    a.units = at<UnitDesc>(ws, L.off_units);
    a.ts_x = at<TileStats>(ws, L.off_ts_x);
    a.ts_q = at<TileStats>(ws, L.off_ts_q);
    a.cand_x = at<Cand>(ws, L.off_cand_x);
    a.cand_q = at<Cand>(ws, L.off_cand_q);
    a.pen_hdr = at<PenHdr>(ws, L.off_pen_hdr);
    a.pen_bm = at<unsigned>(ws, L.off_pen_bm);
    a.pen_ent = at<PenEntry>(ws, L.off_pen_ent);
    a.draft_base = at<int>(ws, L.off_draft_base);
    a.xout = at<XRowOut>(ws, L.off_xout);
    a.kept = at<KeptEntry>(ws, L.off_kept);
    a.qout = at<QRowOut>(ws, L.off_qout);
    a.req = at<ReqOut>(ws, L.off_req);
    a.lp_done = reinterpret_cast<int*>(a.plan + 1);
    a.lp_list = a.lp_done + L.xslots;
    a.lp_part = at<LpPartial>(ws, L.off_lp_part);
    a.t2d = qo.layout == kQReduced ? at<int>(ws, L.off_t2d) : nullptr;
    a.lp_cand = at<unsigned long long>(ws, L.off_lp_cand);

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    sms = sms < 1 ? 1 : (sms > kMaxGrid ? kMaxGrid : sms);
    a.grid_ss = sms;
    a.max_seg = static_cast<int>((L.seg_max + 2LL * sms - 1) / (2LL * sms));

    if (cudaMemsetAsync(p->row_status, 0, sizeof(int32_t) * p->B, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaMemsetAsync(a.plan, 0, L.zero_bytes, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (a.t2d && cudaMemsetAsync(a.t2d, 0xFF, sizeof(int) * static_cast<size_t>(p->V), s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (launch_prep(a, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    cudaEvent_t ev0 = static_cast<cudaEvent_t>(p->stage_events[0]);
    cudaEvent_t ev1 = static_cast<cudaEvent_t>(p->stage_events[1]);
    if (ev0 && cudaEventRecord(ev0, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    // kernels after prep are launched as programmatic dependents of their predecessor, except
    // across the optional stage events (an event between two kernels must see them apart)
    if (launch_stream_stats(a, s, sms, ev0 == nullptr) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (ev1 && cudaEventRecord(ev1, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (launch_row_finalize_warp(a, s, ev1 == nullptr) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (launch_row_finalize(a, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (launch_accept(a, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    if ((a.want_lp || a.n_top > 0) && launch_logprobs(a, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    return DSPARK_OK;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

// Scratch of dspark_verify_sample_static: a fixed device array (one instance per device).
static __device__ __align__(256) unsigned char g_static_workspace[DSPARK_STATIC_WORKSPACE_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};   // cached device address of g_static_workspace, per device
}  // namespace

extern "C" {

size_t dspark_workspace_bytes(const dspark_params_t* params) {
    if (!shapes_ok(params)) return 0;
    return make_layout(params).total;
}

dspark_status_t dspark_verify_sample(const void* logits, const float* q, const int32_t* draft_ids,
                                     const dspark_counts_t* counts, const dspark_params_t* params,
                                     const float* uniforms, int32_t* out_accept_len, int32_t* out_tokens,
                                     float* out_logprobs, int32_t* out_top_ids, float* out_top_logprobs) {
    return run(logits, q, draft_ids, counts, params, uniforms, out_accept_len, out_tokens, out_logprobs,
               out_top_ids, out_top_logprobs);
}

namespace {
struct HostStage {
    size_t x, q, d, rows, hoff, hids, hcnt, u, acc, tok, lp, tid, tlp, st;
    size_t qids, d2t, eos, stopped, counts, total;
};
HostStage host_stage(const dspark_params_t* p, int64_t nnz, size_t base) {
    HostStage h{};
    const size_t B = p->B, Km = p->K_max, V = p->V, W = Km + 1, n = p->n_top_logprobs;
    const size_t sx = p->logits_dtype == DSPARK_BF16 ? 2 : 4;
    size_t o = base;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
    const QOpts qo = q_opts(p);
    const size_t Lq = static_cast<size_t>(qo.Lq);
    h.x = take(B * W * V * sx);
    h.q = take(B * Km * Lq * 4);
    h.d = take(B * Km * 4 + 4);
    h.rows = take(B * sizeof(dspark_row_params_t));
    h.hoff = take((B + 1) * 4);
    h.hids = take(static_cast<size_t>(nnz > 0 ? nnz : 1) * 4);
    h.hcnt = take(static_cast<size_t>(nnz > 0 ? nnz : 1) * 4);
    h.u = take(B * W * 2 * 4);
    h.acc = take(B * 4);
    h.tok = take(B * W * 4);
    h.lp = take(B * W * 4);
    h.tid = take(B * W * n * 4 + 4);
    h.tlp = take(B * W * n * 4 + 4);
    h.st = take(B * 4);
    h.qids = take(qo.layout == kQSparse ? B * Km * Lq * 4 : 0);
    h.d2t = take(qo.layout == kQReduced ? Lq * 4 : 0);
    h.eos = take(B * 4);
    h.stopped = take(B * 4);
    h.counts = take(2 * Km * 8 + 8);
    h.total = o;
    return h;
}
}  // namespace

size_t dspark_host_workspace_bytes(const dspark_params_t* params, int64_t counts_nnz) {
    if (!shapes_ok(params) || counts_nnz < 0) return 0;
    const size_t dev = make_layout(params).total;
    return host_stage(params, counts_nnz, dev).total;
}

dspark_status_t dspark_verify_sample_host(const void* logits, const float* q, const int32_t* draft_ids,
                                          const dspark_counts_t* counts, const dspark_params_t* params,
                                          const float* uniforms, int32_t* out_accept_len, int32_t* out_tokens,
                                          float* out_logprobs, int32_t* out_top_ids, float* out_top_logprobs) {
    if (!shapes_ok(params) || !logits || !uniforms || !params->rows || !params->row_status || !out_accept_len ||
        !out_tokens)
        return DSPARK_ERR_INVALID_ARG;
    if (params->K_max > 0 && !draft_ids) return DSPARK_ERR_INVALID_ARG;
    const bool has_hist = counts && counts->row_offsets;
    const int64_t nnz = has_hist ? counts->row_offsets[params->B] : 0;
    if (nnz < 0) return DSPARK_ERR_INVALID_ARG;
    const size_t dev = make_layout(params).total;
    const HostStage h = host_stage(params, nnz, dev);
    if (!params->workspace || params->workspace_bytes < h.total) return DSPARK_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(params->workspace) % kAlign) return DSPARK_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(params->stream);
    unsigned char* ws = static_cast<unsigned char*>(params->workspace);
    const size_t B = params->B, Km = params->K_max, V = params->V, W = Km + 1, n = params->n_top_logprobs;
    const size_t sx = params->logits_dtype == DSPARK_BF16 ? 2 : 4;
    auto h2d = [&](size_t off, const void* src, size_t bytes) {
        return bytes == 0 || cudaMemcpyAsync(ws + off, src, bytes, cudaMemcpyHostToDevice, s) == cudaSuccess;
    };
    auto d2h = [&](void* dst, size_t off, size_t bytes) {
        return bytes == 0 || cudaMemcpyAsync(dst, ws + off, bytes, cudaMemcpyDeviceToHost, s) == cudaSuccess;
    };
    const dspark_extras_t* ex = params->extras;
    const QOpts qo = q_opts(params);
    const size_t Lq = static_cast<size_t>(qo.Lq);
    if (qo.layout == kQSparse && q && !ex->q_ids) return DSPARK_ERR_INVALID_ARG;
    if (qo.layout == kQReduced && q && !ex->d2t) return DSPARK_ERR_INVALID_ARG;
    bool ok = h2d(h.x, logits, B * W * V * sx);
    if (q) ok = ok && h2d(h.q, q, B * Km * Lq * 4);
    if (q && qo.layout == kQSparse) ok = ok && h2d(h.qids, ex->q_ids, B * Km * Lq * 4);
    if (q && qo.layout == kQReduced) ok = ok && h2d(h.d2t, ex->d2t, Lq * 4);
    if (ex && ex->eos_ids) ok = ok && h2d(h.eos, ex->eos_ids, B * 4);
    if (ex && ex->pos_counts && Km) ok = ok && h2d(h.counts, ex->pos_counts, 2 * Km * 8);
    if (Km) ok = ok && h2d(h.d, draft_ids, B * Km * 4);
    ok = ok && h2d(h.rows, params->rows, B * sizeof(dspark_row_params_t));
    if (has_hist) {
        ok = ok && h2d(h.hoff, counts->row_offsets, (B + 1) * 4);
        ok = ok && h2d(h.hids, counts->token_ids, static_cast<size_t>(nnz) * 4);
        ok = ok && h2d(h.hcnt, counts->counts, static_cast<size_t>(nnz) * 4);
    }
    ok = ok && h2d(h.u, uniforms, B * W * 2 * 4);
    // on any failure after the first copy was enqueued, wait for the stream before returning:
    // the caller may reuse its host buffers as soon as the call returns
    auto fail = [&](dspark_status_t e) { cudaStreamSynchronize(s); return e; };
    if (!ok) return fail(DSPARK_ERR_CUDA);
    dspark_counts_t dc{reinterpret_cast<const int32_t*>(ws + h.hoff), reinterpret_cast<const int32_t*>(ws + h.hids),
                       reinterpret_cast<const int32_t*>(ws + h.hcnt)};
    dspark_params_t dp = *params;
    dp.rows = reinterpret_cast<const dspark_row_params_t*>(ws + h.rows);
    dp.row_status = reinterpret_cast<int32_t*>(ws + h.st);
    dp.workspace_bytes = dev;
    dspark_extras_t dx{};
    if (ex) {
        dx = *ex;
        dx.q_ids = qo.layout == kQSparse ? reinterpret_cast<const int32_t*>(ws + h.qids) : nullptr;
        dx.d2t = qo.layout == kQReduced ? reinterpret_cast<const int32_t*>(ws + h.d2t) : nullptr;
        dx.eos_ids = ex->eos_ids ? reinterpret_cast<const int32_t*>(ws + h.eos) : nullptr;
        dx.out_stopped = ex->out_stopped ? reinterpret_cast<int32_t*>(ws + h.stopped) : nullptr;
        dx.pos_counts = ex->pos_counts ? reinterpret_cast<unsigned long long*>(ws + h.counts) : nullptr;
        dp.extras = &dx;
    }
    dspark_status_t st = run(ws + h.x, q ? reinterpret_cast<const float*>(ws + h.q) : nullptr,
                             Km ? reinterpret_cast<const int32_t*>(ws + h.d) : nullptr, has_hist ? &dc : nullptr, &dp,
                             reinterpret_cast<const float*>(ws + h.u), reinterpret_cast<int32_t*>(ws + h.acc),
                             reinterpret_cast<int32_t*>(ws + h.tok), out_logprobs ? reinterpret_cast<float*>(ws + h.lp) : nullptr,
                             n ? reinterpret_cast<int32_t*>(ws + h.tid) : nullptr,
                             n ? reinterpret_cast<float*>(ws + h.tlp) : nullptr);
    if (st != DSPARK_OK) return fail(st);
    ok = d2h(out_accept_len, h.acc, B * 4) && d2h(out_tokens, h.tok, B * W * 4) && d2h(params->row_status, h.st, B * 4);
    if (out_logprobs) ok = ok && d2h(out_logprobs, h.lp, B * W * 4);
    if (n && out_top_ids) ok = ok && d2h(out_top_ids, h.tid, B * W * n * 4);
    if (n && out_top_logprobs) ok = ok && d2h(out_top_logprobs, h.tlp, B * W * n * 4);
    if (ex && ex->out_stopped) ok = ok && d2h(ex->out_stopped, h.stopped, B * 4);
    if (ex && ex->pos_counts && Km) ok = ok && d2h(ex->pos_counts, h.counts, 2 * Km * 8);
    if (!ok) return fail(DSPARK_ERR_CUDA);
    if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
    return DSPARK_OK;
}

dspark_status_t dspark_verify_sample_static(const void* logits, const float* q, const int32_t* draft_ids,
                                            const dspark_counts_t* counts, const dspark_params_t* params,
                                            const float* uniforms, int32_t* out_accept_len, int32_t* out_tokens,
                                            float* out_logprobs, int32_t* out_top_ids, float* out_top_logprobs) {
    if (!shapes_ok(params)) return DSPARK_ERR_INVALID_ARG;
    if (make_layout(params).total > DSPARK_STATIC_WORKSPACE_BYTES) return DSPARK_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mu);
        const bool cached = dev >= 0 && dev < kMaxDevices;
        if (cached) ws = g_static_ptr[dev];
        if (!ws) {
            if (cudaGetSymbolAddress(&ws, g_static_workspace) != cudaSuccess || !ws) return DSPARK_ERR_CUDA;
            if (cached) g_static_ptr[dev] = ws;
        }
    }
    dspark_params_t p = *params;
    p.workspace = ws;
    p.workspace_bytes = DSPARK_STATIC_WORKSPACE_BYTES;
    return run(logits, q, draft_ids, counts, &p, uniforms, out_accept_len, out_tokens, out_logprobs, out_top_ids,
               out_top_logprobs);
}

const char* dspark_status_string(dspark_status_t status) {
    switch (status) {
        case DSPARK_OK: return "ok";
        case DSPARK_ERR_INVALID_ARG: return "invalid argument";
        case DSPARK_ERR_UNSUPPORTED: return "unsupported shape or option";
        case DSPARK_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case DSPARK_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

int32_t dspark_launches_per_call(void) { return 6; }

}  // extern "C"
