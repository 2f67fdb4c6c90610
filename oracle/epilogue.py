"""Oracle for the batched speculative verify-and-sample epilogue (float64, CPU, numpy).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  It shares no code with the
CUDA path and imports nothing from the product package; the only module both sides
use is ``workloads`` (seeded input synthesis, no epilogue arithmetic).

What is computed, and where the pages say so (mlx-dspark pages):
  * presence / frequency penalties on the TARGET logits, each verify position counted
    with the base completion counts plus its own draft prefix
    (mlx-dspark Changelog, [0.2.0] Added, "presence_penalty / frequency_penalty";
    v0.2.0 release notes, Highlights);
  * temperature, then top-k and top-p truncation of both target and draft
    (Changelog, [0.1.0] Added, "Lossless top-p / top-k sampling"; v0.1.0 release notes,
    Highlights);
  * the top-k threshold and nucleus cutoff give the same truncated distribution as a
    full vocabulary sort (Changelog, [0.20.2] Changed, grouped sorts);
  * greedy accept of the longest prefix where the target argmax equals the draft
    (Changelog, [0.2.0] Changed, "One device sync per speculative round": cumprod of
    positionwise matches);
  * at T>0 accept draft i with probability min(1, p/q), on the first rejection resample
    from the residual, so the output is an exact target sample (v0.0.2 release notes,
    Highlights, "Lossless temperature speculative sampling");
  * raw target log-softmax of each committed token plus the top candidates
    (Changelog, [0.2.0] Added, "logprobs / top_logprobs").

Readings taken where the pages are silent (each listed in the design notes):
  * penalised logits are formed in float32 with the operation order
    x' = fl(x - fl(fl(f*c) + p)) for c > 0 (x' = x for c = 0), on both sides, so that the
    argmax and the top-k threshold are decided on identical values;
  * the draft input q holds probabilities at T=1; the draft distribution at temperature
    T is q^(1/T) normalised, then truncated with the request's top_k / top_p;
  * top-k keeps every token whose value ties the k-th largest; top-p acts on the
    renormalised top-k distribution and keeps token t iff the mass strictly above its
    value is < top_p (crossing token and its ties kept);
  * full acceptance draws a bonus token from the target at position K;
  * the residual / bonus draw is an inverse CDF over ascending token ids, taking the
    smallest t with cumulative mass > u * total;
  * Q'(d) = 0 with P'(d) > 0 accepts; both zero rejects; an all-zero residual draws
    from P';
  * logprobs are the raw (unpenalised, untempered, untruncated) log-softmax.
Every discrete decision that floating point takes (nucleus boundary, accept test,
inverse-CDF boundary, empty residual) records its margin; a request whose smallest
margin is below ``MARGIN_EPS`` is "fragile" and is exempt from bit-exact comparison.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MARGIN_EPS = 1e-6

# per-request status bits (mirrored by the library's row_status word)
ROW_OK = 0
ROW_BAD_PARAMS = 1
ROW_BAD_DRAFT = 2
ROW_NONFINITE = 4
ROW_BAD_HISTORY = 8


# ----------------------------------------------------------------------------- penalties
def count_vector(V, hist_ids, hist_counts, prefix):
    """c(t) = base completion count of t + occurrences of t in the draft prefix.

    mlx-dspark Changelog, [0.2.0] Added (penalties): each verify position is penalised
    by the base completion counts plus its own draft prefix."""
    c = np.zeros(V, np.int64)
    np.add.at(c, np.asarray(hist_ids, np.int64), np.asarray(hist_counts, np.int64))
    for t in prefix:
        c[int(t)] += 1
    return c


def penalised_logits(x32, counts, presence, frequency):
    """OpenAI presence/frequency penalty on target logits, float32 operation order fixed:
    x' = fl(x - fl(fl(f*c) + p)) where c > 0, else x' = x."""
    x32 = np.asarray(x32, np.float32)
    f = np.float32(frequency)
    p = np.float32(presence)
    cf = counts.astype(np.float32)
    pen = (f * cf).astype(np.float32)
    pen = (pen + p).astype(np.float32)
    return np.where(counts > 0, (x32 - pen).astype(np.float32), x32).astype(np.float32)


# ----------------------------------------------------------------------------- truncation
def order_desc(values):
    """Token ids sorted by value descending, id ascending (a full stable sort)."""
    v = np.asarray(values, np.float64)
    return np.lexsort((np.arange(v.size), -v))


def truncate_full_sort(values, weights, top_k, top_p):
    """Top-k then top-p truncation by one full sort of the vocabulary.

    values: the ordering key (penalised logit or draft probability); weights: the
    unnormalised probabilities, monotone non-decreasing in ``values``.
    Returns (keep mask, nucleus margin).  mlx-dspark Changelog, [0.1.0] Added
    (lossless top-p / top-k on draft and target)."""
    V = values.size
    order = order_desc(values)
    keep = np.ones(V, bool)
    if 0 < top_k < V:
        tau_k = values[order[top_k - 1]]
        keep = values >= tau_k
    margin = np.inf
    if top_p < 1.0:
        idx = order[keep[order]]                  # kept ids, value desc / id asc
        vs = values[idx]
        w = weights[idx].astype(np.float64)
        pk = w / w.sum()
        excl = np.concatenate(([0.0], np.cumsum(pk)[:-1]))
        # mass strictly above each token's value = exclusive prefix at its tie group's start
        start = np.ones(vs.size, bool)
        start[1:] = vs[1:] != vs[:-1]
        first = np.maximum.accumulate(np.where(start, np.arange(vs.size), 0))
        above = excl[first]
        kept_sorted = above < top_p
        keep = np.zeros(V, bool)
        keep[idx[kept_sorted]] = True
        # margins: the last kept group's mass-above vs top_p, and the first dropped group's
        g_above = above[start]
        g_kept = g_above < top_p
        last = float(g_above[g_kept].max())
        # the top group's mass-above is exactly 0 on any machine: that decision has no margin
        margin = float(top_p - last) if last > 0.0 else np.inf
        if (~g_kept).any():
            margin = min(margin, float(g_above[~g_kept].min() - top_p))
    return keep, margin


def truncate_grouped(values, weights, top_k, top_p, group=1024):
    """The same truncation from small per-group sorts instead of one full sort.

    mlx-dspark Changelog, [0.20.2] Changed: the top-k threshold and the nucleus cutoff come
    from small grouped sorts and the truncated distribution is bit-identical.  Each group
    of ``group`` consecutive ids is sorted on its own; the k-th largest value of the whole
    row is the k-th largest of the merged per-group leaders (every member of the global
    top-k is within its group's top-k), and the nucleus walks a lazy merge of the sorted
    groups' heads."""
    V = values.size
    vals = np.asarray(values)
    groups = [np.arange(s, min(s + group, V)) for s in range(0, V, group)]
    sorted_groups = []
    for g in groups:
        o = g[np.lexsort((g, -vals[g].astype(np.float64)))]
        sorted_groups.append(o)
    keep = np.ones(V, bool)
    tau_k = -np.inf
    if 0 < top_k < V:
        leaders = np.concatenate([o[:top_k] for o in sorted_groups])
        lv = np.sort(vals[leaders].astype(np.float64))[::-1]
        tau_k = lv[top_k - 1]
        keep = vals >= tau_k
    margin = np.inf
    if top_p < 1.0:
        # survivors of each group, still sorted; lazy k-way merge by (value desc, id asc)
        heads = [o[vals[o] >= tau_k] for o in sorted_groups]
        Z = float(sum(weights[h].astype(np.float64).sum() for h in heads))
        pos = [0] * len(heads)
        keep = np.zeros(V, bool)
        mass_above = 0.0
        last_kept = None
        dropped_first = None
        while True:
            best = None
            for gi, h in enumerate(heads):
                if pos[gi] < h.size:
                    t = h[pos[gi]]
                    if best is None or (vals[t] > vals[best]) or (vals[t] == vals[best] and t < best):
                        best = t
                        bg = gi
            if best is None:
                break
            v = vals[best]
            # take the whole tie group with value v across all groups
            grp = []
            for gi, h in enumerate(heads):
                while pos[gi] < h.size and vals[h[pos[gi]]] == v:
                    grp.append(h[pos[gi]])
                    pos[gi] += 1
            if mass_above < top_p:
                keep[np.array(grp)] = True
                last_kept = mass_above
                mass_above += float(weights[np.array(grp)].astype(np.float64).sum()) / Z
            else:
                dropped_first = mass_above
                break
        margin = float(top_p - last_kept) if last_kept > 0.0 else np.inf
        if dropped_first is not None:
            margin = min(margin, float(dropped_first - top_p))
    return keep, margin


# ----------------------------------------------------------------------------- distributions
def target_probs(xp32, T, top_k, top_p, truncate=truncate_full_sort):
    """P' = truncate(softmax(x'/T)) renormalised.  v0.0.2 release notes, Highlights
    (temperature sampling); Changelog [0.1.0] Added (top-p / top-k on the target)."""
    s = np.asarray(xp32, np.float64)
    w = np.exp((s - s.max()) / float(T))
    keep, margin = truncate(np.asarray(xp32, np.float32), w, top_k, top_p)
    P = np.where(keep, w, 0.0)
    return P / P.sum(), margin


def draft_probs(q32, T, top_k, top_p, truncate=truncate_full_sort):
    """Q' = truncate(q^(1/T)) renormalised: the draft input holds T=1 probabilities and the
    request's temperature and truncation apply to it as to the target (Changelog [0.1.0]
    Added: truncation applied to both draft and target)."""
    q = np.asarray(q32, np.float64)
    w = q ** (1.0 / float(T))
    keep, margin = truncate(np.asarray(q32, np.float32), w, top_k, top_p)
    Q = np.where(keep, w, 0.0)
    Z = Q.sum()
    if not Z > 0:
        return None, margin
    return Q / Z, margin


# ----------------------------------------------------------------------------- accept / draw
def accept_probability(p, q):
    """min(1, p/q) (v0.0.2 release notes, Highlights); q = 0 accepts iff p > 0."""
    if q == 0.0:
        return 1.0 if p > 0.0 else 0.0
    return min(1.0, p / q)


def accept_test(p, q, u):
    """The accept decision for one draft with uniform u, and its margin."""
    if q == 0.0:
        return p > 0.0, np.inf
    ratio = p / q
    return bool(u < ratio), abs(u - ratio)


def residual(P, Q):
    """Unnormalised residual max(0, P - Q) resampled from on the first rejection."""
    return np.maximum(0.0, P - Q)


def inverse_cdf(w, u):
    """Smallest id t with sum_{s<=t} w_s > u * sum(w) (ascending ids); returns (t, margin).

    The margin is the distance, in mass units, from u*sum(w) to the nearer edge of t's
    cumulative interval."""
    C = np.cumsum(np.asarray(w, np.float64))
    total = C[-1]
    target = float(u) * total
    hits = np.nonzero(C > target)[0]
    if hits.size == 0:
        t = int(np.nonzero(w > 0)[0][-1])
        return t, 0.0
    t = int(hits[0])
    lo = C[t - 1] if t > 0 else 0.0
    return t, float(min(target - lo, C[t] - target))


# ----------------------------------------------------------------------------- logprobs
def raw_log_softmax(x32):
    """Log-softmax of the raw target logits in float64 (Changelog [0.2.0] Added, logprobs:
    raw target log-softmax of each committed token)."""
    x = np.asarray(x32, np.float64)
    m = x.max()
    return x - (m + np.log(np.exp(x - m).sum()))


def top_n(x32, n):
    """The n largest raw logits, value descending then id ascending."""
    return order_desc(np.asarray(x32, np.float32))[:n]


# ----------------------------------------------------------------------------- one request
@dataclass
class RequestResult:
    accept_len: int
    tokens: np.ndarray            # int32 [K_max+1], -1 past the emitted token
    logprobs: np.ndarray          # float64 [K_max+1], -inf past the emitted token
    top_ids: np.ndarray           # int32 [K_max+1, n]
    top_logprobs: np.ndarray      # float64 [K_max+1, n]
    status: int = ROW_OK
    min_margin: float = np.inf
    margins: list = field(default_factory=list)

    @property
    def fragile(self):
        return self.min_margin < MARGIN_EPS


def _validate(batch, b):
    r = batch.rows[b]
    T, k, p, K = float(r["temperature"]), int(r["top_k"]), float(r["top_p"]), int(r["num_drafts"])
    st = ROW_OK
    if not (np.isfinite(T) and T >= 0.0) or not (p > 0.0) or not np.isfinite(p) or k < 0 \
            or K < 0 or K > batch.K_max or not np.isfinite(r["presence_penalty"]) \
            or not np.isfinite(r["frequency_penalty"]):
        return ROW_BAD_PARAMS
    ids, cnt = batch.history(b)
    if ids.size and (ids.min() < 0 or ids.max() >= batch.V or np.any(np.diff(ids) <= 0) or cnt.min() <= 0):
        st |= ROW_BAD_HISTORY
    d = batch.draft_ids[b, :K]
    if d.size and (d.min() < 0 or d.max() >= batch.V):
        st |= ROW_BAD_DRAFT
    return st


def verify_request(batch, b, truncate=truncate_full_sort) -> RequestResult:
    """The whole epilogue for request b of a ``workloads`` batch."""
    V, Km = batch.V, batch.K_max
    n = batch.n_top_logprobs
    tokens = np.full(Km + 1, -1, np.int32)
    lps = np.full(Km + 1, -np.inf)
    tids = np.full((Km + 1, n), -1, np.int32)
    tlp = np.full((Km + 1, n), -np.inf)
    st = _validate(batch, b)
    if st != ROW_OK:
        return RequestResult(-1, tokens, lps, tids, tlp, status=st)
    r = batch.rows[b]
    T, k, p = float(r["temperature"]), int(r["top_k"]), float(r["top_p"])
    pres, freq, K = r["presence_penalty"], r["frequency_penalty"], int(r["num_drafts"])
    x = batch.x_f32(b)                        # [K_max+1, V] float32
    d = batch.draft_ids[b].astype(np.int64)
    u = batch.uniforms[b].astype(np.float64)
    hid, hc = batch.history(b)
    for j in range(K + 1):
        if not np.all(np.isfinite(x[j])):
            return RequestResult(-1, tokens, lps, tids, tlp, status=ROW_NONFINITE)
    if T > 0:
        for i in range(K):
            qi = batch.q[b, i]
            if not (np.all(np.isfinite(qi)) and qi.min() >= 0.0):
                return RequestResult(-1, tokens, lps, tids, tlp, status=ROW_NONFINITE)

    def xp(j):
        return penalised_logits(x[j], count_vector(V, hid, hc, d[:j]), pres, freq)

    margins = []
    if T == 0.0:
        # greedy: accept while the draft equals the penalised argmax (lowest id on ties)
        a = K
        for i in range(K):
            if d[i] != int(np.argmax(xp(i))):
                a = i
                break
        tok = int(np.argmax(xp(a)))
    else:
        a = K
        for i in range(K):
            P, mp = target_probs(xp(i), T, k, p, truncate)
            Q, mq = draft_probs(batch.q[b, i], T, k, p, truncate)
            if Q is None:
                return RequestResult(-1, tokens, lps, tids, tlp, status=ROW_NONFINITE)
            margins += [("nucleus_p", i, mp), ("nucleus_q", i, mq)]
            acc, m = accept_test(P[d[i]], Q[d[i]], u[i, 0])
            margins.append(("accept", i, m))
            if not acc:
                a = i
                break
        P, mp = target_probs(xp(a), T, k, p, truncate)
        margins.append(("nucleus_p", a, mp))
        if a < K:
            Q, mq = draft_probs(batch.q[b, a], T, k, p, truncate)
            margins.append(("nucleus_q", a, mq))
            w = residual(P, Q)
            tot = w.sum()
            margins.append(("residual_mass", a, float(tot)))
            if not tot > 0.0:
                w = P
        else:
            w = P
        tok, m = inverse_cdf(w, u[a, 1])
        margins.append(("draw", a, m))
    tokens[:a] = d[:a]
    tokens[a] = tok
    if batch.want_logprobs or n > 0:
        for j in range(a + 1):
            ls = raw_log_softmax(x[j])
            lps[j] = ls[tokens[j]]
            if n > 0:
                ids = top_n(x[j], n)
                tids[j] = ids
                tlp[j] = ls[ids]
    mm = min([m for (_, _, m) in margins], default=np.inf)
    return RequestResult(a, tokens, lps, tids, tlp, status=ROW_OK, min_margin=mm, margins=margins)


def verify_batch(batch, requests=None, truncate=truncate_full_sort):
    """Run ``verify_request`` over the given requests (default: all)."""
    reqs = range(batch.B) if requests is None else requests
    return {b: verify_request(batch, b, truncate) for b in reqs}
