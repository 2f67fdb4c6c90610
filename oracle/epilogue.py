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
  * logprobs are the raw (unpenalised, untempered, untruncated) log-softmax;
  * a target logit of -inf is a token of zero probability (a masked token); NaN or +inf, or a
    row with no finite logit, has no distribution and makes the request non-finite;
  * a draft given sparsely (lookup mode's one-hot proposal, or any m (id, probability)
    pairs) is the dense draft row with zeros elsewhere (Changelog [0.2.0] Added, "--mode
    lookup": one-hot-proposal speculative sampling); a draft over a reduced vocabulary is
    widened onto the target vocabulary, target id = draft id + d2t[draft id], before the
    accept test (Changelog [0.8.0] Added, reduced draft vocabularies);  the widened row then
    goes through the same temperature and truncation;
  * a request with an end-of-sequence token stops after the first accepted draft equal to
    it: the accepted length counts that draft and nothing is drawn after it (Changelog
    [0.2.0] Fixed, stop when an accepted draft contains eos mid-block);
  * per-position acceptance counts (Changelog [0.9.0] Added, per-position acceptance with
    honest denominators): position i is attempted when the request verified its draft i
    (every earlier draft accepted, no stop before it), accepted when that draft was accepted;
  * with logprob_mode "penalised", logprobs and top_logprobs are the log-softmax of the
    penalised logits x' instead of the raw ones (the alternative reading of "raw target
    log-softmax").

Near ties.  Every discrete decision that floating point takes records a ``Decision``: its
distance from the threshold, in the threshold's own unit, and the branch the other side
of the threshold leads to.
  * accept test: |u - P'/Q'| in uniform units;
  * residual / bonus draw: the distance of u from the nearer edge of the drawn token's
    interval [C(t-1)/C(V-1), C(t)/C(V-1)) of the normalised cumulative weights, in uniform
    units;
  * nucleus boundary: top_p minus the mass above the last kept tie group, and the mass
    above the first dropped group minus top_p, in probability units (the unit top_p is
    stated in);
  * empty residual: the residual mass.
A decision whose distance is below ``MARGIN_EPS`` is a near tie.  ``outcomes`` follows
both sides of every near-tie accept test and nucleus boundary, and a near-tie draw admits
every token whose interval reaches within ``MARGIN_EPS`` of u; a result is correct iff it
is one of these outcomes.  Decisions taken on identical float32 values on both sides
(penalised argmax, top-k threshold, top-n ids) have no margin.
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


def _nucleus_groups(g_above, top_p, flip):
    """Number of tie groups the nucleus keeps, and its two margins.

    g_above: mass strictly above each tie group (non-decreasing).  Kept groups are those
    with g_above < top_p, a prefix.  Margins: top_p minus the last kept group's mass above
    (none for the top group, whose mass above is exactly 0 on any machine) and the first
    dropped group's mass above minus top_p.  flip "drop_last" / "keep_next" takes the other
    side of one of those two boundaries."""
    nk = int(np.count_nonzero(g_above < top_p))
    last = float(g_above[nk - 1])
    m_last = float(top_p - last) if last > 0.0 else np.inf
    m_next = float(g_above[nk] - top_p) if nk < g_above.size else np.inf
    if flip == "drop_last" and nk > 1:
        nk -= 1
    elif flip == "keep_next" and nk < g_above.size:
        nk += 1
    return nk, (m_last, m_next)


def truncate_full_sort(values, weights, top_k, top_p, flip=None):
    """Top-k then top-p truncation by one full sort of the vocabulary.

    values: the ordering key (penalised logit or draft probability); weights: the
    unnormalised probabilities, monotone non-decreasing in ``values``.
    Returns (keep mask, (margin of the last kept group, margin of the first dropped
    group)).  mlx-dspark Changelog, [0.1.0] Added (lossless top-p / top-k on draft and
    target)."""
    V = values.size
    order = order_desc(values)
    keep = np.ones(V, bool)
    if 0 < top_k < V:
        tau_k = values[order[top_k - 1]]
        keep = values >= tau_k
    margins = (np.inf, np.inf)
    if top_p < 1.0:
        idx = order[keep[order]]                  # kept ids, value desc / id asc
        vs = values[idx]
        w = weights[idx].astype(np.float64)
        pk = w / w.sum()
        excl = np.concatenate(([0.0], np.cumsum(pk)[:-1]))
        # tie groups: the mass strictly above a group is the exclusive prefix at its start
        start = np.ones(vs.size, bool)
        start[1:] = vs[1:] != vs[:-1]
        starts = np.nonzero(start)[0]
        nk, margins = _nucleus_groups(excl[starts], top_p, flip)
        end = starts[nk] if nk < starts.size else vs.size
        keep = np.zeros(V, bool)
        keep[idx[:end]] = True
    return keep, margins


def truncate_grouped(values, weights, top_k, top_p, group=1024, flip=None):
    """The same truncation from small per-group sorts instead of one full sort.

    mlx-dspark Changelog, [0.20.2] Changed: the top-k threshold and the nucleus cutoff come
    from small grouped sorts and the truncated distribution is bit-identical.  Each group
    of ``group`` consecutive ids is sorted on its own; the k-th largest value of the whole
    row is the k-th largest of the merged per-group leaders (every member of the global
    top-k is within its group's top-k), and the nucleus walks a lazy merge of the sorted
    groups' heads, one tie group (across all groups) at a time."""
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
    margins = (np.inf, np.inf)
    if top_p < 1.0:
        heads = [o[vals[o] >= tau_k] for o in sorted_groups]
        Z = float(sum(weights[h].astype(np.float64).sum() for h in heads))
        pos = [0] * len(heads)
        ties, above = [], []            # tie groups in merge order, mass strictly above each
        mass_above = 0.0
        while True:
            best = None
            for h, p0 in zip(heads, pos):
                if p0 < h.size:
                    t = h[p0]
                    if best is None or (vals[t] > vals[best]) or (vals[t] == vals[best] and t < best):
                        best = t
            if best is None:
                break
            v = vals[best]
            grp = []
            for gi, h in enumerate(heads):
                while pos[gi] < h.size and vals[h[pos[gi]]] == v:
                    grp.append(h[pos[gi]])
                    pos[gi] += 1
            ties.append(np.array(grp))
            above.append(mass_above)
            if mass_above >= top_p:     # first dropped group found: nothing later can be kept
                break
            mass_above += float(weights[np.array(grp)].astype(np.float64).sum()) / Z
        nk, margins = _nucleus_groups(np.array(above), top_p, flip)
        keep = np.zeros(V, bool)
        for grp in ties[:nk]:
            keep[grp] = True
    return keep, margins


# ----------------------------------------------------------------------------- distributions
def target_probs(xp32, T, top_k, top_p, truncate=truncate_full_sort, flip=None):
    """P' = truncate(softmax(x'/T)) renormalised.  v0.0.2 release notes, Highlights
    (temperature sampling); Changelog [0.1.0] Added (top-p / top-k on the target)."""
    s = np.asarray(xp32, np.float64)
    w = np.exp((s - s.max()) / float(T))
    keep, margins = truncate(np.asarray(xp32, np.float32), w, top_k, top_p, flip=flip)
    P = np.where(keep, w, 0.0)
    return P / P.sum(), margins


def draft_probs(q32, T, top_k, top_p, truncate=truncate_full_sort, flip=None):
    """Q' = truncate(q^(1/T)) renormalised: the draft input holds T=1 probabilities and the
    request's temperature and truncation apply to it as to the target (Changelog [0.1.0]
    Added: truncation applied to both draft and target)."""
    q = np.asarray(q32, np.float64)
    w = q ** (1.0 / float(T))
    keep, margins = truncate(np.asarray(q32, np.float32), w, top_k, top_p, flip=flip)
    Q = np.where(keep, w, 0.0)
    Z = Q.sum()
    if not Z > 0:
        return None, margins
    return Q / Z, margins


# ----------------------------------------------------------------------------- accept / draw
def accept_probability(p, q):
    """min(1, p/q) (v0.0.2 release notes, Highlights); q = 0 accepts iff p > 0."""
    if q == 0.0:
        return 1.0 if p > 0.0 else 0.0
    return min(1.0, p / q)


def accept_test(p, q, u):
    """The accept decision for one draft with uniform u, and its margin |u - p/q|."""
    if q == 0.0:
        return p > 0.0, np.inf
    ratio = p / q
    return bool(u < ratio), abs(u - ratio)


def residual(P, Q):
    """Unnormalised residual max(0, P - Q) resampled from on the first rejection."""
    return np.maximum(0.0, P - Q)


def inverse_cdf(w, u):
    """Smallest id t with sum_{s<=t} w_s > u * sum(w) (ascending ids); returns (t, margin).

    The margin is the distance of u from the nearer edge of t's interval
    [C(t-1)/total, C(t)/total), in uniform units."""
    C = np.cumsum(np.asarray(w, np.float64))
    total = C[-1]
    target = float(u) * total
    hits = np.nonzero(C > target)[0]
    if hits.size == 0:
        t = int(np.nonzero(w > 0)[0][-1])
        return t, 0.0
    t = int(hits[0])
    lo = C[t - 1] if t > 0 else 0.0
    return t, float(min(target - lo, C[t] - target) / total)


def draw_admissible(w, u, eps=MARGIN_EPS):
    """Every id t with w_t > 0 whose interval [C(t-1)/total, C(t)/total) reaches within eps
    of u: the tokens an inverse-CDF draw may return when u is moved by at most eps."""
    w = np.asarray(w, np.float64)
    C = np.cumsum(w)
    total = C[-1]
    lo = np.concatenate(([0.0], C[:-1])) / total
    hi = C / total
    return np.nonzero((w > 0) & (lo < float(u) + eps) & (hi > float(u) - eps))[0].astype(np.int64)


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
class Decision:
    """One floating-point decision of a request: the test, its position, the distance of its
    operand from the threshold (in the threshold's unit) and the flip that takes the other
    side ("" for a draw, whose other sides are listed as admissible tokens)."""
    kind: str            # "nucleus_p", "nucleus_q", "accept", "residual_mass", "draw"
    pos: int
    margin: float
    alt: str = ""

    @property
    def fragile(self):
        return self.margin < MARGIN_EPS


@dataclass
class RequestResult:
    accept_len: int
    tokens: np.ndarray            # int32 [K_max+1], -1 past the emitted token
    logprobs: np.ndarray          # float64 [K_max+1], -inf past the emitted token
    top_ids: np.ndarray           # int32 [K_max+1, n]
    top_logprobs: np.ndarray      # float64 [K_max+1, n]
    status: int = ROW_OK
    decisions: list = field(default_factory=list)
    admissible: np.ndarray = None        # ids the emitted token may be (the drawn id first)
    admissible_logprobs: np.ndarray = None
    flips: dict = field(default_factory=dict)
    stopped: bool = False                # an accepted draft was the end-of-sequence token
    attempted: np.ndarray = None         # int [K_max]: drafts verified, by position
    accepted: np.ndarray = None          # int [K_max]: drafts accepted, by position

    @property
    def min_margin(self):
        return min((d.margin for d in self.decisions), default=np.inf)

    @property
    def fragile(self):
        return any(d.fragile for d in self.decisions)

    def near_ties(self):
        """Kinds of the near-tie decisions of this outcome."""
        return [d.kind for d in self.decisions if d.fragile]


def bad_logit_row(x32):
    """NaN or +inf anywhere, or no finite logit at all: the row defines no distribution.
    A logit of -inf is allowed: that token has probability zero."""
    x = np.asarray(x32, np.float32)
    return bool(np.isnan(x).any() or (x == np.inf).any() or not np.isfinite(x).any())


def widened_draft(batch, b, i):
    """Draft probabilities of request b at position i over the target vocabulary (float32):
    the dense row, or the sparse pairs / reduced-vocabulary row scattered onto V with zeros
    elsewhere."""
    if batch.q_layout == "dense":
        return np.asarray(batch.q[b, i], np.float32)
    out = np.zeros(batch.V, np.float32)
    if batch.q_layout == "sparse":
        out[np.asarray(batch.q_ids[b, i], np.int64)] = batch.q[b, i]
    else:
        dv = np.arange(batch.q.shape[-1], dtype=np.int64)
        out[dv + np.asarray(batch.d2t, np.int64)] = batch.q[b, i]
    return out


def draft_layout_ok(batch, b, K):
    """Sparse ids of request b in [0, V) and distinct per row; a d2t table mapping every draft
    id into [0, V) without collisions."""
    if batch.q_layout == "sparse":
        for i in range(K):
            ids = np.asarray(batch.q_ids[b, i], np.int64)
            if ids.min() < 0 or ids.max() >= batch.V or np.unique(ids).size != ids.size:
                return False
    elif batch.q_layout == "reduced":
        t = np.arange(batch.d2t.size, dtype=np.int64) + np.asarray(batch.d2t, np.int64)
        if t.min() < 0 or t.max() >= batch.V or np.unique(t).size != t.size:
            return False
    return True


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
    if T > 0 and K > 0 and not draft_layout_ok(batch, b, K):
        st |= ROW_BAD_DRAFT
    return st


def verify_request(batch, b, truncate=truncate_full_sort, flips=None) -> RequestResult:
    """The whole epilogue for request b of a ``workloads`` batch.

    flips: {(kind, position): alternative} takes the other side of those near-tie decisions
    (used by ``outcomes``); None follows every decision as float64 takes it."""
    flips = dict(flips or {})
    V, Km = batch.V, batch.K_max
    n = batch.n_top_logprobs
    tokens = np.full(Km + 1, -1, np.int32)
    lps = np.full(Km + 1, -np.inf)
    tids = np.full((Km + 1, n), -1, np.int32)
    tlp = np.full((Km + 1, n), -np.inf)
    st = _validate(batch, b)
    if st != ROW_OK:
        return RequestResult(-1, tokens, lps, tids, tlp, status=st, flips=flips)
    r = batch.rows[b]
    T, k, p = float(r["temperature"]), int(r["top_k"]), float(r["top_p"])
    pres, freq, K = r["presence_penalty"], r["frequency_penalty"], int(r["num_drafts"])
    x = batch.x_f32(b)                        # [K_max+1, V] float32
    d = batch.draft_ids[b].astype(np.int64)
    u = batch.uniforms[b].astype(np.float64)
    hid, hc = batch.history(b)
    for j in range(K + 1):
        if bad_logit_row(x[j]):
            return RequestResult(-1, tokens, lps, tids, tlp, status=ROW_NONFINITE, flips=flips)
    if T > 0:
        for i in range(K):
            qi = batch.q[b, i]
            if not (np.all(np.isfinite(qi)) and qi.min() >= 0.0):
                return RequestResult(-1, tokens, lps, tids, tlp, status=ROW_NONFINITE, flips=flips)
    qrows = {}

    def qrow(i):
        if i not in qrows:
            qrows[i] = widened_draft(batch, b, i)
        return qrows[i]

    def xp(j):
        return penalised_logits(x[j], count_vector(V, hid, hc, d[:j]), pres, freq)

    decisions = []
    cache = {}

    def dist(kind, j):
        """P'_j or Q'_j (memoised), recording its nucleus decisions once."""
        if (kind, j) not in cache:
            fl = flips.get((kind, j))
            if kind == "nucleus_p":
                D, (m_last, m_next) = target_probs(xp(j), T, k, p, truncate, flip=fl)
            else:
                D, (m_last, m_next) = draft_probs(qrow(j), T, k, p, truncate, flip=fl)
            decisions.append(Decision(kind, j, m_last, "drop_last"))
            decisions.append(Decision(kind, j, m_next, "keep_next"))
            cache[(kind, j)] = D
        return cache[(kind, j)]

    if T == 0.0:
        # greedy: accept while the draft equals the penalised argmax (lowest id on ties)
        a = K
        for i in range(K):
            if d[i] != int(np.argmax(xp(i))):
                a = i
                break
        tok = int(np.argmax(xp(a)))
        adm = np.array([tok], np.int64)
    else:
        a = K
        for i in range(K):
            P = dist("nucleus_p", i)
            Q = dist("nucleus_q", i)
            if Q is None:
                return RequestResult(-1, tokens, lps, tids, tlp, status=ROW_NONFINITE, flips=flips)
            acc, m = accept_test(P[d[i]], Q[d[i]], u[i, 0])
            decisions.append(Decision("accept", i, m, "flip"))
            if flips.get(("accept", i)) == "flip":
                acc = not acc
            if not acc:
                a = i
                break
        P = dist("nucleus_p", a)
        w = P
        tiny_residual = False
        if a < K:
            Q = dist("nucleus_q", a)
            w = residual(P, Q)
            tot = w.sum()
            decisions.append(Decision("residual_mass", a, float(tot)))
            # a near-empty residual: float32 rounding of P - Q may leave any id of P' standing
            tiny_residual = tot < MARGIN_EPS
            if not tot > 0.0:
                w = P
        tok, m = inverse_cdf(w, u[a, 1])
        decisions.append(Decision("draw", a, m))
        adm = draw_admissible(w, u[a, 1])
        if tiny_residual:
            adm = np.union1d(adm, np.nonzero(P > 0)[0])
        adm = np.concatenate(([tok], adm[adm != tok])).astype(np.int64)
    # per-position acceptance before any stop: drafts 0..a-1 accepted, draft a rejected (a < K)
    attempted = np.zeros(Km, np.int64)
    accepted = np.zeros(Km, np.int64)
    attempted[:min(a + 1, K)] = 1
    accepted[:a] = 1
    # an accepted draft equal to the end-of-sequence token ends the request's output there
    stopped = False
    eos = -1 if batch.eos_ids is None else int(batch.eos_ids[b])
    if eos >= 0:
        hit = np.nonzero(d[:a] == eos)[0]
        if hit.size:
            a = int(hit[0]) + 1
            stopped = True
            attempted[a:] = 0
            accepted[a:] = 0
            adm = np.array([-1], np.int64)
            # decisions past the stop shape nothing that is emitted
            decisions = [dc for dc in decisions if dc.pos < a and dc.kind not in ("draw", "residual_mass")]
    tokens[:a] = d[:a]
    if not stopped:
        tokens[a] = tok
    last = a if not stopped else a - 1                       # last emitted position
    adm_lp = None
    if batch.want_logprobs or n > 0:
        for j in range(last + 1):
            row = xp(j) if batch.logprob_mode == "penalised" else x[j]
            ls = raw_log_softmax(row)
            lps[j] = ls[tokens[j]]
            if j == a:
                adm_lp = ls[adm]
            if n > 0:
                ids = top_n(row, n)
                tids[j] = ids
                tlp[j] = ls[ids]
    return RequestResult(a, tokens, lps, tids, tlp, status=ROW_OK, decisions=decisions, admissible=adm,
                         admissible_logprobs=adm_lp, flips=flips, stopped=stopped, attempted=attempted,
                         accepted=accepted)


def outcomes(batch, b, truncate=truncate_full_sort, max_outcomes=16):
    """Every outcome request b may correctly have: the float64 one first, then, for each
    near-tie accept test or nucleus boundary, the outcome with that decision taken the other
    way (recursively, up to ``max_outcomes``).  Near-tie draws need no branch: each
    outcome lists its admissible emitted tokens."""
    base = verify_request(batch, b, truncate)
    found = [base]
    if base.status != ROW_OK:
        return found
    seen = {frozenset()}
    stack = [base]
    while stack and len(found) < max_outcomes:
        res = stack.pop()
        for dcs in res.decisions:
            if not dcs.fragile or not dcs.alt or (dcs.kind, dcs.pos) in res.flips:
                continue
            nf = dict(res.flips)
            nf[(dcs.kind, dcs.pos)] = dcs.alt
            key = frozenset(nf.items())
            if key in seen:
                continue
            seen.add(key)
            alt = verify_request(batch, b, truncate, flips=nf)
            found.append(alt)
            stack.append(alt)
            if len(found) >= max_outcomes:
                break
    return found


def verify_batch(batch, requests=None, truncate=truncate_full_sort):
    """Run ``verify_request`` over the given requests (default: all)."""
    reqs = range(batch.B) if requests is None else requests
    return {b: verify_request(batch, b, truncate) for b in reqs}


def outcomes_batch(batch, requests=None, truncate=truncate_full_sort):
    """``outcomes`` over the given requests (default: all)."""
    reqs = range(batch.B) if requests is None else requests
    return {b: outcomes(batch, b, truncate) for b in reqs}
