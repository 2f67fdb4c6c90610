"""Pins of the oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: published vectors,
hand-worked examples, library routines, closed forms, exact enumeration of the
speculative-sampling law, or brute force on tiny inputs.
"""
import itertools
import os

import numpy as np
import pytest
import scipy.special

from oracle import epilogue as O
from tests._batches import one_request, replicate
from workloads.philox import philox4x32_10, epilogue_uniforms
from workloads import configs

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


# ------------------------------------------------------------------ Philox
def test_philox_known_answers():
    for ln in _lines("philox4x32_10_kat.txt"):
        w = [int(t, 16) for t in ln.split()]
        out = philox4x32_10(np.array(w[:4], np.uint64), np.array(w[4:6], np.uint64))
        assert [int(v) for v in out] == w[6:10]


def test_uniforms_layout_and_range():
    u = epilogue_uniforms(7, 3, 4)
    assert u.shape == (3, 5, 2) and u.dtype == np.float32
    assert (u >= 0).all() and (u < 1).all()
    words = philox4x32_10(np.array([2, 1, 0, 0], np.uint64), np.array([7, 0], np.uint64))
    assert u[1, 2, 0] == np.float32((int(words[0]) >> 8) * 2.0 ** -24)
    assert u[1, 2, 1] == np.float32((int(words[1]) >> 8) * 2.0 ** -24)


# ------------------------------------------------------------------ penalties + greedy (hand example)
def test_penalty_greedy_hand_example():
    rows = _lines("penalty_greedy_example.txt")
    x = np.tile(np.array([2.0, 1.5, 1.0, 0.5], np.float32), (3, 1))
    d = [1, 0]
    for ln in rows[:3]:
        f = ln.split()
        j = int(f[0])
        want = np.array([float(v) for v in f[1:5]])
        c = O.count_vector(4, [0, 2], [2, 1], d[:j])
        xp = O.penalised_logits(x[j], c, 0.5, 0.3)
        assert np.allclose(xp, want, atol=2e-9, rtol=0)
        assert int(np.argmax(xp)) == int(f[5])
    res = rows[3].split()
    b = one_request(x, np.full((2, 4), 0.25), d, T=0.0, presence=0.5, frequency=0.3,
                    hist_ids=[0, 2], hist_counts=[2, 1])
    r = O.verify_request(b, 0)
    assert r.accept_len == int(res[1])
    assert list(r.tokens) == [int(v) for v in res[2:]]
    # without the penalties the draft is rejected at once (the penalties decide this case)
    b0 = one_request(x, np.full((2, 4), 0.25), d, T=0.0, hist_ids=[0, 2], hist_counts=[2, 1])
    r0 = O.verify_request(b0, 0)
    assert r0.accept_len == 0 and r0.tokens[0] == 0


def test_penalty_float32_operation_order():
    # x' = fl(x - fl(fl(f*c) + p)) with every step rounded to float32
    x = np.float32(10.0625)
    c = O.count_vector(3, [1], [4], [])
    xp = O.penalised_logits(np.array([0, x, 0], np.float32), c, 0.2, 0.2)
    pen = np.float32(np.float32(np.float32(0.2) * np.float32(4)) + np.float32(0.2))
    assert xp[1] == np.float32(x - pen)
    assert xp.dtype == np.float32 and xp[0] == 0 and xp[2] == 0


# ------------------------------------------------------------------ greedy == sequential argmax decoding
@pytest.mark.parametrize("seed", range(6))
def test_greedy_equals_sequential_argmax(seed):
    rng = np.random.default_rng(seed)
    V, K = 50, 4
    x = np.round(rng.normal(0, 2, (K + 1, V)).astype(np.float32) * 4) / 4   # some exact ties
    hist = np.array(sorted(rng.choice(V, 6, replace=False)), np.int32)
    cnt = rng.integers(1, 4, 6).astype(np.int32)
    # sequential penalised argmax decoding from the same logits (np.argmax: first index on ties)
    seq = []
    for j in range(K + 1):
        c = np.zeros(V, np.int64)
        c[hist] += cnt
        for t in seq:
            c[t] += 1
        pen = np.where(c > 0, np.float32(0.4) * c.astype(np.float32) + np.float32(0.3), 0).astype(np.float32)
        xp = np.where(c > 0, x[j] - pen, x[j]).astype(np.float32)
        seq.append(int(np.argmax(xp)))
    m = int(rng.integers(0, K + 1))
    d = list(seq[:K])
    if m < K:
        d[m] = (seq[m] + 1) % V
    b = one_request(x, np.full((K, V), 1.0 / V), d, T=0.0, presence=0.3, frequency=0.4,
                    hist_ids=hist, hist_counts=cnt)
    r = O.verify_request(b, 0)
    assert r.accept_len == m
    assert list(r.tokens[:m + 1]) == seq[:m + 1]


def test_greedy_k0_is_plain_argmax():
    x = np.array([[0.5, 3.0, 3.0, -1.0]], np.float32)
    b = one_request(x, np.zeros((0, 4)), [], T=0.0)
    r = O.verify_request(b, 0)
    assert r.accept_len == 0 and r.tokens[0] == 1


# ------------------------------------------------------------------ truncation
def test_nucleus_hand_examples():
    for ln in _lines("nucleus_examples.txt"):
        name, probs, k, p, kept = [s.strip() for s in ln.split("|")]
        w = np.array([float(v) for v in probs.split()])
        want = sorted(int(v) for v in kept.split())
        for trunc in (O.truncate_full_sort, lambda v, ww, kk, pp: O.truncate_grouped(v, ww, kk, pp, group=2)):
            keep, margins = trunc(w.astype(np.float32), w, int(k), float(p))
            assert sorted(np.nonzero(keep)[0].tolist()) == want, name
            assert min(margins) > 1e-6, name


def _trunc_cases(rng):
    V = 3000
    yield rng.normal(0, 3, V).astype(np.float32)                          # generic
    yield (np.round(rng.normal(0, 2, V) * 2) / 2).astype(np.float32)      # tie-heavy
    yield np.zeros(V, np.float32)                                        # all equal
    xb = rng.normal(0, 3, V).astype(np.float32)
    from workloads.generate import f32_to_bf16_bits, bf16_bits_to_f32
    yield bf16_bits_to_f32(f32_to_bf16_bits(xb))                         # bf16-exact values


@pytest.mark.parametrize("seed", range(3))
def test_grouped_select_equals_full_sort(seed):
    rng = np.random.default_rng(seed)
    for vals in _trunc_cases(rng):
        for T in (0.6, 1.0):
            w = np.exp((vals.astype(np.float64) - vals.max()) / T)
            for k in (0, 1, 20, 64, vals.size):
                for p in (1e-9, 0.5, 0.95, 1.0):
                    a, ma = O.truncate_full_sort(vals, w, k, p)
                    b, mb = O.truncate_grouped(vals, w, k, p, group=256)
                    assert np.array_equal(a, b), (k, p)
                    for x, y in zip(ma, mb):
                        assert abs(x - y) < 1e-12 or (np.isinf(x) and np.isinf(y))


def test_topk_brute_force_small():
    # brute force on every subset: top-k keeps exactly the values >= the k-th largest
    rng = np.random.default_rng(5)
    for _ in range(50):
        V = 7
        vals = rng.integers(0, 4, V).astype(np.float32)
        for k in range(1, V):
            keep, _ = O.truncate_full_sort(vals, np.exp(vals.astype(np.float64)), k, 1.0)
            kth = sorted(vals.tolist(), reverse=True)[k - 1]
            assert keep.tolist() == [v >= kth for v in vals.tolist()]


def test_no_truncation_is_softmax():
    rng = np.random.default_rng(1)
    x = rng.normal(0, 3, 500).astype(np.float32)
    for T in (0.3, 0.7, 1.0, 2.0):
        P, m = O.target_probs(x, T, 0, 1.0)
        assert np.allclose(P, scipy.special.softmax(x.astype(np.float64) / T), rtol=1e-12, atol=1e-300)
        P2, _ = O.target_probs(x, T, x.size, 1.0)
        assert np.array_equal(P, P2)


def test_draft_temperature_closed_form():
    rng = np.random.default_rng(2)
    q = scipy.special.softmax(rng.normal(0, 2, 300)).astype(np.float32)
    Q, _ = O.draft_probs(q, 0.5, 0, 1.0)
    q64 = q.astype(np.float64)
    assert np.allclose(Q, q64 ** 2 / (q64 ** 2).sum(), rtol=1e-12)
    Q1, _ = O.draft_probs(q, 1.0, 0, 1.0)
    assert np.allclose(Q1, q64 / q64.sum(), rtol=1e-15)


def test_topk1_sampling_equals_greedy():
    rng = np.random.default_rng(3)
    V, K = 40, 3
    for s in range(10):
        x = rng.normal(0, 2, (K + 1, V)).astype(np.float32)
        q = scipy.special.softmax(rng.normal(0, 2, (K, V)), axis=1)
        d = [int(np.argmax(x[i])) if rng.random() < 0.7 else int(rng.integers(V)) for i in range(K)]
        u = rng.random((K + 1, 2))
        g = O.verify_request(one_request(x, q, d, T=0.0), 0)
        t1 = O.verify_request(one_request(x, q, d, T=0.8, top_k=1, uniforms=u), 0)
        assert g.accept_len == t1.accept_len
        assert list(g.tokens) == list(t1.tokens)


def test_draft_equal_target_accepts_everything():
    rng = np.random.default_rng(4)
    V, K, T = 30, 4, 0.9
    x = rng.normal(0, 2, (K + 1, V)).astype(np.float32)
    q = scipy.special.softmax(x[:K].astype(np.float64) / 1.0, axis=1).astype(np.float32)
    for s in range(10):
        u = rng.random((K + 1, 2))
        d = [int(rng.integers(V)) for _ in range(K)]
        r = O.verify_request(one_request(x, q, d, T=1.0, uniforms=u), 0)
        # Q' = P' (same softmax at T=1, no truncation) -> ratio 1 up to rounding -> accept all
        assert r.accept_len == K or r.fragile


def test_k0_draw_is_textbook_inverse_cdf():
    rng = np.random.default_rng(6)
    V = 64
    for s in range(20):
        x = rng.normal(0, 2, (1, V)).astype(np.float32)
        u = rng.random((1, 2))
        r = O.verify_request(one_request(x, np.zeros((0, V)), [], T=0.7, top_k=10, top_p=0.9, uniforms=u), 0)
        P, _ = O.target_probs(x[0], 0.7, 10, 0.9)
        C = np.cumsum(P)
        want = int(np.searchsorted(C, np.float32(u[0, 1]) * C[-1], side="right"))
        assert r.tokens[0] == want and r.accept_len == 0


def test_inverse_cdf_boundaries():
    # exact boundaries: u*total equal to a cumulative sum selects the NEXT id (strict >),
    # and a zero-weight leading id is never drawn, even with u = 0
    assert O.inverse_cdf(np.array([1.0, 1.0, 2.0]), 0.25)[0] == 1
    assert O.inverse_cdf(np.array([1.0, 1.0, 2.0]), 0.5)[0] == 2
    assert O.inverse_cdf(np.array([0.0, 0.0, 3.0, 1.0]), 0.0)[0] == 2
    assert O.inverse_cdf(np.array([2.0, 0.0, 2.0]), 0.5)[0] == 2
    assert O.inverse_cdf(np.array([1.0, 1.0, 2.0]), 0.25)[1] == 0.0


def test_inverse_cdf_matches_searchsorted():
    rng = np.random.default_rng(7)
    for _ in range(200):
        w = rng.random(17) * (rng.random(17) < 0.6)
        if w.sum() == 0:
            continue
        u = rng.random()
        t, m = O.inverse_cdf(w, u)
        C = np.cumsum(w)
        assert t == int(np.searchsorted(C, u * C[-1], side="right"))
        assert w[t] > 0 and m >= 0


# ------------------------------------------------------------------ exact law of speculative sampling
def _enum_case(seed, V=5, K=2, T=0.8, top_k=4, top_p=0.9, pres=0.4, freq=0.3):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1.5, (K + 1, V)).astype(np.float32)
    q = scipy.special.softmax(rng.normal(0, 1.5, (K, V)), axis=1).astype(np.float32)
    hist_ids, hist_cnt = np.array([1, V - 1], np.int32), np.array([2, 1], np.int32)
    return x, q, hist_ids, hist_cnt, dict(T=T, top_k=top_k, top_p=top_p, presence=pres, frequency=freq)


def _P(x, j, prefix, hist_ids, hist_cnt, prm):
    V = x.shape[1]
    xp = O.penalised_logits(x[j], O.count_vector(V, hist_ids, hist_cnt, prefix), prm["presence"], prm["frequency"])
    return O.target_probs(xp, prm["T"], prm["top_k"], prm["top_p"])[0]


@pytest.mark.parametrize("seed,V,K", [(0, 5, 2), (1, 4, 3), (2, 6, 2), (3, 3, 3)])
def test_speculative_law_equals_sequential_target(seed, V, K):
    """Speculative round + sequential completion has exactly the law of sequential sampling
    from the penalised, tempered, truncated target (v0.0.2 release notes, Highlights: the
    output distribution equals the target's; Changelog [0.2.0] Added: penalties stay exact)."""
    x, q, hid, hc, prm = _enum_case(seed, V=V, K=K)
    Qs = [O.draft_probs(q[i], prm["T"], prm["top_k"], prm["top_p"])[0] for i in range(K)]

    def seq_prob(s, start, prefix):
        pr = 1.0
        pre = list(prefix)
        for j in range(start, K + 1):
            pr *= _P(x, j, pre, hid, hc, prm)[s[j]]
            pre.append(s[j])
        return pr

    spec = {}
    seqs = list(itertools.product(range(V), repeat=K + 1))
    for d in itertools.product(range(V), repeat=K):
        pd = np.prod([Qs[i][d[i]] for i in range(K)])
        if pd == 0:
            continue
        reach = 1.0                       # probability that positions < i were all accepted
        for i in range(K + 1):
            P = _P(x, i, d[:i], hid, hc, prm)
            if i == K:
                dist, stop_p = P, reach
            else:
                alpha = O.accept_probability(P[d[i]], Qs[i][d[i]])
                r = O.residual(P, Qs[i])
                dist = r / r.sum() if r.sum() > 0 else P
                stop_p = reach * (1 - alpha)
            for s in seqs:
                if tuple(s[:i]) != tuple(d[:i]):
                    continue
                contrib = pd * stop_p * dist[s[i]]
                if contrib:
                    contrib *= seq_prob(s, i + 1, list(s[:i + 1]))
                    spec[s] = spec.get(s, 0.0) + contrib
            if i < K:
                reach *= alpha
    for s in seqs:
        assert abs(spec.get(s, 0.0) - seq_prob(s, 0, [])) < 1e-12


def _outcome_law(x, q, hid, hc, prm, K):
    """Exact law of (accept_len, emitted tokens) with d ~ Q' and uniform draws."""
    V = x.shape[1]
    Qs = [O.draft_probs(q[i], prm["T"], prm["top_k"], prm["top_p"])[0] for i in range(K)]
    law = {}
    for d in itertools.product(range(V), repeat=K):
        pd = np.prod([Qs[i][d[i]] for i in range(K)])
        if pd == 0:
            continue
        reach = 1.0
        for i in range(K + 1):
            P = _P(x, i, d[:i], hid, hc, prm)
            if i == K:
                dist, stop = P, reach
            else:
                alpha = O.accept_probability(P[d[i]], Qs[i][d[i]])
                r = O.residual(P, Qs[i])
                dist = r / r.sum() if r.sum() > 0 else P
                stop = reach * (1 - alpha)
            for t in range(V):
                key = (i,) + tuple(d[:i]) + (t,)
                law[key] = law.get(key, 0.0) + pd * stop * dist[t]
            if i < K:
                reach *= alpha
    return law, Qs


def test_verify_request_wiring_monte_carlo():
    """verify_request with random drafts d ~ Q' and uniforms reproduces the exact outcome law
    (chi-square); a swapped ratio, wrong residual or wrong draw position fails this."""
    V, K = 4, 2
    x, q, hid, hc, prm = _enum_case(11, V=V, K=K)
    law, Qs = _outcome_law(x, q, hid, hc, prm, K)
    rng = np.random.default_rng(12)
    N = 6000
    ds = [[int(rng.choice(V, p=Qs[i])) for i in range(K)] for _ in range(N)]
    us = rng.random((N, K + 1, 2)).astype(np.float32)
    base = one_request(x, q, [0] * K, hist_ids=hid, hist_counts=hc, **prm)
    res = O.verify_batch(replicate(base, ds, us))
    counts = {}
    for r in res.values():
        key = (r.accept_len,) + tuple(int(t) for t in r.tokens[:r.accept_len + 1])
        counts[key] = counts.get(key, 0) + 1
    assert set(counts) <= {k for k, v in law.items() if v > 0}
    keys = [k for k, v in law.items() if v * N >= 5]
    obs = np.array([counts.get(k, 0) for k in keys], float)
    exp = np.array([law[k] * N for k in keys])
    rest_o, rest_e = N - obs.sum(), N - exp.sum()
    if rest_e >= 5:
        obs, exp = np.append(obs, rest_o), np.append(exp, rest_e)
    chi2 = float(((obs - exp) ** 2 / exp).sum())
    dof = len(obs) - 1
    from scipy.stats import chi2 as chi2d
    assert chi2d.sf(chi2, dof) > 1e-4, (chi2, dof)


# ------------------------------------------------------------------ logprobs
def test_raw_log_softmax_matches_library():
    rng = np.random.default_rng(8)
    x = rng.normal(0, 3, 10000).astype(np.float32)
    assert np.allclose(O.raw_log_softmax(x), scipy.special.log_softmax(x.astype(np.float64)), atol=1e-12)


def test_top_n_order():
    x = np.array([1.0, 3.0, 2.0, 3.0, -1.0, 2.0], np.float32)
    assert O.top_n(x, 4).tolist() == [1, 3, 2, 5]


def test_logprobs_use_raw_logits_at_emitted_tokens():
    rng = np.random.default_rng(9)
    V, K = 20, 2
    x = rng.normal(0, 2, (K + 1, V)).astype(np.float32)
    q = scipy.special.softmax(rng.normal(0, 2, (K, V)), axis=1)
    b = one_request(x, q, [int(np.argmax(x[0])), 3], T=0.0, presence=1.0, frequency=1.0,
                    hist_ids=[int(np.argmax(x[0]))], hist_counts=[1], n_top=3, want_logprobs=True)
    r = O.verify_request(b, 0)
    for j in range(r.accept_len + 1):
        ls = scipy.special.log_softmax(x[j].astype(np.float64))
        assert abs(r.logprobs[j] - ls[r.tokens[j]]) < 1e-12
        assert r.top_ids[j].tolist() == np.argsort(-x[j], kind="stable")[:3].tolist()
    assert np.all(np.isneginf(r.logprobs[r.accept_len + 1:]))
    assert np.all(r.tokens[r.accept_len + 1:] == -1)


# ------------------------------------------------------------------ validation
def test_invalid_rows_flagged():
    x = np.zeros((3, 8), np.float32)
    q = np.full((2, 8), 1 / 8)
    assert O.verify_request(one_request(x, q, [1, 2], T=-1.0), 0).status == O.ROW_BAD_PARAMS
    assert O.verify_request(one_request(x, q, [1, 2], T=1.0, top_p=0.0), 0).status == O.ROW_BAD_PARAMS
    assert O.verify_request(one_request(x, q, [1, 9], T=1.0), 0).status == O.ROW_BAD_DRAFT
    xn = x.copy()
    xn[1, 3] = np.nan
    assert O.verify_request(one_request(xn, q, [1, 2], T=1.0), 0).status == O.ROW_NONFINITE
    assert O.verify_request(one_request(x, q, [1, 2], T=1.0, K=3), 0).status == O.ROW_BAD_PARAMS


def test_workloads_smoke_oracle_small():
    b = configs.build("b1k2v4096")
    r = O.verify_request(b, 0)
    assert 0 <= r.accept_len <= 2 and r.tokens[r.accept_len] >= 0
    g = O.verify_request(configs.build("b1k2v4096_greedy"), 0)
    assert 0 <= g.accept_len <= 2


# ------------------------------------------------------------------ near-tie bookkeeping
def test_draw_margin_in_uniform_units():
    """A residual of total mass 0.25 (weights 0.1, 0.15): u * 0.25 lying 5e-7 of mass above
    the first boundary is 2e-6 away in uniform units, so the draw is not a near tie and only
    token 1 is admissible; 2e-7 of mass (8e-7 in u) is a near tie admitting tokens 0 and 1."""
    w = np.array([0.1, 0.15])
    u = (0.1 + 5e-7) / 0.25
    t, m = O.inverse_cdf(w, u)
    assert t == 1 and abs(m - 2e-6) < 1e-12
    assert O.draw_admissible(w, u).tolist() == [1]
    u = (0.1 + 2e-7) / 0.25
    t, m = O.inverse_cdf(w, u)
    assert t == 1 and abs(m - 8e-7) < 1e-12 and m < O.MARGIN_EPS
    assert O.draw_admissible(w, u).tolist() == [0, 1]
    # zero-weight ids are never admissible, even next to u
    assert O.draw_admissible(np.array([0.1, 0.0, 0.15]), u).tolist() == [0, 2]


def _residual_quarter_request(u_draw):
    """K=1, T=1, no truncation: P = softmax(x1), Q = q; the draft is rejected (u0 > P/Q) and
    the residual max(0, P - Q) is drawn with u_draw."""
    x = np.log(np.array([[0.4, 0.35, 0.25], [0.2, 0.3, 0.5]], np.float64)).astype(np.float32)
    q = np.array([[0.3, 0.25, 0.45]], np.float32)
    P = scipy.special.softmax(x[0].astype(np.float64))
    Q = q[0].astype(np.float64) / q[0].astype(np.float64).sum()
    return one_request(x, q, [2], T=1.0, uniforms=[[0.9, u_draw], [0.0, 0.0]]), P, Q


def test_request_draw_margin_uses_uniform_units():
    """Through verify_request: the residual max(0, P - Q) has total ~0.2; u placed 5e-7 of
    mass above its first boundary is a draw with margin ~2.5e-6 in u, not a near tie."""
    _, P, Q = _residual_quarter_request(0.0)
    r = np.maximum(0.0, P - Q)
    u = (r[0] + 5e-7) / r.sum()
    b, _, _ = _residual_quarter_request(u)
    res = O.verify_request(b, 0)
    assert res.accept_len == 0 and res.tokens[0] == 1
    draw = [d for d in res.decisions if d.kind == "draw"][0]
    assert abs(draw.margin - 5e-7 / r.sum()) < 1e-7          # u is rounded to float32
    assert not draw.fragile and res.admissible.tolist() == [1]


def test_nucleus_margins_and_flips_hand_example():
    """Weights 0.5, 0.3, 0.2: the mass above the smallest group is 0.8.  top_p = 0.8 + 3e-7
    keeps it with a last-kept margin of 3e-7 (its flip drops it); top_p = 0.8 - 3e-7 drops it
    with a first-dropped margin of 3e-7 (its flip keeps it)."""
    w = np.array([0.5, 0.3, 0.2])
    v = w.astype(np.float32)
    for trunc in (O.truncate_full_sort, lambda *a, **k: O.truncate_grouped(*a, group=2, **k)):
        keep, (m_last, m_next) = trunc(v, w, 0, 0.8 + 3e-7)
        assert keep.tolist() == [True, True, True]
        assert abs(m_last - 3e-7) < 1e-12 and np.isinf(m_next)
        keep, _ = trunc(v, w, 0, 0.8 + 3e-7, flip="drop_last")
        assert keep.tolist() == [True, True, False]
        keep, (m_last, m_next) = trunc(v, w, 0, 0.8 - 3e-7)
        assert keep.tolist() == [True, True, False]
        assert abs(m_next - 3e-7) < 1e-12 and abs(m_last - (0.3 - 3e-7)) < 1e-12
        keep, _ = trunc(v, w, 0, 0.8 - 3e-7, flip="keep_next")
        assert keep.tolist() == [True, True, True]


def test_accept_near_tie_has_both_outcomes():
    """u within 4e-7 below P'(d)/Q'(d): float64 accepts (then the bonus draw from P'_1); the
    other side rejects and draws from the residual at position 0.  Both outcomes, and only
    these, are correct, each as the closed-form sequential computation gives it."""
    x = np.log(np.array([[0.4, 0.35, 0.25], [0.2, 0.3, 0.5]], np.float64)).astype(np.float32)
    q = np.array([[0.3, 0.25, 0.45]], np.float32)
    P0 = scipy.special.softmax(x[0].astype(np.float64))
    P1 = scipy.special.softmax(x[1].astype(np.float64))
    Q0 = q[0].astype(np.float64) / q[0].astype(np.float64).sum()
    ratio = P0[2] / Q0[2]
    u_draw = 0.55
    b = one_request(x, q, [2], T=1.0, uniforms=[[ratio - 4e-7, u_draw], [0.0, u_draw]])
    outs = O.outcomes(b, 0)
    assert len(outs) == 2
    acc, rej = outs
    assert acc.accept_len == 1 and acc.tokens[0] == 2
    assert acc.tokens[1] == int(np.searchsorted(np.cumsum(P1), u_draw, side="right"))
    assert rej.accept_len == 0
    r = np.maximum(0.0, P0 - Q0)
    assert rej.tokens[0] == int(np.searchsorted(np.cumsum(r), u_draw * r.sum(), side="right"))
    assert [d.kind for d in acc.decisions if d.fragile] == ["accept"]
    # far from the ratio there is one outcome
    far = one_request(x, q, [2], T=1.0, uniforms=[[ratio - 1e-3, u_draw], [0.0, u_draw]])
    assert len(O.outcomes(far, 0)) == 1


def test_subset_batches_equal_the_whole_batch():
    """A request built on its own equals the same request of the whole batch, bit for bit."""
    full = configs.build("b4k8v151936_mixed")
    for b in (0, 3):
        one = configs.build("b4k8v151936_mixed", requests=[b])
        assert one.B == 1 and one.requests == (b,)
        assert np.array_equal(one.x[0], full.x[b]) and np.array_equal(one.q[0], full.q[b])
        assert np.array_equal(one.draft_ids[0], full.draft_ids[b])
        assert np.array_equal(one.uniforms[0], full.uniforms[b])
        assert np.array_equal(one.rows[0], full.rows[b])
        hi, hc = full.history(b)
        oi, oc = one.history(0)
        assert np.array_equal(hi, oi) and np.array_equal(hc, oc)


def test_masked_logits_have_zero_probability():
    """A -inf logit is a token of probability zero: never drawn, never accepted, logprob -inf;
    NaN, +inf or an all -inf row make the request non-finite."""
    x = np.array([[0.0, -np.inf, 1.0, 0.5], [2.0, 0.0, -np.inf, -np.inf]], np.float32)
    q = np.array([[0.1, 0.6, 0.2, 0.1]], np.float32)
    for u0 in (0.0, 0.3, 0.9):
        for u1 in (0.0, 0.4, 0.99):
            r = O.verify_request(one_request(x, q, [1], T=1.0, uniforms=[[u0, u1], [0.0, u1]], n_top=4,
                                             want_logprobs=True), 0)
            assert r.status == O.ROW_OK and r.accept_len == 0       # P'(1) = 0: draft 1 is rejected
            assert r.tokens[0] != 1
            assert r.top_ids[0].tolist() == [2, 3, 0, 1] and np.isneginf(r.top_logprobs[0][3])
    g = O.verify_request(one_request(x, q, [2], T=0.0), 0)
    assert g.accept_len == 1 and g.tokens.tolist() == [2, 0]
    g = O.verify_request(one_request(x, q, [1], T=0.0), 0)
    assert g.accept_len == 0 and g.tokens[0] == 2
    for bad in (np.nan, np.inf):
        xb = x.copy()
        xb[1, 1] = bad
        assert O.verify_request(one_request(xb, q, [2], T=1.0), 0).status == O.ROW_NONFINITE
    xb = x.copy()
    xb[0, :] = -np.inf
    assert O.verify_request(one_request(xb, q, [2], T=1.0), 0).status == O.ROW_NONFINITE
