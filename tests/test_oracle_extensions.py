"""Pins of the oracle's draft layouts, end-of-sequence stop, per-position acceptance counts and
penalised logprob mode.

Sources (mlx-dspark pages): Changelog [0.2.0] Added, "--mode lookup" (drafter-free drafts, T > 0
through a one-hot proposal, still an exact target sample); Changelog [0.8.0] Added, reduced draft
vocabularies (a d2t offset table, target id = draft id + d2t[draft id], the draft distribution
widened onto the target vocabulary before the accept test); Changelog [0.2.0] Fixed (stop when an
accepted draft is the eos token mid-block); Changelog [0.9.0] Added (per-position acceptance with
honest denominators); Changelog [0.2.0] Added, logprobs (the penalised variant is the other
reading of "raw target log-softmax").
"""
import dataclasses

import numpy as np
import pytest
import scipy.special
from scipy.stats import chi2 as chi2d

from oracle import epilogue as O
from tests._batches import one_request, replicate


def _sparse(batch, ids, vals):
    """The batch with its draft rows given as (ids, probabilities) pairs [B, K_max, m]."""
    ids = np.asarray(ids, np.int32).reshape(batch.B, batch.K_max, -1)
    vals = np.asarray(vals, np.float32).reshape(ids.shape)
    return dataclasses.replace(batch, q=vals, q_ids=ids, q_layout="sparse")


def _reduced(batch, qred, d2t):
    qred = np.asarray(qred, np.float32).reshape(batch.B, batch.K_max, -1)
    return dataclasses.replace(batch, q=qred, d2t=np.asarray(d2t, np.int32), q_layout="reduced")


def _same(r0, r1):
    assert r0.status == r1.status and r0.accept_len == r1.accept_len
    assert np.array_equal(r0.tokens, r1.tokens)
    assert [(d.kind, d.pos, d.margin) for d in r0.decisions] == [(d.kind, d.pos, d.margin) for d in r1.decisions]


# ------------------------------------------------------------------ one-hot proposal (lookup drafts)
X0 = np.array([0.0, 1.0, 2.0, 0.5, -1.0, 1.5], np.float32)


def test_one_hot_proposal_hand_example():
    """T = 1, no truncation, one draft d0 = 2 proposed with probability 1.  softmax(X0) =
    [0.05680, 0.15440, 0.41970, 0.09365, 0.02090, 0.25456] (exp sum 17.60563): the draft is
    accepted iff u0 < P(2) = 0.41970; on rejection the residual max(0, P - onehot(2)) is P with
    token 2 removed, whose normalised cumulative masses are 0.0979, 0.3639, 0.3639, 0.5253,
    0.5613, 1 -- so u1 = 0.3, 0.5, 0.55, 0.9 draw tokens 1, 3, 4, 5."""
    x = np.stack([X0, X0])
    base = one_request(x, np.zeros((1, 6)), [2], T=1.0)
    for u0, acc in ((0.4196, 1), (0.4198, 0)):
        for u1, tok in ((0.3, 1), (0.5, 3), (0.55, 4), (0.9, 5)):
            u = np.array([[u0, u1], [0.0, u1]], np.float32)
            b = _sparse(dataclasses.replace(base, uniforms=u[None]), [[2]], [[1.0]])
            r = O.verify_request(b, 0)
            assert r.status == O.ROW_OK and r.accept_len == acc
            if acc == 0:
                assert r.tokens.tolist() == [tok, -1]
            else:
                assert r.tokens[0] == 2
                # the bonus draw is from P'_1 = softmax(X0): cumulative 0.0568, 0.2112, 0.6309, ...
                assert r.tokens[1] == {0.3: 2, 0.5: 2, 0.55: 2, 0.9: 5}[u1]


def test_one_hot_proposal_is_lossless_monte_carlo():
    """With a fixed one-hot proposal, the first emitted token is distributed as P'_0, and given
    that it is the draft d0, the second is distributed as P'_1 after the prefix [d0] (the target's
    sequential law), under penalties, temperature and truncation."""
    rng = np.random.default_rng(21)
    V, K = 5, 2
    x = rng.normal(0, 1.5, (K + 1, V)).astype(np.float32)
    prm = dict(T=0.8, top_k=4, top_p=0.9, presence=0.4, frequency=0.3)
    hid, hc = [1, 4], [2, 1]
    d = [1, 3]
    N = 6000
    us = rng.random((N, K + 1, 2)).astype(np.float32)
    base = one_request(x, np.zeros((K, V)), d, hist_ids=hid, hist_counts=hc, **prm)
    rep = replicate(base, [d] * N, us)
    rep = _sparse(rep, np.tile(np.array(d, np.int32)[None, :, None], (N, 1, 1)), np.ones((N, K, 1)))
    res = O.verify_batch(rep)

    def P(j, prefix):
        xp = O.penalised_logits(x[j], O.count_vector(V, hid, hc, prefix), prm["presence"], prm["frequency"])
        return O.target_probs(xp, prm["T"], prm["top_k"], prm["top_p"])[0]

    def chi2_ok(obs_tokens, p):
        obs = np.bincount(obs_tokens, minlength=V).astype(float)
        exp = p * len(obs_tokens)
        keep = exp > 0
        assert obs[~keep].sum() == 0
        stat = float(((obs[keep] - exp[keep]) ** 2 / exp[keep]).sum())
        return chi2d.sf(stat, keep.sum() - 1) > 1e-4

    first = np.array([r.tokens[0] for r in res.values()])
    assert chi2_ok(first, P(0, []))
    second = np.array([r.tokens[1] for r in res.values() if r.tokens[0] == d[0]])
    assert len(second) > 1000 and chi2_ok(second, P(1, [d[0]]))


# ------------------------------------------------------------------ sparse and reduced layouts
def test_sparse_rows_equal_the_dense_rows_they_stand_for():
    """m = 3 pairs (ids 4, 0, 2; probabilities 0.2, 0.5, 0.3) are the dense row
    [0.5, 0, 0.3, 0, 0.2, 0]; with top_k = 2 the truncated draft is [0.625, 0, 0.375, 0, 0, 0]."""
    rng = np.random.default_rng(22)
    V = 6
    x = rng.normal(0, 1.0, (2, V)).astype(np.float32)
    dense = np.array([[0.5, 0, 0.3, 0, 0.2, 0]], np.float32)
    for T, k, p in ((1.0, 0, 1.0), (0.7, 2, 1.0), (1.3, 0, 0.6)):
        for s in range(40):
            u = rng.random((2, 2)).astype(np.float32)
            bd = one_request(x, dense, [int(rng.choice([0, 2, 4, 1]))], T=T, top_k=k, top_p=p, uniforms=u)
            bs = _sparse(bd, [[4, 0, 2]], [[0.2, 0.5, 0.3]])
            _same(O.verify_request(bd, 0), O.verify_request(bs, 0))
    b = _sparse(one_request(x, dense, [0], T=1.0, top_k=2), [[4, 0, 2]], [[0.2, 0.5, 0.3]])
    Q = O.draft_probs(O.widened_draft(b, 0, 0), 1.0, 2, 1.0)[0]
    assert np.allclose(Q, [0.625, 0, 0.375, 0, 0, 0], atol=1e-7)


def test_reduced_vocabulary_hand_example():
    """Draft vocabulary of 3 over V = 6 with d2t = [1, 3, 3]: draft ids 0, 1, 2 are target ids
    1, 4, 5, so q = [0.5, 0.3, 0.2] widens to [0, 0.5, 0, 0, 0.3, 0.2]; the request then behaves
    exactly as with that dense row."""
    rng = np.random.default_rng(23)
    V = 6
    x = rng.normal(0, 1.0, (3, V)).astype(np.float32)
    wide = np.array([[0, 0.5, 0, 0, 0.3, 0.2], [0, 0.2, 0, 0, 0.1, 0.7]], np.float32)
    red = [[0.5, 0.3, 0.2], [0.2, 0.1, 0.7]]
    b = _reduced(one_request(x, wide, [1, 5], T=1.0), red, [1, 3, 3])
    assert O.widened_draft(b, 0, 0).tolist() == pytest.approx([0, 0.5, 0, 0, 0.3, 0.2])
    assert O.widened_draft(b, 0, 1).tolist() == pytest.approx([0, 0.2, 0, 0, 0.1, 0.7])
    for T, k, p in ((1.0, 0, 1.0), (0.6, 2, 0.9)):
        for s in range(40):
            u = rng.random((3, 2)).astype(np.float32)
            d = [int(rng.choice([1, 4, 5, 0])), int(rng.choice([1, 4, 5, 2]))]
            bd = one_request(x, wide, d, T=T, top_k=k, top_p=p, uniforms=u)
            _same(O.verify_request(bd, 0), O.verify_request(_reduced(bd, red, [1, 3, 3]), 0))


def test_invalid_draft_layouts_flagged():
    x = np.zeros((3, 6), np.float32)
    dense = np.full((2, 6), 1 / 6, np.float32)
    b = one_request(x, dense, [1, 2], T=1.0)
    ok = [[[1, 2], [2, 3]]]
    assert O.verify_request(_sparse(b, ok, np.full((1, 2, 2), 0.5)), 0).status == O.ROW_OK
    for bad in ([[[1, 1], [2, 3]]], [[[1, 2], [6, 3]]], [[[1, 2], [-1, 3]]]):
        assert O.verify_request(_sparse(b, bad, np.full((1, 2, 2), 0.5)), 0).status == O.ROW_BAD_DRAFT
    # rows past num_drafts are not read; a greedy request reads no draft row at all
    b1 = one_request(x, dense, [1, 2], T=1.0, K=1)
    assert O.verify_request(_sparse(b1, [[[1, 2], [3, 3]]], np.full((1, 2, 2), 0.5)), 0).status == O.ROW_OK
    bg = one_request(x, dense, [1, 2], T=0.0)
    assert O.verify_request(_sparse(bg, [[[1, 1], [9, 9]]], np.full((1, 2, 2), 0.5)), 0).status == O.ROW_OK
    red = np.full((1, 2, 3), 1 / 3)
    assert O.verify_request(_reduced(b, red, [1, 3, 3]), 0).status == O.ROW_OK
    assert O.verify_request(_reduced(b, red, [1, 3, 4]), 0).status == O.ROW_BAD_DRAFT   # 2 + 4 = 6 >= V
    assert O.verify_request(_reduced(b, red, [1, 0, 3]), 0).status == O.ROW_BAD_DRAFT   # 0+1 == 1+0
    assert O.verify_request(_reduced(bg, red, [1, 0, 3]), 0).status == O.ROW_OK


# ------------------------------------------------------------------ end-of-sequence stop + counts
def _greedy_rows(argmaxes, V=8):
    x = np.zeros((len(argmaxes), V), np.float32)
    for j, t in enumerate(argmaxes):
        x[j, t] = 3.0
    return x


@pytest.mark.parametrize("drafts,eos,K,acc,tokens,stopped,attempted,accepted", [
    ([5, 7, 2], 7, 3, 2, [5, 7, -1, -1], True, [1, 1, 0], [1, 1, 0]),
    ([5, 7, 2], 2, 3, 3, [5, 7, 2, -1], True, [1, 1, 1], [1, 1, 1]),
    ([5, 7, 2], 5, 3, 1, [5, -1, -1, -1], True, [1, 0, 0], [1, 0, 0]),
    ([5, 7, 2], 6, 3, 3, [5, 7, 2, 6], False, [1, 1, 1], [1, 1, 1]),     # eos only as the bonus token
    ([5, 7, 2], -1, 3, 3, [5, 7, 2, 6], False, [1, 1, 1], [1, 1, 1]),
    ([5, 3, 2], 3, 3, 1, [5, 7, -1, -1], False, [1, 1, 0], [1, 0, 0]),   # eos only as the rejected draft
    ([5, 7, 7], 7, 3, 2, [5, 7, -1, -1], True, [1, 1, 0], [1, 1, 0]),    # the first accepted occurrence
    ([1, 7, 2], 7, 3, 0, [5, -1, -1, -1], False, [1, 0, 0], [0, 0, 0]),
    ([5, 7, 0], 4, 2, 2, [5, 7, 2, -1], False, [1, 1, 0], [1, 1, 0]),    # K_b = 2 < K_max = 3
])
def test_eos_stop_and_position_counts(drafts, eos, K, acc, tokens, stopped, attempted, accepted):
    """Greedy rows with argmaxes 5, 7, 2, 6 at positions 0..3."""
    x = _greedy_rows([5, 7, 2, 6])
    b = one_request(x, np.full((3, 8), 1 / 8), drafts, T=0.0, K=K, want_logprobs=True, n_top=2)
    b = dataclasses.replace(b, eos_ids=np.array([eos], np.int32))
    r = O.verify_request(b, 0)
    assert (r.accept_len, r.tokens.tolist(), r.stopped) == (acc, tokens, stopped)
    assert r.attempted.tolist() == attempted and r.accepted.tolist() == accepted
    emitted = acc if stopped else acc + 1
    assert np.all(np.isfinite(r.logprobs[:emitted])) and np.all(np.isneginf(r.logprobs[emitted:]))
    assert np.all(r.top_ids[:emitted] >= 0) and np.all(r.top_ids[emitted:] == -1)


def test_eos_stop_in_sampled_request():
    """T > 0: the stop cuts the accepted prefix after the eos draft and discards the draw."""
    x = _greedy_rows([5, 7, 2, 6])
    q = np.zeros((3, 8), np.float32)
    q[0, 5] = q[1, 7] = q[2, 2] = 1.0
    u = np.zeros((4, 2), np.float32)                       # accept everything P'(d) > 0 allows
    b = one_request(x, q, [5, 7, 2], T=1.0, uniforms=u)
    full = O.verify_request(b, 0)
    assert full.accept_len == 3 and not full.stopped
    r = O.verify_request(dataclasses.replace(b, eos_ids=np.array([7], np.int32)), 0)
    assert r.accept_len == 2 and r.stopped and r.tokens.tolist() == [5, 7, -1, -1]
    assert r.admissible.tolist() == [-1]
    assert all(d.kind in ("accept", "nucleus_p", "nucleus_q") and d.pos < 2 for d in r.decisions)


# ------------------------------------------------------------------ penalised logprobs
def _golden_penalised_rows():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "penalty_greedy_example.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    return np.array([[float(v) for v in f[1:5]] for f in rows[:3]])


def test_penalised_logprob_mode_hand_example():
    """The penalty hand example (tokens 1, 0, 1 emitted): in penalised mode the logprobs and top
    ids are those of the printed penalised rows x'; in raw mode those of x = [2, 1.5, 1, 0.5]."""
    x = np.tile(np.array([2.0, 1.5, 1.0, 0.5], np.float32), (3, 1))
    xp = _golden_penalised_rows()
    b = one_request(x, np.full((2, 4), 0.25), [1, 0], T=0.0, presence=0.5, frequency=0.3,
                    hist_ids=[0, 2], hist_counts=[2, 1], want_logprobs=True, n_top=4)
    raw = O.verify_request(b, 0)
    pen = O.verify_request(dataclasses.replace(b, logprob_mode="penalised"), 0)
    assert raw.tokens.tolist() == pen.tokens.tolist() == [1, 0, 1]
    for j, t in enumerate([1, 0, 1]):
        assert abs(pen.logprobs[j] - scipy.special.log_softmax(xp[j])[t]) < 1e-7
        assert abs(raw.logprobs[j] - scipy.special.log_softmax(x[j].astype(np.float64))[t]) < 1e-12
        assert raw.top_ids[j].tolist() == [0, 1, 2, 3]
    assert pen.top_ids[0].tolist() == [1, 0, 3, 2]
    assert pen.top_ids[1].tolist() == [0, 1, 3, 2]
    assert pen.top_ids[2].tolist() == [1, 0, 3, 2]
    assert abs(pen.top_logprobs[0][0] - scipy.special.log_softmax(xp[0])[1]) < 1e-7


def test_penalised_mode_without_penalty_is_raw():
    rng = np.random.default_rng(24)
    x = rng.normal(0, 2, (3, 30)).astype(np.float32)
    q = scipy.special.softmax(rng.normal(0, 2, (2, 30)), axis=1)
    b = one_request(x, q, [3, 4], T=0.9, uniforms=rng.random((3, 2)), want_logprobs=True, n_top=5)
    r0 = O.verify_request(b, 0)
    r1 = O.verify_request(dataclasses.replace(b, logprob_mode="penalised"), 0)
    assert np.array_equal(r0.logprobs, r1.logprobs) and np.array_equal(r0.top_ids, r1.top_ids)
