"""The parity comparison accepts exactly the oracle's correct outcomes (CPU only).

A "GPU result" is made on the CPU from the oracle's own outcome, then changed: every
planted difference in accept length, tokens, logprobs or top-logprob ids must be caught,
and a near-tie draw's other admissible token, or the other side of a near-tie accept test,
must be accepted.
"""
import numpy as np
import pytest
import scipy.special

from oracle import epilogue as O
from tests._batches import one_request
from tests._compare import compare
from workloads import configs


def _as_got(batch, outs_by_b):
    B, W, n = batch.B, batch.K_max + 1, batch.n_top_logprobs
    got = {"accept_len": np.zeros(B, np.int32), "tokens": np.full((B, W), -1, np.int32),
           "row_status": np.zeros(B, np.int32), "logprobs": np.full((B, W), -np.inf, np.float32),
           "top_ids": np.full((B, W, n), -1, np.int32), "top_logprobs": np.full((B, W, n), -np.inf, np.float32)}
    if not batch.want_logprobs:
        del got["logprobs"]
    if n == 0:
        del got["top_ids"], got["top_logprobs"]
    for b, outs in outs_by_b.items():
        o = outs[0]
        got["accept_len"][b] = o.accept_len
        got["tokens"][b] = o.tokens
        got["row_status"][b] = o.status
        if "logprobs" in got:
            got["logprobs"][b] = o.logprobs.astype(np.float32)
        if "top_ids" in got:
            got["top_ids"][b] = o.top_ids
            got["top_logprobs"][b] = o.top_logprobs.astype(np.float32)
    return got


@pytest.fixture(scope="module")
def case():
    batch = configs.build("b256k16v262144_mixed", B=18, requests=[1, 3, 7])
    want = O.outcomes_batch(batch)
    return batch, want


def test_oracle_result_passes(case):
    batch, want = case
    t = compare(batch, _as_got(batch, want), want)
    assert t.requests == 3 and t.off_float64 == 0


@pytest.mark.parametrize("plant", ["accept_len", "token", "logprob", "top_id", "top_logprob", "tail", "status"])
def test_planted_difference_is_caught(case, plant):
    batch, want = case
    got = _as_got(batch, want)
    b = 1
    a = int(got["accept_len"][b])
    if plant == "accept_len":
        got["accept_len"][b] = a + 1 if a < int(batch.rows["num_drafts"][b]) else a - 1
    elif plant == "token":
        got["tokens"][b, a] = (got["tokens"][b, a] + 7) % batch.V
    elif plant == "logprob":
        got["logprobs"][b, a] += 3e-4
    elif plant == "top_id":
        got["top_ids"][b, 0, [0, 1]] = got["top_ids"][b, 0, [1, 0]]
    elif plant == "top_logprob":
        got["top_logprobs"][b, 0, 2] -= 3e-4
    elif plant == "tail":
        got["tokens"][b, -1] = 0 if a + 1 < batch.K_max + 1 else got["tokens"][b, -1]
        if a + 1 >= batch.K_max + 1:
            pytest.skip("no position past the emitted token")
    elif plant == "status":
        got["row_status"][b] = 4
    with pytest.raises(AssertionError):
        compare(batch, got, want)


def test_near_tie_draw_admits_neighbour_only():
    """u placed 2e-7 (in u units) above a boundary: both tokens at the boundary pass, a third
    token does not."""
    x = np.log(np.array([[0.1, 0.2, 0.3, 0.4]], np.float64)).astype(np.float32)
    P = scipy.special.softmax(x[0].astype(np.float64))
    C = np.cumsum(P)
    u = np.float32(C[1] + 2e-7)
    b = one_request(x, np.zeros((0, 4)), [], T=1.0, uniforms=[[0.0, u]], n_top=2, want_logprobs=True)
    want = O.outcomes_batch(b)
    assert sorted(want[0][0].admissible.tolist()) == [1, 2]
    for tok, ok in ((2, True), (1, True), (3, False), (0, False)):
        got = _as_got(b, want)
        got["tokens"][0, 0] = tok
        got["logprobs"][0, 0] = np.float32(np.log(P[tok]))
        if ok:
            assert compare(b, got, want).off_float64 == (tok != want[0][0].tokens[0])
        else:
            with pytest.raises(AssertionError):
                compare(b, got, want)


def test_near_tie_accept_admits_both_sides():
    x = np.log(np.array([[0.4, 0.35, 0.25], [0.2, 0.3, 0.5]], np.float64)).astype(np.float32)
    q = np.array([[0.3, 0.25, 0.45]], np.float32)
    P0 = scipy.special.softmax(x[0].astype(np.float64))
    Q0 = q[0].astype(np.float64) / q[0].astype(np.float64).sum()
    ratio = P0[2] / Q0[2]
    b = one_request(x, q, [2], T=1.0, uniforms=[[ratio - 4e-7, 0.55], [0.0, 0.55]])
    want = O.outcomes_batch(b)
    assert len(want[0]) == 2
    for o in want[0]:
        got = _as_got(b, {0: [o]})
        compare(b, got, want)
    got = _as_got(b, want)
    got["accept_len"][0] = 0
    got["tokens"][0] = [2, -1]                # rejected, but the residual draw never emits 2 here
    with pytest.raises(AssertionError):
        compare(b, got, want)


def test_eos_stop_outcome_and_counts():
    """A request stopped by its end-of-sequence draft: the stopped result passes, one that
    ignores the stop (emits the draw) fails, and the tally sums the per-position counts."""
    import dataclasses
    x = np.zeros((4, 8), np.float32)
    for j, t in enumerate([5, 7, 2, 6]):
        x[j, t] = 3.0
    b = one_request(x, np.full((3, 8), 1 / 8), [5, 7, 2], T=0.0, want_logprobs=True, n_top=2)
    b = dataclasses.replace(b, eos_ids=np.array([7], np.int32))
    want = O.outcomes_batch(b)
    got = _as_got(b, want)
    got["stopped"] = np.array([1], np.int32)
    t = compare(b, got, want)
    assert t.stopped == 1 and t.attempted.tolist() == [1, 1, 0] and t.accepted.tolist() == [1, 1, 0]
    bad = {k: v.copy() for k, v in got.items()}
    bad["tokens"][0, 2] = 2
    with pytest.raises(AssertionError):
        compare(b, bad, want)
    bad = {k: v.copy() for k, v in got.items()}
    bad["stopped"][0] = 0
    with pytest.raises(AssertionError):
        compare(b, bad, want)
    bad = {k: v.copy() for k, v in got.items()}
    bad["logprobs"][0, 2] = -1.0
    with pytest.raises(AssertionError):
        compare(b, bad, want)
