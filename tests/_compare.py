"""Element-by-element comparison of the CUDA path's outputs with the oracle's."""
from __future__ import annotations

import numpy as np

LOGPROB_TOL = 1e-4   # absolute, from the logprob agreement the pages quote (~1e-6) with fp32 headroom


def compare(batch, got, want, lp_tol=LOGPROB_TOL):
    """got: results() of an EpilogueCall; want: {b: oracle RequestResult}.

    Non-fragile requests must match bit for bit on status, accept length, tokens and
    top-logprob ids, and within lp_tol on logprobs.  Fragile requests (a floating-point
    decision within the oracle's margin) must still produce a valid output.
    Returns (exact, fragile) request counts."""
    exact = fragile = 0
    W = batch.K_max + 1
    for b, r in want.items():
        st = int(got["row_status"][b])
        assert st == r.status, f"request {b}: status {st} != oracle {r.status}"
        if r.status != 0:
            assert int(got["accept_len"][b]) == -1
            assert np.all(got["tokens"][b] == -1)
            continue
        a_g = int(got["accept_len"][b])
        K = int(batch.rows["num_drafts"][b])
        if r.fragile:
            fragile += 1
            assert 0 <= a_g <= K
            assert np.array_equal(got["tokens"][b][:a_g], batch.draft_ids[b][:a_g])
            assert 0 <= got["tokens"][b][a_g] < batch.V
            assert np.all(got["tokens"][b][a_g + 1:] == -1)
            continue
        exact += 1
        assert a_g == r.accept_len, f"request {b}: accept_len {a_g} != oracle {r.accept_len} (margin {r.min_margin})"
        assert np.array_equal(got["tokens"][b], r.tokens), f"request {b}: tokens {got['tokens'][b]} != {r.tokens}"
        a = r.accept_len
        if "logprobs" in got:
            lp = got["logprobs"][b]
            assert np.all(np.abs(lp[: a + 1] - r.logprobs[: a + 1]) <= lp_tol), (b, lp[: a + 1], r.logprobs[: a + 1])
            assert np.all(np.isneginf(lp[a + 1: W]))
        if "top_ids" in got:
            assert np.array_equal(got["top_ids"][b][: a + 1], r.top_ids[: a + 1]), (b, got["top_ids"][b][: a + 1], r.top_ids[: a + 1])
            assert np.all(np.abs(got["top_logprobs"][b][: a + 1] - r.top_logprobs[: a + 1]) <= lp_tol)
            assert np.all(got["top_ids"][b][a + 1:] == -1)
    return exact, fragile
