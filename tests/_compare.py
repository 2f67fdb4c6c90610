"""Element-by-element comparison of the CUDA path's outputs with the oracle's outcomes.

The oracle (``oracle.epilogue.outcomes``) gives, per request, every outcome that is correct:
the float64 one, plus the other side of each near-tie accept test or nucleus boundary, each
with the emitted tokens its draw admits (a near-tie draw admits the tokens whose intervals
reach within 1e-6 of u).  A request of the CUDA path is correct iff its accept length and
tokens are exactly one of those outcomes; its logprobs and top-logprob lists are then
checked at every emitted position: ids bit for bit, values within LOGPROB_TOL.
Nothing is exempt: every request of every batch is compared.  A request that stopped on its
end-of-sequence token emits positions 0..accept_len-1 only (its token at accept_len is -1);
the per-position acceptance counts of the matched outcomes are summed into the tally, for
comparison with the device's counters.
"""
from __future__ import annotations

from collections import Counter
from dataclasses import dataclass, field

import numpy as np

LOGPROB_TOL = 1e-4   # absolute, from the logprob agreement the pages quote (~1e-6) with fp32 headroom

REPORT = []          # one line per compared batch, printed at the end of the test session


@dataclass
class Tally:
    """Counts of one compared batch."""
    requests: int = 0          # requests compared
    single: int = 0            # requests with one correct outcome and one admissible token
    near_tie_requests: int = 0 # requests with at least one near-tie decision
    decisions: int = 0         # floating-point decisions the oracle took
    near_ties: Counter = field(default_factory=Counter)   # near-tie decisions by kind
    off_float64: int = 0       # requests whose GPU result is not the float64 outcome itself
    attempted: np.ndarray = None   # per draft position: requests that verified it (matched outcomes)
    accepted: np.ndarray = None    # per draft position: requests that accepted it
    stopped: int = 0               # requests stopped by their end-of-sequence token

    def line(self, name):
        kinds = ", ".join(f"{k} {v}" for k, v in sorted(self.near_ties.items())) or "none"
        stop = f"; {self.stopped} stopped at eos" if self.stopped else ""
        return (f"{name}: {self.requests} requests compared, {self.single} with a single correct result; "
                f"near-tie decisions {sum(self.near_ties.values())} of {self.decisions} ({kinds}) in "
                f"{self.near_tie_requests} requests; {self.off_float64} GPU results on the other side of a near tie"
                f"{stop}")


def _close(got, want, tol):
    """Element-wise: equal (both -inf included) or within tol."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return (got == want) | (np.abs(got - np.where(np.isfinite(want), want, 0.0)) <= tol) & np.isfinite(want)


def _matching(outs, a_g, toks):
    for o in outs:
        if o.accept_len != a_g or not np.array_equal(toks[:a_g], o.tokens[:a_g]):
            continue
        hit = np.nonzero(o.admissible == toks[a_g])[0]
        if hit.size:
            return o, int(hit[0])
    return None, -1


def compare(batch, got, want, lp_tol=LOGPROB_TOL, tally=None):
    """got: results() of an EpilogueCall; want: {b: oracle outcomes of request b, the
    float64 one first} (``oracle.epilogue.outcomes``).  Asserts on the first mismatch and
    returns the tally."""
    tally = tally if tally is not None else Tally()
    W = batch.K_max + 1
    if tally.attempted is None:
        tally.attempted = np.zeros(batch.K_max, np.int64)
        tally.accepted = np.zeros(batch.K_max, np.int64)
    for b, outs in want.items():
        base = outs[0]
        st = int(got["row_status"][b])
        assert st == base.status, f"request {b}: status {st} != oracle {base.status}"
        tally.requests += 1
        if base.status != 0:
            assert int(got["accept_len"][b]) == -1
            assert np.all(got["tokens"][b] == -1)
            if "logprobs" in got:
                assert np.all(np.isneginf(got["logprobs"][b]))
            if "top_ids" in got:
                assert np.all(got["top_ids"][b] == -1)
            tally.single += 1
            continue
        a_g = int(got["accept_len"][b])
        toks = got["tokens"][b]
        assert np.all(toks[a_g + 1:] == -1), f"request {b}: tokens past the emitted one: {toks}"
        o, ia = _matching(outs, a_g, toks)
        assert o is not None, (
            f"request {b}: GPU accept_len {a_g}, tokens {toks.tolist()} is none of the oracle's outcomes "
            + "; ".join(f"(a={x.accept_len}, tokens={x.tokens.tolist()}, admissible {x.admissible[:8].tolist()}, "
                        f"near ties {x.near_ties()})" for x in outs))
        ties = base.near_ties()
        tally.decisions += len(base.decisions)
        tally.near_ties.update(ties)
        tally.near_tie_requests += bool(ties)
        tally.single += len(outs) == 1 and base.admissible.size == 1
        tally.off_float64 += not (o is base and ia == 0)
        tally.attempted += o.attempted
        tally.accepted += o.accepted
        tally.stopped += bool(o.stopped)
        if "stopped" in got:
            assert bool(got["stopped"][b]) == o.stopped, f"request {b}: stopped {got['stopped'][b]} != {o.stopped}"
        n_em = a_g if o.stopped else a_g + 1              # emitted positions
        if "logprobs" in got:
            lp = got["logprobs"][b]
            want_lp = np.array(o.logprobs[:n_em])
            if not o.stopped:
                want_lp[a_g] = o.admissible_logprobs[ia]
            assert np.all(_close(lp[:n_em], want_lp, lp_tol)), \
                f"request {b}: logprobs {lp[:n_em]} != oracle {want_lp}"
            assert np.all(np.isneginf(lp[n_em:W]))
        if "top_ids" in got:
            ti, tl = got["top_ids"][b], got["top_logprobs"][b]
            assert np.array_equal(ti[:n_em], o.top_ids[:n_em]), \
                f"request {b}: top ids {ti[:n_em]} != oracle {o.top_ids[:n_em]}"
            assert np.all(_close(tl[:n_em], o.top_logprobs[:n_em], lp_tol)), \
                f"request {b}: top logprobs {tl[:n_em]} != oracle {o.top_logprobs[:n_em]}"
            assert np.all(ti[n_em:] == -1) and np.all(np.isneginf(tl[n_em:]))
    return tally


def report(name, tally):
    """Record a batch's tally for the end-of-session summary."""
    REPORT.append(tally.line(name))
    return tally
