"""GPU parity of the options beyond the dense call, through the C ABI, against the oracle:
sparse (one-hot lookup) and reduced-vocabulary drafts, the end-of-sequence stop with the
per-position acceptance counters, penalised logprobs, and the active-row prefix layout.

Every request is compared as in test_parity_gpu.py (tests/_compare.py); the counters are
compared with the sums of the matched oracle outcomes' per-position counts.
"""
import dataclasses

import numpy as np
import pytest

from oracle import epilogue as O
from tests._compare import compare, report
from tests._oracle_pool import workload_outcomes
from workloads import configs
from workloads.generate import make_batch, row_params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def runner():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from sample_verify_epilogue_gb300.runner import EpilogueCall
    return EpilogueCall


def _run(runner, batch, name, want=None, runs=1):
    call = runner(batch, counters=True)
    for _ in range(runs):
        call.run()
    got = call.results()
    if want is None:
        want = O.outcomes_batch(batch)
    tally = compare(batch, got, want)
    assert tally.requests == batch.B
    # the counters are added to by every run
    assert np.array_equal(got["pos_counts"][0], runs * tally.attempted), (got["pos_counts"], tally.attempted)
    assert np.array_equal(got["pos_counts"][1], runs * tally.accepted), (got["pos_counts"], tally.accepted)
    report(name, tally)
    return got, tally


MIX = [row_params(1.0, 0, 1.0, 0.3, 0.2, 4), row_params(0.7, 20, 0.9, 0.0, 0.0, 4),
       row_params(0.0, 0, 1.0, 0.3, 0.2, 4), row_params(1.3, 0, 0.8, 0.0, 0.0, 3),
       row_params(0.9, 300, 1.0, 0.0, 0.0, 4), row_params(1.0, 1, 1.0, 0.0, 0.0, 2)]


@pytest.mark.parametrize("m", [1, 3, 40])
def test_sparse_drafts(runner, m):
    batch = make_batch(B=6, K_max=4, V=151936, logits_dtype="bf16", rows=MIX, seed=40 + m, philox_seed=m,
                       boost_frac=0.3, argmax_frac=0.6, history_len=300, want_logprobs=True, n_top_logprobs=4,
                       q_layout="sparse", q_m=m)
    _run(runner, batch, f"sparse q m={m} V=151936", runs=2)


def test_onehot_full_size(runner):
    name = "b64k8v262144_onehot"
    _run(runner, configs.build(name), name, want=workload_outcomes(name))


@pytest.mark.parametrize("Vd", [1, 5000, 151936])
def test_reduced_vocabulary(runner, Vd):
    batch = make_batch(B=6, K_max=4, V=151936, logits_dtype="bf16", rows=MIX, seed=50, philox_seed=Vd,
                       history_len=300, want_logprobs=True, n_top_logprobs=4, q_layout="reduced",
                       draft_vocab=Vd, subset_boost=2.0)
    _run(runner, batch, f"reduced draft vocabulary Vd={Vd} V=151936")


def test_d2t_full_size(runner):
    name = "b64k8v262144_d2t32000"
    _run(runner, configs.build(name), name, want=workload_outcomes(name))


def test_invalid_draft_layouts(runner):
    base = make_batch(B=6, K_max=4, V=5000, logits_dtype="fp32", rows=MIX, seed=60, q_layout="sparse", q_m=3)
    ids = base.q_ids.copy()
    ids[0, 1, 2] = ids[0, 1, 0]          # a repeated id (request 0, T > 0): bad
    ids[1, 2, 0] = 5000                  # out of range (request 1, T > 0): bad
    ids[2, 0, 0] = -3                    # request 2 is greedy: its draft rows are not read
    ids[3, 3, 1] = ids[3, 3, 0]          # past request 3's 3 drafts: not read
    sp = dataclasses.replace(base, q_ids=ids)
    _run(runner, sp, "invalid sparse rows")
    want = O.outcomes_batch(sp)
    assert [want[b][0].status for b in range(6)] == [O.ROW_BAD_DRAFT, O.ROW_BAD_DRAFT, 0, 0, 0, 0]
    red = make_batch(B=6, K_max=4, V=5000, logits_dtype="fp32", rows=MIX, seed=61, q_layout="reduced",
                     draft_vocab=300)
    d2t = red.d2t.copy()
    d2t[7] = d2t[8] + 1                  # draft ids 7 and 8 both map to target id S[8]
    bad = dataclasses.replace(red, d2t=d2t)
    _run(runner, bad, "colliding d2t")
    st = [O.outcomes_batch(bad)[b][0].status for b in range(6)]
    assert st == [O.ROW_BAD_DRAFT, O.ROW_BAD_DRAFT, 0, O.ROW_BAD_DRAFT, O.ROW_BAD_DRAFT, O.ROW_BAD_DRAFT]
    d2t = red.d2t.copy()
    d2t[-1] = 5000                       # maps past the target vocabulary
    _run(runner, dataclasses.replace(red, d2t=d2t), "out-of-range d2t")


@pytest.mark.parametrize("eos_pos", [0, 1, 3])
def test_eos_stop_and_counters(runner, eos_pos):
    rows = MIX + [row_params(0.0, 0, 1.0, 0.0, 0.0, 4)] * 2
    batch = make_batch(B=8, K_max=4, V=30000, logits_dtype="bf16", rows=rows, seed=70 + eos_pos,
                       philox_seed=eos_pos, boost_frac=0.6, argmax_frac=0.8, draft_mode="q", history_len=100,
                       want_logprobs=True, n_top_logprobs=3, eos_pos=eos_pos)
    got, tally = _run(runner, batch, f"eos at draft {eos_pos}", runs=3)
    assert tally.stopped > 0


def test_eos_stop_full_size_mixed(runner):
    batch = configs.build("b256k16v262144_mixed", B=36)
    batch = dataclasses.replace(batch, eos_ids=batch.draft_ids[:, 1].copy())
    got, tally = _run(runner, batch, "b256k16v262144_mixed B=36, eos = draft 1")
    assert tally.stopped > 0


def test_penalised_logprobs(runner):
    name = "b1k4v151936"
    for B, mode in ((4, "penalised"), (4, "raw")):
        batch = dataclasses.replace(configs.build(name, B=B), want_logprobs=True, n_top_logprobs=20,
                                    logprob_mode=mode)
        _run(runner, batch, f"{name} B={B} logprobs {mode}")


def test_penalised_logprobs_mixed(runner):
    # penalised requests (b < 9) and unpenalised ones in one call; fp32 and a ragged vocabulary
    batch = dataclasses.replace(configs.build("b256k16v262144_mixed", B=18), logprob_mode="penalised")
    _run(runner, batch, "b256k16v262144_mixed B=18 logprobs penalised")
    rows = [row_params(0.8, 0, 1.0, 1.5, 1.0, 3), row_params(0.0, 0, 1.0, 2.0, 2.0, 3)]
    small = make_batch(B=2, K_max=3, V=4099, logits_dtype="fp32", rows=rows, seed=81, history_len=3000,
                       argmax_frac=0.5, want_logprobs=True, n_top_logprobs=20, logprob_mode="penalised")
    _run(runner, small, "fp32 V=4099 heavy history, logprobs penalised")


def test_active_row_prefix_layout(runner):
    """Retired requests leave the batch; the survivors, compacted to a contiguous prefix of the
    same buffers, give bit for bit what they gave in the full-width call (mlx-dspark Changelog,
    [0.3.0] Added: retirement compacts the active rows to a prefix and every pass runs at the
    active width)."""
    torch = pytest.importorskip("torch")
    batch = configs.build("b256k16v262144_mixed", B=24)
    full = runner(batch)
    full.run()
    want = full.results()
    keep = [b for b in range(24) if b not in (2, 5, 11, 17, 23)]
    n = len(keep)
    call = runner(batch)                                      # capacity-sized buffers (24 requests)
    dev = call.x.device
    idx = torch.tensor(keep, device=dev)
    rows = call.rows.view(24, -1)
    # one row-copy per buffer moves the survivors to the front
    for t in (call.x, call.q, call.d, rows, call.u):
        t[:n] = t.index_select(0, idx).clone()
    sub = batch.subset(keep)
    call.counts[0][: n + 1] = torch.from_numpy(sub.hist_offsets.astype(np.int32)).to(dev)
    call.counts[1][: len(sub.hist_ids)] = torch.from_numpy(sub.hist_ids).to(dev)
    call.counts[2][: len(sub.hist_counts)] = torch.from_numpy(sub.hist_counts).to(dev)
    # the call at the active width: prefixes of the same buffers
    call.x, call.q, call.d, call.u = call.x[:n], call.q[:n], call.d[:n], call.u[:n]
    call.rows = rows[:n].reshape(-1)
    call.counts = (call.counts[0][: n + 1], call.counts[1], call.counts[2])
    call.out = {k: v[:n] for k, v in call.out.items()}
    call.row_status = call.row_status[:n]
    call.B = n
    call.run()
    got = call.results()
    for k in ("accept_len", "tokens", "logprobs", "top_ids", "top_logprobs", "row_status"):
        assert np.array_equal(got[k], want[k][keep]), k


def test_host_entry_point_with_options(runner):
    """dspark_verify_sample_host with a sparse layout, eos tokens and counters equals the device call."""
    torch = pytest.importorskip("torch")
    from sample_verify_epilogue_gb300 import binding
    batch = make_batch(B=6, K_max=4, V=30000, logits_dtype="bf16", rows=MIX, seed=90, philox_seed=9,
                       boost_frac=0.5, argmax_frac=0.7, history_len=100, want_logprobs=True, n_top_logprobs=3,
                       q_layout="sparse", q_m=2, eos_pos=1)
    dev = runner(batch, counters=True)
    dev.run()
    want = dev.results()
    B, W, n = batch.B, batch.K_max + 1, 3
    out = {"accept_len": np.zeros(B, np.int32), "tokens": np.zeros((B, W), np.int32),
           "logprobs": np.zeros((B, W), np.float32), "top_ids": np.zeros((B, W, n), np.int32),
           "top_logprobs": np.zeros((B, W, n), np.float32)}
    status = np.zeros(B, np.int32)
    stopped = np.zeros(B, np.int32)
    counts = np.full(2 * batch.K_max, 5, np.uint64)          # added to, not overwritten
    q_ids = np.ascontiguousarray(batch.q_ids)
    eos = np.ascontiguousarray(batch.eos_ids)
    ex = binding.make_extras(q_layout="sparse", q_row_len=2, q_ids=q_ids.ctypes.data, eos_ids=eos.ctypes.data,
                             out_stopped=stopped.ctypes.data, pos_counts=counts.ctypes.data)
    rows = np.ascontiguousarray(batch.rows).view(np.uint8)
    nbytes = binding.dspark_host_workspace_bytes(B, batch.K_max, batch.V, "bf16", n, len(batch.hist_ids), ex)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    binding.dspark_verify_sample_host(
        np.ascontiguousarray(batch.x), np.ascontiguousarray(batch.q), np.ascontiguousarray(batch.draft_ids),
        (batch.hist_offsets, batch.hist_ids, batch.hist_counts), rows, np.ascontiguousarray(batch.uniforms),
        out=out, row_status=status, workspace=ws, logits_dtype="bf16", want_logprobs=True, n_top_logprobs=n,
        extras=ex)
    for k in out:
        assert np.array_equal(out[k], want[k]), k
    assert np.array_equal(stopped, want["stopped"])
    assert np.array_equal(counts.reshape(2, -1).astype(np.int64) - 5, want["pos_counts"])


def test_logprob_threshold_paths(runner):
    """The logprob pass gathers from a top-k row's k-th largest penalised logit only when that
    bounds the n-th largest logit: k >= n and, in raw mode, no negative penalty.  Rows on
    either side of each condition, in both modes; sparse rows at the largest m."""
    rows = [row_params(1.0, 64, 0.95, 0.3, 0.2, 3),      # bound used
            row_params(1.0, 10, 1.0, 0.3, 0.2, 3),       # k < n: searched
            row_params(0.8, 64, 1.0, -0.5, -0.3, 3),     # negative penalties: searched in raw mode
            row_params(0.0, 0, 1.0, 0.4, 0.4, 3),        # greedy: searched
            row_params(1.2, 0, 0.7, 0.0, 0.0, 3),        # no top-k: searched
            row_params(0.9, 300, 1.0, 0.0, 0.0, 3)]      # k > 256 (block finalize): searched
    for mode in ("raw", "penalised"):
        batch = make_batch(B=6, K_max=3, V=151936, logits_dtype="bf16", rows=rows, seed=101, philox_seed=7,
                           boost_frac=0.3, argmax_frac=0.5, history_len=2048, want_logprobs=True,
                           n_top_logprobs=20, logprob_mode=mode)
        _run(runner, batch, f"logprob threshold paths ({mode})")
    sp = make_batch(B=6, K_max=3, V=151936, logits_dtype="bf16", rows=rows, seed=102, philox_seed=8,
                    argmax_frac=0.5, history_len=500, want_logprobs=True, n_top_logprobs=20,
                    q_layout="sparse", q_m=256)
    _run(runner, sp, "sparse q m=256")
