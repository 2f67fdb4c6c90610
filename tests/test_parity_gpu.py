"""Parity of the CUDA path (through the C ABI) with the float64 oracle, on a GB300.

Every request of every batch is compared with the oracle's outcomes (tests/_compare.py):
accept length and tokens exactly one of the correct outcomes, logprobs and top-logprob
lists at every emitted position.  The near-tie decisions of each batch are counted and
printed in the session summary.
"""
import numpy as np
import pytest

from oracle import epilogue as O
from tests._compare import Tally, compare, report
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


def _run(runner, batch, name, want=None):
    call = runner(batch)
    call.run()
    got = call.results()
    if want is None:
        want = O.outcomes_batch(batch)
    tally = compare(batch, got, want)
    assert tally.requests == batch.B
    report(name, tally)
    return got, tally


@pytest.mark.parametrize("name", ["b1k2v4096", "b1k2v4096_greedy", "b1k4v151936", "b4k8v151936_mixed"])
def test_small_workloads(runner, name):
    _run(runner, configs.build(name), name)


def test_mixed18_all_combinations(runner):
    # every (T, top_k, top_p) combination of the mixed workload, penalties on the first half
    _run(runner, configs.build("b256k16v262144_mixed", B=18), "b256k16v262144_mixed B=18")


def test_signed_zero_draft_probabilities(runner):
    """Draft rows holding -0.0 (a valid zero probability) in top-k and full rows, on both sides
    of a tile: the streaming pass scans top-k draft rows on raw bit patterns, where -0.0 has
    the sign bit set, and must fall back to the float maximum for those tiles."""
    rows = [row_params(1.0, 20, 0.9, 0.0, 0.0, 3), row_params(0.8, 64, 1.0, 0.0, 0.0, 3),
            row_params(1.0, 0, 1.0, 0.0, 0.0, 3), row_params(0.7, 0, 0.8, 0.0, 0.0, 3)]
    batch = make_batch(B=4, K_max=3, V=30011, logits_dtype="bf16", rows=rows, seed=303, philox_seed=303,
                       x_sigma=1.0, argmax_frac=0.5, history_len=0)
    rng = np.random.default_rng(303)
    for b in range(4):
        for i in range(3):
            z = rng.choice(batch.V, size=500, replace=False)
            z = z[z != batch.draft_ids[b, i]]
            batch.q[b, i, z] = -0.0
    assert np.signbit(batch.q).sum() > 0
    _run(runner, batch, "signed-zero draft probabilities")


def test_list_draw_lengths(runner):
    """Kept lists of every length class of the draw from a truncated row: one entry, the
    one-warp path (up to 64 entries, both sides of a half-warp), and the block path above it;
    flat logits so that drafts are often rejected and the residual is drawn from."""
    ks = (1, 2, 31, 33, 63, 64, 65, 128, 1000)
    rows = [row_params(1.0, ks[b % len(ks)], 1.0 if b < len(ks) else 0.9, 0.0, 0.0, 4) for b in range(2 * len(ks))]
    batch = make_batch(B=len(rows), K_max=4, V=20000, logits_dtype="bf16", rows=rows, seed=65, philox_seed=65,
                       x_sigma=0.4, argmax_frac=0.5, history_len=0)
    _run(runner, batch, "kept-list lengths")


@pytest.mark.parametrize("dtype,V", [("fp32", 1003), ("bf16", 5001), ("bf16", 24577), ("fp32", 12289), ("bf16", 17)])
def test_ragged_vocab(runner, dtype, V):
    rows = [row_params(0.9, 10, 0.9, 0.3, 0.2, 3), row_params(0.0, 0, 1.0, 0.3, 0.2, 3),
            row_params(1.0, 0, 1.0, 0.0, 0.0, 2), row_params(0.7, 0, 0.8, 0.0, 0.0, 3)]
    batch = make_batch(B=4, K_max=3, V=V, logits_dtype=dtype, rows=rows, seed=V, philox_seed=V,
                       history_len=min(40, V), want_logprobs=True, n_top_logprobs=min(5, V))
    _run(runner, batch, f"ragged {dtype} V={V}")


def test_tie_heavy_and_all_equal(runner):
    rows = [row_params(0.8, 20, 0.95, 0.0, 0.0, 4), row_params(0.0, 0, 1.0, 0.0, 0.0, 4),
            row_params(1.0, 5, 1.0, 0.0, 0.0, 4), row_params(0.6, 0, 0.5, 0.0, 0.0, 4)]
    batch = make_batch(B=4, K_max=4, V=30000, logits_dtype="bf16", rows=rows, seed=3, philox_seed=3,
                       x_quant=0.5, want_logprobs=True, n_top_logprobs=8)
    _run(runner, batch, "tie-heavy V=30000")
    flat = make_batch(B=4, K_max=4, V=30000, logits_dtype="bf16", rows=rows, seed=4, philox_seed=4,
                      x_sigma=0.0, want_logprobs=True, n_top_logprobs=8)
    _run(runner, flat, "all-equal V=30000")


def test_large_top_k_and_top_k_one(runner):
    rows = [row_params(0.9, 300, 0.9, 0.2, 0.1, 3), row_params(0.9, 1, 1.0, 0.0, 0.0, 3),
            row_params(1.3, 1000, 1.0, 0.0, 0.0, 3), row_params(0.5, 256, 0.99, 0.0, 0.0, 3)]
    batch = make_batch(B=4, K_max=3, V=100000, logits_dtype="bf16", rows=rows, seed=8, philox_seed=8,
                       history_len=500)
    _run(runner, batch, "top_k 300/1/1000/256 V=100000")


def test_long_accepts(runner):
    # drafts equal to the target argmax / draft equal to target: deep accepted prefixes
    rows = [row_params(0.0, 0, 1.0, 0.0, 0.0, 8), row_params(0.0, 0, 1.0, 0.5, 0.5, 8)]
    batch = make_batch(B=2, K_max=8, V=50000, logits_dtype="bf16", rows=rows, seed=9, philox_seed=9,
                       draft_mode="argmax", history_len=100)
    got, _ = _run(runner, batch, "argmax drafts K=8")
    assert got["accept_len"][0] == 8
    rows = [row_params(1.0, 0, 1.0, 0.0, 0.0, 6), row_params(1.0, 40, 1.0, 0.0, 0.0, 6)]
    batch = make_batch(B=2, K_max=6, V=20000, logits_dtype="fp32", rows=rows, seed=10, philox_seed=10,
                       draft_mode="copy")
    _run(runner, batch, "draft == target K=6")


def test_sampled_deep_accepts(runner):
    # a greedy drafter (d = argmax q) with a close draft: sampled acceptance runs deep, so the
    # accept test, the draft-prefix penalty counts and residual draws are exercised at j > 0
    rows = [row_params(0.8, 20, 0.9, 0.3, 0.2, 8), row_params(1.0, 0, 1.0, 0.3, 0.2, 8),
            row_params(0.6, 50, 0.95, 0.0, 0.0, 8), row_params(1.0, 64, 1.0, 0.5, 0.5, 8)] * 3
    batch = make_batch(B=12, K_max=8, V=40000, logits_dtype="bf16", rows=rows, seed=21, philox_seed=21,
                       draft_sigma=0.3, draft_mode="q_argmax", history_len=200, want_logprobs=True,
                       n_top_logprobs=4)
    got, _ = _run(runner, batch, "greedy drafter K=8")
    assert got["accept_len"].max() >= 3


def _sequential_greedy_drafts(batch, b, K):
    """Drafts equal to sequential penalised greedy decoding of request b (oracle functions):
    every one of them is accepted."""
    x = batch.x_f32(b)
    r = batch.rows[b]
    hid, hc = batch.history(b)
    seq = []
    for j in range(K):
        c = O.count_vector(batch.V, hid, hc, seq)
        seq.append(int(np.argmax(O.penalised_logits(x[j], c, r["presence_penalty"], r["frequency_penalty"]))))
    return seq


def test_k64_deep_accepts(runner):
    """K_max = 64, the largest the ABI takes: greedy requests whose drafts are the sequential
    penalised greedy decode over a small vocabulary (tokens repeat, so the draft-prefix counts
    at positions j >= 32 matter), and sampled requests with draft == target."""
    V, K = 48, 64
    rows = [row_params(0.0, 0, 1.0, 0.6, 0.4, K), row_params(0.0, 0, 1.0, 0.05, 0.02, K),
            row_params(1.0, 0, 1.0, 0.0, 0.0, K), row_params(0.0, 0, 1.0, 0.0, 0.0, 40)]
    batch = make_batch(B=4, K_max=K, V=V, logits_dtype="fp32", rows=rows, seed=64, philox_seed=64,
                       x_sigma=0.5, draft_mode="copy", history_len=30, want_logprobs=True, n_top_logprobs=6)
    for b in (0, 1):
        batch.draft_ids[b, :] = _sequential_greedy_drafts(batch, b, K)
    got, _ = _run(runner, batch, "K=64 V=48")
    assert got["accept_len"][0] == K and got["accept_len"][1] == K
    assert got["accept_len"][2] >= 32


def test_max_batch_small_vocab(runner):
    """B = 2048, the largest the ABI takes, every parameter combination, small vocabulary."""
    B, V = 2048, 96
    Ts, ks, ps = (0.0, 0.6, 1.0), (0, 5, 20), (0.9, 1.0)
    rows = [row_params(Ts[c // 6], ks[(c // 2) % 3], ps[c % 2], 0.2 * (b % 2), 0.1 * (b % 3), b % 4)
            for b in range(B) for c in [b % 18]]
    batch = make_batch(B=B, K_max=3, V=V, logits_dtype="bf16", rows=rows, seed=2048, philox_seed=2048,
                       x_sigma=1.5, history_len=8, want_logprobs=True, n_top_logprobs=3)
    _run(runner, batch, "B=2048 V=96")


def test_k0_and_repeated_drafts(runner):
    rows = [row_params(0.7, 20, 0.9, 0.4, 0.4, 0), row_params(0.0, 0, 1.0, 0.4, 0.4, 0)]
    batch = make_batch(B=2, K_max=0, V=9000, logits_dtype="bf16", rows=rows, seed=11, philox_seed=11,
                       history_len=50, want_logprobs=True, n_top_logprobs=3)
    _run(runner, batch, "K=0")
    rows = [row_params(0.0, 0, 1.0, 1.5, 1.0, 5), row_params(0.9, 30, 0.9, 1.5, 1.0, 5)]
    batch = make_batch(B=2, K_max=5, V=3000, logits_dtype="fp32", rows=rows, seed=12, philox_seed=12,
                       history_len=30)
    batch.draft_ids[:, :] = batch.draft_ids[:, :1]          # the same token drafted five times
    _run(runner, batch, "repeated drafts")


def test_invalid_rows(runner):
    rows = [row_params(-1.0, 0, 1.0, 0, 0, 2), row_params(0.8, 0, 0.0, 0, 0, 2), row_params(0.8, 5, 0.9, 0, 0, 2),
            row_params(0.8, 5, 0.9, 0, 0, 2), row_params(0.8, 5, 0.9, 0, 0, 2), row_params(0.0, 0, 1.0, 0, 0, 2)]
    batch = make_batch(B=6, K_max=2, V=2000, logits_dtype="fp32", rows=rows, seed=13, philox_seed=13,
                       want_logprobs=True)
    batch.draft_ids[2, 1] = 2000                            # out of range
    batch.x[3, 1, 17] = np.nan                              # non-finite logit
    batch.q[4, 0, 5] = -0.1                                 # negative draft probability
    batch.rows["num_drafts"][5] = 3                         # K_b > K_max
    _run(runner, batch, "invalid rows")


def test_row_isolation(runner):
    """A request's outputs do not depend on the rest of the batch (mlx-dspark Changelog
    [0.3.0] Added, dynamic batch admission: B=1 bit-exact vs single sequence)."""
    batch = configs.build("b256k16v262144_mixed", B=6)
    call = runner(batch)
    call.run()
    full = call.results()
    for b in range(batch.B):
        one = configs.build("b256k16v262144_mixed", B=6, requests=[b])
        c1 = runner(one)
        c1.run()
        r1 = c1.results()
        for k in ("accept_len", "tokens", "logprobs", "top_ids", "top_logprobs", "row_status"):
            assert np.array_equal(r1[k][0], full[k][b]), (b, k)


def _full_size(runner, name):
    """A workload at full size, in the launch configuration the bench times; the oracle
    (all host cores) gives the outcomes of every request."""
    batch = configs.build(name)
    call = runner(batch)
    call.run()
    got = call.results()
    del call
    want = workload_outcomes(name)
    tally = compare(batch, got, want)
    assert tally.requests == batch.B
    report(f"{name} (full size)", tally)
    return got


def test_b64k8_full_size(runner):
    got = _full_size(runner, "b64k8v262144")
    assert np.all(got["row_status"] == 0)


def test_b256k16_full_size(runner):
    got = _full_size(runner, "b256k16v262144_mixed")
    assert np.all(got["row_status"] == 0)


def test_masked_logits(runner):
    """Logits of -inf are tokens of probability zero (masked vocabulary): 30% of the tokens
    masked in half the requests, and a request whose rows keep only three finite logits (its
    top_logprobs lists run into the masked tokens)."""
    rows = [row_params(1.0, 0, 1.0, 0.2, 0.1, 3), row_params(0.7, 20, 0.9, 0.0, 0.0, 3),
            row_params(0.0, 0, 1.0, 0.3, 0.3, 3), row_params(1.0, 5, 1.0, 0.0, 0.0, 3),
            row_params(0.9, 0, 0.8, 0.0, 0.0, 3), row_params(0.0, 0, 1.0, 0.0, 0.0, 3)]
    batch = make_batch(B=6, K_max=3, V=5000, logits_dtype="bf16", rows=rows, seed=31, philox_seed=31,
                       history_len=40, want_logprobs=True, n_top_logprobs=5)
    rng = np.random.default_rng(31)
    ninf = np.uint16(0xFF80)                                # bf16 -inf
    for b in (0, 1, 2):
        mask = rng.random(batch.V) < 0.3
        batch.x[b][:, mask] = ninf
    keep = np.array([7, 1234, 4999])
    row = np.full(batch.V, ninf, np.uint16)
    batch.x[5][:, :] = row
    batch.x[5][:, keep] = batch.x[4][:, keep]
    _run(runner, batch, "masked logits V=5000")


def test_expired_waits_report_internal(runner):
    """A test build whose streaming-pass waits all count as expired: every valid request reports
    DSPARK_ROW_INTERNAL (an invalid one keeps its own bits too), with no output but the error
    padding, and the GPU context stays usable (the normal build then matches the oracle)."""
    from sample_verify_epilogue_gb300 import binding
    from sample_verify_epilogue_gb300.build import build_variant
    lib = binding.open_library(build_variant("expired_waits", ["-DDSPARK_TEST_EXPIRED_WAITS"], ["stream_stats.cu"]))
    batch = configs.build("b256k16v262144_mixed", B=18)
    batch.rows["temperature"][4] = -1.0                    # an invalid request
    call = runner(batch)
    call.run(lib=lib)
    got = call.results()
    st = got["row_status"]
    assert np.all(st & 16), st
    assert st[4] & 1
    assert np.all(got["accept_len"] == -1) and np.all(got["tokens"] == -1)
    assert np.all(np.isneginf(got["logprobs"])) and np.all(got["top_ids"] == -1)
    call.run()
    want = O.outcomes_batch(batch)
    report("after expired waits (b256k16v262144_mixed B=18)", compare(batch, call.results(), want))
