"""Parity of the CUDA path (through the C ABI) with the float64 oracle, on a GB300."""
import numpy as np
import pytest

from oracle import epilogue as O
from tests._compare import compare
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


def _run(runner, batch, requests=None):
    call = runner(batch)
    call.run()
    got = call.results()
    want = O.verify_batch(batch, requests)
    ex, fr = compare(batch, got, want)
    valid = sum(1 for r in want.values() if r.status == 0)
    assert ex >= valid - max(1, valid // 4), f"only {ex} of {valid} requests compared exactly ({fr} fragile)"
    return got, ex, fr


@pytest.mark.parametrize("name", ["b1k2v4096", "b1k2v4096_greedy", "b1k4v151936", "b4k8v151936_mixed"])
def test_small_workloads(runner, name):
    batch = configs.build(name)
    _, ex, fr = _run(runner, batch)
    assert ex + fr == batch.B and ex >= batch.B - 1


def test_b64k8_reduced(runner):
    batch = configs.build("b64k8v262144", B=4)
    _, ex, fr = _run(runner, batch)
    assert ex >= 3


def test_mixed18_all_combinations(runner):
    # every (T, top_k, top_p) combination of the mixed workload, penalties on the first half
    batch = configs.build("b256k16v262144_mixed", B=18)
    _, ex, fr = _run(runner, batch)
    assert ex >= 15


@pytest.mark.parametrize("dtype,V", [("fp32", 1003), ("bf16", 5001), ("bf16", 24577), ("fp32", 12289), ("bf16", 17)])
def test_ragged_vocab(runner, dtype, V):
    rows = [row_params(0.9, 10, 0.9, 0.3, 0.2, 3), row_params(0.0, 0, 1.0, 0.3, 0.2, 3),
            row_params(1.0, 0, 1.0, 0.0, 0.0, 2), row_params(0.7, 0, 0.8, 0.0, 0.0, 3)]
    batch = make_batch(B=4, K_max=3, V=V, logits_dtype=dtype, rows=rows, seed=V, philox_seed=V,
                       history_len=min(40, V), want_logprobs=True, n_top_logprobs=min(5, V))
    _run(runner, batch)


def test_tie_heavy_and_all_equal(runner):
    rows = [row_params(0.8, 20, 0.95, 0.0, 0.0, 4), row_params(0.0, 0, 1.0, 0.0, 0.0, 4),
            row_params(1.0, 5, 1.0, 0.0, 0.0, 4), row_params(0.6, 0, 0.5, 0.0, 0.0, 4)]
    batch = make_batch(B=4, K_max=4, V=30000, logits_dtype="bf16", rows=rows, seed=3, philox_seed=3,
                       x_quant=0.5, want_logprobs=True, n_top_logprobs=8)
    _run(runner, batch)
    flat = make_batch(B=4, K_max=4, V=30000, logits_dtype="bf16", rows=rows, seed=4, philox_seed=4,
                      x_sigma=0.0, want_logprobs=True, n_top_logprobs=8)
    _run(runner, flat)


def test_large_top_k_and_top_k_one(runner):
    rows = [row_params(0.9, 300, 0.9, 0.2, 0.1, 3), row_params(0.9, 1, 1.0, 0.0, 0.0, 3),
            row_params(1.3, 1000, 1.0, 0.0, 0.0, 3), row_params(0.5, 256, 0.99, 0.0, 0.0, 3)]
    batch = make_batch(B=4, K_max=3, V=100000, logits_dtype="bf16", rows=rows, seed=8, philox_seed=8,
                       history_len=500)
    _run(runner, batch)


def test_long_accepts(runner):
    # drafts equal to the target argmax / draft equal to target: deep accepted prefixes
    rows = [row_params(0.0, 0, 1.0, 0.0, 0.0, 8), row_params(0.0, 0, 1.0, 0.5, 0.5, 8)]
    batch = make_batch(B=2, K_max=8, V=50000, logits_dtype="bf16", rows=rows, seed=9, philox_seed=9,
                       draft_mode="argmax", history_len=100)
    got, _, _ = _run(runner, batch)
    assert got["accept_len"][0] == 8
    rows = [row_params(1.0, 0, 1.0, 0.0, 0.0, 6), row_params(1.0, 40, 1.0, 0.0, 0.0, 6)]
    batch = make_batch(B=2, K_max=6, V=20000, logits_dtype="fp32", rows=rows, seed=10, philox_seed=10,
                       draft_mode="copy")
    _run(runner, batch)


def test_sampled_deep_accepts(runner):
    # a greedy drafter (d = argmax q) with a close draft: sampled acceptance runs deep, so the
    # accept test, the draft-prefix penalty counts and residual draws are exercised at j > 0
    rows = [row_params(0.8, 20, 0.9, 0.3, 0.2, 8), row_params(1.0, 0, 1.0, 0.3, 0.2, 8),
            row_params(0.6, 50, 0.95, 0.0, 0.0, 8), row_params(1.0, 64, 1.0, 0.5, 0.5, 8)] * 3
    batch = make_batch(B=12, K_max=8, V=40000, logits_dtype="bf16", rows=rows, seed=21, philox_seed=21,
                       draft_sigma=0.3, draft_mode="q_argmax", history_len=200, want_logprobs=True,
                       n_top_logprobs=4)
    got, ex, fr = _run(runner, batch)
    assert got["accept_len"].max() >= 3


def test_k0_and_repeated_drafts(runner):
    rows = [row_params(0.7, 20, 0.9, 0.4, 0.4, 0), row_params(0.0, 0, 1.0, 0.4, 0.4, 0)]
    batch = make_batch(B=2, K_max=0, V=9000, logits_dtype="bf16", rows=rows, seed=11, philox_seed=11,
                       history_len=50, want_logprobs=True, n_top_logprobs=3)
    _run(runner, batch)
    rows = [row_params(0.0, 0, 1.0, 1.5, 1.0, 5), row_params(0.9, 30, 0.9, 1.5, 1.0, 5)]
    batch = make_batch(B=2, K_max=5, V=3000, logits_dtype="fp32", rows=rows, seed=12, philox_seed=12,
                       history_len=30)
    batch.draft_ids[:, :] = batch.draft_ids[:, :1]          # the same token drafted five times
    _run(runner, batch)


def test_invalid_rows(runner):
    rows = [row_params(-1.0, 0, 1.0, 0, 0, 2), row_params(0.8, 0, 0.0, 0, 0, 2), row_params(0.8, 5, 0.9, 0, 0, 2),
            row_params(0.8, 5, 0.9, 0, 0, 2), row_params(0.8, 5, 0.9, 0, 0, 2), row_params(0.0, 0, 1.0, 0, 0, 2)]
    batch = make_batch(B=6, K_max=2, V=2000, logits_dtype="fp32", rows=rows, seed=13, philox_seed=13,
                       want_logprobs=True)
    batch.draft_ids[2, 1] = 2000                            # out of range
    batch.x[3, 1, 17] = np.nan                              # non-finite logit
    batch.q[4, 0, 5] = -0.1                                 # negative draft probability
    batch.rows["num_drafts"][5] = 3                         # K_b > K_max
    _run(runner, batch)


def test_row_isolation(runner):
    """A request's outputs do not depend on the rest of the batch (mlx-dspark Changelog
    [0.3.0] Added, dynamic batch admission: B=1 bit-exact vs single sequence)."""
    batch = configs.build("b256k16v262144_mixed", B=6)
    call = runner(batch)
    call.run()
    full = call.results()
    from workloads.generate import Batch
    for b in range(batch.B):
        lo, hi = batch.hist_offsets[b], batch.hist_offsets[b + 1]
        one = Batch(B=1, K_max=batch.K_max, V=batch.V, logits_dtype=batch.logits_dtype, x=batch.x[b:b + 1],
                    q=batch.q[b:b + 1], draft_ids=batch.draft_ids[b:b + 1],
                    hist_offsets=np.array([0, hi - lo], np.int32), hist_ids=batch.hist_ids[lo:hi],
                    hist_counts=batch.hist_counts[lo:hi], rows=batch.rows[b:b + 1], uniforms=batch.uniforms[b:b + 1],
                    want_logprobs=batch.want_logprobs, n_top_logprobs=batch.n_top_logprobs)
        c1 = runner(one)
        c1.run()
        r1 = c1.results()
        for k in ("accept_len", "tokens", "logprobs", "top_ids", "top_logprobs", "row_status"):
            assert np.array_equal(r1[k][0], full[k][b]), (b, k)


def test_b64k8_full_size_sampled(runner):
    """The benchmarked workload at full size, in the launch configuration the bench times;
    the oracle checks a sample of requests one by one."""
    batch = configs.build("b64k8v262144")
    call = runner(batch)
    call.run()
    got = call.results()
    want = O.verify_batch(batch, requests=[0, 17, 42, 63])
    ex, fr = compare(batch, got, want)
    assert ex >= 3
    # properties over every request: accepted prefix equals the drafts, one emitted token
    K = batch.K_max
    assert np.all(got["row_status"] == 0)
    for b in range(batch.B):
        a = int(got["accept_len"][b])
        assert 0 <= a <= K
        assert np.array_equal(got["tokens"][b][:a], batch.draft_ids[b][:a])
        assert 0 <= got["tokens"][b][a] < batch.V
        assert np.all(got["top_ids"][b][: a + 1] >= 0)


def test_b256k16_full_size_sampled(runner):
    """The largest workload (B=256, K=16, V=262144, mixed parameters) at full size: the oracle
    checks requests covering all 18 (T, top_k, top_p) combinations and both penalty halves;
    properties are checked on every request."""
    batch = configs.build("b256k16v262144_mixed")
    call = runner(batch)
    call.run()
    got = call.results()
    sample = list(range(18)) + [137, 255]
    want = O.verify_batch(batch, requests=sample)
    ex, fr = compare(batch, got, want)
    assert ex >= len(sample) - max(1, len(sample) // 4), f"only {ex} of {len(sample)} exact ({fr} fragile)"
    assert np.all(got["row_status"] == 0)
    for b in range(batch.B):
        a = int(got["accept_len"][b])
        K = int(batch.rows[b]["num_drafts"])
        assert 0 <= a <= K
        assert np.array_equal(got["tokens"][b][:a], batch.draft_ids[b][:a])
        assert 0 <= got["tokens"][b][a] < batch.V
        assert np.all(got["tokens"][b][a + 1:] == -1)
