"""The five workloads of the batched verify-and-sample epilogue, plus small variants.

Each workload is named by what it is: batch B, drafts K, vocabulary V, logit dtype
and sampling mix.  The vocabulary sizes stand in for the Qwen3-class (151,936) and
Gemma-class (262,144) vocabularies the mlx-dspark pages sample over (changelog
v0.20.2 "Changed": grouped-select sampling over 150k-262k vocabularies).  No model,
dataset or weights are involved: all inputs are seeded synthetic arrays.
"""
from __future__ import annotations

import numpy as np

from .generate import make_batch, row_params

WORKLOADS = ("b1k2v4096", "b1k2v4096_greedy", "b1k4v151936", "b4k8v151936_mixed",
             "b64k8v262144", "b256k16v262144_mixed", "b64k8v262144_onehot", "b64k8v262144_d2t32000")

DESCRIPTIONS = {
    "b1k2v4096": "B=1 K=2 V=4096 fp32 logits N(0,2^2), draft = target + N(0,0.5^2), T=0.7 top_k=20 top_p=0.95",
    "b1k2v4096_greedy": "as b1k2v4096 with T=0 (greedy)",
    "b1k4v151936": "B=1 K=4 V=151936 bf16 N(0,3^2) with 5% of verify rows' argmax +8, draft = target + N(0,0.7^2), "
                   "T=0.6 top_k=20 top_p=0.95, presence 0.5 / frequency 0.3 over a 2048-token Zipf(1.1) history",
    "b4k8v151936_mixed": "B=4 per-row K in {2..8} V=151936 bf16 as b1k4v151936; rows greedy / T=1 top_k=0 top_p=1 / "
                         "T=0.7 top_k=50 / greedy; 30% of draft tokens forced to the target argmax",
    "b64k8v262144": "B=64 K=8 V=262144 bf16 N(0,3^2), fp32 q from draft = target + N(0,1), T=1 top_k=64 top_p=0.95, "
                    "presence/frequency 0.2/0.2 over 4096-token Zipf(1.1) histories, top_logprobs=20",
    "b256k16v262144_mixed": "B=256 K=16 V=262144 bf16 as b64k8v262144; (T, top_k, top_p) = combination b mod 18 of "
                            "{0,0.6,1}x{0,20,64}x{0.9,1}; penalties 0.2/0.2 on requests b<128; top_logprobs=5",
    "b64k8v262144_onehot": "as b64k8v262144 with prompt-lookup drafts: a one-hot proposal (sparse q, m=1) per "
                           "position; 30% of verify rows' argmax +8, 70% of drafts are the target argmax",
    "b64k8v262144_d2t32000": "as b64k8v262144 with a reduced draft vocabulary of 32000 ids (a seeded ascending "
                             "subset, d2t offsets) from which the drafts are drawn; target logits of those "
                             "ids +2 (the frequent tokens)",
}


def _mixed18(B, K):
    Ts, ks, ps = (0.0, 0.6, 1.0), (0, 20, 64), (0.9, 1.0)
    rows = []
    for b in range(B):
        c = b % 18
        pen = 0.2 if b < B // 2 else 0.0
        rows.append(row_params(Ts[c // 6], ks[(c // 2) % 3], ps[c % 2], pen, pen, K))
    return rows


DEFAULT_B = {"b1k2v4096": 1, "b1k2v4096_greedy": 1, "b1k4v151936": 1, "b4k8v151936_mixed": 4,
             "b64k8v262144": 64, "b256k16v262144_mixed": 256, "b64k8v262144_onehot": 64,
             "b64k8v262144_d2t32000": 64}


def build_size(name: str, B=None) -> int:
    """Number of requests ``build(name, B=B)`` makes."""
    return B or DEFAULT_B[name]


def build(name: str, *, B=None, requests=None):
    """Build a workload by name.  ``B`` overrides the batch size (for bounded samples);
    ``requests`` builds only those requests of the batch (each identical to the same request
    of the whole batch)."""
    i = WORKLOADS.index(name)
    if name in ("b1k2v4096", "b1k2v4096_greedy"):
        T = 0.0 if name.endswith("greedy") else 0.7
        Bn = B or 1
        return make_batch(B=Bn, K_max=2, V=4096, logits_dtype="fp32",
                          rows=[row_params(T, 20, 0.95, 0, 0, 2)] * Bn, seed=1000, philox_seed=0,
                          x_sigma=2.0, draft_sigma=0.5, want_logprobs=False, name=name, requests=requests)
    if name == "b1k4v151936":
        Bn = B or 1
        return make_batch(B=Bn, K_max=4, V=151936, logits_dtype="bf16",
                          rows=[row_params(0.6, 20, 0.95, 0.5, 0.3, 4)] * Bn, seed=1000 + i, philox_seed=i,
                          x_sigma=3.0, draft_sigma=0.7, boost_frac=0.05, history_len=2048, name=name,
                          requests=requests)
    if name == "b4k8v151936_mixed":
        Bn = B or 4
        rng = np.random.default_rng(2000 + i)
        Ks = rng.integers(2, 9, size=Bn)
        kinds = [(0.0, 0, 1.0), (1.0, 0, 1.0), (0.7, 50, 1.0), (0.0, 0, 1.0)]
        rows = [row_params(*kinds[b % 4], 0.0, 0.0, int(Ks[b])) for b in range(Bn)]
        return make_batch(B=Bn, K_max=8, V=151936, logits_dtype="bf16", rows=rows,
                          seed=1000 + i, philox_seed=i, x_sigma=3.0, draft_sigma=0.7, boost_frac=0.05,
                          argmax_frac=0.3, name=name, requests=requests)
    if name == "b64k8v262144":
        Bn = B or 64
        return make_batch(B=Bn, K_max=8, V=262144, logits_dtype="bf16",
                          rows=[row_params(1.0, 64, 0.95, 0.2, 0.2, 8)] * Bn, seed=1000 + i, philox_seed=i,
                          x_sigma=3.0, draft_sigma=1.0, history_len=4096, want_logprobs=True,
                          n_top_logprobs=20, name=name, requests=requests)
    if name == "b256k16v262144_mixed":
        Bn = B or 256
        return make_batch(B=Bn, K_max=16, V=262144, logits_dtype="bf16", rows=_mixed18(Bn, 16),
                          seed=1000 + i, philox_seed=i, x_sigma=3.0, draft_sigma=1.0, history_len=4096,
                          want_logprobs=True, n_top_logprobs=5, name=name, requests=requests)
    if name == "b64k8v262144_onehot":
        Bn = B or 64
        return make_batch(B=Bn, K_max=8, V=262144, logits_dtype="bf16",
                          rows=[row_params(1.0, 64, 0.95, 0.2, 0.2, 8)] * Bn, seed=1000 + i, philox_seed=i,
                          x_sigma=3.0, draft_sigma=1.0, boost_frac=0.3, argmax_frac=0.7, history_len=4096,
                          want_logprobs=True, n_top_logprobs=20, name=name, requests=requests,
                          q_layout="sparse", q_m=1)
    if name == "b64k8v262144_d2t32000":
        Bn = B or 64
        return make_batch(B=Bn, K_max=8, V=262144, logits_dtype="bf16",
                          rows=[row_params(1.0, 64, 0.95, 0.2, 0.2, 8)] * Bn, seed=1000 + i, philox_seed=i,
                          x_sigma=3.0, draft_sigma=1.0, history_len=4096, want_logprobs=True,
                          n_top_logprobs=20, name=name, requests=requests, q_layout="reduced",
                          draft_vocab=32000, subset_boost=2.0)
    raise KeyError(name)
