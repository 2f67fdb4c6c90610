"""Seeded synthetic inputs for the verify-and-sample epilogue.

Input synthesis only (numpy, CPU): target logits, draft probabilities, draft ids,
completion-count histories, per-request sampling parameters and the Philox
uniforms.  Both the oracle and the CUDA path consume these arrays; neither side's
arithmetic lives here.

Shapes (one batch of B requests, K_max drafted tokens at most):
  x      [B, K_max+1, V]  target logits, bf16 (stored as uint16 bit patterns) or fp32
  q      [B, K_max, V]    draft probabilities, fp32 (softmax of synthetic draft logits);
                          sparse layout: [B, K_max, m] values with ids q_ids [B, K_max, m];
                          reduced layout: [B, K_max, Vd] over a draft vocabulary, d2t [Vd]
  d      [B, K_max]       draft token ids, int32 (positions >= K_b are padding, 0)
  hist   CSR over requests: offsets [B+1], ids (ascending per request), counts (>0)
  rows   structured [B]: temperature, top_k, top_p, presence, frequency, num_drafts
  u      [B, K_max+1, 2]  fp32 uniforms (accept draw, resample/bonus draw)
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .philox import epilogue_uniforms

ROW_DTYPE = np.dtype([
    ("temperature", np.float32),
    ("top_k", np.int32),
    ("top_p", np.float32),
    ("presence_penalty", np.float32),
    ("frequency_penalty", np.float32),
    ("num_drafts", np.int32),
])


def row_params(temperature=0.0, top_k=0, top_p=1.0, presence=0.0, frequency=0.0, num_drafts=0):
    return (np.float32(temperature), np.int32(top_k), np.float32(top_p),
            np.float32(presence), np.float32(frequency), np.int32(num_drafts))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Batch:
    B: int
    K_max: int
    V: int
    logits_dtype: str                 # "bf16" or "fp32"
    x: np.ndarray                     # uint16 bits (bf16) or float32
    q: np.ndarray                     # float32 [B, K_max, V]
    draft_ids: np.ndarray             # int32 [B, K_max]
    hist_offsets: np.ndarray          # int32 [B+1]
    hist_ids: np.ndarray              # int32 [nnz]
    hist_counts: np.ndarray           # int32 [nnz]
    rows: np.ndarray                  # ROW_DTYPE [B]
    uniforms: np.ndarray              # float32 [B, K_max+1, 2]
    want_logprobs: bool = False
    n_top_logprobs: int = 0
    name: str = ""
    requests: tuple = ()              # index of each request in the full workload batch
    meta: dict = field(default_factory=dict)
    # draft layout: "dense" q [B, K_max, V]; "sparse" q [B, K_max, m] probabilities of the ids
    # in q_ids [B, K_max, m]; "reduced" q [B, K_max, Vd] over a draft vocabulary with d2t [Vd]
    # (target id = draft id + d2t[draft id])
    q_layout: str = "dense"
    q_ids: np.ndarray = None
    d2t: np.ndarray = None
    eos_ids: np.ndarray = None        # int32 [B]: end-of-sequence token per request (-1: none)
    logprob_mode: str = "raw"         # "raw" or "penalised" log-softmax for logprobs

    def x_f32(self, b=None) -> np.ndarray:
        """Target logits as float32 (exact upcast of bf16)."""
        xs = self.x if b is None else self.x[b]
        return bf16_bits_to_f32(xs) if self.logits_dtype == "bf16" else np.asarray(xs, np.float32)

    def history(self, b):
        lo, hi = int(self.hist_offsets[b]), int(self.hist_offsets[b + 1])
        return self.hist_ids[lo:hi], self.hist_counts[lo:hi]

    def draft_row_len(self) -> int:
        """Entries of one draft row of q: V (dense), m (sparse) or the draft vocabulary."""
        return self.q.shape[-1] if self.q is not None and self.q.ndim == 3 else 0

    def algorithmic_bytes(self) -> int:
        """One read of each needed logit and draft probability (sparse drafts: id + probability)."""
        sx = 2 if self.logits_dtype == "bf16" else 4
        per_q = self.draft_row_len() * (8 if self.q_layout == "sparse" else 4)
        total = 0
        for b in range(self.B):
            K = int(self.rows["num_drafts"][b])
            total += (K + 1) * self.V * sx
            if float(self.rows["temperature"][b]) > 0.0:
                total += K * per_q
        return total

    def verify_rows(self) -> int:
        return int(np.sum(self.rows["num_drafts"].astype(np.int64) + 1))

    def subset(self, reqs) -> "Batch":
        """A batch of the given requests of this one (copies of their arrays)."""
        reqs = [int(b) for b in reqs]
        ids, cnt, offs = [], [], [0]
        for b in reqs:
            i, c = self.history(b)
            ids.append(i)
            cnt.append(c)
            offs.append(offs[-1] + len(i))
        orig = self.requests if self.requests else tuple(range(self.B))
        return Batch(B=len(reqs), K_max=self.K_max, V=self.V, logits_dtype=self.logits_dtype,
                     x=self.x[reqs].copy(), q=self.q[reqs].copy(), draft_ids=self.draft_ids[reqs].copy(),
                     hist_offsets=np.array(offs, np.int32),
                     hist_ids=np.concatenate(ids).astype(np.int32) if ids else np.zeros(0, np.int32),
                     hist_counts=np.concatenate(cnt).astype(np.int32) if cnt else np.zeros(0, np.int32),
                     rows=self.rows[reqs].copy(), uniforms=self.uniforms[reqs].copy(),
                     want_logprobs=self.want_logprobs, n_top_logprobs=self.n_top_logprobs, name=self.name,
                     requests=tuple(orig[b] for b in reqs), meta=dict(self.meta), q_layout=self.q_layout,
                     q_ids=None if self.q_ids is None else self.q_ids[reqs].copy(), d2t=self.d2t,
                     eos_ids=None if self.eos_ids is None else self.eos_ids[reqs].copy(),
                     logprob_mode=self.logprob_mode)


def zipf_history(rng, V, H, s, perm):
    """H tokens with P(rank r) proportional to r^-s over ranks 1..V, mapped to ids by perm.

    Returns (ids ascending, counts)."""
    if H <= 0:
        return np.zeros(0, np.int32), np.zeros(0, np.int32)
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    ranks = np.searchsorted(cdf, rng.random(H), side="right")
    ranks = np.minimum(ranks, V - 1)
    toks = perm[ranks]
    ids, counts = np.unique(toks, return_counts=True)
    return ids.astype(np.int32), counts.astype(np.int32)


def _softmax_f32(z64: np.ndarray) -> np.ndarray:
    m = z64.max(axis=-1, keepdims=True)
    e = np.exp(z64 - m)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def make_batch(*, B, K_max, V, logits_dtype="bf16", rows, seed=0, philox_seed=0,
               x_sigma=3.0, draft_sigma=1.0, boost_frac=0.0, boost=8.0,
               history_len=0, zipf_s=1.1, draft_mode="q", argmax_frac=0.0,
               x_quant=None, want_logprobs=False, n_top_logprobs=0, name="", requests=None,
               q_layout="dense", q_m=1, draft_vocab=None, eos_pos=None, logprob_mode="raw",
               subset_boost=0.0) -> Batch:
    """Build one seeded batch.

    rows: sequence of row_params tuples (length B).
    draft_mode: "q"        -- d_i drawn from q_i (plain categorical draw, generator-side uniforms)
                "argmax"   -- d_i = argmax of the raw target logits at position i
                "q_argmax" -- d_i = argmax of q_i (a greedy drafter)
                "copy"   -- q_i = softmax of the target logits themselves (draft == target)
    argmax_frac: after drawing, that fraction of draft tokens (seeded) is replaced by the
                 raw target argmax at its position.
    x_quant: if set, target logits are rounded to multiples of this step (tie-heavy rows).
    requests: build only these requests of the B-request batch; request i of the result is
              request requests[i] of the full batch, bit for bit (each request draws from
              its own seeded stream, so any subset can be built on its own).
    q_layout: "dense"; "sparse" -- each draft row keeps m = q_m entries: the drafted id and
              the m-1 other largest entries of the dense row, in a seeded order (q_m = 1 is
              a one-hot proposal, q = 1 at the drafted id); "reduced" -- the draft vocabulary
              is a seeded ascending subset S of draft_vocab target ids, d2t[i] = S[i] - i, q
              is the softmax of the draft logits over S and drafts are drawn from it;
              subset_boost is added to the target logits of S (the frequent tokens a
              reduced draft vocabulary keeps) before rounding.
    eos_pos: if set, request b's end-of-sequence token is its draft at position
             min(eos_pos, K_b - 1) (none when K_b = 0).
    """
    # shared draws (boosted rows, the history permutation) come from stream 0, request b's
    # draws from stream 1 + b
    g = np.random.default_rng(np.random.SeedSequence(seed, spawn_key=(0,)))
    rows_all = np.array(list(rows), dtype=ROW_DTYPE)
    assert rows_all.shape == (B,)
    reqs = list(range(B)) if requests is None else [int(b) for b in requests]
    n_rows = B * (K_max + 1)
    boosted = np.zeros(n_rows, bool)
    if boost_frac > 0:
        nb = int(np.ceil(boost_frac * n_rows))
        boosted[g.choice(n_rows, size=nb, replace=False)] = True
    boosted = boosted.reshape(B, K_max + 1)
    perm = g.permutation(V)

    Bn = len(reqs)
    rows_arr = rows_all[reqs]
    x_store = np.empty((Bn, K_max + 1, V), np.uint16 if logits_dtype == "bf16" else np.float32)
    sub = np.sort(g.choice(V, size=draft_vocab, replace=False)) if q_layout == "reduced" else None
    Lq = {"dense": V, "sparse": q_m, "reduced": draft_vocab}[q_layout]
    q = np.empty((Bn, K_max, Lq), np.float32)
    q_ids = np.zeros((Bn, K_max, q_m), np.int32) if q_layout == "sparse" else None
    d = np.zeros((Bn, K_max), np.int32)
    offs = [0]
    h_ids, h_cnt = [], []
    for b, b_full in enumerate(reqs):
        rng = np.random.default_rng(np.random.SeedSequence(seed, spawn_key=(1 + b_full,)))
        xf = rng.standard_normal((K_max + 1, V), dtype=np.float32) * np.float32(x_sigma)
        if x_quant is not None:
            xf = (np.round(xf / np.float32(x_quant)) * np.float32(x_quant)).astype(np.float32)
        if sub is not None and subset_boost:
            xf[:, sub] += np.float32(subset_boost)
        for j in np.nonzero(boosted[b_full])[0]:
            t = int(np.argmax(xf[j]))
            xf[j, t] += np.float32(boost)
        if logits_dtype == "bf16":
            bits = f32_to_bf16_bits(xf)
            x_store[b] = bits
            xr = bf16_bits_to_f32(bits)
        else:
            x_store[b] = xf
            xr = xf
        if K_max > 0:
            cols = sub if sub is not None else slice(None)
            if draft_mode == "copy":
                qd = _softmax_f32(xr[:K_max, cols].astype(np.float64))
            else:
                noise = rng.standard_normal((K_max, V), dtype=np.float32) * np.float32(draft_sigma)
                qd = _softmax_f32(xr[:K_max, cols].astype(np.float64) + noise[:, cols].astype(np.float64))
            K_b = int(rows_arr["num_drafts"][b])
            for i in range(K_max):
                if draft_mode == "argmax":
                    t = int(np.argmax(xr[i]))
                elif draft_mode == "q_argmax":
                    t = int(np.argmax(qd[i]))
                else:
                    cdf = np.cumsum(qd[i], dtype=np.float64)
                    t = int(np.searchsorted(cdf, rng.random() * cdf[-1], side="right"))
                    t = min(t, qd.shape[-1] - 1)
                if sub is not None and draft_mode != "argmax":
                    t = int(sub[t])
                d[b, i] = t
                if argmax_frac > 0 and rng.random() < argmax_frac:
                    d[b, i] = int(np.argmax(xr[i]))
                if i >= K_b:
                    d[b, i] = 0
            if q_layout == "sparse":
                for i in range(K_max):
                    order = np.argsort(-qd[i], kind="stable")
                    ids = [int(d[b, i])] + [int(t) for t in order[:q_m] if t != d[b, i]][: q_m - 1]
                    ids = np.array(ids, np.int32)[rng.permutation(q_m)]
                    q_ids[b, i] = ids
                    q[b, i] = 1.0 if q_m == 1 else qd[i, ids]
            else:
                q[b] = qd
        ids, cnt = zipf_history(rng, V, history_len, zipf_s, perm)
        h_ids.append(ids)
        h_cnt.append(cnt)
        offs.append(offs[-1] + len(ids))
    eos_ids = None
    if eos_pos is not None:
        Ks = rows_arr["num_drafts"].astype(np.int64)
        eos_ids = np.array([d[b, min(eos_pos, Ks[b] - 1)] if Ks[b] > 0 else -1 for b in range(Bn)], np.int32)
    batch = Batch(
        B=Bn, K_max=K_max, V=V, logits_dtype=logits_dtype, x=x_store, q=q, draft_ids=d,
        hist_offsets=np.array(offs, np.int32),
        hist_ids=np.concatenate(h_ids).astype(np.int32) if h_ids else np.zeros(0, np.int32),
        hist_counts=np.concatenate(h_cnt).astype(np.int32) if h_cnt else np.zeros(0, np.int32),
        rows=rows_arr, uniforms=epilogue_uniforms(philox_seed, B, K_max)[reqs],
        want_logprobs=want_logprobs, n_top_logprobs=n_top_logprobs, name=name, requests=tuple(reqs),
        q_layout=q_layout, q_ids=q_ids, d2t=None if sub is None else (sub - np.arange(draft_vocab)).astype(np.int32),
        eos_ids=eos_ids, logprob_mode=logprob_mode,
        meta=dict(seed=seed, philox_seed=philox_seed, x_sigma=x_sigma, draft_sigma=draft_sigma,
                  boost_frac=boost_frac, history_len=history_len, draft_mode=draft_mode,
                  argmax_frac=argmax_frac, q_layout=q_layout, q_m=q_m, draft_vocab=draft_vocab, eos_pos=eos_pos,
                  subset_boost=subset_boost),
    )
    return batch
