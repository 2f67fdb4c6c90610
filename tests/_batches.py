"""Small hand-built batches for the tests (input data only)."""
from __future__ import annotations

import numpy as np

from workloads.generate import ROW_DTYPE, Batch, f32_to_bf16_bits


def one_request(x_rows, q_rows, drafts, *, T, top_k=0, top_p=1.0, presence=0.0, frequency=0.0,
                hist_ids=(), hist_counts=(), uniforms=None, n_top=0, want_logprobs=False,
                bf16=False, K=None):
    """A batch with B=1 from explicit rows: x_rows [K+1, V], q_rows [K, V], drafts [K]."""
    x = np.asarray(x_rows, np.float32)
    K_max = x.shape[0] - 1
    V = x.shape[1]
    q = np.asarray(q_rows, np.float32).reshape(K_max, V)
    d = np.asarray(drafts, np.int32).reshape(K_max)
    rows = np.array([(T, top_k, top_p, presence, frequency, K_max if K is None else K)], dtype=ROW_DTYPE)
    u = np.zeros((1, K_max + 1, 2), np.float32) if uniforms is None else np.asarray(uniforms, np.float32).reshape(1, K_max + 1, 2)
    return Batch(B=1, K_max=K_max, V=V, logits_dtype="bf16" if bf16 else "fp32",
                 x=(f32_to_bf16_bits(x) if bf16 else x)[None], q=q[None], draft_ids=d[None],
                 hist_offsets=np.array([0, len(hist_ids)], np.int32),
                 hist_ids=np.asarray(hist_ids, np.int32), hist_counts=np.asarray(hist_counts, np.int32),
                 rows=rows, uniforms=u, want_logprobs=want_logprobs, n_top_logprobs=n_top)


def replicate(batch_one, d_list, u_list):
    """B copies of a one-request batch with per-copy drafts and uniforms."""
    Bn = len(d_list)
    b = batch_one
    return Batch(B=Bn, K_max=b.K_max, V=b.V, logits_dtype=b.logits_dtype,
                 x=np.repeat(b.x, Bn, axis=0), q=np.repeat(b.q, Bn, axis=0),
                 draft_ids=np.asarray(d_list, np.int32).reshape(Bn, b.K_max),
                 hist_offsets=np.arange(Bn + 1, dtype=np.int32) * len(b.hist_ids),
                 hist_ids=np.tile(b.hist_ids, Bn), hist_counts=np.tile(b.hist_counts, Bn),
                 rows=np.repeat(b.rows, Bn), uniforms=np.asarray(u_list, np.float32).reshape(Bn, b.K_max + 1, 2),
                 want_logprobs=b.want_logprobs, n_top_logprobs=b.n_top_logprobs)
