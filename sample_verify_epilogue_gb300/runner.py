"""Device-side buffers for one batch and one call of the epilogue through the C ABI.

Takes host arrays (numpy) shaped as described in include/dspark.h, allocates the device
inputs, outputs and the workspace once with torch, and calls ``dspark_verify_sample``.
A batch with a sparse or reduced draft layout, eos tokens or penalised logprobs (or
``counters=True``) passes a dspark_extras_t; its per-position counters accumulate over runs.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding


class EpilogueCall:
    """Inputs, outputs and workspace of one batch resident on a CUDA device."""

    def __init__(self, batch, device="cuda", counters=False):
        dev = torch.device(device)
        self.B, self.K_max, self.V = batch.B, batch.K_max, batch.V
        self.dtype = batch.logits_dtype
        self.want_logprobs = bool(batch.want_logprobs)
        self.n_top = int(batch.n_top_logprobs)
        W = self.K_max + 1
        if self.dtype == "bf16":
            xt = torch.from_numpy(np.ascontiguousarray(batch.x).view(np.int16)).view(torch.bfloat16)
        else:
            xt = torch.from_numpy(np.ascontiguousarray(batch.x, dtype=np.float32))
        self.x = xt.to(dev)
        self.q = torch.from_numpy(np.ascontiguousarray(batch.q, dtype=np.float32)).to(dev) if self.K_max > 0 else None
        self.d = torch.from_numpy(np.ascontiguousarray(batch.draft_ids, dtype=np.int32)).to(dev) if self.K_max > 0 else None
        rows = np.ascontiguousarray(batch.rows)
        assert rows.dtype.itemsize == 24
        self.rows = torch.from_numpy(rows.view(np.uint8).copy()).to(dev)
        self.counts = None
        if batch.hist_offsets is not None and len(batch.hist_offsets) == self.B + 1:
            ids = batch.hist_ids if len(batch.hist_ids) else np.zeros(1, np.int32)
            cnt = batch.hist_counts if len(batch.hist_counts) else np.zeros(1, np.int32)
            self.counts = tuple(torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
                                for a in (batch.hist_offsets, ids, cnt))
        self.u = torch.from_numpy(np.ascontiguousarray(batch.uniforms, dtype=np.float32)).to(dev)
        self.out = {
            "accept_len": torch.empty(self.B, dtype=torch.int32, device=dev),
            "tokens": torch.empty(self.B, W, dtype=torch.int32, device=dev),
        }
        if self.want_logprobs:
            self.out["logprobs"] = torch.empty(self.B, W, dtype=torch.float32, device=dev)
        if self.n_top > 0:
            self.out["top_ids"] = torch.empty(self.B, W, self.n_top, dtype=torch.int32, device=dev)
            self.out["top_logprobs"] = torch.empty(self.B, W, self.n_top, dtype=torch.float32, device=dev)
        self.row_status = torch.empty(self.B, dtype=torch.int32, device=dev)
        # options beyond the dense call: draft layout, eos tokens, counters, logprob mode
        layout = getattr(batch, "q_layout", "dense")
        eos = getattr(batch, "eos_ids", None)
        mode = getattr(batch, "logprob_mode", "raw")
        self.extras = None
        self.q_ids = self.d2t = self.eos = None
        if layout != "dense" or eos is not None or mode != "raw" or counters:
            def dev_i32(a):
                return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
            if layout == "sparse":
                self.q_ids = dev_i32(batch.q_ids)
            if layout == "reduced":
                self.d2t = dev_i32(batch.d2t)
            if eos is not None:
                self.eos = dev_i32(eos)
            self.out["stopped"] = torch.empty(self.B, dtype=torch.int32, device=dev)
            self.pos_counts = torch.zeros(2 * max(self.K_max, 1), dtype=torch.int64, device=dev)
            self.extras = binding.make_extras(
                q_layout=layout, q_row_len=batch.q.shape[-1] if layout != "dense" else 0,
                q_ids=None if self.q_ids is None else self.q_ids.data_ptr(),
                d2t=None if self.d2t is None else self.d2t.data_ptr(),
                eos_ids=None if self.eos is None else self.eos.data_ptr(),
                out_stopped=self.out["stopped"].data_ptr(), pos_counts=self.pos_counts.data_ptr(),
                logprob_mode=mode)
        nbytes = binding.dspark_workspace_bytes(self.B, self.K_max, self.V, self.dtype, self.n_top, self.extras)
        if nbytes == 0:
            raise ValueError("unsupported shapes")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def run(self, stream=None, stage_events=(None, None), lib=None):
        """Enqueue one call; ``lib``: another build of the library (``binding.open_library``)."""
        if lib is not None:
            binding._device_call(lib.dspark_verify_sample, self.x, self.q, self.d, self.counts, self.rows, self.u,
                                 self.out, self.row_status, self.workspace, self.want_logprobs, self.n_top,
                                 stream, stage_events, self.extras)
            return
        binding.dspark_verify_sample(
            self.x, self.q, self.d, self.counts, self.rows, self.u, out=self.out, row_status=self.row_status,
            workspace=self.workspace, want_logprobs=self.want_logprobs, n_top_logprobs=self.n_top,
            stream=stream, stage_events=stage_events, extras=self.extras)

    def results(self):
        torch.cuda.synchronize()
        r = {k: v.cpu().numpy() for k, v in self.out.items()}
        r["row_status"] = self.row_status.cpu().numpy()
        if self.extras is not None:
            pc = self.pos_counts.cpu().numpy()
            r["pos_counts"] = pc[: 2 * self.K_max].reshape(2, self.K_max)
        return r

    def algorithmic_bytes(self, batch) -> int:
        return batch.algorithmic_bytes()
