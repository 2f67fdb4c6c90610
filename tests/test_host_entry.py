"""dspark_verify_sample_host: the epilogue from host buffers.

Its outputs must equal those of the device-buffer entry point, bit for bit, from pinned
tensors and from pageable numpy arrays alike, on two calls in a row.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from sample_verify_epilogue_gb300 import binding
    return binding.load_library()


def _batch():
    from workloads.generate import make_batch, row_params
    rows = [row_params(1.0, 64, 0.95, 0.2, 0.2, 4), row_params(0.0, 0, 1.0, 0.1, 0.3, 4),
            row_params(0.7, 0, 0.9, 0.0, 0.0, 3), row_params(1.3, 20, 1.0, 0.0, 0.5, 2)]
    return make_batch(B=4, K_max=4, V=32000, logits_dtype="bf16", rows=rows, seed=91, philox_seed=5,
                      history_len=256, want_logprobs=True, n_top_logprobs=5)


@pytest.mark.parametrize("pinned", [True, False])
def test_host_entry_matches_device_entry(lib, pinned):
    import torch
    from sample_verify_epilogue_gb300 import binding
    from sample_verify_epilogue_gb300.runner import EpilogueCall
    batch = _batch()
    call = EpilogueCall(batch)
    call.run()
    want = call.results()

    def host(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a).pin_memory() if pinned else a

    B, W, n = batch.B, batch.K_max + 1, batch.n_top_logprobs
    hx = host(np.ascontiguousarray(batch.x).view(np.int16))
    hq = host(batch.q)
    hd = host(batch.draft_ids)
    hrows = host(np.ascontiguousarray(batch.rows).view(np.uint8))
    hcounts = (host(batch.hist_offsets), host(batch.hist_ids), host(batch.hist_counts))
    hu = host(batch.uniforms)
    out = {"accept_len": np.full(B, -7, np.int32), "tokens": np.full((B, W), -7, np.int32),
           "logprobs": np.full((B, W), -7, np.float32), "top_ids": np.full((B, W, n), -7, np.int32),
           "top_logprobs": np.full((B, W, n), -7, np.float32)}
    status = np.full(B, -7, np.int32)
    nbytes = binding.dspark_host_workspace_bytes(B, batch.K_max, batch.V, "bf16", n, int(batch.hist_offsets[-1]))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):                                    # the workspace is reused as it stands
        binding.dspark_verify_sample_host(hx, hq, hd, hcounts, hrows, hu, out=out, row_status=status, workspace=ws,
                                          logits_dtype="bf16", want_logprobs=True, n_top_logprobs=n)
        assert np.array_equal(status, want["row_status"])
        for k, v in out.items():
            w = want[k]
            assert np.array_equal(v.view(np.uint32) if v.dtype == np.float32 else v,
                                  w.view(np.uint32) if w.dtype == np.float32 else w), k
