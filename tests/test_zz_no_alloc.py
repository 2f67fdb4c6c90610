"""dspark_verify_sample_static: the epilogue on the library's fixed device scratch.

Its results must equal those of dspark_verify_sample (caller workspace) on the same inputs,
on two calls in a row (the scratch is reused and holds nothing that has to start at zero),
and shapes whose workspace exceeds the fixed size must be refused before any CUDA work.
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


def _batches():
    from workloads.generate import make_batch, row_params
    from workloads import configs
    yield "b1k2v4096", configs.build("b1k2v4096")
    mixed = [row_params(1.0, 64, 0.95, 0.2, 0.2, 4), row_params(0.0, 0, 1.0, 0.1, 0.3, 4),
             row_params(0.7, 0, 0.9, 0.0, 0.0, 3), row_params(1.3, 20, 1.0, 0.0, 0.5, 2)]
    yield "b4k4v32000_mixed", make_batch(B=4, K_max=4, V=32000, logits_dtype="bf16", rows=mixed, seed=77,
                                         philox_seed=9, history_len=256, want_logprobs=True, n_top_logprobs=5)


def _fresh_out(call):
    import torch
    return {k: torch.full_like(v, -7) for k, v in call.out.items()}


@pytest.mark.parametrize("name", ["b1k2v4096", "b4k4v32000_mixed"])
def test_static_scratch_matches_workspace_entry(lib, name):
    import torch
    from sample_verify_epilogue_gb300 import binding
    from sample_verify_epilogue_gb300.runner import EpilogueCall
    batch = dict(_batches())[name]
    call = EpilogueCall(batch)
    call.run()
    want = call.results()
    for _ in range(2):                                   # two calls in a row on the same scratch
        out = _fresh_out(call)
        status = torch.full_like(call.row_status, -7)
        before = torch.cuda.memory_allocated()
        binding.dspark_verify_sample_static(call.x, call.q, call.d, call.counts, call.rows, call.u, out=out,
                                            row_status=status, want_logprobs=call.want_logprobs,
                                            n_top_logprobs=call.n_top)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == before
        assert np.array_equal(status.cpu().numpy(), want["row_status"])
        for k, v in out.items():
            got = v.cpu().numpy()
            assert got.dtype == want[k].dtype
            assert np.array_equal(got.view(np.uint32) if got.dtype == np.float32 else got,
                                  want[k].view(np.uint32) if want[k].dtype == np.float32 else want[k]), k


def test_static_scratch_refuses_oversize_shapes(lib):
    import ctypes
    from sample_verify_epilogue_gb300 import binding
    assert binding.dspark_workspace_bytes(64, 8, 262144, "bf16", 20) > binding.DSPARK_STATIC_WORKSPACE_BYTES
    p = binding.make_params(64, 8, 262144, "bf16", n_top_logprobs=20)
    d = ctypes.c_void_p(256)
    code = lib.dspark_verify_sample_static(d, d, d, None, ctypes.byref(p), d, d, d, None, None, None)
    assert code == 2                                      # DSPARK_ERR_UNSUPPORTED
