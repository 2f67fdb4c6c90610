"""The C ABI library builds, loads and exports every entry point its header declares
(CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sample_verify_epilogue_gb300.build import build
    path = build()
    from sample_verify_epilogue_gb300 import binding
    return binding.load_library(path)


def _declared():
    src = open(os.path.join(ROOT, "include", "dspark.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z_]+)\s*\(", src)))


def test_header_symbols_exported(lib):
    names = _declared()
    assert "dspark_verify_sample" in names and len(names) >= 6
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_sizes(lib):
    from sample_verify_epilogue_gb300 import binding as bd
    w3 = bd.dspark_workspace_bytes(64, 8, 262144, "bf16", 20)
    w4 = bd.dspark_workspace_bytes(256, 16, 262144, "bf16", 5)
    w0 = bd.dspark_workspace_bytes(1, 2, 4096, "fp32", 0)
    assert 0 < w0 < w3 < w4
    assert w3 % 256 == 0
    # shapes out of range report 0
    assert bd.dspark_workspace_bytes(0, 8, 1000, "bf16") == 0
    assert bd.dspark_workspace_bytes(2049, 8, 1000, "bf16") == 0
    assert bd.dspark_workspace_bytes(4, 65, 1000, "bf16") == 0
    assert bd.dspark_workspace_bytes(4, 8, (1 << 24) + 1, "bf16") == 0
    assert bd.dspark_workspace_bytes(4, 8, 1000, "bf16", 21) == 0
    assert bd.dspark_host_workspace_bytes(64, 8, 262144, "bf16", 20, 100000) > w3


def test_status_strings_and_launches(lib):
    from sample_verify_epilogue_gb300 import binding as bd
    assert bd.dspark_status_string(0) == "ok"
    assert "workspace" in bd.dspark_status_string(3)
    assert bd.dspark_launches_per_call() == 6


def test_invalid_arguments_rejected_before_any_cuda_call(lib):
    from sample_verify_epilogue_gb300 import binding as bd
    p = bd.make_params(0, 2, 100, "bf16")
    code = lib.dspark_verify_sample(None, None, None, None, ctypes.byref(p), None, None, None, None, None, None)
    assert code == 1
    p = bd.make_params(2, 2, 100, "bf16")
    code = lib.dspark_verify_sample(ctypes.c_void_p(256), None, None, None, ctypes.byref(p), None, None, None, None,
                                    None, None)
    assert code == 1                       # missing uniforms / outputs / rows / status
    rows = ctypes.create_string_buffer(48)
    st = ctypes.create_string_buffer(8)
    p = bd.make_params(2, 2, 100, "bf16", rows=ctypes.addressof(rows), row_status=ctypes.addressof(st),
                       workspace=None, workspace_bytes=0)
    d = ctypes.c_void_p(512)
    code = lib.dspark_verify_sample(ctypes.c_void_p(256), None, d, None, ctypes.byref(p), ctypes.c_void_p(1024),
                                    ctypes.c_void_p(2048), ctypes.c_void_p(4096), None, None, None)
    assert code == 3                       # no workspace


def test_static_scratch_limits(lib):
    """dspark_verify_sample_static: shapes whose workspace exceeds the fixed 16 MiB scratch are
    refused with DSPARK_ERR_UNSUPPORTED before any CUDA call; the documented shapes fit."""
    from sample_verify_epilogue_gb300 import binding as bd
    cap = bd.DSPARK_STATIC_WORKSPACE_BYTES
    assert cap == 16 << 20
    for shape in [(16, 8, 151936), (12, 8, 262144), (4, 4, 32000), (1, 2, 4096)]:
        assert 0 < bd.dspark_workspace_bytes(*shape, "bf16", 20) <= cap, shape
    assert bd.dspark_workspace_bytes(64, 8, 262144, "bf16", 20) > cap
    p = bd.make_params(64, 8, 262144, "bf16", n_top_logprobs=20)
    d = ctypes.c_void_p(256)
    assert lib.dspark_verify_sample_static(d, d, d, None, ctypes.byref(p), d, d, d, None, None, None) == 2
