"""ctypes binding of libdspark.so: the C ABI of include/dspark.h with the same names.

Argument marshalling only.  Every step of the epilogue runs in the library's sm_103a
kernels; this module passes device pointers (``tensor.data_ptr()``) and the current torch
stream.  It raises if the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB

DSPARK_OK = 0
DSPARK_BF16 = 0
DSPARK_FP32 = 1
DSPARK_MAX_TOP_LOGPROBS = 20
DSPARK_MAX_SPARSE_M = 256
DSPARK_Q_DENSE, DSPARK_Q_SPARSE, DSPARK_Q_REDUCED = 0, 1, 2
DSPARK_LOGPROBS_RAW, DSPARK_LOGPROBS_PENALISED = 0, 1
Q_LAYOUTS = {"dense": DSPARK_Q_DENSE, "sparse": DSPARK_Q_SPARSE, "reduced": DSPARK_Q_REDUCED}
LOGPROB_MODES = {"raw": DSPARK_LOGPROBS_RAW, "penalised": DSPARK_LOGPROBS_PENALISED}

ROW_BAD_PARAMS = 1
ROW_BAD_DRAFT = 2
ROW_NONFINITE = 4
ROW_BAD_HISTORY = 8
ROW_INTERNAL = 16

# dspark_row_params_t: float, int32, float, float, float, int32 (24 bytes)
ROW_PARAMS_DTYPE = np.dtype([
    ("temperature", np.float32), ("top_k", np.int32), ("top_p", np.float32),
    ("presence_penalty", np.float32), ("frequency_penalty", np.float32), ("num_drafts", np.int32),
])


class dspark_counts_t(ctypes.Structure):
    _fields_ = [("row_offsets", ctypes.c_void_p), ("token_ids", ctypes.c_void_p), ("counts", ctypes.c_void_p)]


class dspark_extras_t(ctypes.Structure):
    _fields_ = [
        ("q_layout", ctypes.c_int32), ("q_row_len", ctypes.c_int32), ("q_ids", ctypes.c_void_p),
        ("d2t", ctypes.c_void_p), ("eos_ids", ctypes.c_void_p), ("out_stopped", ctypes.c_void_p),
        ("pos_counts", ctypes.c_void_p), ("logprob_mode", ctypes.c_int32),
    ]


class dspark_params_t(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("K_max", ctypes.c_int32), ("V", ctypes.c_int32), ("logits_dtype", ctypes.c_int32),
        ("rows", ctypes.c_void_p), ("want_logprobs", ctypes.c_int32), ("n_top_logprobs", ctypes.c_int32),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t), ("stream", ctypes.c_void_p),
        ("row_status", ctypes.c_void_p), ("stage_events", ctypes.c_void_p * 2),
        ("extras", ctypes.POINTER(dspark_extras_t)),
    ]


def make_extras(q_layout="dense", q_row_len=0, q_ids=None, d2t=None, eos_ids=None, out_stopped=None,
                pos_counts=None, logprob_mode="raw"):
    """A dspark_extras_t; array arguments are raw addresses (int) or None."""
    x = dspark_extras_t()
    x.q_layout = Q_LAYOUTS[q_layout] if isinstance(q_layout, str) else int(q_layout)
    x.q_row_len = int(q_row_len)
    x.q_ids, x.d2t, x.eos_ids = q_ids, d2t, eos_ids
    x.out_stopped, x.pos_counts = out_stopped, pos_counts
    x.logprob_mode = LOGPROB_MODES[logprob_mode] if isinstance(logprob_mode, str) else int(logprob_mode)
    return x


_lib = None

EXPORTS = ("dspark_workspace_bytes", "dspark_verify_sample", "dspark_host_workspace_bytes",
           "dspark_verify_sample_host", "dspark_verify_sample_static", "dspark_status_string",
           "dspark_launches_per_call")

DSPARK_STATIC_WORKSPACE_BYTES = 16 << 20


def load_library(path: str = LIB):
    """Load libdspark.so (built by ``sample_verify_epilogue_gb300.build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = open_library(path)
    return _lib


def open_library(path: str):
    """A CDLL of a build of the library at ``path`` with the argument types set (not cached)."""
    if not os.path.exists(path):
        raise ImportError(f"{os.path.basename(path)} not found at {path}: build it first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(dspark_params_t)
    C = ctypes.POINTER(dspark_counts_t)
    vp = ctypes.c_void_p
    lib.dspark_workspace_bytes.argtypes = [P]
    lib.dspark_workspace_bytes.restype = ctypes.c_size_t
    lib.dspark_host_workspace_bytes.argtypes = [P, ctypes.c_int64]
    lib.dspark_host_workspace_bytes.restype = ctypes.c_size_t
    sig = [vp, vp, vp, C, P, vp, vp, vp, vp, vp, vp]
    lib.dspark_verify_sample.argtypes = sig
    lib.dspark_verify_sample.restype = ctypes.c_int
    lib.dspark_verify_sample_host.argtypes = sig
    lib.dspark_verify_sample_host.restype = ctypes.c_int
    lib.dspark_verify_sample_static.argtypes = sig
    lib.dspark_verify_sample_static.restype = ctypes.c_int
    lib.dspark_status_string.argtypes = [ctypes.c_int]
    lib.dspark_status_string.restype = ctypes.c_char_p
    lib.dspark_launches_per_call.argtypes = []
    lib.dspark_launches_per_call.restype = ctypes.c_int32
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def make_params(B, K_max, V, logits_dtype, *, rows=None, want_logprobs=False, n_top_logprobs=0,
                workspace=None, workspace_bytes=0, stream=None, row_status=None, stage_events=(None, None),
                extras=None):
    p = dspark_params_t()
    p.B, p.K_max, p.V = int(B), int(K_max), int(V)
    p.logits_dtype = DSPARK_BF16 if logits_dtype in ("bf16", DSPARK_BF16) else DSPARK_FP32
    p.rows = rows
    p.want_logprobs = int(bool(want_logprobs))
    p.n_top_logprobs = int(n_top_logprobs)
    p.workspace = workspace
    p.workspace_bytes = int(workspace_bytes)
    p.stream = stream
    p.row_status = row_status
    p.stage_events[0] = stage_events[0]
    p.stage_events[1] = stage_events[1]
    if extras is not None:
        p.extras = ctypes.pointer(extras)
    return p


def dspark_workspace_bytes(B, K_max, V, logits_dtype, n_top_logprobs=0, extras=None) -> int:
    lib = load_library()
    p = make_params(B, K_max, V, logits_dtype, n_top_logprobs=n_top_logprobs, extras=extras)
    return int(lib.dspark_workspace_bytes(ctypes.byref(p)))


def dspark_host_workspace_bytes(B, K_max, V, logits_dtype, n_top_logprobs=0, counts_nnz=0, extras=None) -> int:
    lib = load_library()
    p = make_params(B, K_max, V, logits_dtype, n_top_logprobs=n_top_logprobs, extras=extras)
    return int(lib.dspark_host_workspace_bytes(ctypes.byref(p), int(counts_nnz)))


def dspark_status_string(code: int) -> str:
    return load_library().dspark_status_string(int(code)).decode()


def dspark_launches_per_call() -> int:
    return int(load_library().dspark_launches_per_call())


def _check(code):
    if code != DSPARK_OK:
        raise RuntimeError(f"dspark: {dspark_status_string(code)} ({code})")


def _device_call(fn, logits, q, draft_ids, counts, rows, uniforms, out, row_status, workspace, want_logprobs,
                 n_top_logprobs, stream, stage_events, extras=None):
    import torch
    B, W, V = logits.shape
    if stream is None:
        stream = torch.cuda.current_stream(logits.device).cuda_stream
    dt = DSPARK_BF16 if logits.dtype == torch.bfloat16 else DSPARK_FP32
    p = make_params(B, W - 1, V, dt, rows=rows.data_ptr(), want_logprobs=want_logprobs,
                    n_top_logprobs=n_top_logprobs,
                    workspace=None if workspace is None else workspace.data_ptr(),
                    workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
                    stream=stream, row_status=row_status.data_ptr(),
                    stage_events=tuple(None if e is None else e for e in stage_events), extras=extras)
    c = None
    if counts is not None:
        c = dspark_counts_t(counts[0].data_ptr(), counts[1].data_ptr(), counts[2].data_ptr())
    code = fn(
        _ptr(logits), _ptr(q), _ptr(draft_ids), ctypes.byref(c) if c is not None else None, ctypes.byref(p),
        _ptr(uniforms), _ptr(out["accept_len"]), _ptr(out["tokens"]), _ptr(out.get("logprobs")),
        _ptr(out.get("top_ids")), _ptr(out.get("top_logprobs")))
    _check(code)


def dspark_verify_sample(logits, q, draft_ids, counts, rows, uniforms, *, out, row_status, workspace,
                         want_logprobs=False, n_top_logprobs=0, stream=None, stage_events=(None, None),
                         extras=None):
    """Enqueue the epilogue on ``stream`` (default: torch's current stream).

    logits [B, K_max+1, V] bf16/fp32, q [B, K_max, V] fp32 or None, draft_ids [B, K_max] int32,
    counts (offsets [B+1], ids, counts) int32 or None, rows: uint8 tensor of B packed
    dspark_row_params_t, uniforms [B, K_max+1, 2] fp32 -- all CUDA tensors.
    out: dict with "accept_len" [B], "tokens" [B, K_max+1] int32, and optionally
    "logprobs" [B, K_max+1], "top_ids" / "top_logprobs" [B, K_max+1, n] tensors.
    extras: a dspark_extras_t (``make_extras``, device addresses) or None.
    """
    _device_call(load_library().dspark_verify_sample, logits, q, draft_ids, counts, rows, uniforms, out,
                 row_status, workspace, want_logprobs, n_top_logprobs, stream, stage_events, extras)


def dspark_verify_sample_static(logits, q, draft_ids, counts, rows, uniforms, *, out, row_status,
                                want_logprobs=False, n_top_logprobs=0, stream=None, stage_events=(None, None),
                                extras=None):
    """The same call with the library's fixed device scratch (no workspace, no allocation);
    shapes needing more than DSPARK_STATIC_WORKSPACE_BYTES are refused.  Calls that overlap
    on the GPU race on that scratch."""
    _device_call(load_library().dspark_verify_sample_static, logits, q, draft_ids, counts, rows, uniforms, out,
                 row_status, None, want_logprobs, n_top_logprobs, stream, stage_events, extras)


def dspark_verify_sample_host(logits, q, draft_ids, counts, rows, uniforms, *, out, row_status, workspace,
                              logits_dtype, want_logprobs=False, n_top_logprobs=0, stream=None, extras=None):
    """The epilogue from host buffers (numpy or pinned torch CPU tensors); synchronous.

    ``workspace`` is a CUDA uint8 tensor of at least dspark_host_workspace_bytes bytes.
    Outputs are written into the host arrays of ``out`` and ``row_status``; ``extras`` holds
    host addresses."""
    lib = load_library()
    B, W, V = logits.shape

    def hp(a):
        if a is None:
            return None
        if isinstance(a, np.ndarray):
            assert a.flags.c_contiguous
            return ctypes.c_void_p(a.ctypes.data)
        return ctypes.c_void_p(a.data_ptr())

    p = make_params(B, W - 1, V, logits_dtype, rows=hp(rows).value, want_logprobs=want_logprobs,
                    n_top_logprobs=n_top_logprobs, workspace=workspace.data_ptr(),
                    workspace_bytes=workspace.numel() * workspace.element_size(), stream=stream,
                    row_status=hp(row_status).value, extras=extras)
    c = None
    if counts is not None:
        c = dspark_counts_t(hp(counts[0]).value, hp(counts[1]).value, hp(counts[2]).value)
    code = lib.dspark_verify_sample_host(
        hp(logits), hp(q), hp(draft_ids), ctypes.byref(c) if c is not None else None, ctypes.byref(p),
        hp(uniforms), hp(out["accept_len"]), hp(out["tokens"]), hp(out.get("logprobs")),
        hp(out.get("top_ids")), hp(out.get("top_logprobs")))
    _check(code)
