"""The oracle's outcomes for the requests of a named workload, on all host cores.

A process pool started with the spawn method, so no worker is ever forked from a process
that has touched the GPU.  Each worker builds its request on its own from the workload's
seeds (``workloads.configs.build(name, requests=[b])`` equals request b of the whole batch)
and returns ``oracle.epilogue.outcomes`` for it, so no batch is copied between processes.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

_pool = None


def _outcomes_of_request(args):
    name, B, b = args
    from oracle import epilogue as O
    from workloads import configs
    batch = configs.build(name, B=B, requests=[b])
    return b, O.outcomes(batch, 0)


def workers() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(32, n))


def pool() -> ProcessPoolExecutor:
    global _pool
    if _pool is None:
        _pool = ProcessPoolExecutor(max_workers=workers(), mp_context=mp.get_context("spawn"))
    return _pool


def workload_outcomes(name, B=None, requests=None):
    """{b: outcomes of request b} for the given requests (default: all) of workload ``name``."""
    from workloads import configs
    if requests is None:
        requests = range(configs.build_size(name, B))
    jobs = [(name, B, int(b)) for b in requests]
    return dict(pool().map(_outcomes_of_request, jobs, chunksize=1))
