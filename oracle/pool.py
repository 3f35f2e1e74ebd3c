"""The oracle's whole step on every host core: ``index.index_step`` run over a
batch's requests by a pool of single-threaded worker processes.

TEST INFRASTRUCTURE ONLY (see the package docstring): the benchmark's CPU
baseline and its reference arm time the oracle with it.  It adds no
arithmetic: each worker calls ``index.index_step`` unchanged on a list of
requests, reading the step's arrays from shared memory (the pool planes are
hundreds of MB to GB, so they are never copied per task), and the parent puts
the per-request results back together.  Workers are started with ``spawn`` (a
process forked from one that has used a GPU can hang) and keep one BLAS thread
each, so the worker count is the number of cores the oracle uses.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np

from . import index

_ARRAY_ARGS = ("q", "q_scale", "payload", "scale", "page_table", "slot_ids", "row_lens")
_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS")

# In a worker: the step's arguments, arrays viewing the shared blocks.
_KW = None
_SHM = []


def _attach(arrays: dict, scalars: dict) -> None:
    global _KW
    kw = dict(scalars)
    for name, spec in arrays.items():
        if spec is None:
            kw[name] = None
            continue
        shm_name, shape, dtype = spec
        shm = shared_memory.SharedMemory(name=shm_name)
        _SHM.append(shm)
        kw[name] = np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf)
    _KW = kw


def _run(requests):
    res = index.index_step(**_KW, requests=list(requests))
    return list(requests), res.ids[list(requests)], res.scores[list(requests)]


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or its machine type."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        vendor = model = ""
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name":
                model = model or v.strip()
            elif k.strip() == "Vendor ID":
                vendor = v.strip()
        if model:
            return f"{vendor} {model}".strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


class OraclePool:
    """index_step over all requests of one set of step arguments, split by
    request across ``workers`` processes.  Use as a context manager."""

    def __init__(self, step_kwargs: dict, workers: int = 0):
        self.workers = workers or host_cores()
        self.R = int(np.asarray(step_kwargs["q"]).shape[0])
        self.M = step_kwargs["packed_queries"] * step_kwargs["gqa"]
        self.topk = step_kwargs["topk"]
        self._blocks = []
        arrays = {}
        for name in _ARRAY_ARGS:
            a = step_kwargs.get(name)
            if a is None:
                arrays[name] = None
                continue
            a = np.ascontiguousarray(a)
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, dtype=a.dtype, buffer=shm.buf)[...] = a
            self._blocks.append(shm)
            arrays[name] = (shm.name, a.shape, a.dtype.str)
        scalars = {k: v for k, v in step_kwargs.items() if k not in _ARRAY_ARGS}
        saved = {v: os.environ.get(v) for v in _THREAD_VARS}
        for v in _THREAD_VARS:
            os.environ[v] = "1"
        try:
            self._pool = mp.get_context("spawn").Pool(self.workers, initializer=_attach,
                                                      initargs=(arrays, scalars))
        finally:
            for v, old in saved.items():
                if old is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = old
        # requests that read keys, longest first (the pool hands them out in order)
        lens = np.asarray(step_kwargs["row_lens"]).reshape(self.R, -1).max(axis=1)
        slots = np.asarray(step_kwargs["slot_ids"])
        n_slots = np.asarray(step_kwargs["page_table"]).shape[0]
        live = [r for r in range(self.R) if 0 <= int(slots[r]) < n_slots and lens[r] > 0]
        self.requests = sorted(live, key=lambda r: -int(lens[r]))

    def step(self, requests=None):
        """The whole step (or only ``requests``): (ids [R, M, topk], scores)."""
        todo = self.requests if requests is None else list(requests)
        ids = np.full((self.R, self.M, self.topk), -1, dtype=np.int64)
        scores = np.full((self.R, self.M, self.topk), -np.inf, dtype=np.float64)
        for rs, i, s in self._pool.imap_unordered(_run, [[r] for r in todo], chunksize=1):
            ids[rs], scores[rs] = i, s
        return ids, scores

    def close(self):
        if self._pool is not None:
            self._pool.close()
            self._pool.join()
            self._pool = None
        for shm in self._blocks:
            shm.close()
            shm.unlink()
        self._blocks = []

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
