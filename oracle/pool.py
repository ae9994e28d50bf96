"""Runs the oracle's functions, unchanged, over the parts of a batch in a process pool.

TEST INFRASTRUCTURE. Only tests/ and bench.py's CPU baseline legs use it. It holds
no attention or addressing arithmetic of its own: every result comes from one call
of a function of ``oracle.paged_ref`` (or another oracle module) on a sub-batch of
the problem, exactly as a caller on one core would make it. The parts are
independent problems (one sequence, or some query rows of one sequence), because
each sequence attends only to its own keys.

Large read-only arrays (the caches) go to the workers as ``.npy`` files that each
worker maps into memory, so a worker only pages in the blocks its sequences read;
the small per-part arguments (a sequence's queries, table row and length) are
pickled with each task. Workers are started with the ``spawn`` method and import
numpy and the oracle only: a process forked from one that holds a CUDA context can
hang.
"""
from __future__ import annotations

import atexit
import importlib
import multiprocessing as mp
import os
import shutil
import tempfile
import time

import numpy as np

_SHARED: dict = {}
_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _init(paths: dict) -> None:
    for name, path in paths.items():
        _SHARED[name] = np.load(path, mmap_mode="r")


def _run(task):
    module, fn, shared_args, kwargs, positional = task
    f = getattr(importlib.import_module(module), fn)
    args = [(_SHARED[a[1]] if isinstance(a, tuple) and a and a[0] == "shared" else a)
            for a in positional]
    kw = dict(kwargs)
    for k, name in shared_args.items():
        kw[k] = _SHARED[name]
    return f(*args, **kw)


def SHARED(name: str):
    """Placeholder for a positional argument that is one of the shared arrays."""
    return ("shared", name)


def default_workers() -> int:
    n = os.cpu_count() or 1
    try:
        n = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        pass
    return max(1, n)


def _scratch_dir(nbytes: int) -> str:
    """A RAM-backed directory when it has room for the shared arrays, else the temp dir."""
    for base in ("/dev/shm", tempfile.gettempdir()):
        try:
            if os.path.isdir(base) and shutil.disk_usage(base).free > 2 * nbytes + (1 << 30):
                return tempfile.mkdtemp(prefix="pkv_oracle_", dir=base)
        except OSError:
            continue
    return tempfile.mkdtemp(prefix="pkv_oracle_")


class OraclePool:
    """``with OraclePool(shared={...}) as pool: results = pool.map(tasks)``.

    ``shared`` maps names to large numpy arrays written once for all workers. A task
    is ``(module, function, shared_kwargs, kwargs, positional)``: the function is
    looked up in ``module`` (an ``oracle.*`` module), ``shared_kwargs`` maps keyword
    names to shared-array names, ``positional`` may hold ``SHARED(name)``
    placeholders. Results come back in task order.
    """

    def __init__(self, shared: dict, workers: int | None = None):
        self.shared = shared
        self.workers = workers or default_workers()
        self.dir = None
        self.pool = None
        self.seconds = 0.0

    def __enter__(self):
        nbytes = sum(int(a.nbytes) for a in self.shared.values())
        self.dir = _scratch_dir(nbytes)
        # The files live in RAM when /dev/shm has room: remove them however this
        # process ends (an exception while starting the pool, or an exit without
        # __exit__), so that they cannot pile up across runs.
        atexit.register(shutil.rmtree, self.dir, True)
        try:
            paths = {}
            for name, arr in self.shared.items():
                path = os.path.join(self.dir, f"{name}.npy")
                np.save(path, np.ascontiguousarray(arr))
                paths[name] = path
            ctx = mp.get_context("spawn")
            # One BLAS thread per worker: the pool already has a process per core,
            # and numpy's threaded matrix-vector products would oversubscribe them.
            saved = {k: os.environ.get(k) for k in _THREAD_VARS}
            os.environ.update({k: "1" for k in _THREAD_VARS})
            try:
                self.pool = ctx.Pool(self.workers, initializer=_init, initargs=(paths,))
            finally:
                for k, v in saved.items():
                    if v is None:
                        os.environ.pop(k, None)
                    else:
                        os.environ[k] = v
        except BaseException:
            shutil.rmtree(self.dir, ignore_errors=True)
            raise
        return self

    def map(self, tasks, chunksize: int = 1):
        t = time.perf_counter()
        out = self.pool.map(_run, tasks, chunksize=chunksize)
        self.seconds += time.perf_counter() - t
        return out

    def __exit__(self, *exc):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()
        if self.dir is not None:
            shutil.rmtree(self.dir, ignore_errors=True)
        return False


def task(fn: str, module: str = "oracle.paged_ref", shared_kwargs=None, positional=(), **kwargs):
    """One call of ``module.fn(*positional, **shared_kwargs-resolved, **kwargs)``."""
    return (module, fn, dict(shared_kwargs or {}), kwargs, tuple(positional))
