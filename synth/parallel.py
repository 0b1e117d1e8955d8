"""Seeded layers generated in worker processes and handed over through shared memory.

Generating one 131072-token layer (32 query heads over 4 KV heads, head_dim 128) takes
seconds of numpy, and a good part of it is serial, so many layers are drawn faster by several
processes than by one.  A worker draws its layer with ``make_layer`` (same seeds, same values
as in the calling process) and writes q, k and v as ``.npy`` files on the /dev/shm tmpfs; the
caller maps them, uses them and removes them.  Files are named after the process that consumes
them, so ``sweep`` removes whatever a failure left behind.  Pools start with ``spawn``: a
caller that has initialised CUDA must not fork.

This module moves the generator's output around; it computes nothing of the method.
"""
from __future__ import annotations

import glob
import os
import uuid
from collections import deque
from contextlib import contextmanager
from multiprocessing import get_context

import numpy as np

SHM_DIR = "/dev/shm"


def worker_count() -> int:
    return max(1, min(8, (os.cpu_count() or 2) - 1))


def threads_per_worker(workers: int) -> int:
    return max(1, (os.cpu_count() or 1) // max(1, workers))


@contextmanager
def pool(n: int | None = None):
    """A spawn pool whose workers run numpy with one BLAS thread each; shared files made for
    the calling process are removed when the pool closes."""
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"
    try:
        p = get_context("spawn").Pool(n or worker_count())
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    try:
        yield p
    finally:
        p.terminate()
        p.join()
        sweep()


def _prefix(owner_pid: int) -> str:
    return f"bsaorc{owner_pid}_"


def to_shared(arr: np.ndarray, owner_pid: int | None = None) -> str:
    """Copy arr into a new shared file owned by ``owner_pid`` (by default the parent of the
    calling process, i.e. the pool's owner); returns its path."""
    owner = os.getppid() if owner_pid is None else owner_pid
    path = os.path.join(SHM_DIR, _prefix(owner) + uuid.uuid4().hex[:16])
    mm = np.lib.format.open_memmap(path, mode="w+", dtype=arr.dtype, shape=arr.shape)
    mm[...] = arr
    mm.flush()
    del mm
    return path


def attach(path: str) -> np.ndarray:
    """Writable memory map of a shared file (writable, so torch.from_numpy takes it)."""
    return np.load(path, mmap_mode="r+")


def discard(path: str) -> None:
    try:
        os.unlink(path)
    except FileNotFoundError:
        pass


def sweep() -> None:
    """Remove every shared file made for this process that is still there."""
    for f in glob.glob(os.path.join(SHM_DIR, _prefix(os.getpid()) + "*")):
        discard(f)


JOB_TIMEOUT_S = 1800  # no job comes near this; a pool whose workers cannot start fails instead of waiting


def bounded_imap(p, fn, arg_list, ahead: int, timeout: float = JOB_TIMEOUT_S):
    """Results of fn(*args) in order, at most ``ahead`` jobs submitted but not yet consumed
    (each layer job holds its layer in shared memory until the caller consumes it).  A job
    that gives no result within ``timeout`` seconds raises multiprocessing.TimeoutError."""
    pending = deque()
    it = iter(arg_list)
    for args in it:
        pending.append(p.apply_async(fn, args))
        if len(pending) >= ahead:
            break
    while pending:
        r = pending.popleft().get(timeout)
        for args in it:
            pending.append(p.apply_async(fn, args))
            break
        yield r


def layer_job(w, layer: int, threads: int) -> dict:
    """Draw layer ``layer`` of workload ``w`` into shared files; returns their paths and the
    needle list."""
    from . import make_layer
    lay = make_layer(w, layer=layer, threads=threads)
    return {"layer": layer, "paths": {x: to_shared(lay[x]) for x in ("q", "k", "v")},
            "needles": lay["needles"], "seed": lay["seed"]}


def layers(w, layer_ids, workers: int | None = None):
    """Yield (layer, dict of q / k / v arrays mapped from shared memory, needles) for each
    seeded layer in order; each layer's files are removed once the caller moves on."""
    n = workers or worker_count()
    th = threads_per_worker(n)
    with pool(n) as p:
        for r in bounded_imap(p, layer_job, [(w, L, th) for L in layer_ids], ahead=n + 2):
            arrays = {x: attach(path) for x, path in r["paths"].items()}
            try:
                yield r["layer"], arrays, r["needles"]
            finally:
                del arrays
                for path in r["paths"].values():
                    discard(path)
