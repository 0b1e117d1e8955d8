"""Process pool that runs the fp64 oracle on the 128K-token seeded layers (test helper).

The long-prefill workload (131072 tokens, 32 query heads over 4 KV heads, head_dim 128,
block 128) names 48 independently seeded layers.  Generating one layer and building its
oracle masks takes seconds of single-core numpy, so the layers are spread over worker
processes.  Each worker generates its layer, leaves q, k and v in shared memory (files on
the /dev/shm tmpfs) for the GPU side (which then never generates the layer itself), and returns the oracle's whole-layer
mask rows plus the oracle attention of sampled rows.  The pool starts with ``spawn``: the
pytest process has already initialised CUDA, and a forked child of it would hang.  Workers
run numpy with one BLAS thread each.
"""
from __future__ import annotations

import os
import uuid
from collections import deque
from contextlib import contextmanager
from multiprocessing import get_context

import numpy as np


def worker_count() -> int:
    return max(1, min(8, (os.cpu_count() or 2) - 1))


@contextmanager
def pool(n: int | None = None):
    """A spawn pool whose workers use one BLAS thread each."""
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


# ---------------------------------------------------------------- shared arrays
#
# Plain memory-mapped files under /dev/shm (tmpfs): any process opens one by name, and
# nothing tracks them but the name prefix of the process that consumes them.

SHM_DIR = "/dev/shm"


def _prefix(owner_pid: int) -> str:
    return f"bsaorc{owner_pid}_"


def to_shared(arr: np.ndarray, owner_pid: int | None = None):
    """Copy arr into a new shared file named after the process that will consume it (the
    pool's parent by default, so ``sweep`` can remove whatever a failure left behind);
    returns a picklable handle."""
    owner = os.getppid() if owner_pid is None else owner_pid
    path = os.path.join(SHM_DIR, _prefix(owner) + uuid.uuid4().hex[:16])
    mm = np.lib.format.open_memmap(path, mode="w+", dtype=arr.dtype, shape=arr.shape)
    mm[...] = arr
    mm.flush()
    del mm
    return path


class Shared:
    """Attached view of a shared array (``.a``); ``release(unlink)`` detaches."""

    def __init__(self, handle):
        self.path = handle
        self.a = np.load(handle, mmap_mode="r+")  # writable view: torch.from_numpy takes it without a warning

    def release(self, unlink: bool = False):
        self.a = None
        if unlink:
            discard(self.path)


def sweep() -> None:
    """Remove every shared file made for this process that is still there (after a failure
    the results still queued in the pool hold files nobody will consume)."""
    import glob
    for f in glob.glob(os.path.join(SHM_DIR, _prefix(os.getpid()) + "*")):
        discard(f)


def discard(handle) -> None:
    """Remove a shared file if it still exists."""
    try:
        os.unlink(handle)
    except FileNotFoundError:
        pass


# ---------------------------------------------------------------- jobs (run in workers)

def _oracle_rows_by_group(w, q_bits, k_bits, v_bits, keep, rows):
    """oracle.sparse_attention_rows for rows (b, h, i), one KV group at a time, widening only
    that group's query heads, keys and values (float32 holds bf16 values exactly; the oracle
    computes in float64 on those values)."""
    import oracle as O
    import synth

    out = {}
    for g in sorted({h // w.group for (_, h, _) in rows}):
        sel = [(b, h, i) for (b, h, i) in rows if h // w.group == g]
        hs = slice(g * w.group, (g + 1) * w.group)
        q = synth.bf16_to_f32(q_bits[:, :, hs])
        k = synth.bf16_to_f32(k_bits[:, :, g:g + 1])
        v = synth.bf16_to_f32(v_bits[:, :, g:g + 1])
        res = O.sparse_attention_rows(q, k, v, keep[:, g:g + 1] != 0, w.block,
                                      [(b, h - g * w.group, i) for (b, h, i) in sel])
        for (b, h, i) in sel:
            out[(b, h, i)] = res[(b, h - g * w.group, i)]
    return out


def layer_job(wname: str, layer: int, att_blocks: int, seed: int):
    """Generate one seeded layer into shared memory, build the oracle's masks for every
    row, and compute the oracle attention of ``att_blocks`` seeded query blocks (first
    and last included) for one head of each KV group, over the oracle's own masks."""
    import synth
    from parity_util import oracle_rows

    w = synth.workload(wname)
    lay = synth.make_layer(w, layer=layer, threads=max(1, (os.cpu_count() or 1) // worker_count()))
    handles = {x: to_shared(lay[x]) for x in ("q", "k", "v")}
    orc = oracle_rows(w, lay, {(b, g): list(range(w.nb)) for b in range(w.batch) for g in range(w.hkv)})
    keep = np.zeros((w.batch, w.hkv, w.nb, w.nb), dtype=np.uint8)
    for (b, g, i), (m, _, _) in orc["rows"].items():
        keep[b, g, i] = m
    att = {}
    if att_blocks > 0:
        rng = np.random.default_rng(seed + layer)
        blocks = sorted({0, w.nb - 1} | set(rng.integers(1, w.nb - 1, att_blocks - 2).tolist()))
        rows = [(b, g * w.group + int(rng.integers(0, w.group)), i)
                for b in range(w.batch) for i in blocks for g in range(w.hkv)]
        att = _oracle_rows_by_group(w, lay["q"], lay["k"], lay["v"], keep, rows)
    return dict(layer=layer, handles=handles, orc=orc, keep=keep, att=att)


def attention_rows_job(wname: str, handles: dict, keep: np.ndarray, rows):
    """Oracle attention of ``rows`` over the oracle's masks ``keep``, compared with the GPU
    output in shared memory (o as bf16 bits [b, N, Hq, d], lse fp32 [b, Hq, N]).  Returns
    (max |o diff|, sum |o diff|, elements, max |lse diff|)."""
    import synth

    w = synth.workload(wname)
    sh = {x: Shared(h) for x, h in handles.items()}
    try:
        ref = _oracle_rows_by_group(w, sh["q"].a, sh["k"].a, sh["v"].a, keep, rows)
        mx = sm = 0.0
        cnt = 0
        lmx = 0.0
        for (b, h, i), (oi, li) in ref.items():
            t = slice(i * w.block, (i + 1) * w.block)
            go = synth.bf16_to_f32(sh["o"].a[b, t, h, :]).astype(np.float64)
            e = np.abs(go - oi)
            mx = max(mx, float(e.max()))
            sm += float(e.sum())
            cnt += e.size
            lmx = max(lmx, float(np.abs(sh["lse"].a[b, h, t] - li).max()))
        return mx, sm, cnt, lmx
    finally:
        for s in sh.values():
            s.release()


def bounded_imap(p, fn, arg_list, ahead: int):
    """Results of fn(*args) in order, with at most ``ahead`` jobs submitted but unconsumed
    (each layer job holds about 1.3 GB of shared memory until its result is consumed)."""
    pending = deque()
    it = iter(arg_list)
    for args in it:
        pending.append(p.apply_async(fn, args))
        if len(pending) >= ahead:
            break
    while pending:
        r = pending.popleft().get()
        for args in it:
            pending.append(p.apply_async(fn, args))
            break
        yield r
