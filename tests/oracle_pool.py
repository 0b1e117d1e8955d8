"""Process pool that runs the fp64 oracle on the 128K-token seeded layers (test helper).

The long-prefill workload (131072 tokens, 32 query heads over 4 KV heads, head_dim 128,
block 128) names 48 independently seeded layers.  Generating one layer and building its
oracle masks takes seconds of single-core numpy, so the layers are spread over worker
processes.  Each worker generates its layer, leaves q, k and v in shared memory (files on
the /dev/shm tmpfs) for the GPU side (which then never generates the layer itself), and returns the oracle's whole-layer
mask rows plus the oracle attention of sampled rows.  The pool and the shared-memory helpers
are those of synth.parallel (spawn start: the pytest process has already initialised CUDA, and
a forked child of it would hang; one BLAS thread per worker).
"""
from __future__ import annotations

import os

import numpy as np

from synth.parallel import (JOB_TIMEOUT_S, attach, bounded_imap, discard, pool, sweep,  # noqa: F401
                            threads_per_worker, to_shared, worker_count)


class Shared:
    """Attached view of a shared array (``.a``); ``release(unlink)`` detaches."""

    def __init__(self, handle):
        self.path = handle
        self.a = attach(handle)

    def release(self, unlink: bool = False):
        self.a = None
        if unlink:
            discard(self.path)


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
    lay = synth.make_layer(w, layer=layer, threads=threads_per_worker(worker_count()))
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
