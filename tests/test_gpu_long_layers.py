"""Whole-workload parity of the 128K-token long prefill (131072 tokens, 32 query heads over
4 KV heads, head_dim 128, block 128, keep-ratios 0.10 / 0.02), GPU against the fp64 oracle.

* All 48 independently seeded layers: every mask row of every KV head under the excuse
  protocol (each layer's excused count is printed at the end of the run), the block
  summaries and the quantile ranks, the kept lists against the mask, and the attention
  of 32 seeded query blocks per layer (the first and last included, one head per KV group)
  through the GPU's own kept lists, on the rows whose GPU mask equals the oracle's.
* Layer 0: every attention row (32 heads x 1024 query blocks) against the oracle's
  explicit softmax on the oracle's masks, max-abs 2e-2 / mean-abs 2e-3 / LSE 1e-3, and
  the run on the GPU's own lists bit-identical to it on every row whose mask agrees.

The rescue coefficient's quantiles are taken per layer and per KV head ("Your 128K Context
Is 6x Slower Than It Needs to Be", section "The rescue branch"), so each seeded layer is a
separate case.  The oracle runs in a spawn process pool (tests/oracle_pool.py).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle_pool as P
import synth
from parity_util import (check_lists_match_mask, check_meta, compare_mask_rows,
                         gpu_mask_build, shape_of, to_dev)

pytestmark = pytest.mark.gpu

W = "gqa32x4_n131072_d128_b128"
SEED = 4242


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_kv_gb300 import build
    build.build()


def _attention_dev(w, q, k, v, kv_idx, kv_cnt):
    """bsa_prefill_fwd on device tensors; returns device o (bf16) and lse."""
    import block_sparse_long_kv_gb300 as bsa
    s = shape_of(w)
    o = torch.empty_like(q)
    lse = torch.empty(w.batch, w.hq, w.seq, dtype=torch.float32, device=q.device)
    st = torch.zeros(1, dtype=torch.int32, device=q.device)
    bsa.prefill_fwd(s, q, k, v, kv_idx, kv_cnt, 1.0 / math.sqrt(w.head_dim), o, lse, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o, lse


def _lists_dev(keep, device="cuda"):
    import oracle as O
    kv_idx, kv_cnt = O.kv_lists(keep)
    return torch.from_numpy(kv_idx).to(device), torch.from_numpy(kv_cnt).to(device)


def _check_rows(w, o, lse, ref, rows):
    errs, lerr = [], 0.0
    for (b, h, i) in rows:
        oi, li = ref[(b, h, i)]
        t = slice(i * w.block, (i + 1) * w.block)
        go = o[b, t, h].float().cpu().numpy().astype(np.float64)
        errs.append(np.abs(go - oi).reshape(-1))
        lerr = max(lerr, float(np.abs(lse[b, h, t].cpu().numpy() - li).max()))
    e = np.concatenate(errs)
    assert e.max() <= 2e-2, f"max-abs {e.max()}"
    assert e.mean() <= 2e-3, f"mean-abs {e.mean()}"
    assert lerr <= 1e-3, f"lse {lerr}"
    return float(e.max()), float(e.mean()), lerr


def test_all_48_layers_masks_and_sampled_attention():
    w = synth.workload(W)
    assert w.layers == 48
    nw = P.worker_count()
    jobs = [(W, layer, 32, SEED) for layer in range(w.layers)]
    seen = []
    leftovers = []
    with P.pool(nw) as pool:
        try:
            for r in P.bounded_imap(pool, P.layer_job, jobs, ahead=nw + 2):
                layer = r["layer"]
                leftovers = list(r["handles"].values())
                sh = {x: P.Shared(h) for x, h in r["handles"].items()}
                try:
                    lay = {x: sh[x].a for x in sh}
                    got = gpu_mask_build(w, lay)
                    check_lists_match_mask(got["mask"], got["kv_idx"], got["kv_cnt"])
                    check_meta(w, lay, got, r["orc"])
                    compared, excused = compare_mask_rows(got["mask"], r["orc"], label=f"L{layer}")
                    assert excused <= max(4, compared // 1000), (layer, compared, excused)
                    # end to end: attention over the GPU's own lists, sampled rows whose mask agrees
                    q, k, v = (to_dev(lay[x]) for x in ("q", "k", "v"))
                    o, lse = _attention_dev(w, q, k, v, torch.from_numpy(got["kv_idx"]).cuda(),
                                            torch.from_numpy(got["kv_cnt"]).cuda())
                    rows = [(b, h, i) for (b, h, i) in r["att"]
                            if np.array_equal(got["mask"][b, h // w.group, i], r["keep"][b, h // w.group, i])]
                    assert len(rows) >= len(r["att"]) // 2, (layer, len(rows), len(r["att"]))
                    _check_rows(w, o, lse, r["att"], rows)
                    del q, k, v, o, lse
                finally:
                    for s in sh.values():
                        s.release(unlink=True)
                    leftovers = []
                seen.append(layer)
        finally:
            for h in leftovers:
                P.discard(h)
    assert seen == list(range(w.layers))


def test_layer0_every_attention_row():
    w = synth.workload(W)
    nw = P.worker_count()
    with P.pool(nw) as pool:
        r = pool.apply_async(P.layer_job, (W, 0, 0, SEED)).get(P.JOB_TIMEOUT_S)
        handles = dict(r["handles"])
        sh = {x: P.Shared(h) for x, h in handles.items()}
        try:
            lay = {x: sh[x].a for x in sh}
            q, k, v = (to_dev(lay[x]) for x in ("q", "k", "v"))
            keep = r["keep"]
            o, lse = _attention_dev(w, q, k, v, *_lists_dev(keep))
            # the GPU's own lists give the same bits on every row whose mask agrees
            got = gpu_mask_build(w, lay)
            o2, lse2 = _attention_dev(w, q, k, v, torch.from_numpy(got["kv_idx"]).cuda(),
                                      torch.from_numpy(got["kv_cnt"]).cuda())
            agree = np.all(got["mask"] == keep, axis=-1)               # [b, hkv, nb]
            assert agree.mean() >= 0.99, agree.mean()
            tok = torch.from_numpy(np.repeat(agree, w.block, axis=-1)).cuda()   # [b, hkv, N]
            tok = tok.repeat_interleave(w.group, dim=1).permute(0, 2, 1)       # [b, N, hq]
            assert torch.equal(o[tok], o2[tok])
            assert torch.equal(lse.permute(0, 2, 1)[tok], lse2.permute(0, 2, 1)[tok])
            del o2, lse2, q, k, v
            handles["o"] = P.to_shared(o.view(torch.int16).cpu().numpy().view(np.uint16), os.getpid())
            handles["lse"] = P.to_shared(lse.cpu().numpy(), os.getpid())
            del o, lse
            torch.cuda.empty_cache()
            # every (head, query block) row, interleaved so each job mixes short and long rows
            jobs = []
            for h in range(w.hq):
                for part in range(4):
                    rows = [(0, h, i) for i in range(part, w.nb, 4)]
                    jobs.append((W, handles, keep, rows))
            res = pool.starmap_async(P.attention_rows_job, jobs).get(P.JOB_TIMEOUT_S)
        finally:
            for s in sh.values():
                s.release(unlink=True)
            for x in ("o", "lse"):
                if x in handles:
                    P.discard(handles[x])
    mx = max(x[0] for x in res)
    mean = sum(x[1] for x in res) / sum(x[2] for x in res)
    lmx = max(x[3] for x in res)
    assert sum(x[2] for x in res) == w.batch * w.seq * w.hq * w.head_dim
    assert mx <= 2e-2 and mean <= 2e-3 and lmx <= 1e-3, (mx, mean, lmx)
    print(f"layer 0, all {w.hq * w.nb} attention rows: max-abs {mx:.3e}, mean-abs {mean:.3e}, "
          f"LSE {lmx:.3e}")
