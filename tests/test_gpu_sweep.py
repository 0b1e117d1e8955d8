"""The block-size x keep-ratio sweep at 64K tokens (GQA 32/4, head_dim 128) on the GPU.

For each block size one layer is drawn; for each of the 9 keep-ratio pairs the GPU
mask is compared with the oracle on every needle query block plus sampled rows
(mask protocol of parity_util), and the GPU's whole-mask density and needle recall
are compared with the oracle's stored figures (tests/golden/sweep_oracle.json,
written by tests/golden/make_sweep_oracle.py from the oracle alone).  One ratio
pair per block size also checks sampled attention rows through the GPU's lists.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
import synth
from parity_util import (check_attention_rows, check_lists_match_mask, compare_mask_rows,
                         gpu_attention, gpu_mask_build, oracle_rows)

pytestmark = pytest.mark.gpu

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "sweep_oracle.json")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_kv_gb300 import build
    build.build()


def needle_pairs(w, needles):
    return [(b, g, i, jb) for (b, g, jb, slot, pos) in needles
            for i in sorted(set((pos // w.block).tolist()))]


def reselect(base, w):
    """The oracle rows of ``base`` re-selected at ``w``'s keep ratios (scores and
    alpha do not depend on the ratios)."""
    pc, pr = O.ratio_ppm(w.centroid_keep), O.ratio_ppm(w.rescue_keep)
    rows = {}
    for (b, g, i), (_, s_c, r) in base["rows"].items():
        cent, resc = O.select_row(s_c, r, base["alpha"][b, g], i, pc, pr)
        m = np.zeros(w.nb, dtype=np.uint8)
        m[0] |= O.FORCED
        m[i] |= O.FORCED
        m[cent] |= O.CENTROID
        m[resc] |= O.RESCUE
        rows[(b, g, i)] = (m, s_c, r)
    return {**base, "rows": rows}


@pytest.mark.parametrize("block", [64, 128, 256])
def test_sweep_masks_density_recall(block):
    gold = json.load(open(GOLD))["workloads"]
    ws = [w for w in synth.sweep_workloads() if w.block == block]
    assert len(ws) == 9
    w0 = ws[0]
    lay = synth.make_layer(w0)
    pairs = needle_pairs(w0, lay["needles"])
    rng = np.random.default_rng(block)
    rows = {}
    for (b, g, i, _) in pairs:
        rows.setdefault((b, g), set()).add(i)
    for g in range(w0.hkv):
        rows.setdefault((0, g), set()).update({0, 1, 2, w0.nb - 1}
                                              | set(rng.integers(0, w0.nb, 12).tolist()))
    base = oracle_rows(w0, lay, {k: sorted(v) for k, v in rows.items()})
    for w in ws:
        got = gpu_mask_build(w, lay)
        check_lists_match_mask(got["mask"][:, :, -4:], got["kv_idx"][:, :, -4:],
                               got["kv_cnt"][:, :, -4:])
        orc = reselect(base, w)
        compared, excused = compare_mask_rows(got["mask"], orc)
        assert excused <= max(4, compared // 1000), (w.name, compared, excused)
        ref = gold[w.name]
        kept = int(got["kv_cnt"].astype(np.int64).sum())
        assert abs(kept - ref["kept_blocks"]) <= max(2, 1e-4 * ref["kept_blocks"]), (w.name, kept, ref)
        hits = sum(bool(got["mask"][b, g, i, jb]) for (b, g, i, jb) in pairs)
        assert len(pairs) == ref["needle_pairs"]
        assert abs(hits - ref["needle_hits"]) <= excused, (w.name, hits, ref["needle_hits"])
        if w.centroid_keep == 0.1 and w.rescue_keep == 0.02:
            o, lse = gpu_attention(w, lay, torch.from_numpy(got["kv_idx"]).cuda(),
                                   torch.from_numpy(got["kv_cnt"]).cuda())
            keep = np.zeros((w.batch, w.hkv, w.nb, w.nb), dtype=np.uint8)
            att = []
            for (b, g, i), (m, _, _) in orc["rows"].items():
                keep[b, g, i] = m
                if i % 5 == 0 and np.array_equal(got["mask"][b, g, i], m):
                    att += [(b, g * w.group, i), (b, g * w.group + w.group - 1, i)]
            assert att
            check_attention_rows(w, lay, o, lse, keep != 0, att)
