"""Write ``sweep_oracle.json``: the oracle's mask density and needle-block recall for
the 27 block-size x keep-ratio combinations at 64K tokens (GQA 32/4, head_dim 128).

Calls only ``oracle`` (and ``synth`` for the seeded inputs).  For each block size the
layer is drawn once; block meta, quantiles, the rescue coefficient, the query
summaries and the two score matrices do not depend on the keep ratios, so they are
computed once per (b, g) and every ratio pair runs only the oracle's per-row
selection over the whole causal mask.

Density   = kept blocks / causal blocks (nb (nb + 1) / 2 per (b, g)).
Recall    = kept (needle query block, needle key block) pairs / all such pairs; a
            needle's query block is any block holding one of its query positions.

Run from the repository root:  python tests/golden/make_sweep_oracle.py
"""
from __future__ import annotations

import json
import math
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "sweep_oracle.json")


def needle_pairs(w, needles):
    out = []
    for (b, g, jb, slot, pos) in needles:
        for i in sorted(set((pos // w.block).tolist())):
            out.append((b, g, i, jb))
    return out


def oracle_sweep(block: int) -> dict:
    """Oracle density and needle recall of the 9 keep-ratio pairs at one block size."""
    group = [w for w in synth.sweep_workloads() if w.block == block]
    w0 = group[0]
    lay = synth.make_layer(w0)
    k = synth.bf16_to_f64(lay["k"])
    centroid, radius = O.block_meta(k, block)
    del k
    med, p90 = O.radius_quantiles(radius)
    alpha = O.rescue_coefficient(radius, med, p90)
    scale = 1.0 / math.sqrt(w0.head_dim)
    grp = w0.group
    pairs = needle_pairs(w0, lay["needles"])
    kept = {w.name: 0 for w in group}
    hits = {w.name: 0 for w in group}
    for b in range(w0.batch):
        for g in range(w0.hkv):
            qg = synth.bf16_to_f64(lay["q"][b:b + 1, :, g * grp:(g + 1) * grp])
            qbar, nbar = O.query_summary(qg, block)          # [1, G, nb, d], [1, G, nb]
            del qg
            # the oracle's [b, Hq, nb, d] layout with this group's heads at g * grp
            qb = np.zeros((b + 1, w0.hq) + qbar.shape[2:])
            nbb = np.zeros((b + 1, w0.hq, nbar.shape[2]))
            qb[b, g * grp:(g + 1) * grp] = qbar[0]
            nbb[b, g * grp:(g + 1) * grp] = nbar[0]
            s_c, r = O.block_scores(qb, nbb, centroid, radius, alpha, scale, b, g)
            del qb, nbb
            want = {}
            for (pb, pg, i, jb) in pairs:
                if pb == b and pg == g:
                    want.setdefault(i, []).append(jb)
            for w in group:
                pc, pr = O.ratio_ppm(w.centroid_keep), O.ratio_ppm(w.rescue_keep)
                for i in range(w.nb):
                    cent, resc = O.select_row(s_c[i], r[i], alpha[b, g], i, pc, pr)
                    row = set(cent.tolist()) | set(resc.tolist()) | {0, i}
                    kept[w.name] += len(row)
                    for jb in want.get(i, ()):
                        hits[w.name] += jb in row
    res = {}
    for w in group:
        causal = w.batch * w.hkv * w.nb * (w.nb + 1) // 2
        res[w.name] = {"block": block, "centroid_keep": w.centroid_keep,
                       "rescue_keep": w.rescue_keep, "kept_blocks": kept[w.name],
                       "density": kept[w.name] / causal, "needle_pairs": len(pairs),
                       "needle_hits": hits[w.name],
                       "needle_recall": hits[w.name] / len(pairs)}
    return res


def main():
    res = {}
    t0 = time.time()
    for block in sorted({w.block for w in synth.sweep_workloads()}):
        res.update(oracle_sweep(block))
        print(f"block {block}: {time.time() - t0:.1f}s", flush=True)
    doc = {"about": "oracle mask density and needle recall, 64K-token sweep, GQA 32/4, d 128, "
                    "seed 4000, written by tests/golden/make_sweep_oracle.py",
           "workloads": res}
    with open(OUT, "w") as f:
        json.dump(doc, f, indent=1, sort_keys=True)
        f.write("\n")


if __name__ == "__main__":
    main()
