"""Helpers for GPU-vs-oracle parity: run the CUDA path through the C ABI on
seeded inputs, run the oracle on the same bf16 values, and apply the mask
comparison protocol.

Mask protocol: masks must agree bit for bit except for excused blocks.  A
mismatched block is excused when
  * its oracle score on the path where it differs lies within 1e-4 relative of
    that row's oracle threshold (the lowest kept score), the denominator being
    max(|threshold|, 1e-3 * rms of the row's candidate scores);
  * its radius lies within 1e-4 relative of the median (rescue eligibility flip);
  * its row holds an excused centroid-path block (the rescue candidate set
    depends on the centroid path).
Forced bits must always match.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
import synth

REL = 1e-4

# (test id, label, compared blocks, excused blocks) of every mask comparison in this
# process; tests/conftest.py prints them at the end of the run.
EXCUSE_LOG = []


def _current_test() -> str:
    import os
    cur = os.environ.get("PYTEST_CURRENT_TEST", "?")
    return cur.rsplit(" ", 1)[0].split("::", 1)[-1]


def to_dev(bits: np.ndarray, device="cuda"):
    return torch.from_numpy(bits.view(np.int16)).to(device).view(torch.bfloat16)


def shape_of(w):
    from block_sparse_long_kv_gb300 import make_shape
    return make_shape(w.batch, w.seq, w.hq, w.hkv, w.head_dim, w.block)


def gpu_mask_build(w, lay, centroid_keep=None, rescue_keep=None, device="cuda", flags=0):
    """Run bsa_block_meta + bsa_select_mask; return numpy results.  With block-mean queries
    (flags 0) also run bsa_mask_build on the same inputs and require the same outputs bit for
    bit (kv_idx up to each row's kv_cnt: entries past it are unspecified)."""
    import block_sparse_long_kv_gb300 as bsa
    s = shape_of(w)
    q, k = to_dev(lay["q"], device), to_dev(lay["k"], device)
    meta = bsa.alloc_meta(s, device)
    sel = bsa.alloc_select(s, device, with_mask=True)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    bsa.block_meta(s, k, meta["centroid"], meta["radius"], meta["quant"], meta["alpha"], status)
    prm = bsa.SelectParams(w.centroid_keep if centroid_keep is None else centroid_keep,
                           w.rescue_keep if rescue_keep is None else rescue_keep, flags)
    bsa.select_mask(s, prm, q, meta["centroid"], meta["radius"], meta["alpha"], sel["kv_idx"],
                    sel["kv_cnt"], sel["mask"], dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    out = {kk: v.cpu().numpy() for kk, v in {**meta, **sel}.items()}
    if flags == 0:
        check_fused_build(s, prm, q, k, out, device)
    return out


def check_fused_build(s, prm, q, k, want, device="cuda"):
    """bsa_mask_build gives `want` (the two-call results) bit for bit."""
    import block_sparse_long_kv_gb300 as bsa
    meta = bsa.alloc_meta(s, device)
    sel = bsa.alloc_select(s, device, with_mask=True)
    for t in (*meta.values(), *sel.values()):
        t.fill_(-7 if t.dtype != torch.uint8 else 0xA5)  # nothing may survive from before the call
    status = torch.zeros(1, dtype=torch.int32, device=device)
    bsa.mask_build(s, prm, q, k, meta["centroid"], meta["radius"], meta["quant"], meta["alpha"],
                   sel["kv_idx"], sel["kv_cnt"], sel["mask"], dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = {kk: v.cpu().numpy() for kk, v in {**meta, **sel}.items()}
    for x in ("centroid", "radius", "quant", "alpha", "kv_cnt", "mask"):
        np.testing.assert_array_equal(got[x], want[x], err_msg=f"bsa_mask_build {x}")
    cnt = want["kv_cnt"]
    live = np.arange(want["kv_idx"].shape[-1]) < cnt[..., None]
    np.testing.assert_array_equal(got["kv_idx"][live], want["kv_idx"][live], err_msg="bsa_mask_build kv_idx")


def check_lists_match_mask(mask, kv_idx, kv_cnt):
    b, h, nb, _ = mask.shape
    for bi in range(b):
        for g in range(h):
            for i in range(nb):
                js = np.nonzero(mask[bi, g, i])[0]
                assert kv_cnt[bi, g, i] == js.size, (bi, g, i)
                np.testing.assert_array_equal(kv_idx[bi, g, i, :js.size], js)


def oracle_rows(w, lay, rows_by_bg, centroid_keep=None, rescue_keep=None, token_max=False):
    """Oracle mask rows for selected query blocks only.

    rows_by_bg: {(b, g): [i, ...]}.  Returns dict with per-(b, g, i) mask rows
    and the row scores, plus the oracle meta (centroid, radius, med, p90, alpha).
    token_max: per-token aggregation of the scores (oracle token_block_scores,
    restricted to the selected rows).
    """
    rc = w.centroid_keep if centroid_keep is None else centroid_keep
    rr = w.rescue_keep if rescue_keep is None else rescue_keep
    k = synth.bf16_to_f64(lay["k"])
    centroid, radius = O.block_meta(k, w.block)
    del k
    med, p90 = O.radius_quantiles(radius)
    alpha = O.rescue_coefficient(radius, med, p90)
    scale = 1.0 / math.sqrt(w.head_dim)
    grp = w.group
    rows = {}
    for (b, g), ilist in rows_by_bg.items():
        ilist = sorted(ilist)
        if token_max:
            for i in ilist:
                # the oracle's per-token scores of block i alone (a one-block query slice)
                qs = synth.bf16_to_f64(lay["q"][b:b + 1, i * w.block:(i + 1) * w.block])
                cen1 = centroid[b:b + 1]
                s_c, r = O.token_block_scores(qs, cen1, radius[b:b + 1], alpha[b:b + 1], w.block,
                                              scale, 0, g)
                cent, resc = O.select_row(s_c[0], r[0], alpha[b, g], i, O.ratio_ppm(rc),
                                          O.ratio_ppm(rr))
                m = np.zeros(w.nb, dtype=np.uint8)
                m[0] |= O.FORCED
                m[i] |= O.FORCED
                m[cent] |= O.CENTROID
                m[resc] |= O.RESCUE
                rows[(b, g, i)] = (m, s_c[0], r[0])
            continue
        # mean query / norm of just these blocks (oracle query_summary on each block's tokens)
        qbar = np.zeros((grp, len(ilist), w.head_dim))
        nbar = np.zeros((grp, len(ilist)))
        for ri, i in enumerate(ilist):
            qs = synth.bf16_to_f64(lay["q"][b:b + 1, i * w.block:(i + 1) * w.block,
                                            g * grp:(g + 1) * grp])
            qb1, nb1 = O.query_summary(qs, w.block)
            qbar[:, ri] = qb1[0, :, 0]
            nbar[:, ri] = nb1[0, :, 0]
        # pad to the oracle's [b, Hq, rows, d] layout with this group's heads at g*grp
        qb = np.zeros((b + 1, w.hq, len(ilist), w.head_dim))
        nbb = np.zeros((b + 1, w.hq, len(ilist)))
        qb[b, g * grp:(g + 1) * grp] = qbar
        nbb[b, g * grp:(g + 1) * grp] = nbar
        s_c, r = O.block_scores(qb, nbb, centroid, radius, alpha, scale, b, g)
        for ri, i in enumerate(ilist):
            cent, resc = O.select_row(s_c[ri], r[ri], alpha[b, g], i, O.ratio_ppm(rc), O.ratio_ppm(rr))
            m = np.zeros(w.nb, dtype=np.uint8)
            m[0] |= O.FORCED
            m[i] |= O.FORCED
            m[cent] |= O.CENTROID
            m[resc] |= O.RESCUE
            rows[(b, g, i)] = (m, s_c[ri], r[ri])
    return dict(rows=rows, centroid=centroid, radius=radius, med=med, p90=p90, alpha=alpha)


def check_meta(w, lay, got, orc):
    """Block summaries within 1e-5 relative of the oracle; quantiles at the oracle's rank (up to
    near-ties within 1e-4); alpha within 1e-3."""
    cen = got["centroid"]                                 # [b, hkv, nb, d]
    scale = np.abs(orc["centroid"]).max()
    assert np.abs(cen - orc["centroid"]).max() <= 1e-5 * max(scale, 1.0)
    np.testing.assert_allclose(got["radius"], orc["radius"], rtol=1e-5)
    # quantiles: the GPU picks the block the oracle's rank names (up to near-ties)
    nb = w.nb
    for b in range(w.batch):
        for g in range(w.hkv):
            order = np.lexsort((np.arange(nb), orc["radius"][b, g]))
            for qi, rank in ((0, O.nearest_rank(nb, 1, 2)), (1, O.nearest_rank(nb, 9, 10))):
                want = got["radius"][b, g, order[rank - 1]]
                if got["quant"][b, g, qi] != want:
                    ref = orc["radius"][b, g, order[rank - 1]]
                    near = np.abs(orc["radius"][b, g] - ref) <= 1e-4 * ref
                    assert near.sum() > 1, ("quantile rank differs", b, g, qi)
    assert np.abs(got["alpha"] - orc["alpha"]).max() <= 1e-3


def compare_mask_rows(gpu_mask, orc, label=""):
    """Apply the protocol; returns (n_compared_blocks, n_excused).  Raises on an unexcused mismatch.
    Every call is recorded in EXCUSE_LOG (with ``label`` naming the layer or case)."""
    compared, excused = _compare_mask_rows(gpu_mask, orc)
    EXCUSE_LOG.append((_current_test(), label, compared, excused))
    return compared, excused


def _compare_mask_rows(gpu_mask, orc):
    excused = 0
    compared = 0
    for (b, g, i), (om, s_c, r) in orc["rows"].items():
        gm = gpu_mask[b, g, i]
        compared += i + 1
        diff = np.nonzero(gm != om)[0]
        if diff.size == 0:
            continue
        assert not np.any((gm[diff] ^ om[diff]) & O.FORCED), ("forced bits differ", b, g, i)
        cands = np.arange(1, i)
        cent = np.nonzero(om & O.CENTROID)[0]
        resc = np.nonzero(om & O.RESCUE)[0]

        def near(score, kept, j):
            if kept.size == 0:
                return False
            t = score[kept].min()
            rms = math.sqrt(float(np.mean(score[cands] ** 2))) if cands.size else 0.0
            den = max(abs(t), 1e-3 * rms)
            return abs(score[j] - t) <= REL * den

        med = orc["med"][b, g]
        cent_excused = False
        row_ok = []
        for j in diff:
            if (gm[j] ^ om[j]) & O.CENTROID:
                ok = near(s_c, cent, j)
                cent_excused |= ok
                row_ok.append((j, ok))
        for j in diff:
            if not ((gm[j] ^ om[j]) & O.CENTROID) and ((gm[j] ^ om[j]) & O.RESCUE):
                ok = (near(r, resc, j) or abs(orc["radius"][b, g, j] - med) <= REL * med
                      or cent_excused)
                row_ok.append((j, ok))
        for j, ok in row_ok:
            assert ok, f"unexcused mask mismatch at b={b} g={g} i={i} j={j}: gpu={gm[j]} oracle={om[j]}"
        excused += len(row_ok)
    return compared, excused


def upload_lists(mask_rows_full, device="cuda"):
    kv_idx, kv_cnt = O.kv_lists(mask_rows_full)
    return (torch.from_numpy(kv_idx).to(device), torch.from_numpy(kv_cnt).to(device))


def gpu_attention(w, lay, kv_idx=None, kv_cnt=None, scale=None, device="cuda"):
    import block_sparse_long_kv_gb300 as bsa
    s = shape_of(w)
    q, k, v = to_dev(lay["q"], device), to_dev(lay["k"], device), to_dev(lay["v"], device)
    o = torch.empty_like(q)
    lse = torch.empty(w.batch, w.hq, w.seq, dtype=torch.float32, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    scale = 1.0 / math.sqrt(w.head_dim) if scale is None else scale
    if kv_idx is None:
        bsa.prefill_dense_fwd(s, q, k, v, scale, o, lse, status)
    else:
        bsa.prefill_fwd(s, q, k, v, kv_idx, kv_cnt, scale, o, lse, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check_attention_rows(w, lay, o_gpu, lse_gpu, keep, rows, scale=None):
    """Compare GPU rows (b, h, i) against the oracle: max-abs 2e-2, mean-abs 2e-3, LSE 1e-3."""
    # float32 holds bf16 values exactly; the oracle widens each slice to float64
    q = synth.bf16_to_f32(lay["q"])
    k = synth.bf16_to_f32(lay["k"])
    v = synth.bf16_to_f32(lay["v"])
    ref = O.sparse_attention_rows(q, k, v, keep, w.block, rows, scale)
    errs = []
    lerr = 0.0
    for (b, h, i), (oi, li) in ref.items():
        go = o_gpu[b, i * w.block:(i + 1) * w.block, h, :]
        errs.append(np.abs(go - oi))
        lerr = max(lerr, float(np.abs(lse_gpu[b, h, i * w.block:(i + 1) * w.block] - li).max()))
    e = np.concatenate([x.reshape(-1) for x in errs])
    assert e.max() <= 2e-2, f"max-abs {e.max()}"
    assert e.mean() <= 2e-3, f"mean-abs {e.mean()}"
    assert lerr <= 1e-3, f"lse {lerr}"
    return float(e.max()), float(e.mean()), lerr
