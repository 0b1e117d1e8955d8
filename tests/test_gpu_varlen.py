"""Packed ragged batches on the GPU against the oracle, through the C ABI.

Sequences of any length (including empty ones and lengths that are not a
multiple of the block) are packed along one token axis; every sequence must
match the oracle run on that sequence alone: meta within 1e-5, masks under
the excuse protocol of parity_util, attention within the bf16 bounds.  A
fixed-length batch sent through the varlen entry points must give the
fixed-length results bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from parity_util import compare_mask_rows, shape_of, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_kv_gb300 import build
    build.build()


def vshape(vw):
    import block_sparse_long_kv_gb300 as bsa
    return bsa.make_varlen_shape(vw.batch, vw.total, vw.max_seqlen, vw.hq, vw.hkv, vw.head_dim,
                                 vw.block)


def gpu_varlen(vw, lay, kv=None, rc=None, rr=None, cu=None, dense=False, flags=0):
    """Mask build + attention of a packed batch; numpy results and the device status."""
    import block_sparse_long_kv_gb300 as bsa
    s = vshape(vw)
    cu_d = torch.from_numpy(lay["cu_seqlens"] if cu is None else cu).cuda()
    q, k, v = (to_dev(lay[x]) for x in ("q", "k", "v"))
    meta = bsa.alloc_varlen_meta(s)
    sel = bsa.alloc_varlen_select(s)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.varlen_block_meta(s, cu_d, k, meta["centroid"], meta["radius"], meta["quant"],
                          meta["alpha"], st)
    prm = bsa.SelectParams(vw.centroid_keep if rc is None else rc,
                           vw.rescue_keep if rr is None else rr, flags)
    bsa.varlen_select_mask(s, prm, cu_d, q, meta["centroid"], meta["radius"], meta["alpha"],
                           sel["kv_idx"], sel["kv_cnt"], sel["mask"], dev_status=st)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((vw.hq, vw.total), float("nan"), dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(vw.head_dim)
    if dense:
        bsa.varlen_prefill_dense_fwd(s, cu_d, q, k, v, scale, o, lse, st)
    else:
        idx, cnt = (sel["kv_idx"], sel["kv_cnt"]) if kv is None else kv
        bsa.varlen_prefill_fwd(s, cu_d, q, k, v, idx, cnt, scale, o, lse, st)
    torch.cuda.synchronize()
    out = {x: t.cpu().numpy() for x, t in {**meta, **sel}.items()}
    out["o"] = o.float().cpu().numpy()
    out["lse"] = lse.cpu().numpy()
    out["status"] = int(st.item())
    out["nbs"] = bsa.varlen_block_stride(s)
    return out


def oracle_varlen(vw, lay, rc=None, rr=None, token_max=False):
    q = synth.bf16_to_f64(lay["q"])
    k = synth.bf16_to_f64(lay["k"])
    return O.varlen_select_blocks(q, k, lay["cu_seqlens"], vw.block,
                                  vw.centroid_keep if rc is None else rc,
                                  vw.rescue_keep if rr is None else rr, with_scores=True,
                                  token_max=token_max)


def padded_oracle(vw, res, nbs):
    """Oracle results in the padded [batch, hkv, nbs, ...] layout of the varlen ABI."""
    b, hkv, d = vw.batch, vw.hkv, vw.head_dim
    cen = np.zeros((b, hkv, nbs, d))
    rad = np.zeros((b, hkv, nbs))
    alpha = np.zeros((b, hkv, nbs))
    med = np.zeros((b, hkv))
    p90 = np.zeros((b, hkv))
    keep = np.zeros((b, hkv, nbs, nbs), dtype=np.uint8)
    rows = {}
    for bi, r in enumerate(res):
        nb = r["mask"].shape[-1]
        cen[bi, :, :nb] = r["centroid"][0]
        rad[bi, :, :nb] = r["radius"][0]
        alpha[bi, :, :nb] = r["alpha"][0]
        med[bi], p90[bi] = r["med"][0], r["p90"][0]
        keep[bi, :, :nb, :nb] = r["mask"][0]
        for g in range(hkv if nb else 0):
            s_c, s_r = r["scores"][(0, g)]
            for i in range(nb):
                m = np.zeros(nbs, dtype=np.uint8)
                m[:nb] = r["mask"][0, g, i]
                sc = np.zeros(nbs)
                sr = np.zeros(nbs)
                sc[:nb], sr[:nb] = s_c[i], s_r[i]
                rows[(bi, g, i)] = (m, sc, sr)
    return dict(centroid=cen, radius=rad, alpha=alpha, med=med, p90=p90, keep=keep, rows=rows)


def lists_of(keep):
    idx, cnt = O.kv_lists(keep)
    return torch.from_numpy(np.ascontiguousarray(idx)).cuda(), torch.from_numpy(cnt).cuda()


def check_varlen_attention(vw, lay, got, keep, rows):
    """rows: (b, h, i).  GPU O / LSE against the oracle with the given per-sequence masks."""
    q, k, v = (synth.bf16_to_f32(lay[x]) for x in ("q", "k", "v"))
    cu = lay["cu_seqlens"]
    masks = [keep[b:b + 1] != 0 for b in range(vw.batch)]
    ref = O.varlen_attention_rows(q, k, v, cu, masks, vw.block, rows)
    errs, lerr = [], 0.0
    for (b, h, i), (oi, li) in ref.items():
        s0 = int(cu[b]) + i * vw.block
        n = oi.shape[0]
        errs.append(np.abs(got["o"][s0:s0 + n, h] - oi).reshape(-1))
        lerr = max(lerr, float(np.abs(got["lse"][h, s0:s0 + n] - li).max()))
    e = np.concatenate(errs)
    assert e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())
    assert lerr <= 1e-3, lerr


def check_meta_and_masks(vw, got, orc):
    scale = max(np.abs(orc["centroid"]).max(), 1.0)
    assert np.abs(got["centroid"] - orc["centroid"]).max() <= 1e-5 * scale
    np.testing.assert_allclose(got["radius"], orc["radius"], rtol=1e-5, atol=1e-7)
    assert np.abs(got["alpha"] - orc["alpha"]).max() <= 1e-3
    compared, excused = compare_mask_rows(got["mask"], orc)
    assert excused <= max(4, compared // 1000), (compared, excused)
    # padding: lists of rows past a sequence's blocks are empty, their mask rows zero
    for b, n in enumerate(vw.lengths):
        nb = -(-n // vw.block)
        assert np.all(got["kv_cnt"][b, :, nb:] == 0)
        assert np.all(got["mask"][b, :, nb:] == 0)
        assert np.all(got["mask"][b, :, :, nb:] == 0)
    return compared, excused


def test_varlen_tiny_full():
    vw = synth.VARLEN_WORKLOADS["varlen_h2x1_d64_b64"]
    lay = synth.make_varlen_layer(vw)
    res = oracle_varlen(vw, lay)
    got = gpu_varlen(vw, lay)
    assert got["status"] == 0
    orc = padded_oracle(vw, res, got["nbs"])
    check_meta_and_masks(vw, got, orc)
    # attention on the oracle's own lists, every row of every sequence
    kv = lists_of(orc["keep"])
    got2 = gpu_varlen(vw, lay, kv=kv)
    rows = [(b, h, i) for b, n in enumerate(vw.lengths) for h in range(vw.hq)
            for i in range(-(-n // vw.block))]
    check_varlen_attention(vw, lay, got2, orc["keep"], rows)
    assert not np.isnan(got2["o"]).any() and not np.isnan(got2["lse"]).any()


def test_varlen_tiny_dense_equals_oracle_dense():
    vw = synth.VARLEN_WORKLOADS["varlen_h2x1_d64_b64"]
    lay = synth.make_varlen_layer(vw)
    got = gpu_varlen(vw, lay, dense=True)
    assert got["status"] == 0
    q, k, v = (synth.bf16_to_f64(lay[x]) for x in ("q", "k", "v"))
    od, ld = O.varlen_dense_attention(q, k, v, lay["cu_seqlens"])
    assert np.abs(got["o"] - od).max() <= 2e-2 and np.abs(got["o"] - od).mean() <= 2e-3
    assert np.abs(got["lse"] - ld).max() <= 1e-3


@pytest.mark.parametrize("name", ["varlen_gqa32x4_d128_b128", "varlen_gqa32x4_d128_b64"])
def test_varlen_gqa_masks_full_attention_sampled(name):
    vw = synth.VARLEN_WORKLOADS[name]
    lay = synth.make_varlen_layer(vw)
    res = oracle_varlen(vw, lay)
    got = gpu_varlen(vw, lay)
    assert got["status"] == 0
    orc = padded_oracle(vw, res, got["nbs"])
    check_meta_and_masks(vw, got, orc)
    rng = np.random.default_rng(3)
    rows = []
    for b, n in enumerate(vw.lengths):
        nb = -(-n // vw.block)
        if nb == 0:
            continue
        for h in (0, vw.hq - 1, int(rng.integers(0, vw.hq))):
            for i in sorted({0, nb - 1, int(rng.integers(0, nb))}):
                rows.append((b, h, i))
    # end to end on rows whose GPU mask equals the oracle's
    same = [(b, h, i) for (b, h, i) in rows
            if np.array_equal(got["mask"][b, h // vw.group, i], orc["keep"][b, h // vw.group, i])]
    assert same
    check_varlen_attention(vw, lay, got, orc["keep"], same)


def test_fixed_batch_through_varlen_is_bit_identical():
    import block_sparse_long_kv_gb300 as bsa
    from parity_util import gpu_mask_build, gpu_attention
    w = synth.Workload("var", 2, 2048, 8, 2, 128, 128, 0.25, 0.05, seed_base=99, needles_fixed=1)
    lay = synth.make_layer(w)
    fixed = gpu_mask_build(w, lay)
    o_f, l_f = gpu_attention(w, lay, torch.from_numpy(fixed["kv_idx"]).cuda(),
                             torch.from_numpy(fixed["kv_cnt"]).cuda())
    vw = synth.VarlenWorkload("as_varlen", (2048, 2048), 8, 2, 128, 128, 0.25, 0.05)
    vlay = {x: np.ascontiguousarray(lay[x].reshape(-1, *lay[x].shape[2:])) for x in ("q", "k", "v")}
    vlay["cu_seqlens"] = vw.cu_seqlens()
    got = gpu_varlen(vw, vlay)
    assert got["status"] == 0 and got["nbs"] == 16
    for x in ("centroid", "radius", "quant", "alpha", "kv_cnt", "mask"):
        np.testing.assert_array_equal(got[x], fixed[x], err_msg=x)
    np.testing.assert_array_equal(got["o"].reshape(o_f.shape), o_f)
    np.testing.assert_array_equal(got["lse"].reshape(8, 2, 2048).transpose(1, 0, 2), l_f)


def test_inconsistent_cu_seqlens_is_reported_not_faulted():
    vw = synth.VARLEN_WORKLOADS["varlen_h2x1_d64_b64"]
    lay = synth.make_varlen_layer(vw)
    bad = lay["cu_seqlens"].copy()
    bad[-1] = vw.total + 100                             # the last sequence runs past the tokens
    got = gpu_varlen(vw, lay, cu=bad)
    assert got["status"] == 1                            # BSA_ERR_INVALID_ARG
    last = vw.batch - 1
    assert np.all(got["kv_cnt"][last] == 0) and np.all(got["centroid"][last] == 0)
    # the other sequences are untouched by the bad entry
    good = gpu_varlen(vw, lay)
    assert good["status"] == 0
    for x in ("mask", "kv_cnt", "centroid", "radius"):
        np.testing.assert_array_equal(got[x][:last], good[x][:last])
    n = int(lay["cu_seqlens"][last])
    np.testing.assert_array_equal(got["o"][:n], good["o"][:n])


def test_varlen_token_max_masks():
    from block_sparse_long_kv_gb300 import SELECT_TOKEN_MAX
    vw = synth.VARLEN_WORKLOADS["varlen_h2x1_d64_b64"]
    lay = synth.make_varlen_layer(vw)
    res = oracle_varlen(vw, lay, token_max=True)
    got = gpu_varlen(vw, lay, flags=SELECT_TOKEN_MAX)
    assert got["status"] == 0
    check_meta_and_masks(vw, got, padded_oracle(vw, res, got["nbs"]))
