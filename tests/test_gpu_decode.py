"""Single-token decode on the GPU against the oracle, through the C ABI.

The cache is a packed batch whose last token per sequence is the new one;
q_new is that token's query.  Selection: the kept lists under the excuse
protocol of parity_util (a decode row is a prefill row with a one-token query
block).  Attention: bf16 output within max-abs 2e-2 / mean-abs 2e-3 of the
fp64 oracle, LSE within 1e-3, first on the oracle's own lists, then end to end
on rows whose GPU list equals the oracle's.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from parity_util import compare_mask_rows, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_kv_gb300 import build
    build.build()


def last_queries(vw, lay):
    cu = lay["cu_seqlens"]
    q = np.zeros((vw.batch, vw.hq, vw.head_dim), dtype=np.uint16)
    for b in range(vw.batch):
        if cu[b + 1] > cu[b]:
            q[b] = lay["q"][cu[b + 1] - 1]
    return q


def gpu_decode(vw, lay, q_new, rc=None, rr=None, lists=None):
    import block_sparse_long_kv_gb300 as bsa
    s = bsa.make_varlen_shape(vw.batch, vw.total, vw.max_seqlen, vw.hq, vw.hkv, vw.head_dim, vw.block)
    nbs = bsa.varlen_block_stride(s)
    cu = torch.from_numpy(lay["cu_seqlens"]).cuda()
    k, v = to_dev(lay["k"]), to_dev(lay["v"])
    qn = to_dev(q_new)
    meta = bsa.alloc_varlen_meta(s)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.varlen_block_meta(s, cu, k, meta["centroid"], meta["radius"], meta["quant"], meta["alpha"], st)
    kv_idx = torch.zeros(vw.batch, vw.hkv, nbs, dtype=torch.int32, device="cuda")
    kv_cnt = torch.zeros(vw.batch, vw.hkv, dtype=torch.int32, device="cuda")
    prm = bsa.SelectParams(vw.centroid_keep if rc is None else rc, vw.rescue_keep if rr is None else rr, 0)
    ws = torch.empty(bsa.decode_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    bsa.decode_select(s, prm, cu, qn, meta["centroid"], meta["radius"], meta["alpha"], kv_idx, kv_cnt,
                      ws, st)
    if lists is not None:
        kv_idx, kv_cnt = lists
    o = torch.full((vw.batch, vw.hq, vw.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((vw.batch, vw.hq), float("nan"), dtype=torch.float32, device="cuda")
    bsa.decode_fwd(s, cu, qn, k, v, kv_idx, kv_cnt, 1.0 / math.sqrt(vw.head_dim), o, lse, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    out = dict(kv_idx=kv_idx.cpu().numpy(), kv_cnt=kv_cnt.cpu().numpy(), o=o.float().cpu().numpy(),
               lse=lse.cpu().numpy(), nbs=nbs, alpha=meta["alpha"].cpu().numpy())
    if lists is None:
        # the one-launch step: the same lists bit for bit, and its own O / LSE (checked against
        # the oracle beside the two calls' by check_outputs)
        idx2 = torch.full_like(kv_idx, -7)
        cnt2 = torch.full_like(kv_cnt, -7)
        o2 = torch.full_like(o, float("nan"))
        lse2 = torch.full_like(lse, float("nan"))
        ws2 = torch.full_like(ws, 0xA5)
        bsa.decode_step(s, prm, cu, qn, k, v, meta["centroid"], meta["radius"], meta["alpha"],
                        1.0 / math.sqrt(vw.head_dim), idx2, cnt2, o2, lse2, ws2, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        cnt = out["kv_cnt"]
        np.testing.assert_array_equal(cnt2.cpu().numpy(), cnt)
        live = np.arange(nbs) < cnt[..., None]
        np.testing.assert_array_equal(idx2.cpu().numpy()[live], out["kv_idx"][live])
        out["o_step"] = o2.float().cpu().numpy()
        out["lse_step"] = lse2.cpu().numpy()
    return out


def oracle_decode(vw, lay, q_new, rc=None, rr=None):
    """Per (b, g): kept list and row scores, plus per-sequence meta, from the oracle."""
    rc = vw.centroid_keep if rc is None else rc
    rr = vw.rescue_keep if rr is None else rr
    k = synth.bf16_to_f64(lay["k"])
    qn = synth.bf16_to_f64(q_new)
    cu = lay["cu_seqlens"]
    out = {}
    for b in range(vw.batch):
        s0, s1 = O.seq_bounds(cu, b)
        n = s1 - s0
        if n == 0:
            continue
        cen, rad = O.block_meta(k[None, s0:s1], vw.block)
        med, p90 = O.radius_quantiles(rad)
        alpha = O.rescue_coefficient(rad, med, p90)
        for g in range(vw.hkv):
            kept, s_c, r = O.decode_select(qn[b], cen[0], rad[0], alpha[0], n, vw.block, rc, rr, g)
            i = (n - 1) // vw.block
            cent, resc = O.select_row(s_c, r, alpha[0, g], i, O.ratio_ppm(rc), O.ratio_ppm(rr))
            out[(b, g)] = dict(kept=kept, s_c=s_c, r=r, med=med[0, g], radius=rad[0, g], n=n,
                               cent=cent, resc=resc)
    return out


def compare_lists(vw, got, orc):
    """Decode rows under the mask protocol: row i of a per-(b, g) one-row mask."""
    nbs = got["nbs"]
    rows, gm = {}, np.zeros((vw.batch, vw.hkv, nbs, nbs), dtype=np.uint8)
    med = np.zeros((vw.batch, vw.hkv))
    rad = np.zeros((vw.batch, vw.hkv, nbs))
    for (b, g), d in orc.items():
        i = (d["n"] - 1) // vw.block
        m = np.zeros(nbs, dtype=np.uint8)
        sc = np.zeros(nbs)
        sr = np.zeros(nbs)
        sc[:d["s_c"].size], sr[:d["r"].size] = d["s_c"], d["r"]
        m[d["cent"]] |= O.CENTROID
        m[d["resc"]] |= O.RESCUE
        m[0] |= O.FORCED
        m[i] |= O.FORCED
        rows[(b, g, i)] = (m, sc, sr)
        c = got["kv_cnt"][b, g]
        js = got["kv_idx"][b, g, :c]
        row = np.zeros(nbs, dtype=np.uint8)
        row[js] = 1
        # the GPU list carries no path bits: a block both keep gets the oracle's bits; a block only
        # the GPU keeps is judged on the centroid path if its S_c sits at the centroid threshold,
        # else on the rescue path
        only = (row != 0) & (m == 0)
        t = sc[d["cent"]].min() if d["cent"].size else np.inf
        cands = sc[1:i]
        den = max(abs(t), 1e-3 * math.sqrt(float(np.mean(cands ** 2)))) if cands.size else 1.0
        at_c = np.abs(sc - t) <= 1e-4 * den
        gb = np.where(row != 0, m, 0).astype(np.uint8)
        gb[only & at_c] = O.CENTROID
        gb[only & ~at_c] = O.RESCUE
        gb[0] |= O.FORCED
        gb[i] |= O.FORCED
        gm[b, g, i] = gb
        med[b, g] = d["med"]
        rad[b, g, :d["radius"].size] = d["radius"]
    return compare_mask_rows(gm, dict(rows=rows, med=med, radius=rad))


def upload(vw, orc, nbs):
    idx = np.zeros((vw.batch, vw.hkv, nbs), dtype=np.int32)
    cnt = np.zeros((vw.batch, vw.hkv), dtype=np.int32)
    for (b, g), d in orc.items():
        idx[b, g, :d["kept"].size] = d["kept"]
        cnt[b, g] = d["kept"].size
    return torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda()


def check_outputs(vw, lay, q_new, got, kept_by_bg, bs=None):
    k, v = synth.bf16_to_f32(lay["k"]), synth.bf16_to_f32(lay["v"])
    qn = synth.bf16_to_f32(q_new)
    cu = lay["cu_seqlens"]
    errs, lerr = [], 0.0
    for b in range(vw.batch) if bs is None else bs:
        s0, s1 = O.seq_bounds(cu, b)
        if s1 == s0:
            continue
        per_g = [kept_by_bg[(b, g)] for g in range(vw.hkv)]
        o, lse = O.decode_attention(qn[b], k[s0:s1], v[s0:s1], per_g, s1 - s0, vw.block)
        for key in ("o", "o_step"):  # the two calls, and the one-launch step when it ran
            if key in got:
                errs.append(np.abs(got[key][b] - o).reshape(-1))
        for key in ("lse", "lse_step"):
            if key in got:
                lerr = max(lerr, float(np.abs(got[key][b] - lse).max()))
    e = np.concatenate(errs)
    assert e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())
    assert lerr <= 1e-3, lerr


@pytest.mark.parametrize("name", ["varlen_h2x1_d64_b64", "varlen_gqa32x4_d128_b128",
                                  "varlen_gqa32x4_d128_b64"])
def test_decode_select_and_attention(name):
    vw = synth.VARLEN_WORKLOADS[name]
    lay = synth.make_varlen_layer(vw)
    q_new = last_queries(vw, lay)
    got = gpu_decode(vw, lay, q_new)
    orc = oracle_decode(vw, lay, q_new)
    compared, excused = compare_lists(vw, got, orc)
    assert excused <= max(4, compared // 1000), (compared, excused)
    # attention on the oracle's lists
    lists = upload(vw, orc, got["nbs"])
    got2 = gpu_decode(vw, lay, q_new, lists=lists)
    check_outputs(vw, lay, q_new, got2, {bg: d["kept"] for bg, d in orc.items()})
    # end to end on the sequences whose GPU lists all equal the oracle's
    same = [b for b in range(vw.batch) if vw.lengths[b] > 0 and all(
        np.array_equal(got["kv_idx"][b, g, :got["kv_cnt"][b, g]], orc[(b, g)]["kept"])
        for g in range(vw.hkv))]
    assert same
    check_outputs(vw, lay, q_new, got, {bg: d["kept"] for bg, d in orc.items()}, bs=same)
    # an empty sequence decodes to zeros, in both paths
    for b, n in enumerate(vw.lengths):
        if n == 0:
            assert np.all(got["o"][b] == 0) and np.all(np.isneginf(got["lse"][b]))
            assert np.all(got["o_step"][b] == 0) and np.all(np.isneginf(got["lse_step"][b]))


def test_decode_keep_all_equals_dense():
    vw = synth.VARLEN_WORKLOADS["varlen_gqa32x4_d128_b128"]
    lay = synth.make_varlen_layer(vw)
    q_new = last_queries(vw, lay)
    got = gpu_decode(vw, lay, q_new, rc=1.0, rr=0.0)
    for b, n in enumerate(vw.lengths):
        nb = -(-n // vw.block)
        for g in range(vw.hkv):
            np.testing.assert_array_equal(got["kv_idx"][b, g, :got["kv_cnt"][b, g]], np.arange(nb))
    kept = {(b, g): np.arange(-(-n // vw.block)) for b, n in enumerate(vw.lengths) for g in range(vw.hkv)}
    check_outputs(vw, lay, q_new, got, kept)


@pytest.mark.parametrize("cfg", [
    dict(hq=16, hkv=1, head_dim=128, block=128),   # G = 16
    dict(hq=8, hkv=8, head_dim=64, block=256),     # G = 1, d = 64, block 256
    dict(hq=8, hkv=2, head_dim=128, block=64),     # G = 4, block 64
    dict(hq=4, hkv=2, head_dim=64, block=128),     # G = 2, d = 64
])
def test_decode_shape_variants(cfg):
    vw = synth.VarlenWorkload("dec", (3000, 777, 4096), cfg["hq"], cfg["hkv"], cfg["head_dim"],
                              cfg["block"], 0.2, 0.05, seed_base=321, needles_fixed=1)
    lay = synth.make_varlen_layer(vw)
    q_new = last_queries(vw, lay)
    got = gpu_decode(vw, lay, q_new)
    orc = oracle_decode(vw, lay, q_new)
    compared, excused = compare_lists(vw, got, orc)
    assert excused <= max(4, compared // 1000), (compared, excused)
    lists = upload(vw, orc, got["nbs"])
    got2 = gpu_decode(vw, lay, q_new, lists=lists)
    check_outputs(vw, lay, q_new, got2, {bg: d["kept"] for bg, d in orc.items()})


@pytest.mark.parametrize("nb", [1000, 2000, 3000, 4096])
def test_decode_select_long_rows_synthetic_meta(nb):
    """Rows of 1000 to 4096 blocks (every register width of the CTA-wide select, up to the
    library's block limit) on synthetic block summaries: sequence 0 random, sequence 1 with
    every centroid, radius and alpha equal so both paths rank pure ties (lowest index
    first)."""
    import block_sparse_long_kv_gb300 as bsa
    block, hq, hkv, d = 64, 8, 2, 64
    lengths = (nb * block, nb * block - 37)
    vw = synth.VarlenWorkload("dec_meta", lengths, hq, hkv, d, block, 0.1, 0.05)
    s = bsa.make_varlen_shape(vw.batch, vw.total, vw.max_seqlen, hq, hkv, d, block)
    nbs = bsa.varlen_block_stride(s)
    rng = np.random.default_rng(nb)
    cen = rng.standard_normal((2, hkv, nbs, d)).astype(np.float32)
    rad = np.exp(rng.uniform(-1, 1, (2, hkv, nbs))).astype(np.float32)
    alpha = np.where(rng.random((2, hkv, nbs)) < 0.5, 0.0, rng.random((2, hkv, nbs))).astype(np.float32)
    cen[1] = cen[1, :, :1]
    rad[1] = 1.5
    alpha[1] = 0.5
    q_new = synth.bf16_bits(rng.standard_normal((2, hq, d)).astype(np.float32))
    cu = torch.tensor(vw.cu_seqlens(), dtype=torch.int32, device="cuda")
    kv_idx = torch.zeros(2, hkv, nbs, dtype=torch.int32, device="cuda")
    kv_cnt = torch.zeros(2, hkv, dtype=torch.int32, device="cuda")
    ws = torch.empty(bsa.decode_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.decode_select(s, bsa.SelectParams(vw.centroid_keep, vw.rescue_keep, 0), cu, to_dev(q_new),
                      torch.from_numpy(cen).cuda(), torch.from_numpy(rad).cuda(),
                      torch.from_numpy(alpha).cuda(), kv_idx, kv_cnt, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = dict(kv_idx=kv_idx.cpu().numpy(), kv_cnt=kv_cnt.cpu().numpy(), nbs=nbs)
    qn = synth.bf16_to_f64(q_new)
    orc = {}
    for b, n in enumerate(lengths):
        nbb = -(-n // block)
        i = (n - 1) // block
        for g in range(hkv):
            c64, r64, a64 = (x[b, :, :nbb].astype(np.float64) for x in (cen, rad, alpha))
            kept, s_c, r = O.decode_select(qn[b], c64, r64, a64, n, block, vw.centroid_keep,
                                           vw.rescue_keep, g)
            cent, resc = O.select_row(s_c, r, a64[g], i, O.ratio_ppm(vw.centroid_keep),
                                      O.ratio_ppm(vw.rescue_keep))
            orc[(b, g)] = dict(kept=kept, s_c=s_c, r=r, med=-1.0, radius=r64[g], n=n, cent=cent,
                               resc=resc)
    compared, excused = compare_lists(vw, got, orc)
    assert excused <= max(4, compared // 1000), (compared, excused)
    for g in range(hkv):  # pure ties: bit-exact, lowest indices first
        np.testing.assert_array_equal(got["kv_idx"][1, g, :got["kv_cnt"][1, g]], orc[(1, g)]["kept"])
    # the one-launch step selects with a team of warps (P = 8, 16 or 32 entries per lane at these
    # row lengths): the same lists bit for bit (a zero cache: only the selection is compared)
    kz = torch.zeros(vw.total, hkv, d, dtype=torch.bfloat16, device="cuda")
    idx2 = torch.full_like(kv_idx, -7)
    cnt2 = torch.full_like(kv_cnt, -7)
    o2 = torch.empty(2, hq, d, dtype=torch.bfloat16, device="cuda")
    bsa.decode_step(s, bsa.SelectParams(vw.centroid_keep, vw.rescue_keep, 0), cu, to_dev(q_new), kz, kz,
                    torch.from_numpy(cen).cuda(), torch.from_numpy(rad).cuda(), torch.from_numpy(alpha).cuda(),
                    1.0 / math.sqrt(d), idx2, cnt2, o2, None, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(cnt2.cpu().numpy(), got["kv_cnt"])
    live = np.arange(nbs) < got["kv_cnt"][..., None]
    np.testing.assert_array_equal(idx2.cpu().numpy()[live], got["kv_idx"][live])


def test_decode_many_rows_and_malformed_entries():
    """64 sequences (some empty, some one block, some long) so the even cut of all
    rows' entries over the CTAs falls both inside rows and between them; then the same
    lists with malformed entries appended (a block past the sequence, a negative index):
    the attention skips them and still equals the oracle over the valid entries."""
    rng = np.random.default_rng(77)
    lengths = tuple(int(x) for x in rng.choice([0, 1, 63, 64, 65, 700, 3000, 9000, 20000], size=64))
    vw = synth.VarlenWorkload("dec_many", lengths, 16, 2, 128, 64, 0.15, 0.05, seed_base=909,
                              needles_fixed=1)
    lay = synth.make_varlen_layer(vw)
    q_new = last_queries(vw, lay)
    got = gpu_decode(vw, lay, q_new)
    orc = oracle_decode(vw, lay, q_new)
    compared, excused = compare_lists(vw, got, orc)
    assert excused <= max(4, compared // 1000), (compared, excused)
    lists = upload(vw, orc, got["nbs"])
    got2 = gpu_decode(vw, lay, q_new, lists=lists)
    kept = {bg: d["kept"] for bg, d in orc.items()}
    check_outputs(vw, lay, q_new, got2, kept)
    for b, n in enumerate(vw.lengths):
        if n == 0:
            assert np.all(got2["o"][b] == 0) and np.all(np.isneginf(got2["lse"][b]))
            assert np.all(got["o_step"][b] == 0) and np.all(np.isneginf(got["lse_step"][b]))
    # end to end, both paths, on the sequences whose GPU lists all equal the oracle's
    same = [b for b in range(vw.batch) if vw.lengths[b] > 0 and all(
        np.array_equal(got["kv_idx"][b, g, :got["kv_cnt"][b, g]], orc[(b, g)]["kept"])
        for g in range(vw.hkv))]
    assert len(same) >= sum(1 for n in vw.lengths if n > 0) // 2
    check_outputs(vw, lay, q_new, got, kept, bs=same)
    # malformed entries after the valid ones: skipped by the attention
    idx, cnt = (x.cpu().numpy().copy() for x in lists)
    for (b, g), d in orc.items():
        c = d["kept"].size
        nb = -(-vw.lengths[b] // vw.block)
        extra = [nb + 3, -1]
        room = min(len(extra), got["nbs"] - c)
        idx[b, g, c:c + room] = extra[:room]
        cnt[b, g] = c + room
    got3 = gpu_decode(vw, lay, q_new, lists=(torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda()))
    check_outputs(vw, lay, q_new, got3, kept)


@pytest.mark.parametrize("nb", [500, 1024])
def test_decode_step_tied_templates_exact(nb):
    """Exact ties inside small threshold bins (ranked directly by one warp): block j's summary is
    template j % 48, centroid (m + 1) / 64 along dimension 0, radius 0.5 with alpha 1 on every
    fourth template and 0.125 with alpha 0 elsewhere, and the new token is e_0 in every head.  All
    scores are exact in fp32 and fp64, so the one-launch step's lists equal the oracle's bit for
    bit: of equal scores the lowest block indices are kept, in both paths."""
    import block_sparse_long_kv_gb300 as bsa
    block, hq, hkv, d, templates = 64, 8, 2, 64, 48
    lengths = (nb * block,)
    vw = synth.VarlenWorkload("dec_ties", lengths, hq, hkv, d, block, 0.1, 0.05)
    s = bsa.make_varlen_shape(vw.batch, vw.total, vw.max_seqlen, hq, hkv, d, block)
    nbs = bsa.varlen_block_stride(s)
    m = np.arange(nbs) % templates
    cen = np.zeros((1, hkv, nbs, d), dtype=np.float32)
    cen[..., 0] = ((m + 1) / 64.0)[None, None, :]
    wide = m % 4 == 0
    rad = np.broadcast_to(np.where(wide, 0.5, 0.125).astype(np.float32), (1, hkv, nbs)).copy()
    alpha = np.broadcast_to(np.where(wide, 1.0, 0.0).astype(np.float32), (1, hkv, nbs)).copy()
    qf = np.zeros((1, hq, d), dtype=np.float32)
    qf[..., 0] = 1.0
    q_new = synth.bf16_bits(qf)
    cu = torch.tensor(vw.cu_seqlens(), dtype=torch.int32, device="cuda")
    kz = torch.zeros(vw.total, hkv, d, dtype=torch.bfloat16, device="cuda")
    kv_idx = torch.full((1, hkv, nbs), -7, dtype=torch.int32, device="cuda")
    kv_cnt = torch.full((1, hkv), -7, dtype=torch.int32, device="cuda")
    o = torch.empty(1, hq, d, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(bsa.decode_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.decode_step(s, bsa.SelectParams(vw.centroid_keep, vw.rescue_keep, 0), cu, to_dev(q_new), kz, kz,
                    torch.from_numpy(cen).cuda(), torch.from_numpy(rad).cuda(), torch.from_numpy(alpha).cuda(),
                    1.0 / math.sqrt(d), kv_idx, kv_cnt, o, None, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    n = lengths[0]
    i = (n - 1) // block
    qn = synth.bf16_to_f64(q_new)
    c64, r64, a64 = (x[0, :, :nb].astype(np.float64) for x in (cen, rad, alpha))
    for g in range(hkv):
        kept, _, _ = O.decode_select(qn[0], c64, r64, a64, n, block, vw.centroid_keep, vw.rescue_keep, g)
        cnt = int(kv_cnt[0, g].item())
        np.testing.assert_array_equal(kv_idx[0, g, :cnt].cpu().numpy(), kept, err_msg=f"g {g}")
    # the rows do split tie groups: some template is only partly kept
    kept_set = set(kept.tolist())
    cands = [[j for j in range(1, i) if j % templates == t] for t in range(templates)]
    split = [t for t in range(templates) if 0 < sum(j in kept_set for j in cands[t]) < len(cands[t])]
    assert split, "no tie group is split at the thresholds"
