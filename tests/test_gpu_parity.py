"""GPU-vs-oracle parity through the C ABI (needs a GB300 and the built library).

Masks: bit-exact up to the excuse protocol in parity_util.  Attention: bf16
output within max-abs 2e-2 and mean-abs 2e-3 of the fp64 oracle, LSE within
1e-3.  Meta: centroid / radius within 1e-5 relative, quantiles at the same rank.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from parity_util import (check_attention_rows, check_lists_match_mask, check_meta,
                         compare_mask_rows, gpu_attention, gpu_mask_build, oracle_rows, shape_of,
                         to_dev, upload_lists)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_kv_gb300 import build
    build.build()


def all_rows(w):
    return {(b, g): list(range(w.nb)) for b in range(w.batch) for g in range(w.hkv)}


def full_mask_parity(w, lay, rc=None, rr=None, rows=None):
    got = gpu_mask_build(w, lay, rc, rr)
    check_lists_match_mask(got["mask"], got["kv_idx"], got["kv_cnt"])
    orc = oracle_rows(w, lay, rows or all_rows(w), rc, rr)
    check_meta(w, lay, got, orc)
    compared, excused = compare_mask_rows(got["mask"], orc)
    assert excused <= max(4, compared // 1000), (compared, excused)
    return got, orc, excused


def oracle_keep(w, orc):
    keep = np.zeros((w.batch, w.hkv, w.nb, w.nb), dtype=np.uint8)
    for (b, g, i), (m, _, _) in orc["rows"].items():
        keep[b, g, i] = m
    return keep


def sample_rows(w, per_group, seed=0):
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(w.batch):
        for h in range(w.hq):
            iss = {0, w.nb - 1, w.nb // 2} | set(rng.integers(0, w.nb, per_group).tolist())
            rows += [(b, h, int(i)) for i in sorted(iss)]
    return rows


# ------------------------------------------------------------------ tiny, full coverage

def test_tiny_mask_and_attention_full():
    w = synth.workload("tiny_h2x1_n1024_d64_b64")
    lay = synth.make_layer(w)
    got, orc, _ = full_mask_parity(w, lay)
    keep = oracle_keep(w, orc)
    kv_idx, kv_cnt = upload_lists(keep)
    o, lse = gpu_attention(w, lay, kv_idx, kv_cnt)
    rows = [(0, h, i) for h in range(w.hq) for i in range(w.nb)]
    check_attention_rows(w, lay, o, lse, keep != 0, rows)


def test_tiny_dense_equals_oracle_dense():
    w = synth.workload("tiny_h2x1_n1024_d64_b64")
    lay = synth.make_layer(w)
    o, lse = gpu_attention(w, lay)
    q, k, v = (synth.bf16_to_f64(lay[x]) for x in ("q", "k", "v"))
    od, ld = O.dense_attention(q, k, v)
    assert np.abs(o - od).max() <= 2e-2 and np.abs(o - od).mean() <= 2e-3
    assert np.abs(lse - ld).max() <= 1e-3


def test_tiny_needles_kept():
    w = synth.workload("tiny_h2x1_n1024_d64_b64")
    lay = synth.make_layer(w)
    got = gpu_mask_build(w, lay)
    hit = tot = 0
    for (b, g, jb, slot, pos) in lay["needles"]:
        for i in sorted(set((pos // w.block).tolist())):
            tot += 1
            hit += bool(got["mask"][b, g, i, jb])
    assert tot > 0 and hit / tot >= 0.5


# ------------------------------------------------------------------ GQA 32/4, head_dim 128

@pytest.mark.parametrize("name", ["gqa32x4_n8192_d128_b128", "gqa32x4_n32768_d128_b128"])
def test_gqa_mask_full_attention_sampled(name):
    w = synth.workload(name)
    lay = synth.make_layer(w)
    got, orc, excused = full_mask_parity(w, lay)
    keep = oracle_keep(w, orc)
    kv_idx, kv_cnt = upload_lists(keep)
    o, lse = gpu_attention(w, lay, kv_idx, kv_cnt)
    check_attention_rows(w, lay, o, lse, keep != 0, sample_rows(w, 3))
    # end to end through the GPU's own lists on rows whose masks match the oracle's
    o2, lse2 = gpu_attention(w, lay, torch.from_numpy(got["kv_idx"]).cuda(),
                             torch.from_numpy(got["kv_cnt"]).cuda())
    rows = [(b, h, i) for (b, h, i) in sample_rows(w, 3, seed=1)
            if np.array_equal(got["mask"][b, h // w.group, i], keep[b, h // w.group, i])]
    assert rows
    check_attention_rows(w, lay, o2, lse2, keep != 0, rows)


@pytest.mark.parametrize("block", [64, 256])
def test_block_size_variants(block):
    w = synth.Workload(f"gqa_b{block}", 1, 8192, 32, 4, 128, block, 0.1, 0.02, seed_base=4000)
    lay = synth.make_layer(w)
    got, orc, _ = full_mask_parity(w, lay)
    keep = oracle_keep(w, orc)
    kv_idx, kv_cnt = upload_lists(keep)
    o, lse = gpu_attention(w, lay, kv_idx, kv_cnt)
    check_attention_rows(w, lay, o, lse, keep != 0, sample_rows(w, 2))


@pytest.mark.parametrize("rc, rr", [(0.0, 0.0), (0.05, 0.0), (0.2, 0.05), (1.0, 0.0)])
def test_keep_ratio_variants(rc, rr):
    w = synth.workload("gqa32x4_n8192_d128_b128")
    lay = synth.make_layer(w, seed=77)
    got, orc, _ = full_mask_parity(w, lay, rc, rr)
    if rc == 1.0:
        # every causal block kept: the sparse path must equal the dense path bit for bit
        o_s, l_s = gpu_attention(w, lay, torch.from_numpy(got["kv_idx"]).cuda(),
                                 torch.from_numpy(got["kv_cnt"]).cuda())
        o_d, l_d = gpu_attention(w, lay)
        np.testing.assert_array_equal(o_s, o_d)
        np.testing.assert_array_equal(l_s, l_d)
    if rc == 0.0 and rr == 0.0:
        assert np.all(got["kv_cnt"][..., 1:] == 2) and np.all(got["kv_cnt"][..., 0] == 1)


@pytest.mark.parametrize("cfg", [
    dict(batch=2, seq=2048, hq=8, hkv=8, head_dim=128, block=128),   # G = 1
    dict(batch=1, seq=4096, hq=16, hkv=1, head_dim=128, block=128),  # G = 16
    dict(batch=1, seq=2048, hq=8, hkv=2, head_dim=64, block=128),    # d = 64, block 128
    dict(batch=1, seq=4096, hq=8, hkv=2, head_dim=64, block=256),    # d = 64, block 256
    dict(batch=2, seq=256, hq=4, hkv=2, head_dim=128, block=64),     # nb = 4, minimum
])
def test_shape_variants(cfg):
    w = synth.Workload("var", cfg["batch"], cfg["seq"], cfg["hq"], cfg["hkv"], cfg["head_dim"],
                       cfg["block"], 0.25, 0.05, seed_base=99, needles_fixed=1)
    lay = synth.make_layer(w)
    got, orc, _ = full_mask_parity(w, lay)
    keep = oracle_keep(w, orc)
    kv_idx, kv_cnt = upload_lists(keep)
    o, lse = gpu_attention(w, lay, kv_idx, kv_cnt)
    check_attention_rows(w, lay, o, lse, keep != 0, sample_rows(w, 2))
    o_d, l_d = gpu_attention(w, lay)
    rows = sample_rows(w, 1, seed=3)
    check_attention_rows(w, lay, o_d, l_d, np.ones_like(keep, dtype=bool), rows)


def test_deterministic_and_layer_entry_point():
    import block_sparse_long_kv_gb300 as bsa
    w = synth.workload("gqa32x4_n8192_d128_b128")
    lay = synth.make_layer(w)
    s = shape_of(w)
    q, k, v = (to_dev(lay[x]) for x in ("q", "k", "v"))
    ws = bsa.alloc_layer_workspace(s)
    prm = bsa.SelectParams(w.centroid_keep, w.rescue_keep, 0)
    outs = []
    for _ in range(2):
        o = torch.empty_like(q)
        lse = torch.empty(w.batch, w.hq, w.seq, dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        bsa.prefill_layer(s, prm, q, k, v, 1 / math.sqrt(w.head_dim), o, lse, ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs.append((o.clone(), lse.clone(), bsa.layer_views(s, ws)["kv_cnt"].clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    got = gpu_mask_build(w, lay)
    np.testing.assert_array_equal(outs[0][2].cpu().numpy(), got["kv_cnt"])


def test_concurrent_streams_match_sequential():
    """Two layers in flight at once on two streams, each with its own workspace, give the same
    bits as the same calls one after the other: the layer path keeps no state across calls
    outside the caller's buffers."""
    import block_sparse_long_kv_gb300 as bsa
    w = synth.workload("gqa32x4_n8192_d128_b128")
    s = shape_of(w)
    prm = bsa.SelectParams(w.centroid_keep, w.rescue_keep, 0)
    scale = 1 / math.sqrt(w.head_dim)
    inputs = []
    for layer in range(2):
        lay = synth.make_layer(w, layer=layer)
        inputs.append(tuple(to_dev(lay[x]) for x in ("q", "k", "v")))

    def run(q, k, v, stream):
        ws = bsa.alloc_layer_workspace(s)
        o = torch.empty_like(q)
        lse = torch.empty(w.batch, w.hq, w.seq, dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            bsa.prefill_layer(s, prm, q, k, v, scale, o, lse, ws, st, stream=stream)
        return o, lse, ws, st

    seq = []
    for q, k, v in inputs:
        o, lse, ws, st = run(q, k, v, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        seq.append((o, lse, bsa.layer_views(s, ws)["kv_idx"].clone(), bsa.layer_views(s, ws)["kv_cnt"].clone()))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):  # a few rounds, so the two streams' kernels overlap in different ways
        res = [run(q, k, v, st_) for (q, k, v), st_ in zip(inputs, streams)]
        torch.cuda.synchronize()
        for (o, lse, ws, st), (o0, lse0, idx0, cnt0) in zip(res, seq):
            assert int(st.item()) == 0
            assert torch.equal(o, o0) and torch.equal(lse, lse0)
            cnt = bsa.layer_views(s, ws)["kv_cnt"]
            assert torch.equal(cnt, cnt0)
            idx = bsa.layer_views(s, ws)["kv_idx"]
            live = torch.arange(idx.shape[-1], device="cuda") < cnt[..., None]
            assert torch.equal(idx[live], idx0[live])


# ------------------------------------------------------------------ any block count

@pytest.mark.parametrize("cfg", [
    dict(batch=2, seq=9 * 128, hq=32, hkv=4, head_dim=128, block=128),   # nb = 9 (1152-token prompt)
    dict(batch=1, seq=65 * 64, hq=32, hkv=4, head_dim=128, block=64),    # nb = 65 (4160 tokens)
    dict(batch=1, seq=3 * 256, hq=8, hkv=2, head_dim=64, block=256),     # nb = 3
    dict(batch=3, seq=2 * 128, hq=4, hkv=1, head_dim=128, block=128),    # nb = 2
    dict(batch=2, seq=128, hq=4, hkv=2, head_dim=64, block=128),         # nb = 1
])
def test_block_counts_not_multiple_of_four(cfg):
    """seq % block == 0 is the only shape rule: block counts that are not a multiple of 4 give
    every mask row and every attention row of the oracle (oracle lists), the GPU's own lists on
    the rows whose masks agree, per-token aggregation masks, and the whole-layer entry point."""
    import block_sparse_long_kv_gb300 as bsa
    w = synth.Workload("nb_any", cfg["batch"], cfg["seq"], cfg["hq"], cfg["hkv"], cfg["head_dim"],
                       cfg["block"], 0.25, 0.1, seed_base=909, needles_fixed=1)
    lay = synth.make_layer(w)
    got, orc, _ = full_mask_parity(w, lay)
    keep = oracle_keep(w, orc)
    kv_idx, kv_cnt = upload_lists(keep)
    o, lse = gpu_attention(w, lay, kv_idx, kv_cnt)
    rows = [(b, h, i) for b in range(w.batch) for h in range(w.hq) for i in range(w.nb)]
    check_attention_rows(w, lay, o, lse, keep != 0, rows)
    o2, lse2 = gpu_attention(w, lay, torch.from_numpy(got["kv_idx"]).cuda(),
                             torch.from_numpy(got["kv_cnt"]).cuda())
    same = [(b, h, i) for (b, h, i) in rows
            if np.array_equal(got["mask"][b, h // w.group, i], keep[b, h // w.group, i])]
    assert len(same) >= len(rows) // 2
    check_attention_rows(w, lay, o2, lse2, keep != 0, same)
    token_parity(w, lay)
    # the whole-layer call equals the three separate calls bit for bit
    s = shape_of(w)
    q, k, v = (to_dev(lay[x]) for x in ("q", "k", "v"))
    ws = bsa.alloc_layer_workspace(s)
    o3 = torch.empty_like(q)
    lse3 = torch.empty(w.batch, w.hq, w.seq, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.prefill_layer(s, bsa.SelectParams(w.centroid_keep, w.rescue_keep, 0), q, k, v,
                      1 / math.sqrt(w.head_dim), o3, lse3, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(bsa.layer_views(s, ws)["kv_cnt"].cpu().numpy(), got["kv_cnt"])
    np.testing.assert_array_equal(o3.float().cpu().numpy(), o2)
    np.testing.assert_array_equal(lse3.cpu().numpy(), lse2)


# ------------------------------------------------------------------ maximum block count

def test_maximum_block_count():
    """The largest row the library takes: 4096 key blocks (262144 tokens at block 64), sampled
    mask rows (the first, the last and the longest included) and attention rows against the
    oracle."""
    w = synth.Workload("max_nb", 1, 4096 * 64, 2, 1, 64, 64, 0.02, 0.01, seed_base=4242, needles_fixed=4)
    lay = synth.make_layer(w)
    got = gpu_mask_build(w, lay)
    rng = np.random.default_rng(11)
    rows = {(0, 0): sorted({0, 1, 2, w.nb // 2, w.nb - 2, w.nb - 1} | set(rng.integers(0, w.nb, 10).tolist()))}
    orc = oracle_rows(w, lay, rows)
    compared, excused = compare_mask_rows(got["mask"], orc)
    assert excused <= max(4, compared // 1000), (compared, excused)
    check_lists_match_mask(got["mask"][:, :, -2:], got["kv_idx"][:, :, -2:], got["kv_cnt"][:, :, -2:])
    o, lse = gpu_attention(w, lay, torch.from_numpy(got["kv_idx"]).cuda(),
                           torch.from_numpy(got["kv_cnt"]).cuda())
    keep = oracle_keep(w, orc)
    att = [(0, h, i) for i in rows[(0, 0)] for h in range(w.hq)
           if np.array_equal(got["mask"][0, 0, i], keep[0, 0, i])]
    assert att
    check_attention_rows(w, lay, o, lse, keep != 0, att)


# ------------------------------------------------------------------ per-token aggregation

def token_parity(w, lay, rc=None, rr=None):
    from block_sparse_long_kv_gb300 import SELECT_TOKEN_MAX
    got = gpu_mask_build(w, lay, rc, rr, flags=SELECT_TOKEN_MAX)
    check_lists_match_mask(got["mask"], got["kv_idx"], got["kv_cnt"])
    orc = oracle_rows(w, lay, all_rows(w), rc, rr, token_max=True)
    compared, excused = compare_mask_rows(got["mask"], orc)
    assert excused <= max(4, compared // 1000), (compared, excused)
    return got, orc


@pytest.mark.parametrize("name", ["tiny_h2x1_n1024_d64_b64", "gqa32x4_n8192_d128_b128"])
def test_token_max_masks_full(name):
    w = synth.workload(name)
    lay = synth.make_layer(w)
    got, orc = token_parity(w, lay)
    # the per-token selection differs from the block-mean one and keeps the planted needles
    mean = gpu_mask_build(w, lay)
    assert not np.array_equal(got["mask"], mean["mask"])
    keep = oracle_keep(w, orc)
    kv_idx, kv_cnt = upload_lists(keep)
    o, lse = gpu_attention(w, lay, kv_idx, kv_cnt)
    check_attention_rows(w, lay, o, lse, keep != 0, sample_rows(w, 2))


@pytest.mark.parametrize("cfg", [
    dict(batch=2, seq=2048, hq=8, hkv=8, head_dim=128, block=128),   # G = 1
    dict(batch=1, seq=4096, hq=16, hkv=1, head_dim=128, block=128),  # G = 16
    dict(batch=1, seq=2048, hq=8, hkv=2, head_dim=64, block=64),     # d = 64, block 64
    dict(batch=1, seq=4096, hq=8, hkv=2, head_dim=128, block=256),   # block 256
    dict(batch=2, seq=256, hq=4, hkv=2, head_dim=128, block=64),     # nb = 4, minimum
])
def test_token_max_shape_variants(cfg):
    w = synth.Workload("tok", cfg["batch"], cfg["seq"], cfg["hq"], cfg["hkv"], cfg["head_dim"],
                       cfg["block"], 0.25, 0.05, seed_base=123, needles_fixed=1)
    token_parity(w, synth.make_layer(w))


def test_token_max_long_rows_sampled():
    # 32K tokens: 256 key blocks, two 128-block key tiles per CTA; sampled rows
    w = synth.workload("gqa32x4_n32768_d128_b128")
    lay = synth.make_layer(w)
    from block_sparse_long_kv_gb300 import SELECT_TOKEN_MAX
    got = gpu_mask_build(w, lay, flags=SELECT_TOKEN_MAX)
    rng = np.random.default_rng(11)
    rows = {(0, g): sorted({1, 2, 129, 130, 255} | set(rng.integers(0, w.nb, 12).tolist()))
            for g in range(w.hkv)}
    orc = oracle_rows(w, lay, rows, token_max=True)
    compared, excused = compare_mask_rows(got["mask"], orc)
    assert excused <= max(4, compared // 1000), (compared, excused)


def _tied_layer(nb, block, d, hq, templates):
    """K blocks copied from `templates` template blocks (block j is template j % templates), each
    an exactly representable centroid (m + 1) / 64 along dimension 0 plus a zero-mean +-a pattern
    on dimension 1 (a = 0.5 on every fourth template, else 0.125); every query token is e_0 plus a
    zero-mean +-1/16 pattern.  Every score is then exact in bf16, tf32 and fp64, the templates'
    scores are at least 2 % apart, and the copies of one template tie exactly."""
    n = nb * block
    t = np.arange(block)
    sign = np.where(t < block // 2, 1.0, -1.0).astype(np.float32)  # zero mean over a block
    k = np.zeros((1, n, 1, d), dtype=np.float32)
    for j in range(nb):
        m = j % templates
        a = 0.5 if m % 4 == 0 else 0.125
        k[0, j * block:(j + 1) * block, 0, 0] = (m + 1) / 64.0
        k[0, j * block:(j + 1) * block, 0, 1] = a * sign
    q = np.zeros((1, n, hq, d), dtype=np.float32)
    q[..., 0] = 1.0
    qs = np.where((np.arange(n) // 2) % 2 == 0, 1.0, -1.0).astype(np.float32)  # zero mean per block
    q[..., 2] = (qs / 16.0)[:, None]
    v = np.zeros((1, n, 1, d), dtype=np.float32)
    return {"q": synth.bf16_bits(q), "k": synth.bf16_bits(k), "v": synth.bf16_bits(v)}


@pytest.mark.parametrize("nb", [300, 1024])
def test_tied_blocks_exact(nb):
    """Exact ties at the selection thresholds of both paths: rows of up to 1024 blocks whose
    threshold bin holds up to 22 copies of one template (ranked directly by one warp, not by
    radix passes).  Masks and lists equal the oracle's bit for bit, no excuse: of equal scores
    the lowest block indices are kept."""
    block, d, hq, templates = 64, 64, 2, 48
    w = synth.Workload("tied", 1, nb * block, hq, 1, d, block, 0.10, 0.02)
    lay = _tied_layer(nb, block, d, hq, templates)
    got = gpu_mask_build(w, lay)
    check_lists_match_mask(got["mask"], got["kv_idx"], got["kv_cnt"])
    q64, k64 = synth.bf16_to_f64(lay["q"]), synth.bf16_to_f64(lay["k"])
    orc = O.select_blocks(q64, k64, block, w.centroid_keep, w.rescue_keep)
    assert float(orc["alpha"].max()) == 1.0 and float(orc["alpha"].min()) == 0.0  # both paths select
    rescued = int(((orc["mask"] & O.RESCUE) != 0).sum())
    assert rescued > 0
    bad = np.argwhere(got["mask"] != orc["mask"])
    assert bad.size == 0, f"{len(bad)} mask entries differ, first (b, g, i, j) {bad[:4].tolist()}"
