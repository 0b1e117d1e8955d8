"""FP8 (e4m3) inputs on the GPU against the oracle run on the dequantised values.

Inputs are the synthetic layers quantised to e4m3 with one power-of-two scale
per tensor (synth.fp8_layer).  The oracle sees value = e4m3(code) * scale in
fp64; the GPU path must match it under the same bars as the bf16 path: masks
under the excuse protocol, meta within 1e-5, bf16 O within max-abs 2e-2 and
mean-abs 2e-3, LSE within 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from parity_util import compare_mask_rows, shape_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_kv_gb300 import build
    build.build()


def dev8(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).cuda()


def deq(f8, name):
    return synth.e4m3_to_f64(f8[name]) * f8[name + "_scale"]


def gpu_fp8_mask(w, f8):
    import block_sparse_long_kv_gb300 as bsa
    s = shape_of(w)
    meta = bsa.alloc_meta(s)
    sel = bsa.alloc_select(s, with_mask=True)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.block_meta_fp8(s, dev8(f8["k"]), f8["k_scale"], meta["centroid"], meta["radius"], meta["quant"],
                       meta["alpha"], st)
    prm = bsa.SelectParams(w.centroid_keep, w.rescue_keep, 0)
    bsa.select_mask_fp8(s, prm, dev8(f8["q"]), f8["q_scale"], meta["centroid"], meta["radius"],
                        meta["alpha"], sel["kv_idx"], sel["kv_cnt"], sel["mask"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return {x: t.cpu().numpy() for x, t in {**meta, **sel}.items()}


def gpu_fp8_attention(w, f8, kv=None):
    import block_sparse_long_kv_gb300 as bsa
    s = shape_of(w)
    q, k, v = dev8(f8["q"]), dev8(f8["k"]), dev8(f8["v"])
    o = torch.full((w.batch, w.seq, w.hq, w.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.batch, w.hq, w.seq, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = 1.0 / math.sqrt(w.head_dim)
    if kv is None:
        bsa.prefill_dense_fwd_fp8(s, q, k, v, f8["q_scale"], f8["k_scale"], f8["v_scale"], sc, o, lse,
                                  dev_status=st)
    else:
        bsa.prefill_fwd_fp8(s, q, k, v, f8["q_scale"], f8["k_scale"], f8["v_scale"], kv[0], kv[1], sc,
                            o, lse, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def oracle_fp8(w, f8):
    return O.select_blocks(deq(f8, "q"), deq(f8, "k"), w.block, w.centroid_keep, w.rescue_keep,
                           with_scores=True)


def rows_of(w, res):
    rows = {}
    for b in range(w.batch):
        for g in range(w.hkv):
            s_c, r = res["scores"][(b, g)]
            for i in range(w.nb):
                rows[(b, g, i)] = (res["mask"][b, g, i], s_c[i], r[i])
    return dict(rows=rows, med=res["med"], radius=res["radius"])


def check_rows(w, f8, o, lse, keep, rows):
    q, k, v = deq(f8, "q"), deq(f8, "k"), deq(f8, "v")
    ref = O.sparse_attention_rows(q, k, v, keep, w.block, rows)
    errs, lerr = [], 0.0
    for (b, h, i), (oi, li) in ref.items():
        errs.append(np.abs(o[b, i * w.block:(i + 1) * w.block, h] - oi).reshape(-1))
        lerr = max(lerr, float(np.abs(lse[b, h, i * w.block:(i + 1) * w.block] - li).max()))
    e = np.concatenate(errs)
    assert e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())
    assert lerr <= 1e-3, lerr


def sample(w, per, seed=0):
    rng = np.random.default_rng(seed)
    out = []
    for b in range(w.batch):
        for h in range(w.hq):
            out += [(b, h, int(i)) for i in sorted({0, w.nb - 1} | set(rng.integers(0, w.nb, per).tolist()))]
    return out


@pytest.mark.parametrize("name", ["tiny_h2x1_n1024_d64_b64", "gqa32x4_n8192_d128_b128"])
def test_fp8_meta_and_masks(name):
    w = synth.workload(name)
    f8 = synth.fp8_layer(synth.make_layer(w))
    got = gpu_fp8_mask(w, f8)
    res = oracle_fp8(w, f8)
    scale = max(np.abs(res["centroid"]).max(), 1.0)
    assert np.abs(got["centroid"] - res["centroid"]).max() <= 1e-5 * scale
    np.testing.assert_allclose(got["radius"], res["radius"], rtol=1e-5)
    compared, excused = compare_mask_rows(got["mask"], rows_of(w, res))
    assert excused <= max(4, compared // 1000), (compared, excused)


@pytest.mark.parametrize("block", [64, 128, 256])
def test_fp8_sparse_attention(block):
    w = synth.Workload(f"f8_b{block}", 1, 4096, 16, 2, 128, block, 0.2, 0.05, seed_base=55, needles_fixed=1)
    f8 = synth.fp8_layer(synth.make_layer(w))
    res = oracle_fp8(w, f8)
    idx, cnt = O.kv_lists(res["mask"])
    o, lse = gpu_fp8_attention(w, f8, (torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda()))
    assert not np.isnan(o).any()
    check_rows(w, f8, o, lse, res["mask"] != 0, sample(w, 3))


def test_fp8_dense_attention_and_gqa_mask_end_to_end():
    w = synth.workload("gqa32x4_n8192_d128_b128")
    f8 = synth.fp8_layer(synth.make_layer(w))
    o, lse = gpu_fp8_attention(w, f8)
    check_rows(w, f8, o, lse, np.ones((1, w.hkv, w.nb, w.nb), dtype=bool), sample(w, 1, seed=1))
    # the GPU's own fp8 selection feeding the fp8 attention, on rows whose masks match
    got = gpu_fp8_mask(w, f8)
    res = oracle_fp8(w, f8)
    o2, lse2 = gpu_fp8_attention(w, f8, (torch.from_numpy(got["kv_idx"]).cuda(),
                                         torch.from_numpy(got["kv_cnt"]).cuda()))
    rows = [(b, h, i) for (b, h, i) in sample(w, 2, seed=2)
            if np.array_equal(got["mask"][b, h // w.group, i], res["mask"][b, h // w.group, i])]
    assert rows
    check_rows(w, f8, o2, lse2, res["mask"] != 0, rows)
