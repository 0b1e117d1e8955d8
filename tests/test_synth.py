"""The seeded generator: determinism, shapes and bf16 rounding."""
import numpy as np
import torch

import synth


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).normal(size=100000).astype(np.float32) * 7.0
    x[:4] = [1.00390625, 1.01171875, -2.0078125, 0.0]        # exact ties
    ours = synth.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_generator_deterministic_across_threads():
    w = synth.Workload("t", 1, 9216, 4, 2, 16, 64, 0.25, 0.05)   # 2.25 chunks
    a = synth.make_layer(w, seed=5, threads=1)
    b = synth.make_layer(w, seed=5, threads=4)
    for key in ("q", "k", "v"):
        np.testing.assert_array_equal(a[key], b[key])
    c = synth.make_layer(w, seed=6, threads=1)
    assert not np.array_equal(a["q"], c["q"])


def test_generator_shapes_and_needles():
    w = synth.workload("tiny_h2x1_n1024_d64_b64")
    lay = synth.make_layer(w)
    assert lay["q"].shape == (1, 1024, 2, 64) and lay["q"].dtype == np.uint16
    assert lay["k"].shape == (1, 1024, 1, 64) and lay["v"].shape == (1, 1024, 1, 64)
    assert len(lay["needles"]) == 3
    k = synth.bf16_to_f64(lay["k"])
    for (b, g, jb, slot, pos) in lay["needles"]:
        assert 1 <= jb <= w.nb - 2
        assert np.linalg.norm(k[b, jb * w.block + slot, g]) > 7.9
        assert pos.size == 16 and np.all(pos >= (jb + 1) * w.block)


def test_named_workloads():
    w = synth.workload("gqa32x4_n131072_d128_b128")
    assert (w.seq, w.hq, w.hkv, w.head_dim, w.block, w.nb, w.layers) == (131072, 32, 4, 128, 128, 1024, 48)
    assert w.needles_per_group() == 20
    assert len(synth.sweep_workloads()) == 27


def test_varlen_layer_packs_truncated_sequences():
    vw = synth.VARLEN_WORKLOADS["varlen_h2x1_d64_b64"]
    lay = synth.make_varlen_layer(vw)
    cu = lay["cu_seqlens"]
    assert cu[0] == 0 and cu[-1] == vw.total == lay["q"].shape[0]
    assert np.all(np.diff(cu) == np.array(vw.lengths))
    again = synth.make_varlen_layer(vw, threads=1)
    for x in ("q", "k", "v"):
        np.testing.assert_array_equal(lay[x], again[x])
    # sequence 4 (513 tokens) is the single-sequence draw at 576 tokens, cut to 513
    w = synth.Workload("x", 1, 576, vw.hq, vw.hkv, vw.head_dim, vw.block, 0.25, 0.05,
                       needles_fixed=vw.needles_fixed)
    ref = synth.make_layer(w, seed=vw.seed_base + 4)
    np.testing.assert_array_equal(lay["k"][cu[4]:cu[5]], ref["k"][0, :513])
    for (b, g, jb, slot, pos) in lay["needles"]:
        assert np.all(pos < vw.lengths[b]) and jb * vw.block + slot < vw.lengths[b]
