"""The e4m3 codec the fp8 inputs use, pinned by the format's definition and by
torch's float8_e4m3fn conversion (an independent implementation)."""
import numpy as np
import pytest
import torch

import synth


def test_known_codes():
    v = synth.E4M3_VALUES
    assert v[0x7E] == 448.0 and v[0x38] == 1.0 and v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert v[0x07] == 7 * 2.0 ** -9 and v[0x3F] == 1.875 and np.isnan(v[0x7F])
    assert np.all(np.diff(v[:127]) > 0)


def test_roundtrip_of_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = synth.e4m3_to_f64(codes)
    back = synth.e4m3_bits(vals)
    # -0 encodes as +0
    np.testing.assert_array_equal(np.where(codes == 0x80, 0, codes), back)


def test_ties_to_even_and_saturation():
    # 1.0625 lies halfway between 1.0 (code 0x38) and 1.125 (0x39): the even code wins
    assert synth.e4m3_bits(np.array([1.0625]))[0] == 0x38
    assert synth.e4m3_bits(np.array([1.1875]))[0] == 0x3A      # between 0x39 and 0x3A -> 0x3A
    assert synth.e4m3_bits(np.array([1e6, -1e6]))[0] == 0x7E
    assert synth.e4m3_bits(np.array([-1e6]))[0] == 0xFE


def test_matches_torch_float8_e4m3fn():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(size=20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 200.0)])
    x = x[np.abs(x) < 448.0]
    ours = synth.e4m3_bits(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref = np.where(ref == 0x80, 0, ref)                         # -0 -> +0
    np.testing.assert_array_equal(ours, ref)


def test_fp8_layer_scales_keep_values_in_range():
    w = synth.workload("tiny_h2x1_n1024_d64_b64")
    lay = synth.make_layer(w)
    f8 = synth.fp8_layer(lay)
    for name in ("q", "k", "v"):
        s = f8[name + "_scale"]
        assert np.log2(s) == int(np.log2(s))
        deq = synth.e4m3_to_f64(f8[name]) * s
        x = synth.bf16_to_f64(lay[name])
        assert np.abs(deq).max() <= 448.0 * s
        # e4m3 keeps 3 mantissa bits: relative error below 2^-4 above the subnormal range
        big = np.abs(x) > 2.0 ** -6 * s
        assert np.all(np.abs(deq[big] - x[big]) <= 2.0 ** -4 * np.abs(x[big]))
