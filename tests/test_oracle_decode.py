"""Pins for the oracle's single-token decode step.

Facts used: a decode token that starts a new block is a one-token query block,
so its kept set and its output equal the prefill oracle's last row (itself
pinned by brute force and SDPA); keep-all equals dense causal attention of the
last token; zero ratios keep the sink and the current block only; a
pure-Python softmax over the kept keys; the Cauchy-Schwarz bound of the rescue
score for a single query.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O


def _cache(seed, n=70, hq=4, hkv=2, d=8):
    rng = np.random.default_rng(seed)
    k = rng.normal(size=(n, hkv, d)) * rng.uniform(0.2, 2.0, size=(n, 1, 1))
    return rng.normal(size=(n, hq, d)), k, rng.normal(size=(n, hkv, d))


@pytest.mark.parametrize("n", [65, 129, 17])
def test_decode_equals_prefill_last_row_when_token_opens_a_block(n):
    blk = 16 if n == 17 else 64
    q, k, v = _cache(1, n=n)
    pre = O.select_blocks(q[None], k[None], blk, 0.3, 0.2)
    i = (n - 1) // blk
    assert (n - 1) % blk == 0                          # the new token is alone in its block
    cu = np.array([0, n])
    kept, o, lse = O.varlen_decode(q[n - 1:n], k, v, cu, blk, 0.3, 0.2)
    for g in range(2):
        np.testing.assert_array_equal(kept[(0, g)], np.nonzero(pre["mask"][0, g, i])[0])
    op, lp = O.sparse_attention(q[None], k[None], v[None], pre["mask"] != 0, blk)
    np.testing.assert_allclose(o[0], op[0, n - 1], atol=1e-12)
    np.testing.assert_allclose(lse[0], lp[0, :, n - 1], atol=1e-12)


def test_decode_keep_all_equals_dense_and_sdpa():
    q, k, v = _cache(2, n=90)
    cu = np.array([0, 90])
    kept, o, lse = O.varlen_decode(q[89:90], k, v, cu, 16, 1.0, 0.0)
    assert all(np.array_equal(kept[(0, g)], np.arange(6)) for g in range(2))
    od, ld = O.dense_attention(q[None], k[None], v[None])
    np.testing.assert_allclose(o[0], od[0, 89], atol=1e-12)
    tq = torch.from_numpy(q[89:90]).permute(1, 0, 2)[None]                 # [1, Hq, 1, d]
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)       # the last token sees all
    np.testing.assert_allclose(o[0], ref[0, :, 0].numpy(), atol=1e-12)


def test_decode_zero_ratios_keep_sink_and_current_block():
    q, k, v = _cache(3, n=100)
    kept, _, _ = O.varlen_decode(q[99:100], k, v, np.array([0, 100]), 16, 0.0, 0.0)
    for g in range(2):
        np.testing.assert_array_equal(kept[(0, g)], [0, 6])


def test_decode_attention_bruteforce():
    q, k, v = _cache(4, n=40)
    kept = [np.array([0, 1]), np.array([0, 2])]
    o, lse = O.decode_attention(q[39], k, v, kept, 40, 16, 0.3)
    for h in range(4):
        g = h // 2
        keys = [s for s in range(40) if s // 16 in kept[g]]
        logit = [0.3 * sum(q[39, h, x] * k[s, g, x] for x in range(8)) for s in keys]
        mx = max(logit)
        z = sum(math.exp(a - mx) for a in logit)
        want = sum(math.exp(a - mx) / z * v[s, g] for a, s in zip(logit, keys))
        np.testing.assert_allclose(o[h], want, atol=1e-12)
        assert lse[h] == pytest.approx(mx + math.log(z), abs=1e-12)


def test_decode_rescue_score_bounds_every_logit():
    q, k, v = _cache(5, n=96)
    cen, rad = O.block_meta(k[None], 16)
    ones = np.ones_like(rad[0])
    _, s_c, r = O.decode_select(q[95], cen[0], rad[0], ones, 96, 16, 0.2, 0.1, 1, 1.0)
    for j in range(6):
        logits = q[95, 2:4] @ k[j * 16:(j + 1) * 16, 1].T
        assert logits.max() <= r[j] + 1e-12
        assert s_c[j] <= r[j] + 1e-12
