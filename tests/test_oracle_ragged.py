"""Pins for the oracle's partial last blocks and packed ragged batches.

The facts used: a one-token block is its own centroid with radius 0; the
token counts times the block centroids sum to the sum of all keys (so the
partial block divides by its own count); brute-force loops over the tail
block; dense attention, the pure-python softmax and torch SDPA agree with the
sparse path on lengths that are not a multiple of the block; and a sequence of
a packed batch is unaffected by the tokens of the other sequences.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from test_oracle_pins import _brute_attention


def _rand(seed, *shape):
    return np.random.default_rng(seed).normal(size=shape)


def test_one_token_tail_block_is_its_own_centroid():
    k = _rand(1, 1, 17, 2, 6)                      # 2 full blocks of 8, then 1 token
    cen, rad = O.block_meta(k, 8)
    assert cen.shape == (1, 2, 3, 6) and rad.shape == (1, 2, 3)
    np.testing.assert_array_equal(cen[0, :, 2], k[0, 16])
    np.testing.assert_array_equal(rad[0, :, 2], 0.0)


@pytest.mark.parametrize("n", [9, 23, 31, 40, 63])
def test_counts_times_centroids_sum_to_key_sum(n):
    blk = 8
    k = _rand(n, 2, n, 3, 5)
    cen, rad = O.block_meta(k, blk)
    nb = -(-n // blk)
    counts = np.array([min(blk, n - j * blk) for j in range(nb)], dtype=np.float64)
    lhs = np.einsum("j,bgjd->bgd", counts, cen)
    rhs = k.sum(axis=1)
    np.testing.assert_allclose(lhs, rhs, atol=1e-12)
    # the full blocks are those of the truncated prefix (vectorised path)
    full = n // blk
    if full:
        c2, r2 = O.block_meta(k[:, :full * blk], blk)
        np.testing.assert_array_equal(cen[:, :, :full], c2)
        np.testing.assert_array_equal(rad[:, :, :full], r2)


def test_tail_radius_and_query_summary_bruteforce():
    n, blk, d = 21, 8, 4
    k = _rand(3, 1, n, 1, d)
    q = _rand(4, 1, n, 2, d)
    cen, rad = O.block_meta(k, blk)
    qbar, nbar = O.query_summary(q, blk)
    tail = list(range(16, 21))
    c = [sum(k[0, t, 0, x] for t in tail) / len(tail) for x in range(d)]
    r = max(math.sqrt(sum((k[0, t, 0, x] - c[x]) ** 2 for x in range(d))) for t in tail)
    assert rad[0, 0, 2] == pytest.approx(r, rel=1e-12)
    for h in range(2):
        qb = [sum(q[0, t, h, x] for t in tail) / len(tail) for x in range(d)]
        nb_ = sum(math.sqrt(sum(q[0, t, h, x] ** 2 for x in range(d))) for t in tail) / len(tail)
        np.testing.assert_allclose(qbar[0, h, 2], qb, rtol=1e-12)
        assert nbar[0, h, 2] == pytest.approx(nb_, rel=1e-12)


def test_quantiles_count_the_partial_block():
    k = _rand(5, 1, 8 * 9 + 3, 1, 4)
    k[0, 72:] *= 10.0                              # a wide tail block
    _, rad = O.block_meta(k, 8)
    med, p90 = O.radius_quantiles(rad)
    assert rad.shape[-1] == 10
    assert med[0, 0] == np.quantile(rad[0, 0], 0.5, method="inverted_cdf")
    assert p90[0, 0] == np.quantile(rad[0, 0], 0.9, method="inverted_cdf")


@pytest.mark.parametrize("n", [13, 45])
def test_ragged_all_ones_equals_dense_bruteforce_and_sdpa(n):
    blk = 8
    q, k, v = _rand(6, 1, n, 4, 4), _rand(7, 1, n, 2, 4), _rand(8, 1, n, 2, 4)
    nb = -(-n // blk)
    keep = np.ones((1, 2, nb, nb), dtype=bool)
    o_s, l_s = O.sparse_attention(q, k, v, keep, blk, 0.4)
    o_d, l_d = O.dense_attention(q, k, v, 0.4)
    o_b, l_b = _brute_attention(q, k, v, keep, blk, 0.4)
    np.testing.assert_allclose(o_s, o_b, atol=1e-12)
    np.testing.assert_allclose(l_s, l_b, atol=1e-12)
    np.testing.assert_allclose(o_d, o_b, atol=1e-12)
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(2, dim=1)
    tv = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(2, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=0.4)
    np.testing.assert_allclose(o_s, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12)


def test_ragged_masked_equals_bruteforce():
    n, blk = 37, 8
    q, k, v = _rand(9, 1, n, 4, 4), _rand(10, 1, n, 2, 4), _rand(11, 1, n, 2, 4)
    nb = -(-n // blk)
    keep = np.random.default_rng(12).random((1, 2, nb, nb)) < 0.5
    for i in range(nb):
        keep[:, :, i, i] = True
    o_s, l_s = O.sparse_attention(q, k, v, keep, blk, 0.5)
    o_b, l_b = _brute_attention(q, k, v, keep, blk, 0.5)
    np.testing.assert_allclose(o_s, o_b, atol=1e-12)
    np.testing.assert_allclose(l_s, l_b, atol=1e-12)


def test_varlen_sequences_are_independent():
    lens = [13, 0, 40, 8, 1, 29]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    t = int(cu[-1])
    q, k, v = _rand(13, t, 4, 8), _rand(14, t, 2, 8), _rand(15, t, 2, 8)
    res = O.varlen_select_blocks(q, k, cu, 8, 0.3, 0.1)
    o, lse = O.varlen_dense_attention(q, k, v, cu)
    # scramble every token outside sequence 2: its results must not move
    s0, s1 = O.seq_bounds(cu, 2)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for a in (q2, k2, v2):
        a[:s0] = _rand(16, *a[:s0].shape)
        a[s1:] = _rand(17, *a[s1:].shape)
    res2 = O.varlen_select_blocks(q2, k2, cu, 8, 0.3, 0.1)
    o2, lse2 = O.varlen_dense_attention(q2, k2, v2, cu)
    np.testing.assert_array_equal(res[2]["mask"], res2[2]["mask"])
    np.testing.assert_array_equal(res[2]["radius"], res2[2]["radius"])
    np.testing.assert_array_equal(o[s0:s1], o2[s0:s1])
    np.testing.assert_array_equal(lse[:, s0:s1], lse2[:, s0:s1])
    # an empty sequence has no blocks
    assert res[1]["mask"].shape == (1, 2, 0, 0)
    # each sequence's dense attention is the batch-of-one result
    for b in range(len(lens)):
        s0, s1 = O.seq_bounds(cu, b)
        if s1 > s0:
            ob, lb = O.dense_attention(q[None, s0:s1], k[None, s0:s1], v[None, s0:s1])
            np.testing.assert_array_equal(o[s0:s1], ob[0])
            np.testing.assert_array_equal(lse[:, s0:s1], lb[0])
    # the varlen attention rows of a sequence follow its own mask
    rows = [(2, h, i) for h in range(4) for i in range(5)]
    got = O.varlen_attention_rows(q, k, v, cu, [r["mask"] != 0 for r in res], 8, rows)
    for (b, h, i), (oi, li) in got.items():
        s0, s1 = O.seq_bounds(cu, b)
        want = O.sparse_attention_rows(q[None, s0:s1], k[None, s0:s1], v[None, s0:s1],
                                       res[b]["mask"] != 0, 8, [(0, h, i)])[(0, h, i)]
        np.testing.assert_array_equal(oi, want[0])
