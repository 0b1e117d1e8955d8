"""Pins for the fp64 oracle against facts fixed outside the oracle itself.

Each test names the mathematical fact it relies on: closed forms built by
construction, invariances, the Cauchy-Schwarz bound behind the rescue score,
brute-force loops on tiny inputs, an independent library routine (torch SDPA,
numpy's inverted-CDF quantile) and a planted-needle case.  Together they are
chosen so a dropped term, a wrong sign, a wrong index or a transposed operand
in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth


RNG = np.random.default_rng(12345)


# ----------------------------------------------------------------- meta

def test_centroid_radius_closed_form():
    # Keys c +/- a_m e_m come in symmetric pairs, so the mean is c exactly and
    # the farthest key sits at max(a_m) from it.
    d, blk = 8, 8
    c = np.array([1.0, -2.0, 0.5, 3.0, 0.0, -1.0, 2.0, 0.25])
    amps = [4.0, 1.0, 2.5, 0.5]
    keys = []
    for m, a in enumerate(amps):
        e = np.zeros(d)
        e[m] = a
        keys += [c + e, c - e]
    k = np.array(keys)[None, :, None, :]           # [1, 8, 1, 8]
    k2 = np.concatenate([k, k[:, ::-1] * 2.0], axis=1)  # second block: scaled copy
    cen, rad = O.block_meta(k2, blk)
    np.testing.assert_allclose(cen[0, 0, 0], c, atol=1e-14)
    np.testing.assert_allclose(cen[0, 0, 1], 2.0 * c, atol=1e-14)
    assert rad[0, 0, 0] == pytest.approx(4.0, abs=1e-14)
    assert rad[0, 0, 1] == pytest.approx(8.0, abs=1e-14)


def test_radius_is_max_not_mean_distance():
    # One far key among close ones: radius is that key's distance.
    d, blk = 4, 16
    k = np.zeros((1, blk, 1, d))
    k[0, 3, 0, 0] = 16.0                     # mean = (1, 0, 0, 0)
    cen, rad = O.block_meta(k, blk)
    np.testing.assert_allclose(cen[0, 0, 0], [1.0, 0, 0, 0], atol=1e-15)
    assert rad[0, 0, 0] == pytest.approx(15.0, abs=1e-13)


def test_query_summary_closed_form():
    d, blk = 6, 4
    u = np.zeros(d)
    u[2] = 1.0
    w = np.zeros(d)
    w[5] = 1.0
    # norms 3, 1, 2, 2 ; mean of vectors is (3u + w + 2u - 2u... )/4
    qs = np.array([3 * u, w, 2 * u, -2 * w])
    q = qs[None, :, None, :]
    qbar, nbar = O.query_summary(q, blk)
    np.testing.assert_allclose(qbar[0, 0, 0], (3 * u + w + 2 * u - 2 * w) / 4, atol=1e-15)
    assert nbar[0, 0, 0] == pytest.approx(2.0, abs=1e-15)


# ----------------------------------------------------------------- quantiles

@pytest.mark.parametrize("r, med, p90", [
    ([5, 1, 4, 2, 3], 3, 5),                 # ranks ceil(2.5)=3, ceil(4.5)=5
    ([4, 3, 2, 1], 2, 4),                    # lower median; ceil(3.6)=4
    (list(range(1, 11)), 5, 9),              # ranks 5 and 9
    ([7.0], 7.0, 7.0),
    (list(range(20, 0, -1)), 10, 18),        # ranks 10 and 18
])
def test_quantiles_worked_examples(r, med, p90):
    m, p = O.radius_quantiles(np.array(r, dtype=np.float64)[None, None, :])
    assert m[0, 0] == med and p[0, 0] == p90


@pytest.mark.parametrize("nb", [1, 2, 3, 16, 64, 255, 256, 1024])
def test_quantiles_match_numpy_inverted_cdf(nb):
    r = RNG.random((2, 3, nb))
    m, p = O.radius_quantiles(r)
    np.testing.assert_array_equal(m, np.quantile(r, 0.5, axis=-1, method="inverted_cdf"))
    np.testing.assert_array_equal(p, np.quantile(r, 0.9, axis=-1, method="inverted_cdf"))


# ----------------------------------------------------------------- alpha

def test_alpha_closed_form():
    r = np.array([[[0.5, 1.0, 2.0, 3.0, 5.0]]])
    a = O.rescue_coefficient(r, np.array([[1.0]]), np.array([[3.0]]))
    np.testing.assert_allclose(a[0, 0], [0.0, 0.0, 0.5, 1.0, 1.0], atol=1e-15)
    # a degenerate spread (p90 == median) gives no rescue bonus at all
    a = O.rescue_coefficient(r, np.array([[2.0]]), np.array([[2.0]]))
    np.testing.assert_array_equal(a, 0.0)


def _alpha_of(k, blk):
    cen, rad = O.block_meta(k, blk)
    med, p90 = O.radius_quantiles(rad)
    return O.rescue_coefficient(rad, med, p90)


def test_alpha_invariances():
    w = synth.Workload("pin", 1, 256, 2, 2, 16, 16, 0.25, 0.05, needles_fixed=2)
    lay = synth.make_layer(w, seed=7)
    k = synth.bf16_to_f64(lay["k"])
    a0 = _alpha_of(k, 16)
    assert np.any(a0 > 0) and np.any(a0 == 0) and np.any((a0 > 0) & (a0 < 1))
    np.testing.assert_allclose(_alpha_of(3.5 * k, 16), a0, atol=1e-12)
    np.testing.assert_allclose(_alpha_of(k + RNG.normal(size=16), 16), a0, atol=1e-9)
    perm = k.reshape(1, 16, 16, 2, 16)[:, :, RNG.permutation(16)].reshape(k.shape)
    np.testing.assert_allclose(_alpha_of(perm, 16), a0, atol=1e-12)


# ----------------------------------------------------------------- scores

def _tiny(seed=3, n=512, hq=4, hkv=2, d=16, blk=16, needles=3):
    w = synth.Workload("pin", 1, n, hq, hkv, d, blk, 0.25, 0.05, needles_fixed=needles)
    lay = synth.make_layer(w, seed=seed)
    return (synth.bf16_to_f64(lay["q"]), synth.bf16_to_f64(lay["k"]),
            synth.bf16_to_f64(lay["v"]), w, lay)


def test_cauchy_schwarz_bound_and_ordering():
    # With alpha_j = 1 the rescue score bounds every key of block j:
    # qbar.c + nbar*r >= qbar.c + |qbar||k - c| >= qbar.k.   Also S_c <= R.
    q, k, v, w, _ = _tiny()
    res = O.select_blocks(q, k, w.block, 0.25, 0.05, with_scores=True)
    scale = res["scale"]
    nb = w.nb
    kb = k.reshape(1, nb, w.block, w.hkv, w.head_dim)
    grp = w.group
    checked = 0
    for g in range(w.hkv):
        s_c, r = res["scores"][(0, g)]
        assert np.all(s_c <= r + 1e-12)
        for j in np.nonzero(res["alpha"][0, g] == 1.0)[0]:
            keys = kb[0, j, :, g, :]
            for h in range(g * grp, (g + 1) * grp):
                best = scale * (res["qbar"][0, h] @ keys.T).max(axis=1)   # [nb]
                assert np.all(r[:, j] >= best - 1e-12)
                checked += 1
    assert checked > 0


def test_scores_use_every_head_of_the_group():
    # Max over heads: a signal on one head alone must reach the group score.
    q, k, v, w, _ = _tiny()
    q2 = q.copy()
    res0 = O.select_blocks(q, k, w.block, 0.25, 0.05, with_scores=True)
    h_last = w.group - 1                           # last head of group 0
    c5 = res0["centroid"][0, 0, 5]
    blk = w.block
    q2[0, 9 * blk:10 * blk, h_last, :] += 50.0 * c5 / np.linalg.norm(c5)
    res1 = O.select_blocks(q2, k, w.block, 0.25, 0.05, with_scores=True)
    s0, _ = res0["scores"][(0, 0)]
    s1, _ = res1["scores"][(0, 0)]
    assert s1[9, 5] > s0[9, 5] + 1.0
    assert s1[9].argmax() == 5 or s1[9, 5] == s1[9, :10].max()


# ----------------------------------------------------------------- selection

@pytest.mark.parametrize("ratio, i, want", [
    (0.05, 19, 1),       # 0.05 * 20 = 1 exactly, not 2
    (0.25, 3, 1), (0.25, 4, 2), (0.1, 9, 1), (0.1, 10, 2), (0.03, 99, 3),
    (0.02, 1023, 21), (0.0, 500, 0), (1.0, 7, 8), (0.15, 19, 3),
])
def test_keep_count_integer_ceiling(ratio, i, want):
    assert O.keep_count(O.ratio_ppm(ratio), i) == want


def _check_row_properties(mask_row, s_c, r, alpha, i, ppm_c, ppm_r):
    forced = {0, i}
    cent = set(np.nonzero(mask_row & O.CENTROID)[0].tolist())
    resc = set(np.nonzero(mask_row & O.RESCUE)[0].tolist())
    assert set(np.nonzero(mask_row & O.FORCED)[0].tolist()) == forced
    cands = set(range(1, i))
    assert cent <= cands and resc <= cands and not (cent & resc)
    assert len(cent) == min(O.keep_count(ppm_c, i), len(cands))
    # every kept candidate beats every dropped one (score desc, then lower j)
    for a in cent:
        for b in cands - cent:
            assert (s_c[a], -a) > (s_c[b], -b)
    eligible = {j for j in cands - cent if alpha[j] > 0}
    assert resc <= eligible
    assert len(resc) == min(O.keep_count(ppm_r, i), len(eligible))
    for a in resc:
        for b in eligible - resc:
            assert (r[a], -a) > (r[b], -b)
    assert not np.any(mask_row[i + 1:])


@pytest.mark.parametrize("rc, rr", [(0.25, 0.05), (0.1, 0.2), (0.5, 0.5), (0.0, 0.3)])
def test_selection_is_the_specified_top_k(rc, rr):
    q, k, v, w, _ = _tiny(seed=11)
    res = O.select_blocks(q, k, w.block, rc, rr, with_scores=True)
    for g in range(w.hkv):
        s_c, r = res["scores"][(0, g)]
        for i in range(w.nb):
            _check_row_properties(res["mask"][0, g, i], s_c[i], r[i], res["alpha"][0, g], i,
                                  O.ratio_ppm(rc), O.ratio_ppm(rr))


def test_selection_tie_break_prefers_lower_index():
    s = np.array([0.0, 1.0, 2.0, 2.0, 1.0, 2.0, 0.0, 0.0, 0.0])
    cent, resc = O.select_row(s, s, np.ones(9), 8, O.ratio_ppm(0.25), 0)
    # ceil(0.25 * 9) = 3 of candidates 1..7: the three 2.0s at j = 2, 3, 5
    np.testing.assert_array_equal(cent, [2, 3, 5])
    cent, resc = O.select_row(s, s, np.ones(9), 8, O.ratio_ppm(0.2), O.ratio_ppm(0.12))
    np.testing.assert_array_equal(cent, [2, 3])
    # rescue: ceil(0.12 * 9) = 2 of the dropped {1, 4, 5, 6, 7}: 5 (2.0), then 1 (1.0, before 4)
    np.testing.assert_array_equal(resc, [1, 5])


def test_rescue_ranks_only_blocks_the_centroid_path_dropped():
    # R's best block is already kept by the centroid path; rescue takes the next.
    s_c = np.array([0, 5.0, 4.0, 1.0, 0.0, 0])
    r = np.array([0, 9.0, 1.0, 3.0, 2.0, 0])
    # ceil(0.1 * 6) = 1 block per path
    cent, resc = O.select_row(s_c, r, np.ones(6), 5, O.ratio_ppm(0.1), O.ratio_ppm(0.1))
    np.testing.assert_array_equal(cent, [1])
    np.testing.assert_array_equal(resc, [3])
    # blocks at or below the median radius (alpha = 0) are never rescued
    cent, resc = O.select_row(s_c, r, np.array([1, 1, 1, 0, 1, 1.0]), 5,
                              O.ratio_ppm(0.1), O.ratio_ppm(0.1))
    np.testing.assert_array_equal(resc, [4])


def test_zero_ratios_keep_sink_and_diagonal_only():
    q, k, v, w, _ = _tiny()
    m = O.select_blocks(q, k, w.block, 0.0, 0.0)["mask"]
    want = np.zeros_like(m)
    for i in range(w.nb):
        want[:, :, i, 0] = O.FORCED
        want[:, :, i, i] = O.FORCED
    np.testing.assert_array_equal(m, want)


def test_planted_needle_rescued_but_not_by_centroid():
    # Queries all point along u.  Key block 3 is centred at -u (lowest centroid
    # score) but holds one key at 8u: its radius is by far the widest, so the
    # rescue path keeps it while the centroid path alone drops it.
    d, blk, nb = 16, 16, 8
    n = nb * blk
    rng = np.random.default_rng(0)
    u = np.zeros(d)
    u[0] = 1.0
    k = np.zeros((1, n, 1, d))
    for j in range(nb):
        cen = 0.3 * rng.normal(size=d)
        cen[0] = 0.2 + 0.05 * j
        k[0, j * blk:(j + 1) * blk, 0] = cen + 0.1 * rng.normal(size=(blk, d))
    k[0, 3 * blk:4 * blk, 0] = -u + 0.1 * rng.normal(size=(blk, d))
    k[0, 3 * blk + 7, 0] = 8.0 * u
    q = np.tile(u, (1, n, 2, 1)) + 0.05 * rng.normal(size=(1, n, 2, d))
    v = rng.normal(size=(1, n, 1, d))
    res = O.select_blocks(q, k, blk, 0.25, 0.15)
    row = res["mask"][0, 0, 7]
    assert res["alpha"][0, 0, 3] == 1.0
    assert not (row[3] & O.CENTROID) and (row[3] & O.RESCUE)
    assert not O.select_blocks(q, k, blk, 0.25, 0.0)["mask"][0, 0, 7, 3]
    # and the needle key carries the largest attention weight of a late query
    o, lse = O.sparse_attention(q, k, v, res["mask"] != 0, blk)
    t = 7 * blk + 5
    kept = [s for s in range(t + 1) if res["mask"][0, 0, 7, s // blk]]
    w = {s: math.exp((q[0, t, 0] @ k[0, s, 0]) / math.sqrt(d) - lse[0, 0, t]) for s in kept}
    assert max(w, key=w.get) == 3 * blk + 7
    assert w[3 * blk + 7] > 5.0 / len(kept)


def test_generator_needles_are_rescued_more_often():
    w = synth.workload("tiny_h2x1_n1024_d64_b64")
    lay = synth.make_layer(w)
    q, k = synth.bf16_to_f64(lay["q"]), synth.bf16_to_f64(lay["k"])
    with_r = O.select_blocks(q, k, w.block, w.centroid_keep, w.rescue_keep)["mask"]
    no_r = O.select_blocks(q, k, w.block, w.centroid_keep, 0.0)["mask"]
    hit_r = hit_c = total = 0
    for (b, g, jb, slot, pos) in lay["needles"]:
        for i in sorted(set((pos // w.block).tolist())):
            total += 1
            hit_r += bool(with_r[b, g, i, jb])
            hit_c += bool(no_r[b, g, i, jb])
    assert total > 0 and hit_r >= hit_c


# ----------------------------------------------------------------- attention

def _brute_attention(q, k, v, keep, blk, scale):
    """Pure-python loops: softmax over visible kept keys, one query at a time."""
    b, n, hq, d = q.shape
    grp = hq // k.shape[2]
    o = np.zeros_like(q)
    lse = np.zeros((b, hq, n))
    for bi in range(b):
        for h in range(hq):
            g = h // grp
            for t in range(n):
                ss = []
                for s in range(t + 1):
                    if keep[bi, g, t // blk, s // blk]:
                        ss.append((s, scale * sum(q[bi, t, h, x] * k[bi, s, g, x] for x in range(d))))
                mx = max(val for _, val in ss)
                z = sum(math.exp(val - mx) for _, val in ss)
                for s, val in ss:
                    o[bi, t, h] += math.exp(val - mx) / z * v[bi, s, g]
                lse[bi, h, t] = mx + math.log(z)
    return o, lse


def _tiny_attn_inputs(seed, n=32, hq=4, hkv=2, d=4, blk=8):
    rng = np.random.default_rng(seed)
    return (rng.normal(size=(1, n, hq, d)), rng.normal(size=(1, n, hkv, d)),
            rng.normal(size=(1, n, hkv, d)), blk)


def test_all_ones_mask_equals_dense_bruteforce():
    q, k, v, blk = _tiny_attn_inputs(1)
    nb = q.shape[1] // blk
    keep = np.ones((1, 2, nb, nb), dtype=bool)
    scale = 0.37
    o_s, l_s = O.sparse_attention(q, k, v, keep, blk, scale)
    o_d, l_d = O.dense_attention(q, k, v, scale)
    o_b, l_b = _brute_attention(q, k, v, keep, blk, scale)
    np.testing.assert_allclose(o_s, o_b, atol=1e-12)
    np.testing.assert_allclose(l_s, l_b, atol=1e-12)
    np.testing.assert_allclose(o_d, o_b, atol=1e-12)
    np.testing.assert_allclose(l_d, l_b, atol=1e-12)
    # rho_c = 1 selects every causal block
    m = O.select_blocks(q, k, blk, 1.0, 0.0)["mask"]
    assert all(m[0, g, i, j] for g in range(2) for i in range(nb) for j in range(i + 1))


def test_dense_matches_torch_sdpa_fp64():
    rng = np.random.default_rng(5)
    q = rng.normal(size=(2, 48, 6, 8))
    k = rng.normal(size=(2, 48, 2, 8))
    v = rng.normal(size=(2, 48, 2, 8))
    o, _ = O.dense_attention(q, k, v)
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(3, dim=1)
    tv = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(3, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12)


def test_masked_equals_bruteforce_with_excluded_blocks():
    q, k, v, blk = _tiny_attn_inputs(2)
    nb = q.shape[1] // blk
    rng = np.random.default_rng(9)
    keep = rng.random((1, 2, nb, nb)) < 0.5
    for i in range(nb):
        keep[:, :, i, i] = True
    o_s, l_s = O.sparse_attention(q, k, v, keep, blk, 0.5)
    o_b, l_b = _brute_attention(q, k, v, keep, blk, 0.5)
    np.testing.assert_allclose(o_s, o_b, atol=1e-12)
    np.testing.assert_allclose(l_s, l_b, atol=1e-12)


def test_softmax_rows_sum_to_one_via_lse():
    q, k, v, w, _ = _tiny(n=256)
    res = O.select_blocks(q, k, w.block, 0.25, 0.05)
    keep = res["mask"] != 0
    o, lse = O.sparse_attention(q, k, v, keep, w.block)
    scale = 1 / math.sqrt(w.head_dim)
    grp = w.group
    for h in range(w.hq):
        g = h // grp
        for t in range(0, w.seq, 37):
            kept = [s for s in range(t + 1) if keep[0, g, t // w.block, s // w.block]]
            z = sum(math.exp(scale * float(q[0, t, h] @ k[0, s, g]) - lse[0, h, t]) for s in kept)
            assert z == pytest.approx(1.0, abs=1e-12)


# ----------------------------------------------------------------- per-token aggregation

def _token_case(seed, n=40, hq=4, hkv=2, d=6, blk=8):
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(1, n, hq, d))
    k = rng.normal(size=(1, n, hkv, d)) * rng.uniform(0.2, 2.0, size=(1, n, 1, 1))
    cen, rad = O.block_meta(k, blk)
    med, p90 = O.radius_quantiles(rad)
    alpha = O.rescue_coefficient(rad, med, p90)
    return q, k, cen, rad, alpha, blk


def test_token_scores_bruteforce():
    q, k, cen, rad, alpha, blk = _token_case(1, n=37)           # a partial last block too
    s = 0.3
    nb = cen.shape[2]
    for g in range(2):
        s_c, r = O.token_block_scores(q, cen, rad, alpha, blk, s, 0, g)
        for i in range(nb):
            toks = range(i * blk, min((i + 1) * blk, 37))
            for j in range(nb):
                best_c = best_r = -math.inf
                for t in toks:
                    for h in (2 * g, 2 * g + 1):
                        dot = sum(q[0, t, h, x] * cen[0, g, j, x] for x in range(6))
                        nq = math.sqrt(sum(q[0, t, h, x] ** 2 for x in range(6)))
                        best_c = max(best_c, dot)
                        best_r = max(best_r, dot + alpha[0, g, j] * rad[0, g, j] * nq)
                assert s_c[i, j] == pytest.approx(s * best_c, rel=1e-12, abs=1e-12)
                assert r[i, j] == pytest.approx(s * best_r, rel=1e-12, abs=1e-12)


def test_token_scores_dominate_block_mean_scores():
    # max over tokens >= mean over tokens, for both paths
    q, k, cen, rad, alpha, blk = _token_case(2)
    qbar, nbar = O.query_summary(q, blk)
    for g in range(2):
        t_c, t_r = O.token_block_scores(q, cen, rad, alpha, blk, 1.0, 0, g)
        m_c, m_r = O.block_scores(qbar, nbar, cen, rad, alpha, 1.0, 0, g)
        assert np.all(t_c >= m_c - 1e-12) and np.all(t_r >= m_r - 1e-12)


def test_token_scores_equal_mean_scores_for_uniform_blocks():
    # every query of a block identical: the best token is the mean query
    q, k, cen, rad, alpha, blk = _token_case(3)
    q = np.repeat(q[:, ::blk], blk, axis=1)[:, :q.shape[1]]
    qbar, nbar = O.query_summary(q, blk)
    for g in range(2):
        t_c, t_r = O.token_block_scores(q, cen, rad, alpha, blk, 0.7, 0, g)
        m_c, m_r = O.block_scores(qbar, nbar, cen, rad, alpha, 0.7, 0, g)
        np.testing.assert_allclose(t_c, m_c, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(t_r, m_r, rtol=1e-12, atol=1e-12)


def test_token_rescue_score_bounds_every_logit_when_alpha_is_one():
    q, k, cen, rad, _, blk = _token_case(4)
    ones = np.ones_like(rad)
    nb = cen.shape[2]
    for g in range(2):
        _, r = O.token_block_scores(q, cen, rad, ones, blk, 1.0, 0, g)
        for i in range(nb):
            qt = q[0, i * blk:(i + 1) * blk, 2 * g:2 * g + 2]
            for j in range(nb):
                logits = np.einsum("thd,sd->ths", qt, k[0, j * blk:(j + 1) * blk, g])
                assert logits.max() <= r[i, j] + 1e-12


def test_token_select_blocks_flag_and_permutation_invariance():
    q, k, cen, rad, alpha, blk = _token_case(5, n=64)
    a = O.select_blocks(q, k, blk, 0.3, 0.2, token_max=True, with_scores=True)
    perm = np.concatenate([np.random.default_rng(6).permutation(blk) + i * blk
                           for i in range(64 // blk)])
    b = O.select_blocks(q[:, perm], k, blk, 0.3, 0.2, token_max=True, with_scores=True)
    np.testing.assert_array_equal(a["mask"], b["mask"])
    for key in a["scores"]:
        np.testing.assert_allclose(a["scores"][key][0], b["scores"][key][0], rtol=1e-13)
    # the per-token masks differ from the block-mean masks somewhere on this input
    m = O.select_blocks(q, k, blk, 0.3, 0.2)
    assert not np.array_equal(a["mask"], m["mask"])


# ----------------------------------------------------------------- kept lists

def _lists_bruteforce(mask):
    """Kept lists by explicit enumeration: walk each row left to right and append every
    block whose mask byte is nonzero."""
    b, h, nq, nk = mask.shape
    out = {}
    for bi in range(b):
        for g in range(h):
            for i in range(nq):
                row = []
                for j in range(nk):
                    if int(mask[bi, g, i, j]) != 0:
                        row.append(j)
                out[(bi, g, i)] = row
    return out


@pytest.mark.parametrize("nk, density", [(1, 0.5), (5, 0.3), (16, 0.0), (16, 1.0), (37, 0.2), (64, 0.7)])
def test_kv_lists_match_enumeration(nk, density):
    """oracle.kv_lists (the lists the GPU attention is fed in the parity tests) against a
    brute-force enumeration: ascending kept blocks, count = number of nonzero mask bytes,
    -1 after the count; empty and full rows; any combination of the mask bits counts."""
    rng = np.random.default_rng(nk * 1000 + int(density * 100))
    mask = np.zeros((2, 3, nk, nk), dtype=np.uint8)
    keep = rng.random(mask.shape) < density
    bits = rng.integers(1, 8, mask.shape).astype(np.uint8)   # any nonzero combination of bits
    mask[keep] = bits[keep]
    mask[0, 0, 0] = 0                                        # an empty row
    mask[1, 2, nk - 1] = O.FORCED | O.CENTROID               # a full row
    kv_idx, kv_cnt = O.kv_lists(mask)
    assert kv_idx.shape == mask.shape and kv_idx.dtype == np.int32
    assert kv_cnt.shape == mask.shape[:3] and kv_cnt.dtype == np.int32
    ref = _lists_bruteforce(mask)
    for (bi, g, i), row in ref.items():
        c = int(kv_cnt[bi, g, i])
        assert c == len(row)
        assert list(kv_idx[bi, g, i, :c]) == row
        assert all(kv_idx[bi, g, i, x] < kv_idx[bi, g, i, x + 1] for x in range(c - 1))
        assert np.all(kv_idx[bi, g, i, c:] == -1)
    assert kv_cnt[0, 0, 0] == 0 and np.all(kv_idx[0, 0, 0] == -1)
    assert kv_cnt[1, 2, nk - 1] == nk and list(kv_idx[1, 2, nk - 1]) == list(range(nk))


def test_kv_lists_of_a_selection_cover_sink_and_diagonal():
    """On a real selection every row's list starts with block 0 and ends with the diagonal
    block i, and its length equals forced + centroid + rescue blocks (disjoint paths)."""
    w = synth.Workload("lists", 1, 1024, 4, 2, 32, 64, 0.25, 0.1, seed_base=5, needles_fixed=2)
    lay = synth.make_layer(w)
    q, k = synth.bf16_to_f64(lay["q"]), synth.bf16_to_f64(lay["k"])
    res = O.select_blocks(q, k, w.block, w.centroid_keep, w.rescue_keep)
    kv_idx, kv_cnt = O.kv_lists(res["mask"])
    for g in range(w.hkv):
        for i in range(w.nb):
            c = kv_cnt[0, g, i]
            row = kv_idx[0, g, i, :c]
            assert row[0] == 0 and row[-1] == i
            m = res["mask"][0, g, i]
            nforced = 1 if i == 0 else 2
            ncent = int(np.count_nonzero(m & O.CENTROID))
            nresc = int(np.count_nonzero(m & O.RESCUE))
            assert not np.any((m & O.CENTROID) & ((m & O.RESCUE) >> 1))
            assert c == nforced + ncent + nresc
