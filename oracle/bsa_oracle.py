"""fp64 CPU oracle: radius-rescued block selection + explicit softmax attention.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, ``smoke()`` and
the benchmark's CPU-baseline leg may import or run this module.  It shares no
code with the CUDA path.

Source: the article "Your 128K Context Is 6x Slower Than It Needs to Be"
(articles.phantom-byte.com), sections "Why block-sparse attention
underperforms: the mean-dilution trap" and "The rescue branch: two selection
paths, one mask", and the FlashAttention description in
"attention-kernel-optimization" (skill-vault.co.in), section "FlashAttention
(1 -> 2 -> 3)", which fixes that tiled online softmax equals the explicit
softmax computed here.

The article gives prose, not formulas.  Each function states the reading it
implements and cites it by number (reading 1 .. 19 of the repository's
specification), so that the oracle and the CUDA path follow one definition.
All arithmetic is float64 on the bf16-rounded inputs.

Layouts: q [b, N, Hq, d], k and v [b, N, Hkv, d]; per-block tensors are
[b, H, nb, ...]; masks are [b, Hkv, nb_q, nb_k] uint8 with bit 0 = forced
(first or diagonal block), bit 1 = kept by the centroid path, bit 2 = kept by
the rescue path.  N need not be a multiple of the block size: nb = ceil(N / B)
and the last block holds the N - (nb - 1) B remaining tokens (reading 3: a
partial block is summarised, ranked and attended over its own tokens only).
Packed ragged batches ("varlen") hold sequence b in tokens
cu_seqlens[b] .. cu_seqlens[b+1] - 1 of q [T, Hq, d], k and v [T, Hkv, d];
each sequence is processed on its own, exactly like a batch of one.
"""
from __future__ import annotations

import math

import numpy as np

FORCED, CENTROID, RESCUE = 1, 2, 4


# ------------------------------------------------------------ block summaries

def block_meta(k: np.ndarray, block: int):
    """Centroid and radius of every key block.

    Rescue branch section: every key block is summarised by its centroid and
    by the largest distance from one of its keys to that centroid.  The
    centroid is the mean of the block's keys (reading 1, mean-dilution
    section); the distance is read as plain Euclidean (reading 2).

    k: [b, N, Hkv, d].  Returns centroid [b, Hkv, nb, d], radius [b, Hkv, nb].
    """
    b, n, h, d = k.shape
    nfull = n // block
    kf = np.asarray(k, dtype=np.float64)
    kb = kf[:, :nfull * block].reshape(b, nfull, block, h, d).transpose(0, 3, 1, 2, 4)
    centroid = kb.mean(axis=3)
    dist = np.sqrt(np.sum((kb - centroid[:, :, :, None, :]) ** 2, axis=-1))
    radius = dist.max(axis=-1)
    if n % block:
        # partial last block: its own n - nfull * block keys
        kt = kf[:, nfull * block:].transpose(0, 2, 1, 3)          # [b, Hkv, rest, d]
        ct = kt.mean(axis=2)
        rt = np.sqrt(np.sum((kt - ct[:, :, None, :]) ** 2, axis=-1)).max(axis=-1)
        centroid = np.concatenate([centroid, ct[:, :, None, :]], axis=2)
        radius = np.concatenate([radius, rt[:, :, None]], axis=2)
    return centroid, radius


def nearest_rank(count: int, num: int, den: int) -> int:
    """1-based nearest rank ceil(num/den * count), at least 1."""
    return max(1, (num * count + den - 1) // den)


def radius_quantiles(radius: np.ndarray):
    """Median and 90th-percentile radius per (batch, KV head).

    Rescue branch section: the coefficient is anchored at the median and the
    90th percentile of the radii, taken per layer and per KV head over the
    prompt's blocks.  Reading 4: nearest-rank
    quantiles over all nb blocks, q(p) = r_(ceil(p nb)) of the ascending sort
    (so the median is the lower median for even nb).

    radius: [b, Hkv, nb].  Returns (med, p90), each [b, Hkv].
    """
    nb = radius.shape[-1]
    srt = np.sort(radius, axis=-1)
    med = srt[..., nearest_rank(nb, 1, 2) - 1]
    p90 = srt[..., nearest_rank(nb, 9, 10) - 1]
    return med, p90


def rescue_coefficient(radius: np.ndarray, med: np.ndarray, p90: np.ndarray):
    """Radius-adaptive rescue coefficient alpha_j in [0, 1].

    Rescue branch section: the coefficient adapts to where a block's radius
    falls between the median and the 90th percentile.  Reading 5: a block
    no wider than the median gets no bonus, a block at or beyond p90 the full
    bonus, linear in between:
        alpha_j = clamp((r_j - med) / (p90 - med), 0, 1),
    and alpha = 0 for every block when p90 - med <= 1e-12 * p90.
    """
    med = np.asarray(med, dtype=np.float64)[..., None]
    p90 = np.asarray(p90, dtype=np.float64)[..., None]
    span = p90 - med
    degenerate = span <= 1e-12 * p90
    safe = np.where(degenerate, 1.0, span)
    alpha = np.clip((radius - med) / safe, 0.0, 1.0)
    return np.where(degenerate, 0.0, alpha)


def query_summary(q: np.ndarray, block: int):
    """Per query block: mean query and mean query norm.

    Rescue branch section: the centroid branch ranks blocks by how relevant
    they are on average.  Reading 6: the query side of a block is summarised by the mean
    of its queries (qbar) and the mean of their Euclidean norms (nbar).

    q: [b, N, Hq, d].  Returns qbar [b, Hq, nb, d], nbar [b, Hq, nb].
    """
    b, n, h, d = q.shape
    nfull = n // block
    qf = np.asarray(q, dtype=np.float64)
    qb = qf[:, :nfull * block].reshape(b, nfull, block, h, d).transpose(0, 3, 1, 2, 4)
    qbar = qb.mean(axis=3)
    nbar = np.sqrt(np.sum(qb * qb, axis=-1)).mean(axis=-1)
    if n % block:
        qt = qf[:, nfull * block:].transpose(0, 2, 1, 3)          # [b, Hq, rest, d]
        qbar = np.concatenate([qbar, qt.mean(axis=2)[:, :, None, :]], axis=2)
        nbar = np.concatenate([nbar, np.sqrt(np.sum(qt * qt, axis=-1)).mean(axis=-1)[:, :, None]],
                              axis=2)
    return qbar, nbar


def block_scores(qbar, nbar, centroid, radius, alpha, scale: float, b: int, g: int):
    """Centroid-path and rescue-path scores for one (batch, KV head).

    Centroid path (rescue branch section: blocks ranked by average
    relevance):  S_c[i, j] = max over the group's query heads h of
    scale * (qbar_{h,i} . c_j).
    Rescue path (the base score plus the radius term weighted by the
    coefficient):  R[i, j] = max_h scale * (qbar_{h,i} . c_j +
    alpha_j * nbar_{h,i} * r_j) (reading 7).  Since |qbar| <= nbar, with
    alpha_j = 1 the rescue score bounds every key of block j (Cauchy-Schwarz),
    so a single outlier key cannot be diluted away.  Reading 8: the group's
    heads are combined by a max, so one head is not diluted by the others (GQA sharing,
    32 query heads over 4 KV heads).

    Returns (S_c, R), each [nb, nb] float64 (row i = query block, column j =
    key block; entries with j > i are meaningless).
    """
    hq = qbar.shape[1]
    hkv = centroid.shape[1]
    grp = hq // hkv
    heads = slice(g * grp, (g + 1) * grp)
    dots = np.einsum("hid,jd->hij", qbar[b, heads], centroid[b, g])
    s_c = scale * dots.max(axis=0)
    bonus = nbar[b, heads][:, :, None] * (alpha[b, g] * radius[b, g])[None, None, :]
    r = scale * (dots + bonus).max(axis=0)
    return s_c, r


def token_block_scores(q, centroid, radius, alpha, block: int, scale: float, b: int, g: int):
    """Per-token query aggregation of the two scores for one (batch, KV head).

    The article's selection summarises a query block by its mean; the
    per-token variant ranks key block j for query block i by the best single
    query instead:
        S_c[i, j] = scale * max over the group's heads h and the tokens t of
                    block i of q_{h,t} . c_j
        R[i, j]   = scale * max_{h,t} (q_{h,t} . c_j + alpha_j |q_{h,t}| r_j).
    With alpha_j = 1, R bounds scale * q_{h,t} . k for every key k of block j
    (Cauchy-Schwarz, |k - c_j| <= r_j), i.e. the block's largest logit.
    Reading 15: the maximum over tokens is the plain reading of the article's
    token-to-centroid comparison (section "The numbers, stated honestly").

    q: [b, N, Hq, d].  Returns (S_c, R), each [ceil(N / block), nb] (row i =
    query block of q, column j = key block of centroid).
    """
    n, hq = q.shape[1], q.shape[2]
    hkv = centroid.shape[1]
    grp = hq // hkv
    nq = -(-n // block)
    c = centroid[b, g]                                      # [nb, d]
    bonus = alpha[b, g] * radius[b, g]                      # [nb]
    s_c = np.empty((nq, c.shape[0]))
    r = np.empty((nq, c.shape[0]))
    for i in range(nq):
        qt = np.asarray(q[b, i * block:min((i + 1) * block, n), g * grp:(g + 1) * grp],
                        dtype=np.float64)                   # [t, G, d]
        dots = np.einsum("thd,jd->thj", qt, c)
        norms = np.sqrt(np.sum(qt * qt, axis=-1))           # [t, G]
        s_c[i] = scale * dots.max(axis=(0, 1))
        r[i] = scale * (dots + norms[:, :, None] * bonus[None, None, :]).max(axis=(0, 1))
    return s_c, r


# ------------------------------------------------------------ selection

PPM = 1_000_000


def ratio_ppm(ratio: float) -> int:
    """Keep-ratio in parts per million, rounded half up."""
    return int(math.floor(ratio * PPM + 0.5))


def keep_count(ppm: int, i: int) -> int:
    """ceil(ratio * (i + 1)) in integer arithmetic (ratio = ppm / 1e6).

    Reading 10, of the independent per-path thresholds: each path keeps a fixed fraction
    of the causal row (i + 1 blocks), rounded up.
    """
    return (ppm * (i + 1) + PPM - 1) // PPM


def _top(cands: np.ndarray, score: np.ndarray, k: int) -> np.ndarray:
    """The k best candidates: higher score first, ties to the lower index."""
    if k <= 0 or cands.size == 0:
        return cands[:0]
    s = score[cands]
    order = np.lexsort((cands, -s))
    return cands[order[:k]]


def select_row(s_c_row, r_row, alpha_row, i: int, ppm_c: int, ppm_r: int):
    """Blocks kept for query block i (one batch, one KV head).

    * Forced: key block 0 and the diagonal block i are always kept and take
      part in neither ranking (reading 9; the article does not say).
    * Centroid path (reading 11): the top k_c = min(ceil(rho_c (i+1)), i-1)
      candidates j in 1..i-1 by S_c.
    * Rescue path (reading 12): among the candidates the centroid path dropped and whose
      radius is above the median (alpha_j > 0), the top
      k_r = min(ceil(rho_r (i+1)), #eligible) by R (wide blocks come back
      even when their mean score alone would drop them).
    * The two paths are thresholded independently and combined by OR (reading 13).

    Returns (centroid_kept, rescue_kept) as ascending int arrays.
    """
    cands = np.arange(1, i, dtype=np.int64)
    kc = min(keep_count(ppm_c, i), cands.size)
    cent = np.sort(_top(cands, s_c_row, kc))
    dropped = np.setdiff1d(cands, cent)
    eligible = dropped[alpha_row[dropped] > 0.0]
    kr = min(keep_count(ppm_r, i), eligible.size)
    resc = np.sort(_top(eligible, r_row, kr))
    return cent, resc


def select_blocks(q, k, block: int, centroid_keep: float, rescue_keep: float,
                  scale: float | None = None, with_scores: bool = False, token_max: bool = False):
    """Whole mask build for one layer: meta, quantiles, alpha, scores, select.

    ``token_max`` scores with the per-token aggregation (token_block_scores)
    instead of the block-mean query.  Returns a dict with centroid, radius,
    med, p90, alpha, qbar, nbar and the uint8 mask [b, Hkv, nb, nb] (bits
    FORCED | CENTROID | RESCUE); with ``with_scores`` also the per-(b, g)
    score matrices.
    """
    b, n, hq, d = q.shape
    hkv = k.shape[2]
    nb = -(-n // block)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if nb == 0:
        z = np.zeros
        return dict(centroid=z((b, hkv, 0, d)), radius=z((b, hkv, 0)), med=z((b, hkv)),
                    p90=z((b, hkv)), alpha=z((b, hkv, 0)), qbar=z((b, hq, 0, d)),
                    nbar=z((b, hq, 0)), mask=np.zeros((b, hkv, 0, 0), dtype=np.uint8), scale=scale,
                    **({"scores": {}} if with_scores else {}))
    centroid, radius = block_meta(k, block)
    med, p90 = radius_quantiles(radius)
    alpha = rescue_coefficient(radius, med, p90)
    qbar, nbar = query_summary(q, block)
    ppm_c, ppm_r = ratio_ppm(centroid_keep), ratio_ppm(rescue_keep)
    mask = np.zeros((b, hkv, nb, nb), dtype=np.uint8)
    scores = {}
    for bi in range(b):
        for g in range(hkv):
            if token_max:
                s_c, r = token_block_scores(q, centroid, radius, alpha, block, scale, bi, g)
            else:
                s_c, r = block_scores(qbar, nbar, centroid, radius, alpha, scale, bi, g)
            if with_scores:
                scores[(bi, g)] = (s_c, r)
            for i in range(nb):
                mask[bi, g, i, 0] |= FORCED
                mask[bi, g, i, i] |= FORCED
                cent, resc = select_row(s_c[i], r[i], alpha[bi, g], i, ppm_c, ppm_r)
                mask[bi, g, i, cent] |= CENTROID
                mask[bi, g, i, resc] |= RESCUE
    out = dict(centroid=centroid, radius=radius, med=med, p90=p90, alpha=alpha,
               qbar=qbar, nbar=nbar, mask=mask, scale=scale)
    if with_scores:
        out["scores"] = scores
    return out


def kv_lists(mask: np.ndarray):
    """Kept key blocks per row, ascending.  Returns (kv_idx, kv_cnt).

    kv_idx is [b, Hkv, nb, nb] int32 with the first kv_cnt entries of a row
    valid and the rest set to -1.
    """
    b, h, nq, nk = mask.shape
    kv_idx = np.full((b, h, nq, nk), -1, dtype=np.int32)
    kv_cnt = np.zeros((b, h, nq), dtype=np.int32)
    for bi in range(b):
        for g in range(h):
            for i in range(nq):
                js = np.nonzero(mask[bi, g, i])[0]
                kv_idx[bi, g, i, :js.size] = js
                kv_cnt[bi, g, i] = js.size
    return kv_idx, kv_cnt


# ------------------------------------------------------------ attention

def _attend(qi, keys, vals, qpos, kpos, scale):
    """Explicit causal softmax attention of queries qi over the given keys."""
    s = scale * (qi @ keys.T)
    s = np.where(kpos[None, :] <= qpos[:, None], s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ vals) / l
    lse = (m + np.log(l))[:, 0]
    return o, lse


def sparse_attention_rows(q, k, v, mask, block: int, rows, scale: float | None = None):
    """Attention for selected (batch, query head, query block) rows only.

    Rescue branch section: the OR-combined mask is consumed by an ordinary
    block-sparse FlashAttention.  For each query token t of block i and head
    h (KV head g = h // (Hq/Hkv)) the keys are the tokens s <= t of the key
    blocks kept in mask[b, g, i]; the output is the explicit softmax-weighted
    sum of their values and lse the natural log of the softmax normaliser
    (reading 14).

    mask: boolean-like [b, Hkv, nb, nb].  rows: iterable of (b, h, i).
    Returns {(b, h, i): (o [block, d], lse [block])}.
    """
    b, n, hq, d = q.shape
    hkv = k.shape[2]
    grp = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = {}
    for (bi, h, i) in rows:
        g = h // grp
        kept = np.nonzero(mask[bi, g, i])[0]
        kpos = (kept[:, None] * block + np.arange(block)[None, :]).reshape(-1)
        kpos = kpos[kpos < n]                      # a partial last block has fewer keys
        qpos = i * block + np.arange(block)
        qpos = qpos[qpos < n]
        qi = np.asarray(q[bi, qpos, h, :], dtype=np.float64)
        keys = np.asarray(k[bi, kpos, g, :], dtype=np.float64)
        vals = np.asarray(v[bi, kpos, g, :], dtype=np.float64)
        out[(bi, h, i)] = _attend(qi, keys, vals, qpos, kpos, scale)
    return out


def sparse_attention(q, k, v, mask, block: int, scale: float | None = None):
    """Full sparse attention.  Returns o [b, N, Hq, d], lse [b, Hq, N]."""
    b, n, hq, d = q.shape
    nb = -(-n // block)
    o = np.zeros((b, n, hq, d), dtype=np.float64)
    lse = np.zeros((b, hq, n), dtype=np.float64)
    rows = [(bi, h, i) for bi in range(b) for h in range(hq) for i in range(nb)]
    res = sparse_attention_rows(q, k, v, mask, block, rows, scale)
    for (bi, h, i), (oi, li) in res.items():
        o[bi, i * block:(i + 1) * block, h, :] = oi
        lse[bi, h, i * block:(i + 1) * block] = li
    return o, lse


def dense_attention(q, k, v, scale: float | None = None):
    """Dense causal softmax attention with GQA (every key s <= t).

    Returns o [b, N, Hq, d], lse [b, Hq, N].
    """
    b, n, hq, d = q.shape
    hkv = k.shape[2]
    grp = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((b, n, hq, d), dtype=np.float64)
    lse = np.zeros((b, hq, n), dtype=np.float64)
    pos = np.arange(n)
    for bi in range(b):
        for h in range(hq):
            g = h // grp
            oi, li = _attend(np.asarray(q[bi, :, h, :], dtype=np.float64),
                             np.asarray(k[bi, :, g, :], dtype=np.float64),
                             np.asarray(v[bi, :, g, :], dtype=np.float64), pos, pos, scale)
            o[bi, :, h, :] = oi
            lse[bi, h, :] = li
    return o, lse


# ------------------------------------------------------------ packed ragged batches

def seq_bounds(cu_seqlens, b: int):
    """Token range [start, end) of sequence b of a packed batch."""
    return int(cu_seqlens[b]), int(cu_seqlens[b + 1])


def varlen_select_blocks(q, k, cu_seqlens, block: int, centroid_keep: float, rescue_keep: float,
                         scale: float | None = None, with_scores: bool = False,
                         token_max: bool = False):
    """Mask build of every sequence of a packed batch, each as a batch of one.

    q: [T, Hq, d], k: [T, Hkv, d].  Returns a list with one ``select_blocks``
    result per sequence (its arrays keep a leading batch dimension of 1).
    """
    out = []
    for b in range(len(cu_seqlens) - 1):
        s0, s1 = seq_bounds(cu_seqlens, b)
        out.append(select_blocks(q[None, s0:s1], k[None, s0:s1], block, centroid_keep, rescue_keep,
                                 scale, with_scores, token_max))
    return out


def varlen_attention_rows(q, k, v, cu_seqlens, masks, block: int, rows, scale: float | None = None):
    """Sparse attention rows of a packed batch.

    masks[b]: boolean-like [1, Hkv, nb_b, nb_b] for sequence b.  rows: iterable
    of (b, h, i).  Returns {(b, h, i): (o [tokens of block i, d], lse)}.
    """
    out = {}
    for (b, h, i) in rows:
        s0, s1 = seq_bounds(cu_seqlens, b)
        res = sparse_attention_rows(q[None, s0:s1], k[None, s0:s1], v[None, s0:s1], masks[b], block,
                                    [(0, h, i)], scale)
        out[(b, h, i)] = res[(0, h, i)]
    return out


def varlen_dense_attention(q, k, v, cu_seqlens, scale: float | None = None):
    """Dense causal attention of every sequence of a packed batch.

    Returns o [T, Hq, d] and lse [Hq, T].
    """
    t, hq, d = q.shape
    o = np.zeros((t, hq, d), dtype=np.float64)
    lse = np.zeros((hq, t), dtype=np.float64)
    for b in range(len(cu_seqlens) - 1):
        s0, s1 = seq_bounds(cu_seqlens, b)
        if s1 == s0:
            continue
        ob, lb = dense_attention(q[None, s0:s1], k[None, s0:s1], v[None, s0:s1], scale)
        o[s0:s1] = ob[0]
        lse[:, s0:s1] = lb[0]
    return o, lse


# ------------------------------------------------------------ decode (one new token)

def decode_select(q_tok, centroid, radius, alpha, n: int, block: int, centroid_keep: float,
                  rescue_keep: float, g: int, scale: float | None = None):
    """Kept key blocks of one KV head for a single new query token.

    The new token sits at position n - 1 of a sequence whose cache (including
    the token's own key) holds n tokens, so its row is the block
    i = (n - 1) // block.  Reading 16: the decode query is a query block of one
    token, so its summary is the token itself (mean = q, mean norm = |q|) and
    the row is selected exactly like a prefill row: forced 0 and i, the top
    k_c of 1..i-1 by S_c, the top k_r of the dropped blocks with alpha > 0 by R.

    q_tok: [Hq, d]; centroid [Hkv, nb, d], radius and alpha [Hkv, nb] of the
    cache.  Returns (kept ascending int array, S_c row, R row).
    """
    hq, d = q_tok.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    i = (n - 1) // block
    qbar = np.asarray(q_tok, dtype=np.float64)[None, :, None, :]        # [1, Hq, 1, d]
    nbar = np.sqrt(np.sum(qbar * qbar, axis=-1))                         # [1, Hq, 1]
    s_c, r = block_scores(qbar, nbar, centroid[None], radius[None], alpha[None], scale, 0, g)
    cent, resc = select_row(s_c[0], r[0], alpha[g], i, ratio_ppm(centroid_keep),
                            ratio_ppm(rescue_keep))
    kept = np.union1d(np.union1d(cent, resc), np.array([0, i]))
    return kept, s_c[0], r[0]


def decode_attention(q_tok, k, v, kept_by_g, n: int, block: int, scale: float | None = None):
    """Attention of one new token (position n - 1) over the kept key blocks.

    q_tok: [Hq, d]; k, v: [n', Hkv, d] with n' >= n (tokens past n - 1 are
    ignored); kept_by_g[g]: kept key blocks of KV head g.  Returns o [Hq, d]
    and lse [Hq].
    """
    hq, d = q_tok.shape
    hkv = k.shape[1]
    grp = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((hq, d))
    lse = np.zeros(hq)
    for h in range(hq):
        g = h // grp
        kept = np.asarray(kept_by_g[g])
        kpos = (kept[:, None] * block + np.arange(block)[None, :]).reshape(-1)
        kpos = kpos[kpos < n]
        oi, li = _attend(np.asarray(q_tok[h:h + 1], dtype=np.float64),
                         np.asarray(k[kpos, g], dtype=np.float64),
                         np.asarray(v[kpos, g], dtype=np.float64), np.array([n - 1]), kpos, scale)
        o[h] = oi[0]
        lse[h] = li[0]
    return o, lse


def varlen_decode(q_new, k, v, cu_seqlens, block: int, centroid_keep: float, rescue_keep: float,
                  scale: float | None = None):
    """One decode step of a packed batch: the cache of sequence b is tokens
    cu_seqlens[b] .. cu_seqlens[b+1]-1 of k, v (its last token is the new one);
    q_new [batch, Hq, d].  Block summaries and the rescue coefficient are those
    of the whole cache (block_meta, quantiles over its blocks).  Returns the
    kept lists [(b, g) -> array], o [batch, Hq, d] and lse [batch, Hq]."""
    bsz, hq, d = q_new.shape
    hkv = k.shape[1]
    kept = {}
    o = np.zeros((bsz, hq, d))
    lse = np.zeros((bsz, hq))
    for b in range(bsz):
        s0, s1 = seq_bounds(cu_seqlens, b)
        n = s1 - s0
        if n == 0:
            continue
        kc, vc = k[s0:s1], v[s0:s1]
        cen, rad = block_meta(np.asarray(kc, dtype=np.float64)[None], block)
        med, p90 = radius_quantiles(rad)
        alpha = rescue_coefficient(rad, med, p90)
        per_g = []
        for g in range(hkv):
            kp, _, _ = decode_select(q_new[b], cen[0], rad[0], alpha[0], n, block, centroid_keep,
                                     rescue_keep, g, scale)
            kept[(b, g)] = kp
            per_g.append(kp)
        o[b], lse[b] = decode_attention(q_new[b], kc, vc, per_g, n, block, scale)
    return kept, o, lse
