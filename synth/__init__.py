"""Seeded synthetic inputs for long-context block-sparse causal prefill.

This module is shared by the CPU oracle, the tests and the benchmark, and it
holds none of the method's arithmetic: it only draws Q, K and V, plants
needles, and rounds once to bf16 (round-to-nearest-even).

Recipe (shaped like the GQA prefill workload the article
"Your 128K Context Is 6x Slower Than It Needs to Be" measures on, section
"The rescue branch": 32 query heads over 4 KV heads; head_dim 128):

* Q and V are i.i.d. N(0, 1).
* Keys are clustered per key block: K[b, jB+t, g, :] = c + sigma * z with
  c ~ N(0, 0.5^2 I), sigma = exp(U[ln 0.2, ln 1.5]) drawn per (b, g, j) and
  z ~ N(0, I) per key.  Blocks therefore differ in spread, which is what
  makes the radius signal informative (section "The mean-dilution trap").
* Needles per (b, g): in each chosen key block (drawn without replacement
  from 1..nb-2) one uniformly chosen key slot is replaced by 8u, u a unit
  vector drawn per needle; 16 query positions drawn without replacement from
  the tokens after that block get +2u on every query head of group g.
* Everything is cast to bf16 once; the oracle reads those exact bf16 values.

Every tensor draws from its own child of ``numpy.random.SeedSequence(seed)``
and large tensors are drawn in fixed 4096-token chunks with one child seed per
chunk, so the values do not depend on the thread count or the draw order.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "sweep_workloads", "make_layer",
    "VarlenWorkload", "VARLEN_WORKLOADS", "make_varlen_layer",
    "bf16_bits", "bf16_to_f64", "bf16_to_f32",
    "E4M3_VALUES", "e4m3_bits", "e4m3_to_f64", "fp8_layer",
]

_CHUNK_TOKENS = 4096


@dataclasses.dataclass(frozen=True)
class Workload:
    """One prefill shape plus its selection ratios and needle recipe."""
    name: str
    batch: int
    seq: int
    hq: int
    hkv: int
    head_dim: int
    block: int
    centroid_keep: float
    rescue_keep: float
    layers: int = 1
    seed_base: int = 0
    needles_fixed: int | None = None   # fixed needle count per (b, g); else 2% of nb

    @property
    def nb(self) -> int:
        return self.seq // self.block

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    def needles_per_group(self) -> int:
        if self.needles_fixed is not None:
            return self.needles_fixed
        return max(1, int(round(0.02 * self.nb)))

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# Workloads named by shape.  Ratios: centroid keep-ratio / rescue keep-ratio.
WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_h2x1_n1024_d64_b64", 1, 1024, 2, 1, 64, 64, 0.25, 0.05,
                 seed_base=0, needles_fixed=3),
        Workload("gqa32x4_n8192_d128_b128", 1, 8192, 32, 4, 128, 128, 0.25, 0.05,
                 seed_base=1000),
        Workload("gqa32x4_n32768_d128_b128", 1, 32768, 32, 4, 128, 128, 0.15, 0.03,
                 seed_base=2000),
        Workload("gqa32x4_n131072_d128_b128", 1, 131072, 32, 4, 128, 128, 0.10, 0.02,
                 layers=48, seed_base=3000),
    ]
}


def workload(name: str) -> Workload:
    """A named workload: one of WORKLOADS or a point of the 64K sweep."""
    if name in WORKLOADS:
        return WORKLOADS[name]
    for w in sweep_workloads():
        if w.name == name:
            return w
    raise KeyError(name)


def sweep_workloads():
    """Block-size x keep-ratio sweep at 64K tokens, GQA 32/4, head_dim 128."""
    out = []
    for block in (64, 128, 256):
        for rc in (0.05, 0.1, 0.2):
            for rr in (0.0, 0.02, 0.05):
                out.append(Workload(
                    f"sweep_n65536_b{block}_c{rc:g}_r{rr:g}", 1, 65536, 32, 4, 128,
                    block, rc, rr, seed_base=4000))
    return out


# ---------------------------------------------------------------- bf16 helpers

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------- fp8 (e4m3) helpers
#
# OCP FP8 E4M3 as used by the tensor cores' e4m3 type: 1 sign bit, 4 exponent
# bits (bias 7), 3 mantissa bits, no infinities, S.1111.111 is NaN, largest
# finite 448, subnormals m * 2^-9.

def _e4m3_table() -> np.ndarray:
    vals = np.zeros(128)
    for code in range(128):
        e, m = code >> 3, code & 7
        vals[code] = m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    vals[127] = np.nan
    return vals


E4M3_VALUES = _e4m3_table()  # value of each non-negative code 0..127 (127 is NaN)


def e4m3_bits(x: np.ndarray) -> np.ndarray:
    """float -> e4m3 codes (uint8): round to nearest, ties to the even code, saturating at
    +-448 (finite inputs only)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    finite = E4M3_VALUES[:127]                        # ascending, codes 0..126
    hi = np.clip(np.searchsorted(finite, a, side="left"), 0, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - finite[lo]
    d_hi = finite[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(a == finite[hi], hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    return np.where(np.signbit(x) & (code != 0), code | np.uint8(0x80), code).astype(np.uint8)


def e4m3_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint8)
    v = E4M3_VALUES[b & 0x7F]
    return np.where(b & 0x80, -v, v)


def fp8_layer(lay: dict, threads: int | None = None) -> dict:
    """The layer's Q, K, V (bf16 bits) as e4m3 codes with one power-of-two scale per tensor:
    value = e4m3 * scale, scale = 2^ceil(log2(max|x| / 448))."""
    if threads is None:
        threads = min(16, os.cpu_count() or 1)
    out = {}
    for name in ("q", "k", "v"):
        bits = lay[name]
        flat = bits.reshape(-1)
        mx = float(np.abs(bf16_to_f32(flat)).max()) if flat.size else 1.0
        scale = 2.0 ** int(np.ceil(np.log2(max(mx, 1e-30) / 448.0)))
        codes = np.empty(flat.shape, dtype=np.uint8)
        step = 1 << 22

        def conv(lo):
            hi = min(lo + step, flat.size)
            codes[lo:hi] = e4m3_bits(bf16_to_f64(flat[lo:hi]) / scale)   # exact division by 2^k

        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(conv, range(0, flat.size, step)))
        out[name] = codes.reshape(bits.shape)
        out[name + "_scale"] = scale
    return out


# ---------------------------------------------------------------- generator

def _normal_chunks(ss: np.random.SeedSequence, shape, threads: int) -> np.ndarray:
    """N(0,1) float32 of ``shape`` ([b, N, H, d]) drawn in fixed token chunks."""
    b, n, h, d = shape
    out = np.empty(shape, dtype=np.float32)
    nchunk = (n + _CHUNK_TOKENS - 1) // _CHUNK_TOKENS
    children = ss.spawn(b * nchunk)

    def fill(idx):
        bi, ci = divmod(idx, nchunk)
        t0 = ci * _CHUNK_TOKENS
        t1 = min(n, t0 + _CHUNK_TOKENS)
        g = np.random.Generator(np.random.PCG64(children[idx]))
        out[bi, t0:t1] = g.standard_normal((t1 - t0, h, d), dtype=np.float32)

    if threads <= 1 or b * nchunk == 1:
        for i in range(b * nchunk):
            fill(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(b * nchunk)))
    return out


def make_layer(w: Workload, layer: int = 0, seed: int | None = None,
               threads: int | None = None) -> dict:
    """Draw one layer's Q, K, V for workload ``w``.

    Returns a dict with ``q``, ``k``, ``v`` (uint16 bf16 bits, [b, N, H, d]
    contiguous), ``needles`` (list of (b, g, key_block, key_slot, query
    positions)) and ``seed``.
    """
    if seed is None:
        seed = w.seed_base + layer
    if threads is None:
        threads = min(16, os.cpu_count() or 1)
    b, n, hq, hkv, d, blk = w.batch, w.seq, w.hq, w.hkv, w.head_dim, w.block
    nb = n // blk
    ss = np.random.SeedSequence(seed)
    s_q, s_v, s_kz, s_kc, s_need = ss.spawn(5)

    q = _normal_chunks(s_q, (b, n, hq, d), threads)
    v = _normal_chunks(s_v, (b, n, hkv, d), threads)
    k = _normal_chunks(s_kz, (b, n, hkv, d), threads)

    # per-(b, g) block centres and spreads
    gc = np.random.Generator(np.random.PCG64(s_kc))
    centre = gc.standard_normal((b, nb, hkv, d)) * 0.5
    sigma = np.exp(gc.uniform(np.log(0.2), np.log(1.5), size=(b, nb, hkv)))
    k = k.reshape(b, nb, blk, hkv, d)
    k *= sigma[:, :, None, :, None].astype(np.float32)
    k += centre[:, :, None, :, :].astype(np.float32)
    k = k.reshape(b, n, hkv, d)

    needles = []
    count = w.needles_per_group()
    group = hq // hkv
    need_children = s_need.spawn(b * hkv)
    for bi in range(b):
        for g in range(hkv):
            gn = np.random.Generator(np.random.PCG64(need_children[bi * hkv + g]))
            if nb < 3:
                continue
            cnt = min(count, nb - 2)
            blocks = np.sort(gn.choice(np.arange(1, nb - 1), size=cnt, replace=False))
            for jb in blocks:
                z = gn.standard_normal(d)
                u = z / np.sqrt(np.sum(z * z))
                slot = int(gn.integers(0, blk))
                k[bi, int(jb) * blk + slot, g, :] = (8.0 * u).astype(np.float32)
                first = (int(jb) + 1) * blk
                npos = min(16, n - first)
                pos = np.sort(gn.choice(np.arange(first, n), size=npos, replace=False))
                for h in range(g * group, (g + 1) * group):
                    q[bi, pos, h, :] += (2.0 * u).astype(np.float32)
                needles.append((bi, g, int(jb), slot, pos.astype(np.int64)))

    return {
        "q": bf16_bits(q), "k": bf16_bits(k), "v": bf16_bits(v),
        "needles": needles, "seed": seed, "workload": w,
    }


# ---------------------------------------------------------------- packed ragged batches

@dataclasses.dataclass(frozen=True)
class VarlenWorkload:
    """A packed batch of sequences of mixed lengths (any length, not only
    multiples of the block), one shape of heads, block and ratios."""
    name: str
    lengths: tuple
    hq: int
    hkv: int
    head_dim: int
    block: int
    centroid_keep: float
    rescue_keep: float
    seed_base: int = 0
    needles_fixed: int | None = None

    @property
    def batch(self) -> int:
        return len(self.lengths)

    @property
    def total(self) -> int:
        return int(sum(self.lengths))

    @property
    def max_seqlen(self) -> int:
        return int(max(self.lengths))

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)


VARLEN_WORKLOADS = {
    w.name: w for w in [
        VarlenWorkload("varlen_h2x1_d64_b64", (1000, 64, 1, 130, 513, 0, 257), 2, 1, 64, 64,
                       0.25, 0.05, seed_base=5000, needles_fixed=2),
        VarlenWorkload("varlen_gqa32x4_d128_b128", (8192, 3000, 12345, 128, 700, 20001, 1),
                       32, 4, 128, 128, 0.15, 0.03, seed_base=6000),
        VarlenWorkload("varlen_gqa32x4_d128_b64", (4000, 2113, 65, 6000), 32, 4, 128, 64,
                       0.15, 0.03, seed_base=7000),
        # a serving mix of 19 prompts, 15 to 32768 tokens, 131072 tokens in all
        VarlenWorkload("varlen_mix19_gqa32x4_d128_b128_t131072",
                       (32768, 20000, 16384, 12345, 9000, 8192, 6000, 5000, 4096, 3500, 3000,
                        2500, 2048, 1800, 1500, 1200, 1024, 700, 15),
                       32, 4, 128, 128, 0.15, 0.03, seed_base=8000),
    ]
}


def make_varlen_layer(vw: VarlenWorkload, layer: int = 0, threads: int | None = None) -> dict:
    """Draw one layer of a packed ragged batch.

    Sequence b is drawn with the single-sequence recipe above at its length
    rounded up to whole blocks (seed ``seed_base + 1000 * layer + b``), then
    cut to its length; needle query positions past the cut are dropped.
    Returns ``q``, ``k``, ``v`` (uint16 bf16 bits, [T, H, d]), ``cu_seqlens``
    (int32 [batch + 1]) and ``needles`` as (b, g, key_block, key_slot, query
    positions within the sequence).
    """
    qs, ks, vs, needles = [], [], [], []
    for b, n in enumerate(vw.lengths):
        if n == 0:
            continue
        padded = -(-n // vw.block) * vw.block
        w = Workload(f"{vw.name}_seq{b}", 1, padded, vw.hq, vw.hkv, vw.head_dim, vw.block,
                     vw.centroid_keep, vw.rescue_keep, needles_fixed=vw.needles_fixed)
        lay = make_layer(w, seed=vw.seed_base + 1000 * layer + b, threads=threads)
        qs.append(lay["q"][0, :n])
        ks.append(lay["k"][0, :n])
        vs.append(lay["v"][0, :n])
        for (_, g, jb, slot, pos) in lay["needles"]:
            pos = pos[pos < n]
            if pos.size:
                needles.append((b, g, jb, slot, pos))
    d = vw.head_dim
    cat = lambda xs, h: (np.ascontiguousarray(np.concatenate(xs, axis=0)) if xs
                         else np.zeros((0, h, d), dtype=np.uint16))
    return {"q": cat(qs, vw.hq), "k": cat(ks, vw.hkv), "v": cat(vs, vw.hkv),
            "cu_seqlens": vw.cu_seqlens(), "needles": needles, "workload": vw}
