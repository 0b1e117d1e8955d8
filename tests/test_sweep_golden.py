"""Pins for the stored sweep figures (tests/golden/sweep_oracle.json).

* With a zero rescue ratio every row keeps exactly the forced blocks plus
  min(ceil(rho_c (i + 1)), i - 1) centroid-path blocks, whatever the data, so the
  stored kept-block counts must equal that sum computed here in exact integer
  arithmetic (article, rescue branch section: per-path keep ratios over the
  causal row; sink and diagonal always kept).
* The rescue path only adds blocks: per row at most min(ceil(rho_r (i + 1)),
  (i - 1) - k_c) of them, and a larger rescue ratio keeps a superset, so density
  and needle hits cannot fall as rho_r grows; with rho_r = 0 a larger rho_c keeps
  a superset too.
* The block-256 entries are recomputed from the oracle and must equal the file.
"""
import json
import os
from fractions import Fraction

import pytest

import synth

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = os.path.join(HERE, "golden", "sweep_oracle.json")


def ceil_frac(x: Fraction) -> int:
    return -((-x.numerator) // x.denominator)


def centroid_only_kept(nb: int, rho: Fraction) -> int:
    total = 0
    for i in range(nb):
        forced = 1 if i == 0 else 2
        total += forced + min(ceil_frac(rho * (i + 1)), max(i - 1, 0))
    return total


def rescue_cap(nb: int, rc: Fraction, rr: Fraction) -> int:
    total = 0
    for i in range(nb):
        kc = min(ceil_frac(rc * (i + 1)), max(i - 1, 0))
        total += min(ceil_frac(rr * (i + 1)), max(i - 1, 0) - kc)
    return total


@pytest.fixture(scope="module")
def gold():
    return json.load(open(GOLD))["workloads"]


def test_every_sweep_point_is_stored(gold):
    assert sorted(gold) == sorted(w.name for w in synth.sweep_workloads())


def test_centroid_only_counts_closed_form(gold):
    for w in synth.sweep_workloads():
        g = gold[w.name]
        groups = w.batch * w.hkv
        base = groups * centroid_only_kept(w.nb, Fraction(str(w.centroid_keep)))
        if w.rescue_keep == 0:
            assert g["kept_blocks"] == base, w.name
        else:
            extra = g["kept_blocks"] - base
            cap = groups * rescue_cap(w.nb, Fraction(str(w.centroid_keep)), Fraction(str(w.rescue_keep)))
            assert 0 < extra <= cap, (w.name, extra, cap)
        assert g["density"] == pytest.approx(g["kept_blocks"] / (groups * w.nb * (w.nb + 1) // 2))


def test_monotone_in_the_ratios(gold):
    ws = synth.sweep_workloads()
    for block in (64, 128, 256):
        for rc in (0.05, 0.1, 0.2):
            pts = sorted((w for w in ws if w.block == block and w.centroid_keep == rc),
                         key=lambda w: w.rescue_keep)
            for a, b in zip(pts, pts[1:]):
                assert gold[a.name]["kept_blocks"] < gold[b.name]["kept_blocks"]
                assert gold[a.name]["needle_hits"] <= gold[b.name]["needle_hits"]
        pts = sorted((w for w in ws if w.block == block and w.rescue_keep == 0),
                     key=lambda w: w.centroid_keep)
        for a, b in zip(pts, pts[1:]):
            assert gold[a.name]["needle_hits"] <= gold[b.name]["needle_hits"]


def test_block256_entries_reproduce(gold):
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_sweep_oracle",
                                                  os.path.join(HERE, "golden", "make_sweep_oracle.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    got = mod.oracle_sweep(256)
    for name, v in got.items():
        assert v == gold[name], name
