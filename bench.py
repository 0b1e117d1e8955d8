#!/usr/bin/env python
"""Benchmark one layer of radius-rescued block-sparse long-context prefill.

A step is one pass of the whole hot path over one layer of seeded synthetic
input resident in HBM: bsa_block_meta (centroids, radii, quantiles, rescue
coefficient), bsa_select_mask (query pooling, two-path scores, top-k, kept
lists) and bsa_prefill_fwd (sparse attention over the kept blocks).  Default
workload: 131072 tokens, 32 query heads over 4 KV heads, head_dim 128, block
128, keep-ratios 0.10 / 0.02 (the long-prefill shape of the article "Your 128K
Context Is 6x Slower Than It Needs to Be").

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill ms/layer & kept-block TFLOPS at 128K GQA 32/4; mask-build HBM GB/s"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa32x4_n131072_d128_b128")
    ap.add_argument("--layers", type=int, default=None,
                    help="distinct seeded layers resident and rotated per step (default: every seeded "
                         "layer of the workload, 48 for the 128K one; 2 for the e4m3 and packed modes)")
    ap.add_argument("--e2e-steps", type=int, default=48,
                    help="layers streamed end to end (48: one pass over the 128K configuration's layers)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--token-max", action="store_true",
                    help="score query blocks by their best token (BSA_SELECT_TOKEN_MAX)")
    ap.add_argument("--fp8", action="store_true",
                    help="e4m3 Q / K / V inputs with per-tensor scales (the *_fp8 entry points)")
    ap.add_argument("--sweep", action="store_true",
                    help="block size x keep-ratio sweep at 64K tokens: density, ms/layer, needle recall")
    ap.add_argument("--crossover", action="store_true",
                    help="sparse vs dense path at 32K over a centroid keep-ratio sweep; break-even density")
    ap.add_argument("--decode", action="store_true",
                    help="time one decode step (new token per sequence) over the workload as a cache")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def peak_value(d, *keys):
    for k in keys:
        if k in d and isinstance(d[k], (int, float)):
            return float(d[k])
    return None


def kept_flops(kv_cnt: np.ndarray, block: int, d: int, group: int) -> float:
    """Kept-block FLOPs: 4 B^2 d per off-diagonal block, 2 B^2 d for the diagonal, per query head."""
    cnt = kv_cnt.astype(np.int64)
    per = 4.0 * block * block * d
    return float(group * (per * (cnt - 1).clip(min=0).sum() + 0.5 * per * (cnt > 0).sum()))


def replica_layers(rank: int, layers: int) -> list:
    """Seeded layer indices of one replica: each rank draws its own layers, disjoint across ranks."""
    return [rank * layers + li for li in range(layers)]


def reduce_max(value: float, dist=None, device="cpu") -> float:
    """The maximum of ``value`` over the ranks (the slowest rank sets the job's time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_ms_per_layer(max_total_ms: float, steps: int, world: int) -> float:
    """Whole-job ms per layer: every rank ran ``steps`` layers in at most ``max_total_ms``."""
    return max_total_ms / (steps * world)


def source_sha(*files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


ATTN_SOURCES = ("block_sparse_long_kv_gb300/csrc/bsa_attn.cu", "block_sparse_long_kv_gb300/csrc/sm103_ptx.cuh")


def profiled_traffic():
    """DRAM bytes per attention launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "attn_traffic.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        d = json.load(f)
    if d.get("source_sha") != source_sha(*ATTN_SOURCES):
        return None, d
    return d.get("bytes_per_launch_full"), d


class ClockSampler:
    """nvidia-smi sampling during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            try:
                pw.append(float(parts[2]))
            except ValueError:
                pass
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        out = {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "sm_min_mhz": float(min(sm)),
               "samples": len(sm), "reasons": sorted(reasons)}
        if pw:
            out["power_w_median"] = float(np.median(pw))
        return out


# ------------------------------------------------------------------ CPU oracle sample

def oracle_sample(w, lay, budget_s: float, rng_seed: int = 0):
    """Time the fp64 oracle on a bounded sample of one layer; extrapolate to ms/layer.

    Sample: key-block meta for a slice of key blocks (scaled by block count),
    query summary + scores + selection for random rows (scaled by row count),
    attention for random (head, query block) rows of those (scaled by kept FLOPs).
    """
    import oracle as O
    import synth
    rng = np.random.default_rng(rng_seed)
    nb, B, d, G = w.nb, w.block, w.head_dim, w.group
    scale = 1.0 / math.sqrt(d)
    t0 = time.perf_counter()
    # meta on a slice of key blocks of KV head 0
    nbs = min(nb, 64)
    kslice = synth.bf16_to_f64(lay["k"][:, :nbs * B, 0:1])
    O.block_meta(kslice, B)
    t_meta = (time.perf_counter() - t0) * (nb / nbs) * w.hkv * w.batch
    # full radii are needed for the quantiles the selection uses
    k32 = synth.bf16_to_f32(lay["k"])
    centroid, radius = O.block_meta(k32, B)
    med, p90 = O.radius_quantiles(radius)
    alpha = O.rescue_coefficient(radius, med, p90)
    del k32
    # selection rows
    t1 = time.perf_counter()
    rows = []
    nsel = 0
    while time.perf_counter() - t1 < budget_s * 0.3 or nsel < 4:
        g = int(rng.integers(0, w.hkv))
        i = int(rng.integers(1, nb))
        qs = synth.bf16_to_f64(lay["q"][0:1, i * B:(i + 1) * B, g * G:(g + 1) * G])
        qb, nbar = O.query_summary(qs, B)
        qfull = np.zeros((1, w.hq, 1, d))
        nfull = np.zeros((1, w.hq, 1))
        qfull[0, g * G:(g + 1) * G] = qb[0]
        nfull[0, g * G:(g + 1) * G] = nbar[0]
        s_c, r = O.block_scores(qfull, nfull, centroid, radius, alpha, scale, 0, g)
        cent, resc = O.select_row(s_c[0], r[0], alpha[0, g], i, O.ratio_ppm(w.centroid_keep),
                                  O.ratio_ppm(w.rescue_keep))
        rows.append((g, i, np.union1d(np.union1d(cent, resc), [0, i])))
        nsel += 1
        if nsel >= 256:
            break
    t_sel = (time.perf_counter() - t1) * (nb * w.hkv * w.batch / nsel)
    # attention rows, FLOP-weighted
    q32, v32 = synth.bf16_to_f32(lay["q"]), synth.bf16_to_f32(lay["v"])
    k32 = synth.bf16_to_f32(lay["k"])
    t2 = time.perf_counter()
    flops_done = 0.0
    nat = 0
    for (g, i, kept) in rows:
        mask = np.zeros((1, w.hkv, nb, nb), dtype=bool)
        mask[0, g, i, kept] = True
        h = g * G + int(rng.integers(0, G))
        O.sparse_attention_rows(q32, k32, v32, mask, B, [(0, h, i)], scale)
        flops_done += 4.0 * B * B * d * (len(kept) - 1) + 2.0 * B * B * d
        nat += 1
        if time.perf_counter() - t2 > budget_s * 0.6:
            break
    t_att_per_flop = (time.perf_counter() - t2) / flops_done
    return {"t_meta": t_meta, "t_sel": t_sel, "t_att_per_flop": t_att_per_flop,
            "sample": f"meta over {nbs} of {nb} key blocks (1 KV head), selection for {nsel} "
                      f"random query-block rows, attention for {nat} random (head, query block) rows; "
                      f"extrapolated to the whole layer by block count, row count and kept FLOPs"}


def host_placement(index: int) -> dict:
    """Where the pinned host buffers sit relative to the GPU: the host's NUMA nodes, the GPU's
    NUMA node (from its PCI device), transparent huge pages, and how the buffers were made."""
    out = {"pinned_alloc": "torch pin_memory (cudaHostAlloc), allocated before the layers are drawn"}
    try:
        out["numa_nodes"] = len([d for d in os.listdir("/sys/devices/system/node") if d.startswith("node")])
    except OSError:
        pass
    try:
        bus = subprocess.run(["nvidia-smi", "-i", str(index), "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=10).stdout.strip()
        dom, rest = bus.split(":", 1)
        path = f"/sys/bus/pci/devices/{dom[-4:].lower()}:{rest.lower()}/numa_node"
        with open(path) as f:
            out["gpu_numa_node"] = int(f.read().strip())
        out["gpu_pci"] = bus
    except Exception:
        pass
    try:
        with open("/sys/kernel/mm/transparent_hugepage/enabled") as f:
            out["thp"] = f.read().strip()
    except OSError:
        pass
    return out


def threads_used():
    try:
        from threadpoolctl import threadpool_info
        n = [x.get("num_threads", 1) for x in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ reference arm

def expected_counts(nb: int, centroid_keep: float, rescue_keep: float):
    """Kept blocks per row when every path fills its quota (an upper bound of kv_cnt)."""
    import oracle as O
    cnt = np.zeros(nb, dtype=np.int64)
    for i in range(nb):
        nc = max(i - 1, 0)
        kc = min(O.keep_count(O.ratio_ppm(centroid_keep), i), nc)
        kr = min(O.keep_count(O.ratio_ppm(rescue_keep), i), max(nc - kc, 0))
        cnt[i] = (1 if i == 0 else 2) + kc + kr
    return cnt


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import synth
    if args.workload in synth.VARLEN_WORKLOADS:
        vw = synth.VARLEN_WORKLOADS[args.workload]
        b = int(np.argmax(vw.lengths))
        w = synth.Workload(f"{vw.name}_seq{b}", 1, vw.lengths[b], vw.hq, vw.hkv, vw.head_dim,
                           vw.block, vw.centroid_keep, vw.rescue_keep, needles_fixed=vw.needles_fixed)
        lay = synth.make_layer(w, seed=vw.seed_base + b)
        factor = sum(-(-n // vw.block) for n in vw.lengths) / w.nb
        nbs = max(-(-n // vw.block) for n in vw.lengths)
        cnt = np.zeros((vw.batch, vw.hkv, nbs), dtype=np.int64)
        for bi, n in enumerate(vw.lengths):
            nb = -(-n // vw.block)
            cnt[bi, :, :nb] = expected_counts(nb, vw.centroid_keep, vw.rescue_keep)
        fl = kept_flops_varlen(cnt, vw.lengths, vw.block, vw.head_dim, vw.group)
        cfg = {"workload": vw.name, "batch": vw.batch, "total_tokens": vw.total,
               "max_seqlen": vw.max_seqlen, "lengths": list(vw.lengths), "hq": vw.hq,
               "hkv": vw.hkv, "head_dim": vw.head_dim, "block": vw.block,
               "centroid_keep": vw.centroid_keep, "rescue_keep": vw.rescue_keep}
        extra = (f"; taken on the longest sequence ({w.seq} tokens) and scaled to the packed batch "
                 f"by its block count (x{factor:.2f}) and its kept FLOPs")
    else:
        w = synth.workload(args.workload)
        lay = synth.make_layer(w, layer=0)
        factor = 1.0
        cnt = np.broadcast_to(expected_counts(w.nb, w.centroid_keep, w.rescue_keep),
                              (w.batch, w.hkv, w.nb))
        fl = kept_flops(cnt, w.block, w.head_dim, w.group)
        cfg = {"workload": w.name, "batch": w.batch, "seq": w.seq, "hq": w.hq, "hkv": w.hkv,
               "head_dim": w.head_dim, "block": w.block, "centroid_keep": w.centroid_keep,
               "rescue_keep": w.rescue_keep}
        extra = ""
    # each step times the oracle on a bounded sample of the layer (a few seconds of CPU work),
    # so the whole run stays within minutes; the per-layer value is extrapolated from the sample
    per_step = max(3.0, min(args.cpu_budget, 120.0 / max(1, args.steps + args.warmup)))
    est, wall = [], []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        r = oracle_sample(w, lay, per_step, rng_seed=s)
        if s >= args.warmup:
            est.append(r)
            wall.append(time.perf_counter() - t0)
    ms = [1e3 * (factor * (r["t_meta"] + r["t_sel"]) + r["t_att_per_flop"] * fl) for r in est]
    val = float(np.median(ms))
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "ms/layer",
        "extrapolated": True,
        "n_gpus": args.gpus, "steps": len(est), "warmup": args.warmup,
        "ms_per_step": float(1e3 * np.mean(wall)), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded generator, same workload)",
        "config": cfg,
        "cpu_baseline": {"value": val, "unit": "ms/layer", "cores": threads_used(),
                         "kind": "oracle", "sample": est[0]["sample"] + extra},
        "e2e": {"value": val, "unit": "ms/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "fp64 numpy oracle: each timed step is one bounded sample of the layer "
                "(ms_per_step is that sample's wall time); value extrapolates the samples to a whole "
                "layer by block count, row count and kept FLOPs (upper bound of keep counts for the "
                "FLOP scale)",
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm

def kept_flops_varlen(kv_cnt: np.ndarray, lengths, block: int, d: int, group: int) -> float:
    """Kept-block FLOPs of a packed batch, counted over each block's real tokens: per query
    head 4 n_q B d for a kept block before the diagonal and 2 n_q^2 d for the diagonal, n_q the
    query block's tokens."""
    tot = 0.0
    for b, n in enumerate(lengths):
        nb = -(-n // block)
        for i in range(nb):
            nq = min(block, n - i * block)
            cnt = kv_cnt[b, :, i].astype(np.int64)                 # [hkv]
            tot += group * float((4.0 * nq * block * d * (cnt - 1).clip(min=0)).sum()
                                 + (2.0 * nq * nq * d * (cnt > 0)).sum())
    return tot


def token_score_flops(run) -> float:
    """2 d FLOPs per (query token, head, key block j < its block i)."""
    w = run.w
    lengths = w.lengths if isinstance(run, VarlenRunner) else [w.seq] * w.batch
    tot = 0
    for n in lengths:
        nb = -(-n // w.block)
        for i in range(nb):
            tot += min(w.block, n - i * w.block) * i
    return float(2.0 * w.head_dim * w.hq * tot)


class FixedRunner:
    """One fixed-length layer per step: bsa_mask_build (block-mean queries; bsa_block_meta and
    bsa_select_mask with per-token aggregation), then bsa_prefill_fwd."""

    def __init__(self, bsa, torch, w, dev, flags=0):
        self.bsa, self.torch, self.w, self.dev = bsa, torch, w, dev
        self.s = bsa.make_shape(w.batch, w.seq, w.hq, w.hkv, w.head_dim, w.block)
        self.prm = bsa.SelectParams(w.centroid_keep, w.rescue_keep, flags)
        self.scale = 1.0 / math.sqrt(w.head_dim)
        self.meta = bsa.alloc_meta(self.s, dev)
        self.sel = bsa.alloc_select(self.s, dev, with_mask=False)
        self.fused = flags == 0
        ws_bytes = bsa.mask_build_workspace_bytes(self.s) if self.fused else bsa.select_workspace_bytes(self.s)
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        self.lse = torch.empty(w.batch, w.hq, w.seq, dtype=torch.float32, device=dev)
        self.tokens = w.batch * w.seq

    def make_layer(self, synth, layer):
        return synth.make_layer(self.w, layer=layer)

    def upload(self, lay):
        up = lambda x: self.torch.from_numpy(lay[x].view(np.int16)).to(self.dev).view(self.torch.bfloat16)
        return {x: up(x) for x in ("q", "k", "v")}

    def host_shapes(self):
        """Shape and dtype of the host-side q, k, v and o of one step."""
        w = self.w
        return {"q": ((w.batch, w.seq, w.hq, w.head_dim), self.torch.bfloat16),
                "k": ((w.batch, w.seq, w.hkv, w.head_dim), self.torch.bfloat16),
                "v": ((w.batch, w.seq, w.hkv, w.head_dim), self.torch.bfloat16),
                "o": ((w.batch, w.seq, w.hq, w.head_dim), self.torch.bfloat16)}

    def to_host(self, lay, x):
        return self.torch.from_numpy(lay[x].view(np.int16)).view(self.torch.bfloat16)

    def build(self, L, status):
        """The whole mask build: one call when fused, else the meta and select calls."""
        if self.fused:
            self.mask_call(L, status)
        else:
            self.meta_call(L, status)
            self.select_call(L, status)

    def mask_call(self, L, status):
        m, sl = self.meta, self.sel
        self.bsa.mask_build(self.s, self.prm, L["q"], L["k"], m["centroid"], m["radius"], m["quant"],
                            m["alpha"], sl["kv_idx"], sl["kv_cnt"], None, self.ws, status)

    def meta_call(self, L, status):
        m = self.meta
        self.bsa.block_meta(self.s, L["k"], m["centroid"], m["radius"], m["quant"], m["alpha"], status)

    def select_call(self, L, status):
        m, sl = self.meta, self.sel
        self.bsa.select_mask(self.s, self.prm, L["q"], m["centroid"], m["radius"], m["alpha"],
                             sl["kv_idx"], sl["kv_cnt"], None, self.ws, status)

    def attn_call(self, L, o, status):
        sl = self.sel
        self.bsa.prefill_fwd(self.s, L["q"], L["k"], L["v"], sl["kv_idx"], sl["kv_cnt"], self.scale,
                             o, self.lse, status)

    def stats(self):
        w = self.w
        cnt = self.sel["kv_cnt"].cpu().numpy()
        return (kept_flops(cnt, w.block, w.head_dim, w.group), float(cnt.sum()) * 4 + cnt.size * 4,
                float(cnt.sum()) / (w.batch * w.hkv * w.nb * (w.nb + 1) / 2))

    def e2e_setup(self):
        self.layer_ws = self.bsa.alloc_layer_workspace(self.s, self.dev)

    def e2e_call(self, L, o, status, stream):
        self.bsa.prefill_layer(self.s, self.prm, L["q"], L["k"], L["v"], self.scale, o, self.lse,
                               self.layer_ws, status, stream=stream)

    e2e_api = "bsa_prefill_layer (C ABI)"

    def config(self):
        w = self.w
        return {"workload": w.name, "batch": w.batch, "seq": w.seq, "hq": w.hq, "hkv": w.hkv,
                "head_dim": w.head_dim, "block": w.block, "centroid_keep": w.centroid_keep,
                "rescue_keep": w.rescue_keep}

    def cpu_sample_workload(self):
        return self.w, None


class Fp8Runner(FixedRunner):
    """FixedRunner on e4m3 inputs: bsa_block_meta_fp8, bsa_select_mask_fp8, bsa_prefill_fwd_fp8."""

    def __init__(self, *args, **kwargs):
        super().__init__(*args, **kwargs)
        self.fused = False  # the e4m3 entry points build the mask in two calls

    def make_layer(self, synth, layer):
        lay = synth.make_layer(self.w, layer=layer)
        f8 = synth.fp8_layer(lay)
        out = dict(lay)
        out.update({x: f8[x] for x in ("q", "k", "v")})
        out.update({x + "16": lay[x] for x in ("q", "k", "v")})   # bf16 originals for the CPU oracle
        out["scales"] = {x: f8[x + "_scale"] for x in ("q", "k", "v")}  # each layer its own
        return out

    def upload(self, lay):
        L = {x: self.torch.from_numpy(lay[x]).to(self.dev) for x in ("q", "k", "v")}
        L["scales"] = lay["scales"]
        return L

    def host_shapes(self):
        shp = super().host_shapes()
        return {x: (v[0], self.torch.uint8 if x != "o" else v[1]) for x, v in shp.items()}

    def to_host(self, lay, x):
        return self.torch.from_numpy(lay[x])

    def meta_call(self, L, status):
        m = self.meta
        self.bsa.block_meta_fp8(self.s, L["k"], L["scales"]["k"], m["centroid"], m["radius"], m["quant"],
                                m["alpha"], status)

    def select_call(self, L, status):
        m, sl = self.meta, self.sel
        self.bsa.select_mask_fp8(self.s, self.prm, L["q"], L["scales"]["q"], m["centroid"], m["radius"],
                                 m["alpha"], sl["kv_idx"], sl["kv_cnt"], None, self.ws, status)

    def attn_call(self, L, o, status):
        sl, sc = self.sel, L["scales"]
        if not hasattr(self, "wide_v"):
            self.wide_v = self.torch.empty(self.bsa.prefill_fp8_workspace_bytes(self.s), dtype=self.torch.uint8,
                                           device=self.dev)
        self.bsa.prefill_fwd_fp8(self.s, L["q"], L["k"], L["v"], sc["q"], sc["k"], sc["v"], sl["kv_idx"],
                                 sl["kv_cnt"], self.scale, o, self.lse, self.wide_v, status)

    def e2e_setup(self):
        pass

    def e2e_call(self, L, o, status, stream):
        self.meta_call(L, status)
        self.select_call(L, status)
        self.attn_call(L, o, status)

    e2e_api = "bsa_block_meta_fp8 + bsa_select_mask_fp8 + bsa_prefill_fwd_fp8 (C ABI)"


class VarlenRunner(FixedRunner):
    """One packed ragged batch per step: the bsa_varlen_* entry points."""

    def __init__(self, bsa, torch, vw, dev, flags=0):
        self.bsa, self.torch, self.w, self.dev = bsa, torch, vw, dev
        self.s = bsa.make_varlen_shape(vw.batch, vw.total, vw.max_seqlen, vw.hq, vw.hkv,
                                       vw.head_dim, vw.block)
        self.prm = bsa.SelectParams(vw.centroid_keep, vw.rescue_keep, flags)
        self.scale = 1.0 / math.sqrt(vw.head_dim)
        self.meta = bsa.alloc_varlen_meta(self.s, dev)
        self.sel = bsa.alloc_varlen_select(self.s, dev, with_mask=False)
        self.ws = torch.empty(bsa.varlen_select_workspace_bytes(self.s), dtype=torch.uint8, device=dev)
        self.lse = torch.empty(vw.hq, vw.total, dtype=torch.float32, device=dev)
        self.cu = torch.from_numpy(vw.cu_seqlens()).to(dev)
        self.tokens = vw.total

    def make_layer(self, synth, layer):
        return synth.make_varlen_layer(self.w, layer=layer)

    def host_shapes(self):
        vw = self.w
        return {"q": ((vw.total, vw.hq, vw.head_dim), self.torch.bfloat16),
                "k": ((vw.total, vw.hkv, vw.head_dim), self.torch.bfloat16),
                "v": ((vw.total, vw.hkv, vw.head_dim), self.torch.bfloat16),
                "o": ((vw.total, vw.hq, vw.head_dim), self.torch.bfloat16)}

    def meta_call(self, L, status):
        m = self.meta
        self.bsa.varlen_block_meta(self.s, self.cu, L["k"], m["centroid"], m["radius"], m["quant"],
                                   m["alpha"], status)

    def select_call(self, L, status):
        m, sl = self.meta, self.sel
        self.bsa.varlen_select_mask(self.s, self.prm, self.cu, L["q"], m["centroid"], m["radius"],
                                    m["alpha"], sl["kv_idx"], sl["kv_cnt"], None, self.ws, status)

    def attn_call(self, L, o, status):
        sl = self.sel
        self.bsa.varlen_prefill_fwd(self.s, self.cu, L["q"], L["k"], L["v"], sl["kv_idx"],
                                    sl["kv_cnt"], self.scale, o, self.lse, status)

    def stats(self):
        vw = self.w
        cnt = self.sel["kv_cnt"].cpu().numpy()
        causal = sum(vw.hkv * nb * (nb + 1) / 2 for nb in (-(-n // vw.block) for n in vw.lengths))
        return (kept_flops_varlen(cnt, vw.lengths, vw.block, vw.head_dim, vw.group),
                float(cnt.sum()) * 4 + cnt.size * 4, float(cnt.sum()) / causal)

    def e2e_setup(self):
        pass

    def e2e_call(self, L, o, status, stream):
        self.meta_call(L, status)
        self.select_call(L, status)
        self.attn_call(L, o, status)

    e2e_api = "bsa_varlen_block_meta + bsa_varlen_select_mask + bsa_varlen_prefill_fwd (C ABI)"

    def config(self):
        vw = self.w
        return {"workload": vw.name, "batch": vw.batch, "total_tokens": vw.total,
                "max_seqlen": vw.max_seqlen, "lengths": list(vw.lengths), "hq": vw.hq,
                "hkv": vw.hkv, "head_dim": vw.head_dim, "block": vw.block,
                "centroid_keep": vw.centroid_keep, "rescue_keep": vw.rescue_keep}

    def cpu_sample_workload(self):
        """The longest sequence as a fixed-length batch of one, and the factors that scale its
        per-block and per-row times to the whole packed batch."""
        import synth
        vw = self.w
        b = int(np.argmax(vw.lengths))
        n = vw.lengths[b]
        w = synth.Workload(f"{vw.name}_seq{b}", 1, n, vw.hq, vw.hkv, vw.head_dim, vw.block,
                           vw.centroid_keep, vw.rescue_keep, needles_fixed=vw.needles_fixed)
        blocks = sum(-(-m // vw.block) for m in vw.lengths)
        return w, blocks / w.nb


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import block_sparse_long_kv_gb300 as bsa
    from block_sparse_long_kv_gb300 import build as bld
    import synth
    if rank == 0:
        bld.build()
    if world > 1:
        dist.barrier()

    flags = bsa.SELECT_TOKEN_MAX if args.token_max else 0
    if args.workload in synth.VARLEN_WORKLOADS:
        run = VarlenRunner(bsa, torch, synth.VARLEN_WORKLOADS[args.workload], dev, flags)
    elif args.fp8:
        run = Fp8Runner(bsa, torch, synth.workload(args.workload), dev, flags)
    else:
        run = FixedRunner(bsa, torch, synth.workload(args.workload), dev, flags)
    w = run.w
    n_layers = args.layers or (w.layers if type(run) is FixedRunner else 2)

    # pinned host buffers of the end-to-end leg come first, while the host's free memory is
    # still in long contiguous runs: the layers drawn below leave it fragmented, and a pinned
    # buffer made of scattered small pages copies markedly slower over the host link
    NBUF = 3
    e2e_host = None
    if not args.no_e2e:
        shp = run.host_shapes()
        e2e_host = {"in": [{x: torch.empty(shp[x][0], dtype=shp[x][1], pin_memory=True) for x in ("q", "k", "v")}
                           for _ in range(2)],
                    "o": [torch.empty(shp["o"][0], dtype=shp["o"][1], pin_memory=True) for _ in range(NBUF)]}

    # resident inputs: `n_layers` distinct seeded layers per rank (replicas process their own
    # layers), drawn in worker processes when there are many; host copies are kept for two
    host_layers = []
    dev_layers = []
    ids = replica_layers(rank, n_layers)
    if type(run) is FixedRunner and n_layers > 2:
        from synth import parallel
        for _, arrays, needles in parallel.layers(w, ids):
            dev_layers.append(run.upload(arrays))
            if len(host_layers) < 2:
                host_layers.append({**{x: np.array(arrays[x]) for x in ("q", "k", "v")}, "needles": needles})
            del arrays
    else:
        for li in ids:
            lay = run.make_layer(synth, li)
            host_layers.append(lay)
            dev_layers.append(run.upload(lay))
    o = torch.empty(dev_layers[0]["q"].shape, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    fused = getattr(run, "fused", False)

    def step(L, evs=None):
        if evs:
            evs[0].record(stream)
        if fused:  # the whole mask build in one call (events 1 and 2 coincide)
            run.mask_call(L, status)
        else:
            run.meta_call(L, status)
        if evs:
            evs[1].record(stream)
        if not fused:
            run.select_call(L, status)
        if evs:
            evs[2].record(stream)
        run.attn_call(L, o, status)
        if evs:
            evs[3].record(stream)

    # kept FLOPs and list bytes per layer (exact, from the kernels' own kv_cnt)
    flops, list_bytes, density = [], [], []
    for L in dev_layers:
        step(L)
        torch.cuda.synchronize(dev)
        f, lb, dn = run.stats()
        flops.append(f)
        list_bytes.append(lb)
        density.append(dn)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    for i in range(args.warmup):
        step(dev_layers[i % len(dev_layers)])
    torch.cuda.synchronize(dev)

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for i in range(K):
        step(dev_layers[i % len(dev_layers)], evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = reduce_max(t_start.elapsed_time(t_end), dist if world > 1 else None, dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    meta_ms = np.array([evs[i][0].elapsed_time(evs[i][1]) for i in range(K)])
    sel_ms = np.array([evs[i][1].elapsed_time(evs[i][2]) for i in range(K)])
    att_ms = np.array([evs[i][2].elapsed_time(evs[i][3]) for i in range(K)])
    fl = np.array([flops[i % len(flops)] for i in range(K)])
    lb = np.array([list_bytes[i % len(list_bytes)] for i in range(K)])
    in_bytes = 1 if args.fp8 else 2
    mask_bytes = run.tokens * (w.hq + w.hkv) * w.head_dim * in_bytes + lb
    kept_tflops = float((fl / (att_ms * 1e-3)).mean() / 1e12)
    mask_ms = meta_ms + sel_ms
    mask_gbs = float((mask_bytes / (mask_ms * 1e-3)).mean() / 1e9)

    pk, src = peaks()
    bf16_peak = peak_value(pk, "bf16_tflops", "bf16_tflops_burst")
    hbm_peak = peak_value(pk, "hbm_gbs", "hbm_GBs", "hbm_gb_s")
    peak_note = f"{src} bf16 burst"
    # the seconds-long figure, for context: the timed loop runs tenths of a second per call and
    # draws far less power than a back-to-back GEMM, so the burst figure stays the denominator
    bf16_sustained = peak_value(pk, "bf16_tflops_sustained")
    if args.fp8 and bf16_peak:
        # half the kept FLOPs (S = Q K^T) run on the e4m3 path at the nominal 2x bf16 rate, half
        # (P V) on bf16: the time-weighted peak is 4/3 of the bf16 peak
        bf16_peak = bf16_peak * 4.0 / 3.0
        bf16_sustained = bf16_sustained * 4.0 / 3.0 if bf16_sustained else None
        peak_note = f"{src} bf16 burst x 4/3 (S on e4m3 at 2x, P V on bf16)"
    # the committed DRAM-traffic capture covers the default 128K workload only
    default = (not isinstance(run, (VarlenRunner, Fp8Runner)) and w.name == "gqa32x4_n131072_d128_b128")
    traffic, _ = profiled_traffic() if default else (None, None)
    ms_per_layer = job_ms_per_layer(total_ms, K, world)
    q_gb = run.tokens * w.hq * w.head_dim * in_bytes / 1e9
    cfg = run.config()
    cfg.update({"aggregation": "token_max" if args.token_max else "block_mean",
                "inputs": "e4m3 + per-tensor scales" if args.fp8 else "bf16",
                "layers_rotated": n_layers,
                "layers_timed": min(K, n_layers),
                "l2": f"inputs larger than L2 (Q alone is {q_gb:.2f} GB per layer), layers rotated"})
    result = {
        "metric": METRIC, "value": ms_per_layer, "unit": "ms/layer", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 inputs, bf16 P / O" if args.fp8 else "bf16",
        "data": "synthetic (seeded generator: clustered keys with log-uniform block spreads, planted needles)",
        "config": cfg,
        "kept_block_tflops": kept_tflops,
        "attention_ms": float(att_ms.mean()),
        "mask_build_ms": float(mask_ms.mean()),
        "mask_build_gbs": mask_gbs,
        "density": float(np.mean(density)),
        "density_range": [float(np.min(density)), float(np.max(density))],
        "roofline": {"kernel": "attn_kernel (bsa_prefill_fwd)", "bound": "tensor",
                     "achieved": kept_tflops, "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": kept_tflops / bf16_peak if bf16_peak else None,
                     "frac_of_sustained": kept_tflops / bf16_sustained if bf16_sustained else None,
                     "peak_source": peak_note, "traffic": traffic,
                     "flops_per_launch": float(np.mean(flops))},
        "roofline_mask_build": {"kernels": ("meta_pool_kernel + score_kernel + select_kernel" if fused else
                                             "meta_kernel + quant_kernel + qpool_kernel + score_kernel + select_kernel"),
                                "bound": "hbm", "achieved": mask_gbs, "peak": hbm_peak,
                                "unit": "GB/s", "frac": mask_gbs / hbm_peak if hbm_peak else None,
                                "peak_source": f"{src} hbm copy",
                                "bytes_per_launch": float(np.mean(mask_bytes))},
        # fused: meta + pooling, scores, select, attention (plus a counter memset node); otherwise
        # meta, quant, qpool or centroid split, scores, select, (V widening,) attention
        "gpu_launches": (4 if fused else (7 if args.fp8 else 6)) * K,
        "clocks": clk,
    }
    # the softmax's exponentials: one ex2 on the MUFU units per needed S element (the diagonal
    # block's causal half counted), i.e. kept FLOPs / (4 d).  MUFU peak: 32 ex2 results per
    # clock per SM on this part (twice the 16 of earlier Blackwell SMs); ncu agrees: the XU pipe
    # (sm__inst_executed_pipe_xu) runs at about 30 % of its peak when this rate is 0.29 of 32
    exps = fl / (4.0 * w.head_dim)
    sm_mhz = clk.get("sm_mhz") if isinstance(clk, dict) else None
    mufu_peak = 32 * 152 * (sm_mhz or 2070.0) * 1e6 / 1e9
    exp_rate = float((exps / (att_ms * 1e-3)).mean() / 1e9)
    result["roofline_exp"] = {
        "kernel": "attn_kernel softmax (ex2.approx on MUFU)", "bound": "alu", "achieved": exp_rate,
        "peak": mufu_peak, "unit": "Gexp/s", "frac": exp_rate / mufu_peak,
        "exps_per_launch": float(np.mean(exps)),
        "peak_source": "32 MUFU ex2 results per clock per SM x 152 SMs x the median SM clock of the "
                       "timed region" + ("" if sm_mhz else " (not sampled: 2070 MHz maximum)")}
    if args.token_max:
        # per-token scores are a dense contraction: report the select call against the bf16 peak
        # (FLOPs of q . c for every query token and every key block j < i of its block, per head)
        tf = token_score_flops(run)
        sel_tflops = float((tf / (sel_ms * 1e-3)).mean() / 1e12)
        result["roofline_token_scores"] = {
            "kernels": "centroid_split16_kernel + token_score_kernel + select_kernel (select call)",
            "bound": "tensor", "achieved": sel_tflops, "peak": bf16_peak, "unit": "TFLOP/s",
            "frac": sel_tflops / bf16_peak if bf16_peak else None, "flops_per_launch": tf,
            "note": "algorithmic FLOPs (one product per (token, head, key block)); the kernel runs "
                    "two (bf16 hi and lo centroid splits) and whole 128-block tiles"}

    # end to end through the C ABI: every step copies its Q, K, V from pinned host memory, runs the
    # layer through the library's entry points and copies O back to pinned host memory.  Two buffer
    # sets and two copy streams let the input copy of step s+1 and the output copy of step s-1
    # overlap step s, as a serving loop that prefetches the next layer would.
    if not args.no_e2e:
        run.e2e_setup()
        n_e2e = max(1, args.e2e_steps)
        pinned = e2e_host["in"]
        for x in range(2):
            hl = host_layers[x % len(host_layers)]
            for n in ("q", "k", "v"):
                pinned[x][n].copy_(run.to_host(hl, n))
        # three device buffer sets: a step's inputs are requested two steps ahead, so one slow
        # host copy does not hold up the compute
        o_host = e2e_host["o"]
        dbuf = [{n: (torch.empty_like(o) if n == "o" else torch.empty_like(dev_layers[0][n]))
                 for n in ("q", "k", "v", "o")} for _ in range(NBUF)]
        h2d_s = torch.cuda.Stream(dev)
        d2h_s = torch.cuda.Stream(dev)

        e2e_steps_ms = []  # interval between consecutive steps' compute ends

        def e2e_run(nsteps):
            ev_in = [torch.cuda.Event() for _ in range(nsteps)]
            ev_done = [torch.cuda.Event(enable_timing=True) for _ in range(nsteps)]
            ev_out = [torch.cuda.Event() for _ in range(nsteps)]
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            h2d_s.wait_event(start)
            d2h_s.wait_event(start)

            def issue_h2d(t):
                buf = dbuf[t % NBUF]
                if t >= NBUF:
                    h2d_s.wait_event(ev_done[t - NBUF])     # step t-NBUF no longer reads this buffer
                with torch.cuda.stream(h2d_s):
                    for n in ("q", "k", "v"):
                        buf[n].copy_(pinned[t % 2][n], non_blocking=True)
                hl = host_layers[(t % 2) % len(host_layers)]
                if "scales" in hl:  # per-layer input scales travel with the buffers they describe (e4m3)
                    buf["scales"] = hl["scales"]
                ev_in[t].record(h2d_s)

            for t in range(min(2, nsteps)):
                issue_h2d(t)
            for t in range(nsteps):
                if t + 2 < nsteps:
                    issue_h2d(t + 2)
                buf = dbuf[t % NBUF]
                stream.wait_event(ev_in[t])
                if t >= NBUF:
                    stream.wait_event(ev_out[t - NBUF])       # O of step t-NBUF has reached the host
                run.e2e_call(buf, buf["o"], status, stream)
                ev_done[t].record(stream)
                d2h_s.wait_event(ev_done[t])
                with torch.cuda.stream(d2h_s):
                    o_host[t % NBUF].copy_(buf["o"], non_blocking=True)
                ev_out[t].record(d2h_s)
            stream.wait_event(ev_out[nsteps - 1])
            stream.wait_event(ev_in[nsteps - 1])
            end.record(stream)
            torch.cuda.synchronize(dev)
            e2e_steps_ms[:] = [ev_done[t].elapsed_time(ev_done[t + 1]) for t in range(nsteps - 1)]
            return start.elapsed_time(end)

        e2e_run(2)
        if world > 1:
            dist.barrier()
        e2e_clocks = ClockSampler(local)
        e2e_clocks.start()
        time.sleep(0.3)
        e2e_ms = reduce_max(e2e_run(n_e2e), dist if world > 1 else None, dev)
        e2e_clk = e2e_clocks.stop()
        h2d = sum(pinned[0][n].numel() * pinned[0][n].element_size() for n in ("q", "k", "v"))
        result["e2e"] = {"value": job_ms_per_layer(e2e_ms, n_e2e, world), "unit": "ms/layer",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": o_host[0].numel() * 2,
                         "steps": n_e2e, "clocks": e2e_clk,
                         "api": run.e2e_api + " + pinned host copies on two copy streams, "
                                "three device buffer sets (the input copies of steps s+1 and s+2 and "
                                "the output copy of step s-1 overlap step s)"}
        # the host link on its own, after the timed region: each direction alone, 5 copies
        def copy_rate(fn, nbytes, reps=5):
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(reps):
                fn()
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            return nbytes * reps / (ev0.elapsed_time(ev1) * 1e-3) / 1e9

        def h2d_only():
            for n in ("q", "k", "v"):
                dbuf[0][n].copy_(pinned[0][n], non_blocking=True)

        if len(e2e_steps_ms) >= 8:
            q4 = len(e2e_steps_ms) // 4
            result["e2e"]["step_ms_median_first_quarter"] = float(np.median(e2e_steps_ms[:q4]))
            result["e2e"]["step_ms_median_last_quarter"] = float(np.median(e2e_steps_ms[-q4:]))
            result["e2e"]["step_ms_mean"] = float(np.mean(e2e_steps_ms))
            result["e2e"]["step_ms_max"] = float(np.max(e2e_steps_ms))
        result["e2e"]["host"] = host_placement(local)
        result["e2e"]["copies_alone_gbs"] = {
            "h2d": copy_rate(h2d_only, h2d),
            "d2h": copy_rate(lambda: o_host[0].copy_(dbuf[0]["o"], non_blocking=True), o_host[0].numel() * 2)}
        result["gpu_launches_e2e_per_step"] = 4 if fused else 6
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())}")

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sw, factor = run.cpu_sample_workload()
        lay0 = host_layers[0] if factor is None else synth.make_layer(sw, seed=w.seed_base + int(
            np.argmax(w.lengths)))
        if "q16" in lay0:  # time the oracle on the same layer's bf16 values
            lay0 = {x: lay0[x + "16"] for x in ("q", "k", "v")}
        r = oracle_sample(sw, lay0, args.cpu_budget)
        f = 1.0 if factor is None else factor
        cpu_ms = 1e3 * (f * (r["t_meta"] + r["t_sel"]) + r["t_att_per_flop"] * float(np.mean(flops)))
        sample = r["sample"] if factor is None else (
            r["sample"] + f"; taken on the longest sequence ({sw.seq} tokens) and scaled to the "
            f"packed batch by its block count (x{f:.2f}) and its kept FLOPs")
        result["cpu_baseline"] = {"value": cpu_ms, "unit": "ms/layer", "cores": threads_used(),
                                  "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_decode(args):
    """One decode step per timed step for the last token of every sequence of the workload
    (taken as the KV cache; its block summaries are computed once, as a server keeps them
    between steps): bsa_decode_step (one cooperative launch) for the line's value, then
    bsa_decode_select + bsa_decode_fwd (four launches) timed the same way beside it."""
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import block_sparse_long_kv_gb300 as bsa
    from block_sparse_long_kv_gb300 import build as bld
    import synth
    bld.build()
    if args.workload in synth.VARLEN_WORKLOADS:
        vw = synth.VARLEN_WORKLOADS[args.workload]
        lay = synth.make_varlen_layer(vw)
    else:
        w = synth.workload(args.workload)
        lay0 = synth.make_layer(w)
        vw = synth.VarlenWorkload(w.name, tuple([w.seq] * w.batch), w.hq, w.hkv, w.head_dim, w.block,
                                  w.centroid_keep, w.rescue_keep)
        lay = {x: np.ascontiguousarray(lay0[x].reshape(-1, *lay0[x].shape[2:])) for x in ("q", "k", "v")}
        lay["cu_seqlens"] = vw.cu_seqlens()
        del lay0
    s = bsa.make_varlen_shape(vw.batch, vw.total, vw.max_seqlen, vw.hq, vw.hkv, vw.head_dim, vw.block)
    nbs = bsa.varlen_block_stride(s)
    up = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    k, v = up(lay["k"]), up(lay["v"])
    cu = torch.from_numpy(lay["cu_seqlens"]).to(dev)
    q_new_h = np.zeros((vw.batch, vw.hq, vw.head_dim), dtype=np.uint16)
    for b in range(vw.batch):
        if lay["cu_seqlens"][b + 1] > lay["cu_seqlens"][b]:
            q_new_h[b] = lay["q"][lay["cu_seqlens"][b + 1] - 1]
    q_new = up(q_new_h)
    meta = bsa.alloc_varlen_meta(s, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    bsa.varlen_block_meta(s, cu, k, meta["centroid"], meta["radius"], meta["quant"], meta["alpha"], st)
    kv_idx = torch.zeros(vw.batch, vw.hkv, nbs, dtype=torch.int32, device=dev)
    kv_cnt = torch.zeros(vw.batch, vw.hkv, dtype=torch.int32, device=dev)
    o = torch.empty(vw.batch, vw.hq, vw.head_dim, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(vw.batch, vw.hq, dtype=torch.float32, device=dev)
    ws = torch.empty(bsa.decode_workspace_bytes(s), dtype=torch.uint8, device=dev)
    prm = bsa.SelectParams(vw.centroid_keep, vw.rescue_keep, 0)
    scale = 1.0 / math.sqrt(vw.head_dim)
    stream = torch.cuda.current_stream(dev)
    # an L2-sized buffer rewritten between steps: every step reads its K / V from HBM
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        bsa.decode_select(s, prm, cu, q_new, meta["centroid"], meta["radius"], meta["alpha"], kv_idx,
                          kv_cnt, ws, st)
        if evs:
            evs[1].record(stream)
        bsa.decode_fwd(s, cu, q_new, k, v, kv_idx, kv_cnt, scale, o, lse, ws, st)
        if evs:
            evs[2].record(stream)

    def fused(evs=None):
        if evs:
            evs[0].record(stream)
        bsa.decode_step(s, prm, cu, q_new, k, v, meta["centroid"], meta["radius"], meta["alpha"], scale,
                        kv_idx, kv_cnt, o, lse, ws, st)
        if evs:
            evs[1].record(stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
        flush.zero_()
        fused()
    torch.cuda.synchronize(dev)
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    evf = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    # a step is a few tens of microseconds of GPU work, less than the host needs to issue it, so
    # each timed region starts behind a GPU-side wait long enough for the host to enqueue all of
    # its steps: the events then time the GPU, not the Python calls that feed it
    torch.cuda._sleep(100_000_000)
    for i in range(K):
        flush.zero_()
        fused(evf[i])
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(100_000_000)
    for i in range(K):
        flush.zero_()
        step(evs[i])
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    fused_us = np.array([1e3 * e[0].elapsed_time(e[1]) for e in evf])
    sel_us = np.array([1e3 * e[0].elapsed_time(e[1]) for e in evs])
    att_us = np.array([1e3 * e[1].elapsed_time(e[2]) for e in evs])
    cnt = kv_cnt.cpu().numpy()
    # algorithmic bytes: the kept blocks' keys and values (the current block only up to the new
    # token), the candidates' centroids, radii and alphas, q and o
    kept_tokens = 0
    for b, n in enumerate(vw.lengths):
        if n == 0:
            continue
        last = (n - 1) // vw.block
        idx = kv_idx[b].cpu().numpy()
        for g in range(vw.hkv):
            js = idx[g, :cnt[b, g]]
            kept_tokens += sum(min(vw.block, n - j * vw.block) for j in js)
    kv_bytes = kept_tokens * vw.head_dim * 2 * 2
    meta_bytes = sum(vw.hkv * (-(-n // vw.block)) * (vw.head_dim + 2) * 4 for n in vw.lengths)
    io_bytes = vw.batch * vw.hq * vw.head_dim * 2 * 2
    step_us = sel_us + att_us
    hbm = float(((kv_bytes + meta_bytes + io_bytes) / (fused_us * 1e-6)).mean() / 1e9)
    hbm_two = float(((kv_bytes + meta_bytes + io_bytes) / (step_us * 1e-6)).mean() / 1e9)
    att_gbs = float((kv_bytes / (att_us * 1e-6)).mean() / 1e9)
    pk, src = peaks()
    hbm_peak = peak_value(pk, "hbm_gbs", "hbm_GBs", "hbm_gb_s")
    result = {
        "metric": "decode us/step (new token per sequence, block-sparse split-KV)",
        "value": float(fused_us.mean()), "unit": "us/step", "n_gpus": 1, "steps": K,
        "warmup": max(3, args.warmup), "higher_is_better": False, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": vw.name, "batch": vw.batch, "max_seqlen": vw.max_seqlen,
                   "total_tokens": vw.total, "hq": vw.hq, "hkv": vw.hkv, "head_dim": vw.head_dim,
                   "block": vw.block, "centroid_keep": vw.centroid_keep, "rescue_keep": vw.rescue_keep,
                   "l2": "a 256 MB buffer is rewritten before every step",
                   "issue": "each timed region starts behind a GPU-side wait, so the host has enqueued "
                            "its steps before the GPU reaches them"},
        "two_call_us": float(step_us.mean()), "select_us": float(sel_us.mean()),
        "attention_us": float(att_us.mean()),
        "kept_fraction": float(cnt.sum()) / sum(vw.hkv * (-(-n // vw.block)) for n in vw.lengths),
        "roofline": {"kernel": "decode_step_kernel (bsa_decode_step: scores, selection, attention, merge)",
                     "bound": "hbm", "achieved": hbm, "peak": hbm_peak, "unit": "GB/s",
                     "frac": hbm / hbm_peak if hbm_peak else None, "peak_source": f"{src} hbm copy",
                     "traffic": None, "bytes_per_launch": float(kv_bytes + meta_bytes + io_bytes)},
        "two_call_roofline": {"kernel": "decode_attn_kernel + decode_combine_kernel (bsa_decode_fwd)",
                              "achieved": att_gbs, "unit": "GB/s", "bytes": float(kv_bytes),
                              "step_hbm_gbs": hbm_two},
        "gpu_launches": 5 * K,      # K fused steps (one kernel each, after its barrier memset node)
                                    # and K two-call steps (four kernels each)
        "clocks": clk,
    }
    print(json.dumps(result), flush=True)
    return 0


def needle_recall(w, needles, mask):
    """Fraction of (needle query block, needle key block) pairs the mask keeps."""
    hit = tot = 0
    for (b, g, jb, slot, pos) in needles:
        for i in sorted(set((pos // w.block).tolist())):
            tot += 1
            hit += bool(mask[b, g, i, jb])
    return hit / tot if tot else float("nan")


def run_sweep(args):
    """The 27 block-size x keep-ratio combinations at 64K tokens (GQA 32/4, d 128): per
    combination the kept density, ms per layer (mask build + attention, CUDA events) and the
    needle recall of the GPU mask; one JSON line each, then a summary line."""
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import block_sparse_long_kv_gb300 as bsa
    from block_sparse_long_kv_gb300 import build as bld
    import synth
    bld.build()
    # the oracle's figures, stored by tests/golden/make_sweep_oracle.py (oracle only)
    gold_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tests", "golden",
                             "sweep_oracle.json")
    gold = json.load(open(gold_path))["workloads"]
    rows = []
    layers = {}
    for w in synth.sweep_workloads():
        if w.block not in layers:
            lay = synth.make_layer(w)
            up = lambda x: torch.from_numpy(lay[x].view(np.int16)).to(dev).view(torch.bfloat16)
            layers.clear()
            layers[w.block] = (lay, {x: up(x) for x in ("q", "k", "v")})
        lay, L = layers[w.block]
        run = FixedRunner(bsa, torch, w, dev)
        o = torch.empty_like(L["q"])
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        masked = bsa.alloc_select(run.s, dev, with_mask=True)
        m = run.meta
        bsa.block_meta(run.s, L["k"], m["centroid"], m["radius"], m["quant"], m["alpha"], st)
        bsa.select_mask(run.s, run.prm, L["q"], m["centroid"], m["radius"], m["alpha"], masked["kv_idx"],
                        masked["kv_cnt"], masked["mask"], run.ws, st)
        torch.cuda.synchronize(dev)
        recall = needle_recall(w, lay["needles"], masked["mask"].cpu().numpy())
        for _ in range(max(3, args.warmup)):
            run.build(L, st)
            run.attn_call(L, o, st)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        steps = max(3, min(args.steps, 10))
        times = []
        for _ in range(steps):
            ev[0].record()
            run.build(L, st)
            ev[1].record()
            run.attn_call(L, o, st)
            ev[2].record()
            torch.cuda.synchronize(dev)
            times.append((ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])))
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        f, _, dens = run.stats()
        mk = float(np.median([t[0] for t in times]))
        at = float(np.median([t[1] for t in times]))
        row = {"workload": w.name, "block": w.block, "centroid_keep": w.centroid_keep,
               "rescue_keep": w.rescue_keep, "density": dens, "ms_per_layer": mk + at,
               "mask_build_ms": mk, "attention_ms": at, "kept_block_tflops": f / (at * 1e-3) / 1e12,
               "needle_recall": recall, "oracle_density": gold[w.name]["density"],
               "oracle_needle_recall": gold[w.name]["needle_recall"]}
        rows.append(row)
        print(json.dumps(row), flush=True)
    # the rescue path's contribution: recall with rho_r > 0 against the centroid-only run (rho_r = 0)
    summary = {"metric": "sweep: block size x keep ratios at 64K GQA 32/4 (density, ms/layer, needle recall)",
               "configs": len(rows), "data": "synthetic",
               "recall_centroid_only_mean": float(np.mean([r["needle_recall"] for r in rows if r["rescue_keep"] == 0])),
               "recall_with_rescue_mean": float(np.mean([r["needle_recall"] for r in rows if r["rescue_keep"] > 0]))}
    print(json.dumps(summary), flush=True)
    return 0


def _time_calls(torch, calls, steps, warmup):
    """Median CUDA-event time (ms) of each callable in ``calls`` run back to back."""
    for _ in range(warmup):
        for c in calls:
            c()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
    times = [[] for _ in calls]
    for _ in range(steps):
        ev[0].record()
        for n, c in enumerate(calls):
            c()
            ev[n + 1].record()
        torch.cuda.synchronize()
        for n in range(len(calls)):
            times[n].append(ev[n].elapsed_time(ev[n + 1]))
    return [float(np.median(t)) for t in times]


def run_crossover(args):
    """The sparse path (mask build + attention over the kept blocks) against the dense causal
    path at 32K tokens (GQA 32/4, d 128, block 128, rescue keep-ratio 0.03) while the centroid
    keep-ratio grows to 1; reports density, times, and the density where the two cross."""
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import block_sparse_long_kv_gb300 as bsa
    from block_sparse_long_kv_gb300 import build as bld
    import synth
    bld.build()
    w0 = synth.workload("gqa32x4_n32768_d128_b128")
    lay = synth.make_layer(w0)
    L = {x: torch.from_numpy(lay[x].view(np.int16)).to(dev).view(torch.bfloat16) for x in ("q", "k", "v")}
    o = torch.empty_like(L["q"])
    lse = torch.empty(w0.batch, w0.hq, w0.seq, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    s = bsa.make_shape(w0.batch, w0.seq, w0.hq, w0.hkv, w0.head_dim, w0.block)
    scale = 1.0 / math.sqrt(w0.head_dim)
    steps, warm = max(3, min(args.steps, 20)), max(3, args.warmup)
    dense_ms, = _time_calls(torch, [lambda: bsa.prefill_dense_fwd(s, L["q"], L["k"], L["v"], scale, o,
                                                                    lse, st)], steps, warm)
    dense_flops = 4.0 * w0.batch * w0.hq * w0.head_dim * w0.seq * (w0.seq + 1) / 2
    rows = []
    for rc in (0.02, 0.05, 0.1, 0.15, 0.2, 0.3, 0.4, 0.5, 0.6, 0.7, 0.8, 0.9, 1.0):
        w = w0.with_(centroid_keep=rc)
        run = FixedRunner(bsa, torch, w, dev)
        mk, at = _time_calls(torch, [lambda: run.build(L, st), lambda: run.attn_call(L, o, st)], steps, warm)
        sl = 0.0
        f, _, dens = run.stats()
        row = {"centroid_keep": rc, "rescue_keep": w.rescue_keep, "density": dens,
               "mask_build_ms": mk + sl, "attention_ms": at, "sparse_ms": mk + sl + at,
               "dense_ms": dense_ms, "speedup_vs_dense": dense_ms / (mk + sl + at),
               "kept_block_tflops": f / (at * 1e-3) / 1e12}
        rows.append(row)
        print(json.dumps(row), flush=True)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    # break-even: the first density where the sparse path is no faster, by linear interpolation
    cross = None
    for a, b in zip(rows, rows[1:]):
        if a["sparse_ms"] < dense_ms <= b["sparse_ms"]:
            t = (dense_ms - a["sparse_ms"]) / (b["sparse_ms"] - a["sparse_ms"])
            cross = a["density"] + t * (b["density"] - a["density"])
            break
    print(json.dumps({"metric": "sparse vs dense crossover at 32K GQA 32/4 d128 b128",
                      "dense_ms": dense_ms, "dense_tflops": dense_flops / (dense_ms * 1e-3) / 1e12,
                      "break_even_density": cross, "points": len(rows), "data": "synthetic"}),
          flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.decode:
        return run_decode(args)
    if args.sweep:
        return run_sweep(args)
    if args.crossover:
        return run_crossover(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
