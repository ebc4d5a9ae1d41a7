#!/usr/bin/env python
"""Benchmark of the quantised decode GEMV hot path on GB300.

One step = one pass of a decode layer's projections through libqgemv on one
batch of M tokens:
  dense (default): 27B-class layer, NVFP4 -- QKV 7168x5120, O 5120x6144,
                   gate+up 34816x5120 with the SwiGLU epilogue, down 5120x17408
                   with the residual epilogue; every projection reads its own
                   bf16 N(0, 1) activations;
  q45:             the same shapes under the mixed Q4/Q5 recipe;
  tiny:            one NVFP4 256x512 GEMV;
  moe:             35B-A3B-class MoE layer at M = 8 (device router, then the
                   expert-gathered gate/up + SwiGLU, down and combine).
Metric: effective weight-bytes GB/s (weight bytes per step / step time).
The JSON line is the selected workload (default: dense, M = 1); its "sweep"
array holds the same measurements for every other configuration (dense at
M = 2, 4, 8; Q4/Q5 at M = 1, 8; tiny; MoE), each with its roofline and its
oracle baseline (--no-sweep skips them).

Timing: W untimed warm-up steps, then exactly K steps captured in one CUDA
graph and bracketed by CUDA events on the launching stream (barrier +
synchronize on both sides, max over ranks). Each step reads a different copy
of the layer's weights from a rotation whose total exceeds L2 several times,
so every step streams its weights from HBM. Per-kernel durations come from
events recorded between the kernels inside the graph.

e2e: the same metric through the public Python API with pinned host buffers:
every step copies its activations host->device, runs the projections, and
copies the outputs device->host, all inside the timed region.

cpu_baseline: the fp64 oracle on the host cores over whole steps of the same
workload (repeated to about 12 s; 4 s in the sweep), and with one thread.
--impl reference: the same oracle as the reference arm, K whole steps.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized decode GEMV effective HBM GB/s (% of GB300 peak) and µs/call, M=1–8"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["dense", "q45", "q45ffn", "tiny", "moe"], default="dense")
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-read-probe", action="store_true")
    ap.add_argument("--sweep", dest="sweep", action="store_true", default=True,
                    help="also measure every other configuration (default)")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--no-chain", dest="chain", action="store_false", default=True,
                    help="one launch per projection instead of one qgemv_chain call per step")
    return ap.parse_args()


# ------------------------------------------------------------------ environment
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.strip().split(",") for r in self.f.read().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for i, nm in enumerate(names):
                    if r[5 + i].strip().lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# Kernel sources behind each workload's launches (one or two tokens: the
# CUDA-core kernels; NVFP4 with three to eight tokens and Q4/Q5 with three to
# six: the warp-MMA kernel; Q4/Q5 with seven or eight: the mma.sync kernel;
# the MoE: the grouped CUDA-core expert kernels; the chained layer: its
# kernel at one or two tokens, the workspace kernels at three to eight); a
# committed traffic figure is used only while these files are unchanged.
KERNEL_SOURCES = {
    "simple": ("qgemv_simple.cu", "common.cuh", "qgemv_internal.h"),
    "cc": ("qgemv_cc.cu", "cc_core.cuh", "common.cuh", "qgemv_internal.h"),
    "tc": ("qgemv_tc.cu", "tcgen05.cuh", "common.cuh", "qgemv_internal.h"),
    "mma": ("qgemv_dense.cu", "common.cuh", "qgemv_internal.h"),
    "mt": ("qgemv_mt.cu", "mt_core.cuh", "cc_core.cuh", "common.cuh", "qgemv_internal.h"),
    "moe": ("moe_cc.cu", "moe.cu", "cc_core.cuh", "common.cuh", "qgemv_internal.h"),
    "chain": ("qgemv_chain.cu", "cc_core.cuh", "mt_core.cuh", "common.cuh", "qgemv_internal.h"),
    "chain_ws": ("qgemv_chain_ws.cu", "mt_core.cuh", "cc_core.cuh", "common.cuh", "qgemv_internal.h"),
}


def one_launch_chain(workload, M):
    """Whether the layer's qgemv_chain call runs as one persistent layer
    kernel (it does for every layer of this bench at one to eight tokens; at
    three to eight a small activation conversion kernel runs before it)."""
    return M <= 8


def kernel_family(workload, M):
    if workload == "moe":
        return "moe"
    if workload == "q45ffn" and M > 2:
        return "mt"
    if M <= 2:
        return "cc"
    if workload == "q45":
        return "mt" if M <= 6 else "mma"
    return "mt"


def kernel_source_hash(family):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, "bit_quantized_weight_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag, family):
    """DRAM bytes per launch of `kernel_tag` from the committed ncu summary,
    or None if there is none or the kernel sources changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[kernel_tag]
        if e.get("source_hash") != kernel_source_hash(family):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ workloads
class Workload:
    """Host inputs, device weight copies and the per-step call sequence."""

    def __init__(self, kind, M, copies_min_bytes):
        import numpy as np
        import torch
        import synth
        self.kind, self.M = kind, M
        self.np, self.torch = np, torch
        dev = torch.device("cuda", torch.cuda.current_device())
        self.dev = dev
        # -------- host inputs
        self.projs = []  # (name, N, K, epi, host weights)
        if kind == "dense":
            for name, N, K, epi in synth.dense_layer_shapes():
                self.projs.append((name, N, K, epi, synth.nvfp4_weights(1, f"dense.{name}", N, K)))
        elif kind == "tiny":
            c = synth.TINY
            self.projs.append(("tiny", c.N, c.K, "none", synth.nvfp4_weights(0, "tiny.w", c.N, c.K)))
        elif kind == "q45ffn":
            # the recipe's layer with its FFN fused (Q5 gate + Q4 up, SwiGLU)
            # and RMSNorm prologues ahead of QK, V and the FFN
            W = {name: synth.q45_weights(3, f"q45.{name}", N, K, bits) for name, N, K, bits in synth.Q45_RECIPE}
            sh = {name: (N, K) for name, N, K, bits in synth.Q45_RECIPE}
            for name in ("qk", "v", "o"):
                self.projs.append((name, *sh[name], "none", W[name]))
            ffn = dict(W["gate"])
            ffn["up"] = W["up"]
            self.projs.append(("ffn", *sh["gate"], "swiglu", ffn))
            self.projs.append(("down", *sh["down"], "residual", W["down"]))
            H = synth.DENSE27B.hidden
            r = np.random.default_rng(3)
            gam = [np.round(r.uniform(0.5, 1.5, H) * 128.0) / 128.0 for _ in range(2)]
            self.norms = [torch.from_numpy(g.astype(np.float32)).to(torch.bfloat16).to(dev) for g in gam]
            self.norm_of = {"qk": 0, "v": 0, "ffn": 1}
        else:
            for name, N, K, bits in synth.Q45_RECIPE:
                epi = "residual" if name == "down" else "none"
                self.projs.append((name, N, K, epi, synth.q45_weights(3, f"q45.{name}", N, K, bits)))
        self.weight_bytes = sum(self._wbytes(w) for *_, w in self.projs)
        # -------- activation inputs, packed in one buffer (one H2D copy per step)
        self.in_layout, off = {}, 0
        for name, N, K, epi, _ in self.projs:
            self.in_layout[f"x.{name}"] = (off, (M, K))
            off += M * K
            if epi == "residual":
                self.in_layout[f"r.{name}"] = (off, (M, N))
                off += M * N
        self.in_elems = off
        host_in = np.zeros(off, np.uint16)
        for key, (o, shp) in self.in_layout.items():
            host_in[o:o + shp[0] * shp[1]] = synth.bf16_normal(2, f"bench.{kind}.{key}.M{M}", shp).ravel()
        self.host_in = host_in
        # -------- outputs packed in one buffer (one D2H copy per step)
        self.out_layout, off = {}, 0
        for name, N, K, epi, w in self.projs:
            n_out = N // 2 if (epi == "swiglu" and "up" not in w) else N
            self.out_layout[name] = (off, (M, n_out))
            off += M * n_out
        self.out_elems = off
        # -------- device buffers
        self.d_in = torch.from_numpy(host_in.view(np.int16)).view(torch.bfloat16).to(dev)
        self.d_out = torch.empty(self.out_elems, dtype=torch.bfloat16, device=dev)
        self._views = {}
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 * 2 ** 20)
        self.l2_bytes = int(l2)
        self.copies = max(2, math.ceil(copies_min_bytes * self.l2_bytes / max(self.weight_bytes, 1)))
        self.chains = []
        self.dev_w = [[self._upload(w) for *_, w in self.projs]]

        def clone(d):
            return {k: (clone(v) if isinstance(v, dict) else v.clone() if hasattr(v, "clone") else v)
                    for k, v in d.items()}
        for _ in range(self.copies - 1):
            self.dev_w.append([clone(d) for d in self.dev_w[0]])

    def _wbytes(self, w):
        if "codes" in w:
            return w["codes"].nbytes + w["scales"].nbytes
        b = w["q_lo"].nbytes + w["scale"].nbytes + w["min"].nbytes
        b += w["q_hi"].nbytes if w.get("q_hi") is not None else 0
        return b + (self._wbytes(w["up"]) if "up" in w else 0)

    def _upload(self, w):
        np, torch = self.np, self.torch
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)
        if "codes" in w:
            return {"codes": t(w["codes"]), "scales": t(w["scales"]), "g": w["g"]}
        d = {"q_lo": t(w["q_lo"]), "q_hi": None if w.get("q_hi") is None else t(w["q_hi"]),
             "scale": t(w["scale"].view(np.int16)).view(torch.float16),
             "min": t(w["min"].view(np.int16)).view(torch.float16), "bits": w["bits"]}
        if "up" in w:
            d["up"] = self._upload(w["up"])
        return d

    def view_in(self, key):
        # views are made once: a caller holds its tensors, it does not re-slice
        v = self._views.get(("in", key))
        if v is None:
            o, shp = self.in_layout[key]
            v = self._views[("in", key)] = self.d_in[o:o + shp[0] * shp[1]].view(shp)
        return v

    def view_out(self, name):
        v = self._views.get(("out", name))
        if v is None:
            o, shp = self.out_layout[name]
            v = self._views[("out", name)] = self.d_out[o:o + shp[0] * shp[1]].view(shp)
        return v

    def kernel_names(self):
        return [p[0] for p in self.projs]

    def call(self, idx, copy):
        """Enqueue call idx of the step on the current stream."""
        import bit_quantized_weight_gb300 as q
        name, N, K, epi, _ = self.projs[idx]
        w = self.dev_w[copy % self.copies][idx]
        y = self.view_out(name)
        x = self.view_in(f"x.{name}")
        r = self.view_in(f"r.{name}") if epi == "residual" else None
        nw = self.norms[self.norm_of[name]] if name in getattr(self, "norm_of", {}) else None
        if "codes" in w:
            if epi == "swiglu":
                q.qgemv_swiglu_nvfp4(w["codes"], w["scales"], w["g"], x, y)
            else:
                q.qgemv_nvfp4(w["codes"], w["scales"], w["g"], x, y, residual=r)
        elif "up" in w:
            q.qgemv_swiglu_q45(w, w["up"], x, y, norm=nw)
        elif nw is not None:
            q.GemvChain([{**w, "x": x, "y": y, "norm": nw}]).run()
        else:
            q.qgemv_q45(w["q_lo"], w["q_hi"], w["scale"], w["min"], w["bits"], x, y, residual=r)

    def build_chains(self):
        """One prepared qgemv_chain call per weight copy: the layer's
        projections as the library's single layer call."""
        import bit_quantized_weight_gb300 as q
        self.chains = []
        for c in range(self.copies):
            ops = []
            for idx, (name, N, K, epi, _) in enumerate(self.projs):
                w = self.dev_w[c][idx]
                op = dict(w)
                op.update({"x": self.view_in(f"x.{name}"), "y": self.view_out(name), "epilogue": epi})
                if epi == "residual":
                    op["residual"] = self.view_in(f"r.{name}")
                if "codes" not in op and op.get("q_hi") is None:
                    op.pop("q_hi", None)
                if name in getattr(self, "norm_of", {}):
                    op["norm"] = self.norms[self.norm_of[name]]
                ops.append(op)
            self.chains.append(q.GemvChain(ops))

    def step(self, copy, events=None):
        """Enqueue one step on the current stream: one qgemv_chain call, or
        (with events, or without chains) one call per projection with
        events[i] recorded before call i and events[-1] after the last."""
        if events is None and self.chains:
            self.chains[copy % self.copies].run()
            return
        for i in range(len(self.projs)):
            if events is not None:
                events[i].record()
            self.call(i, copy)
        if events is not None:
            events[-1].record()

    def launches_per_step(self):
        # a chained layer: one launch at one or two tokens; at three to eight
        # the activation conversion kernel and the layer kernel
        if self.chains and one_launch_chain(self.kind, self.M):
            return 1 if self.M <= 2 else 2
        return len(self.projs)

    def alg_bytes(self, idx):
        """Algorithmic bytes of call idx: weights + activations in + outputs."""
        name, N, K, epi, w = self.projs[idx]
        n_out = N // 2 if (epi == "swiglu" and "up" not in w) else N
        b = self._wbytes(w) + 2 * self.M * K + 2 * self.M * n_out
        if epi == "residual":
            b += 2 * self.M * n_out
        return b

    def describe(self):
        return WORKLOAD_NAMES[self.kind](self.M)


class MoeWorkload:
    """35B-A3B-class MoE decode layer: device router (softmax, top-8,
    renormalise) then the expert-gathered NVFP4 gate/up + SwiGLU, down and
    weighted combine. Weight bytes per step = the distinct experts the router
    picks x the bytes of one expert."""

    def __init__(self, M, copies_min_bytes):
        import numpy as np
        import torch
        import synth
        import bit_quantized_weight_gb300 as q
        c = synth.MOE35B
        self.M, self.E, self.H, self.I, self.topk = M, c.experts, c.hidden, c.inter, c.topk
        dev = torch.device("cuda", torch.cuda.current_device())
        E, H, I = self.E, self.H, self.I
        gu = synth.nvfp4_weights(4, "moe.gu", E * 2 * I, H)
        dn = synth.nvfp4_weights(4, "moe.dn", E * H, I)
        self.expert_bytes = (gu["codes"].nbytes + gu["scales"].nbytes + dn["codes"].nbytes
                             + dn["scales"].nbytes) // E
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        base = {"gc": up(gu["codes"]).view(E, 2 * I, H // 2), "gs": up(gu["scales"]).view(E, 2 * I, H // 16),
                "dc": up(dn["codes"]).view(E, H, I // 2), "ds": up(dn["scales"]).view(E, H, I // 16)}
        self.gg = torch.ones(E, dtype=torch.float32, device=dev)
        self.dg = torch.ones(E, dtype=torch.float32, device=dev)
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 * 2 ** 20)
        self.l2_bytes = int(l2)
        total = self.expert_bytes * E
        self.copies = max(2, math.ceil(copies_min_bytes * self.l2_bytes / total))
        self.w = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(self.copies - 1)]
        # activations and router logits, packed for one H2D copy per step
        x = synth.bf16_normal(4, "moe.x", (M, H))
        lg = synth.router_logits(4, "moe.logits", M, E)
        self.host_in = np.concatenate([x.view(np.uint16).ravel(), lg.view(np.uint16).ravel()])
        self.in_elems = self.host_in.size
        self.d_in = torch.from_numpy(self.host_in.view(np.int16)).view(torch.bfloat16).to(dev)
        self.x = self.d_in[: M * H].view(M, H)
        self.logits = self.d_in[M * H:].view(torch.float32).view(M, E)
        self.ids = torch.empty((M, self.topk), dtype=torch.int32, device=dev)
        self.tw = torch.empty((M, self.topk), dtype=torch.float32, device=dev)
        self.d_out = torch.empty(M * H, dtype=torch.bfloat16, device=dev)
        self.out_elems = M * H
        self.ws = torch.empty(q.moe_qgemv_nvfp4_workspace_size(M, self.topk, H, I, E), dtype=torch.uint8, device=dev)
        q.moe_route_topk(self.logits, self.topk, self.ids, self.tw)
        torch.cuda.synchronize()
        self.n_active = int(np.unique(self.ids.cpu().numpy()).size)
        self.weight_bytes = self.n_active * self.expert_bytes
        self.projs = [("router",), ("moe",)]

    def kernel_names(self):
        return ["router", "moe"]

    def launches_per_step(self):
        return 5  # router, grouping, gate/up + SwiGLU, down, combine

    def call(self, idx, copy):
        import bit_quantized_weight_gb300 as q
        w = self.w[copy % self.copies]
        if idx == 0:
            q.moe_route_topk(self.logits, self.topk, self.ids, self.tw)
        else:
            q.moe_qgemv_nvfp4(w["gc"], w["gs"], self.gg, w["dc"], w["ds"], self.dg, self.x, self.ids, self.tw,
                              self.d_out.view(self.M, self.H), self.ws)

    def step(self, copy, events=None):
        for i in range(2):
            if events is not None:
                events[i].record()
            self.call(i, copy)
        if events is not None:
            events[-1].record()

    def alg_bytes(self, idx):
        if idx == 0:
            return self.M * self.E * 4 + self.M * self.topk * 8
        return self.weight_bytes + 2 * self.M * self.H * 2

    def describe(self):
        return WORKLOAD_NAMES["moe"](self.M) + f"; {self.n_active} distinct experts active"


# ------------------------------------------------------------------ CPU oracle
def oracle_step_sample(wl_projs, M, frac, threads):
    """Run the fp64 oracle on every `frac`-th output row of each projection
    (frac = 1: the whole step); returns (seconds, weight bytes processed)."""
    import numpy as np
    import oracle as O
    import synth
    t_total, bytes_done = 0.0, 0
    for name, N, K, epi, w in wl_projs:
        rows = np.arange(0, N, frac)
        x = synth.bf16_normal(2, f"oracle.{name}.M{M}", (M, K))
        if "codes" in w:
            ws = w if frac == 1 else {"codes": w["codes"][rows], "scales": w["scales"][rows], "g": w["g"]}
            t0 = time.perf_counter()
            O.gemv_nvfp4(ws, x, threads=threads)
            t_total += time.perf_counter() - t0
            bytes_done += ws["codes"].nbytes + ws["scales"].nbytes
        else:
            ws = w if frac == 1 else {
                "q_lo": w["q_lo"][rows], "q_hi": None if w.get("q_hi") is None else w["q_hi"][rows],
                "scale": w["scale"][rows], "min": w["min"][rows], "bits": w["bits"]}
            t0 = time.perf_counter()
            O.gemv_q45(ws, x, threads=threads)
            t_total += time.perf_counter() - t0
            bytes_done += sum(a.nbytes for a in (ws["q_lo"], ws["scale"], ws["min"]))
            if ws.get("q_hi") is not None:
                bytes_done += ws["q_hi"].nbytes
    return t_total, bytes_done


def host_projs(kind):
    import synth
    out = []
    if kind == "dense":
        for name, N, K, epi in synth.dense_layer_shapes():
            out.append((name, N, K, epi, synth.nvfp4_weights(1, f"dense.{name}", N, K)))
    elif kind == "tiny":
        c = synth.TINY
        out.append(("tiny", c.N, c.K, "none", synth.nvfp4_weights(0, "tiny.w", c.N, c.K)))
    else:
        for name, N, K, bits in synth.Q45_RECIPE:
            out.append((name, N, K, "none", synth.q45_weights(3, f"q45.{name}", N, K, bits)))
    return out


class OracleMoe:
    """The MoE step on the oracle: the same seeded experts and routing as the
    GPU workload, gate/up + SwiGLU for every (token, slot), then the down
    projections combined in slot order. Weight bytes per step = distinct
    experts x bytes per expert (the metric's definition)."""

    def __init__(self, M):
        import numpy as np
        import oracle as O
        import synth
        c = synth.MOE35B
        E, H, I = c.experts, c.hidden, c.inter
        gu = synth.nvfp4_weights(4, "moe.gu", E * 2 * I, H)
        dn = synth.nvfp4_weights(4, "moe.dn", E * H, I)
        self.expert_bytes = (gu["codes"].nbytes + gu["scales"].nbytes + dn["codes"].nbytes
                             + dn["scales"].nbytes) // E
        self.gu = {"codes": gu["codes"].reshape(E, 2 * I, H // 2), "scales": gu["scales"].reshape(E, 2 * I, H // 16),
                   "g": np.ones(E)}
        self.dn = {"codes": dn["codes"].reshape(E, H, I // 2), "scales": dn["scales"].reshape(E, H, I // 16),
                   "g": np.ones(E)}
        self.x = synth.bf16_normal(4, "moe.x", (M, H))
        lg = synth.router_logits(4, "moe.logits", M, E)
        self.ids, self.w = O.route_topk(lg, c.topk)
        self.n_active = int(np.unique(self.ids).size)
        self.step_bytes = self.n_active * self.expert_bytes

    def step(self, threads):
        import oracle as O
        t0 = time.perf_counter()
        _, _, _, _, h = O.moe_gate_up(self.gu, self.x, self.ids, threads=threads)
        O.moe_down(self.dn, O.bf16_array(h), self.ids, self.w, threads=threads)
        return time.perf_counter() - t0, self.step_bytes


def oracle_runner(kind, M):
    """A callable (threads, frac) -> (seconds, weight bytes) for one oracle
    step of the workload (frac > 1: every frac-th output row only; the MoE
    step is always whole), the workload's name and its weight bytes per step."""
    if kind == "moe":
        om = OracleMoe(M)
        name = WORKLOAD_NAMES["moe"](M) + f"; {om.n_active} distinct experts active"
        return (lambda threads, frac: om.step(threads)), name, om.step_bytes
    projs = host_projs("q45" if kind == "q45ffn" else kind)
    wb = 0
    for *_, w in projs:
        wb += sum(w[k].nbytes for k in ("codes", "scales", "q_lo", "q_hi", "scale", "min")
                  if w.get(k) is not None and hasattr(w[k], "nbytes"))
    return (lambda threads, frac: oracle_step_sample(projs, M, frac, threads)), WORKLOAD_NAMES[kind](M), wb


def cpu_baseline(kind, M, budget_s=12.0, single_thread_budget_s=6.0):
    # the fused-FFN layer streams the same weights through the same GEMV definition
    # (its RMSNorm prologues cost O(K) each): the oracle runs the recipe's projections
    """Oracle throughput on this host's cores: whole steps of the workload,
    repeated until about budget_s of CPU work (a row sample only if one step
    alone exceeds the budget), plus the same with one thread."""
    import oracle as O
    threads = O.default_threads()
    run, _, _ = oracle_runner(kind, M)

    def timed(nthreads, budget):
        t, b = run(nthreads, 1)
        frac, passes = 1, 1
        if t > budget and kind != "moe":               # one whole step is too long: sample rows
            frac = max(2, int(math.ceil(t / budget)))
            t, b = run(nthreads, frac)
        elif t < budget / 2:                           # a whole step is short: repeat it
            passes = max(1, min(5000, int(budget / max(t, 1e-4))))
            for _ in range(passes - 1):
                t1, b1 = run(nthreads, 1)
                t += t1
                b += b1
        return b / t / 1e9, frac, passes, t, b

    v, frac, passes, t, b = timed(threads, budget_s)
    v1, frac1, passes1, t1, b1 = timed(1, single_thread_budget_s)
    what = "whole steps" if frac == 1 else f"every {frac}th output row of each projection"
    return {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{what} of the workload (M={M}), {passes} pass(es), {b / 1e6:.1f} MB of weights in {t:.1f} s",
            "single_thread": {"value": v1, "unit": "GB/s", "cores": 1,
                              "sample": f"{'whole steps' if frac1 == 1 else f'every {frac1}th row'}, "
                                        f"{passes1} pass(es), {b1 / 1e6:.1f} MB in {t1:.1f} s"}}


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle (the method's plain definition)
    timed on the host cores, W untimed then K timed whole steps of the same
    workload as the GPU arm (rows sampled only if K whole steps would take
    more than about two minutes)."""
    if rank != 0:
        return
    import oracle as O
    threads = O.default_threads()
    kind = args.workload
    M = 8 if kind == "moe" else (1 if kind == "tiny" else args.M)
    run, name, step_bytes = oracle_runner(kind, M)
    t1, _ = run(threads, 1)
    frac = 1
    if kind != "moe" and t1 * (args.steps + args.warmup) > 120.0:
        frac = max(2, int(math.ceil(t1 * (args.steps + args.warmup) / 120.0)))
    for _ in range(args.warmup):
        run(threads, frac)
    tt, bb = 0.0, 0
    for _ in range(args.steps):
        t, b = run(threads, frac)
        tt += t
        bb += b
    v = bb / tt / 1e9
    sample = ("whole steps of the workload" if frac == 1 else
              f"every {frac}th output row of each projection per step")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": name, "M": M, "weight_bytes_per_step": step_bytes, "sample": sample},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


WORKLOAD_NAMES = {
    "dense": lambda M: ("dense 27B-class decode layer, NVFP4: QKV 7168x5120, O 5120x6144, "
                        f"gate+up 34816x5120 + SwiGLU, down 5120x17408 + residual, M={M}"),
    "q45": lambda M: ("mixed Q4/Q5 groupwise-int layer on the 27B-class shapes (QK Q4, V Q5, O Q4, "
                      f"gate Q5, up Q4, down Q4 + residual), M={M}"),
    "q45ffn": lambda M: ("mixed Q4/Q5 groupwise-int layer on the 27B-class shapes with the FFN fused (Q5 gate + "
                         "Q4 up, SwiGLU) and RMSNorm prologues on QK, V and the FFN; O Q4, down Q4 + residual, "
                         f"M={M}"),
    "tiny": lambda M: f"tiny NVFP4 GEMV 256x512, M={M}",
    "moe": lambda M: (f"MoE decode layer (35B-A3B-class): hidden 2048, 128 experts, intermediate 768, "
                      f"top-8, M={M}"),
}


# ------------------------------------------------------------------ main
def read_probe_bandwidth(torch, q, stream, peak, nbytes=2 << 30, reps=10):
    """Read-only HBM bandwidth of the library's streaming-read probe (128-bit
    loads from every SM over a 2 GiB buffer, far larger than L2): median of
    `reps` single launches timed with events on the launching stream."""
    buf = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    times = []
    with torch.cuda.stream(stream):
        for _ in range(2):
            q.read_probe(buf, sink, stream=stream)
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            q.read_probe(buf, sink, stream=stream)
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
    t = sorted(times)[len(times) // 2]
    del buf
    gbs = nbytes / (t * 1e-3) / 1e9
    return {"value": gbs, "unit": "GB/s", "bytes": nbytes, "frac_of_measured_copy": gbs / peak,
            "what": "library streaming-read probe (qg_read_probe), median of 10 launches"}


def arithmetic(workload, M, chained=False):
    if workload in ("dense", "tiny") and M <= 2:
        return "f16 x f16 -> f32 FMA on CUDA cores (exact decoded weights, prescaled activations)"
    if workload in ("q45", "q45ffn") and M <= 2:
        return "f16 x f16 -> f32 FMA on CUDA cores (codes as exact f16, prescaled activations)"
    if workload == "q45ffn":
        return "fp32 FMA on CUDA cores (exact fallback kernel for the normalised and fused ops), bf16 mma.sync for the rest"
    if workload == "q45" and (M <= 6 or chained):
        return "f16 mma.sync m16n8k16, f32 accumulate (codes as exact f16, prescaled activations)"
    if workload == "q45":
        return "bf16 mma.sync, f32 accumulate (codes exact in bf16, raw bf16 activations)"
    if workload == "moe":
        return "f16 x f16 -> f32 FMA on CUDA cores (exact decoded weights, prescaled activations)"
    return "f16 mma.sync m16n8k16, f32 accumulate (exact decoded weights, prescaled activations)"


def measure(args, kind, M, world, rank, stream, cpu=True, e2e=True):
    """Time one workload: K steps in one CUDA graph (the headline), per-kernel
    durations, the dominant kernel alone for the roofline, the end-to-end
    loop through the Python API, and the oracle beside it."""
    import torch
    import bit_quantized_weight_gb300 as q
    if kind == "moe":
        wl = MoeWorkload(M, copies_min_bytes=4)
    else:
        wl = Workload(kind, M, copies_min_bytes=4)
        if args.chain and kind != "tiny":
            wl.build_chains()
    chained = bool(getattr(wl, "chains", None))
    n_calls = len(wl.kernel_names())

    with torch.cuda.stream(stream):
        for i in range(args.warmup):                 # eager warm-up
            wl.step(i)
    stream.synchronize()
    assert q.qg_last_device_status(stream) == q.QG_OK

    def make_events(n):
        try:
            return [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n)]
        except (TypeError, RuntimeError):
            return None

    # The headline graph holds only the kernels (events between kernels would
    # serialise them and hide the programmatic-dependent-launch overlap); a
    # second graph of the same steps with events between the calls gives the
    # per-kernel durations.
    ev_steps = [make_events(n_calls + 1) for _ in range(args.steps)]
    per_kernel = ev_steps[0] is not None
    g_warm, g_main, g_ev = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_warm, stream=stream):
        for i in range(args.warmup):
            wl.step(i)
    with torch.cuda.graph(g_main, stream=stream):
        for i in range(args.steps):
            wl.step(args.warmup + i)
    if per_kernel:
        with torch.cuda.graph(g_ev, stream=stream):
            for i in range(args.steps):
                wl.step(args.warmup + i, ev_steps[i])
    g_warm.replay()
    stream.synchronize()

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)                                  # let the sampler take its first reading
    with torch.cuda.stream(stream):
        t0.record(stream)
        g_main.replay()
        t1.record(stream)
    stream.synchronize()
    clk = clocks.stop()
    barrier(world)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    ms = max_over_ranks(ms, world)
    st = q.qg_last_device_status(stream)
    if st != q.QG_OK:
        raise RuntimeError(f"device status {q.qg_status_string(st)} after the timed region")

    value = wl.weight_bytes * args.steps * world / (ms * 1e-3) / 1e9
    ms_per_step = ms / args.steps

    # ---- per-kernel durations (in-graph events) and the dominant kernel's roofline
    us_per_call, dom = {}, None
    if per_kernel:
        with torch.cuda.stream(stream):
            g_ev.replay()
        stream.synchronize()
        names = wl.kernel_names()
        sums = [0.0] * n_calls
        for evs in ev_steps:
            for i in range(n_calls):
                sums[i] += evs[i].elapsed_time(evs[i + 1])
        for i, nm in enumerate(names):
            us_per_call[nm] = sums[i] / args.steps * 1e3
        dom = max(range(n_calls), key=lambda i: sums[i])
    else:
        dom = max(range(n_calls), key=lambda i: wl.alg_bytes(i))
    # The dominant kernel's launch duration for the roofline: K launches of
    # it alone (weights rotating over the same copies) in one graph, CUDA
    # events around the replay on the launching stream. Back to back, each
    # launch overlaps the previous one's tail exactly as inside the step.
    def alone_us(idx):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(args.steps):
                # copies the timed step did not just touch (small weights
                # would otherwise still sit in L2)
                wl.call(idx, i + args.steps)
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) / args.steps * 1e3

    dom_us = alone_us(dom)
    g_dom = None
    sum_alone = None
    if chained:
        sum_alone = sum(dom_us if i == dom else alone_us(i) for i in range(n_calls))
    peak, peak_kind = measured_peaks()
    dom_name = wl.kernel_names()[dom]
    achieved = wl.alg_bytes(dom) / (dom_us * 1e-6) / 1e9
    traffic = profiled_traffic(f"{kind}.{dom_name}.M{M}", kernel_family(kind, M))
    peak_src = (f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback 6.8 TB/s")
    alone = {"kernel": dom_name, "achieved": achieved, "frac": achieved / peak, "alg_bytes_per_launch": wl.alg_bytes(dom),
             "us_per_launch": dom_us, "traffic": traffic,
             "timing": "the projection alone, K launches in one CUDA graph, events on its stream"}
    if chained and one_launch_chain(kind, M):
        # the step is the chained-layer kernel (at three to eight tokens with
        # the conversion kernel ahead of it): it is the
        # dominant (only) kernel, timed by the headline graph itself
        step_bytes = sum(wl.alg_bytes(i) for i in range(n_calls))
        ach = step_bytes / (ms_per_step * 1e-3) / 1e9
        roofline = {"bound": "hbm",
                    "kernel": ("chain_kernel (whole layer, one launch)" if M <= 2 else
                               "chain_ws_convert_kernel + chain_ws_kernel (whole layer, two launches)"),
                    "achieved": ach,
                    "peak": peak, "unit": "GB/s", "frac": ach / peak, "peak_source": peak_src,
                    "traffic": profiled_traffic(f"{kind}.chain.M{M}", "chain" if M <= 2 else "chain_ws"),
                    "alg_bytes_per_launch": step_bytes, "us_per_launch": ms_per_step * 1e3,
                    "timing": "K launches in one CUDA graph (the headline region), events on its stream",
                    "largest_projection_alone": alone}
    else:
        roofline = {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "peak_source": peak_src, "traffic": traffic,
                    "alg_bytes_per_launch": wl.alg_bytes(dom), "us_per_launch": dom_us,
                    "timing": "the kernel alone, K launches in one CUDA graph, events on its stream"}
    if chained:
        roofline["projections_sum_alone_us"] = sum_alone
        roofline["step_vs_sum_alone"] = ms_per_step * 1e3 / sum_alone

    # ---- end to end through the public API with pinned host buffers
    e2e_line = None
    if e2e:
        h_in = torch.from_numpy(wl.host_in.view("int16")).view(torch.bfloat16).pin_memory()
        h_out = torch.empty(wl.out_elems, dtype=torch.bfloat16).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                wl.d_in.copy_(h_in, non_blocking=True)
                wl.step(i)
                h_out.copy_(wl.d_out, non_blocking=True)
            stream.synchronize()
            barrier(world)
            e0.record(stream)
            for i in range(args.steps):
                wl.d_in.copy_(h_in, non_blocking=True)
                wl.step(i)
                h_out.copy_(wl.d_out, non_blocking=True)
            e1.record(stream)
        stream.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), world)
        e2e_line = {"value": wl.weight_bytes * args.steps * world / (ems * 1e-3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": wl.in_elems * 2, "d2h_bytes_per_step": wl.out_elems * 2,
                    "ms_per_step": ems / args.steps}

    cpu_line = cpu_baseline(kind, M, **({} if args.sweep_entry_budget is None else
                                        {"budget_s": args.sweep_entry_budget,
                                         "single_thread_budget_s": args.sweep_entry_budget / 2})) \
        if (cpu and rank == 0 and world == 1) else None
    out = {"workload": wl.describe(), "kind": kind, "M": M, "chained": chained, "value": value, "unit": "GB/s",
           "ms_per_step": ms_per_step, "weight_bytes_per_step": wl.weight_bytes,
           "frac_of_measured_hbm": value / world / peak, "frac_of_8tbs": value / world / NOMINAL_HBM_GBS,
           "us_per_call": us_per_call, "roofline": roofline, "e2e": e2e_line, "cpu_baseline": cpu_line,
           "clocks": clk, "gpu_launches": wl.launches_per_step() * args.steps,
           "dtype": arithmetic(kind, M, chained and one_launch_chain(kind, M)), "l2": f"weights rotate over {wl.copies} copies "
           f"({wl.copies * wl.weight_bytes / 1e6:.0f} MB vs {wl.l2_bytes / 1e6:.0f} MB L2)"}
    del wl, g_warm, g_main, g_ev, g_dom
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


# Every configuration besides the headline one, measured in the same run.
SWEEP = [("dense", 2), ("dense", 4), ("dense", 8), ("q45", 1), ("q45", 2), ("q45", 8), ("q45ffn", 1), ("tiny", 1), ("moe", 8)]


def main():
    args = parse_args()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    assert args.warmup >= 3, "at least 3 warm-up steps"
    import torch
    import bit_quantized_weight_gb300 as q
    torch.cuda.set_device(local)
    if args.workload == "tiny":
        args.M = 1
    if args.workload == "moe":
        args.M = 8
    stream = torch.cuda.Stream()
    args.sweep_entry_budget = None
    head = measure(args, args.workload, args.M, world, rank, stream, cpu=not args.no_cpu_baseline,
                   e2e=not args.no_e2e)
    peak, _ = measured_peaks()
    probe = read_probe_bandwidth(torch, q, stream, peak) if rank == 0 and not args.no_read_probe else None

    sweep = []
    if args.sweep and world == 1:
        args.sweep_entry_budget = 4.0
        for kind, M in SWEEP:
            if (kind, M) == (args.workload, args.M):
                continue
            try:
                sweep.append(measure(args, kind, M, world, rank, stream, cpu=not args.no_cpu_baseline))
            except Exception as ex:                  # one configuration failing must not hide the rest
                sweep.append({"kind": kind, "M": M, "error": f"{type(ex).__name__}: {ex}"})

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
            "data": "synthetic",
            "config": {"workload": head["workload"], "M": args.M,
                       "weight_bytes_per_step": head["weight_bytes_per_step"], "l2": head["l2"],
                       "parallelism": "one independent replica per GPU" if world > 1 else "single GPU",
                       "step": "one qgemv_chain call (the layer's projections in one persistent kernel)"
                               if head["chained"] else "one library call per projection",
                       "graph": "K steps captured in one CUDA graph (kernels only); us_per_call from a "
                                "second graph with events between the calls (which serialise them)"},
            "frac_of_8tbs": head["frac_of_8tbs"],
            "frac_of_measured_hbm": head["frac_of_measured_hbm"],
            "us_per_call": head["us_per_call"],
            "roofline": head["roofline"],
            "read_probe": probe,
            "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"],
            "e2e": head["e2e"],
            "cpu_baseline": head["cpu_baseline"],
            "sweep": sweep,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
