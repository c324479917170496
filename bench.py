#!/usr/bin/env python3
"""Benchmark of the CSA + HCA attention hot path on B300.

The headline step is one query chunk of the 1M-context interleaved layer pair
(context 1,048,576 tokens, the last 4096 positions queried, bf16):
  CSA layer: csa_compress (the chunk's 4096 tokens -> 1024 new entries)
             -> lightning_index fused with topk_select (8 x 64 indexer, k=1024,
                over 262,144 entries) -> sparse_mqa_attn (128 heads x 128,
                1024 selected entries + 128-token window)
  HCA layer: hca_compress (chunk -> 32 new entries)
             -> hca_dense_attn (128 heads x 128 over <= 8192 entries + window)
Entries of the positions before the chunk come from the same compressors in
an untimed set-up (they are the layer's KV cache).  Metric: query tokens per
second (4096 per step per GPU).

The default run also measures six other full-size settings and prints each
as a sub-record of the same JSON line (same fields as the main record):
  decode       one decode step of 64 sequences (one query each at its last
               position, contexts ~U[65536, 262144], compressed caches and
               indexer keys resident): lightning_index fused with topk_select
               (k=1024) -> sparse_mqa_attn (128 heads, window 128).  HBM-bound:
               its roofline is the whole step's algorithmic bytes over the
               step's time against the measured copy bandwidth.
  decode_incremental  the decode setting token by token: each step appends
               one new token per request to the decode state (decode_append:
               window ring, open block, the block's entry every fourth token)
               before the index + top-k and the attention.
  decode_mxfp4, decode_mxfp8  the decode setting with the low-precision
               indexer: indexer keys stored in MXFP4 / MXFP8 (OCP MX, blocks of 32
               values with a power-of-two scale), the step's q_I quantized,
               scores and top-k on the quantized values, bf16 attention; the
               record adds the recall of the quantized selection against the
               exact one.
  csa_prefill  a 32,768-token CSA prefill (64 heads x 128, indexer 8 x 64,
               k=512, window 128): csa_compress -> lightning_index + top-k ->
               sparse_mqa_attn.
  hca_prefill  a 131,072-token HCA prefill (64 heads x 128, m'=128, window
               128): hca_compress -> hca_dense_attn.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload all|layer_pair_1m|csa_decode|csa_decode_incremental|
                              csa_decode_mxfp4|csa_decode_mxfp8|csa_prefill|hca_prefill]

Prints ONE JSON line on rank 0.  `--impl reference` times the CPU oracle on a
bounded sample of the layer-pair workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "CSA+HCA attention query-tokens/s (prefill & decode) and % of B300 roofline"
UNIT = "query-tokens/s"


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per step of the
# kernels of each workload's roofline stage, from one ncu capture of the
# current kernels at the full benchmarked size (traffic well above the
# algorithmic bytes would mean re-reads).  An entry is removed when one of its
# kernels changes, until it is measured again.
NCU_STAGE_TRAFFIC = {
    # the decode step's kernels at the full benchmarked size: streaming
    # indexer 2504.1 MB, cluster top-k 9.8 MB, CSA attention 40.2 MB
    ("csa_decode", "step"): 2554.0e6,
    # the layer pair at 1M: k_hca_tc 140.9 MB read + 84.2 MB written
    ("layer_pair_1m", "hca_dense_attn"): 225.1e6,
    # index + top-k: candidate pass 341.8, 16-bit sample 23.7, thresholds
    # 67.1, candidate pick 79.9 (its 512-thread build; the 256-thread one
    # reads the same candidates), fallback 0 (MB read + written)
    ("layer_pair_1m", "lightning_index+topk"): 512.5e6,
    # k_sparse_tc 1121.8 MB read + 128.1 MB written
    ("layer_pair_1m", "sparse_mqa_attn"): 1249.9e6,
    # the 32K CSA prefill: k_sparse_tc 625.3 + 503.6 MB
    ("csa_prefill", "sparse_mqa_attn"): 1128.9e6,
    # the 128K HCA prefill: k_hca_tc 2215.7 MB read + 2127.5 MB written
    ("hca_prefill", "hca_dense_attn"): 4343.2e6,
}


# --decode-ctx LO,HI: the decode workloads on a shorter context range (a
# smaller case of the same kernels for profiler captures); None = the
# configured ~U[65536, 262144]
DECODE_CTX = None


def decode_config(device):
    if DECODE_CTX is None:
        return wl.CONFIGS["csa_decode"](device=device)
    lo, hi = DECODE_CTX
    return wl.csa_decode(B=64, ctx_lo=lo, ctx_hi=hi, H=128, d=128, HI=8, dI=64, m=4, k=1024,
                         W=128, dtype="bf16", seed=3, device=device)


def gather_bound(keys_sum, d, n_tokens, H, k, ms, peaks):
    """The CSA attention's gathered bytes over its time, against the measured
    copy bandwidth: each token reads the K and V rows of its keys (selected
    entries and window tokens, d bf16 values each) once, its selection (k
    int32), its Q and writes its O.  The gather of random 256-byte rows, not
    the tensor cores, bounds that kernel."""
    b = float(keys_sum * d * 2 * 2 + n_tokens * (k * 4 + 2 * H * d * 2))
    gbs = b / (ms / 1e3) / 1e9
    return {"sparse_mqa_attn_gather": {"bytes": b, "achieved": gbs, "unit": "GB/s",
                                       "peak": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"]}}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        # nvidia-smi's own start-up (driver queries) must not overlap the timed
        # region: wait for its first sample
        t0 = time.perf_counter()
        while not self.lines and self.proc.poll() is None and time.perf_counter() - t0 < 10:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def _n_window(t, W):
    return np.minimum(np.asarray(t, dtype=np.int64) + 1, W)


def _cpu(d):
    return {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in d.items()}


def layer_pair_config(ctx, chunk, H, d, world):
    return {"workload": f"layer_pair_{ctx // 1024}k: CSA (m=4, indexer 8x64, top-k 1024, "
                        f"window 128) + HCA (m'=128, window 128) over a {ctx:,}-token context, "
                        f"last {chunk} positions queried, Q [{chunk},{H},{d}] per layer",
            "context": ctx, "query_chunk": chunk, "heads": H, "head_dim": d,
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (raw K/V 256 MiB each, indexer keys 256 MiB)"}


def tensor_roofline(stages, stage_ms, flops_of, peaks, region_ms, traffic_key=None):
    """Tensor roofline of the stage (among flops_of) with the longest time."""
    dom = max(flops_of, key=lambda s: stage_ms[stages.index(s)])
    dom_ms = stage_ms[stages.index(dom)]
    achieved = flops_of[dom] / (dom_ms / 1e3) / 1e12
    long_region = region_ms > 1000.0
    peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    traffic = NCU_STAGE_TRAFFIC.get((traffic_key, dom)) if traffic_key else None
    return {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
            "traffic_unit": "DRAM bytes per launch of the stage's kernels (ncu)",
            "algorithmic_flop": flops_of[dom],
            "peak_source": peaks["source"] + (" sustained" if long_region else " burst")}


# ---------------------------------------------------------------- workloads

class LayerPair:
    """Device buffers and the step of the 1M-context layer pair."""

    STAGES = ["csa_compress", "lightning_index+topk", "sparse_mqa_attn", "hca_compress",
              "hca_dense_attn"]

    def __init__(self, lc, device, seed=4, ctx=1 << 20, chunk=4096):
        self.lc = lc
        P = wl.layer_pair(ctx=ctx, chunk=chunk, seed=seed, device=device)
        self.P = P
        c, h = P["csa"], P["hca"]
        self.ctx, self.chunk = ctx, chunk
        self.q0 = ctx - chunk
        self.m_c, self.m_h = c["m"], h["m"]
        self.k, self.W = c["k"], c["W"]
        self.H, self.d = c["H"], c["d"]
        d = self.d
        # compressed caches: entries before the chunk come from an untimed
        # compression of the prefix
        self.Kc = torch.empty((ctx // self.m_c, d), dtype=torch.bfloat16, device=device)
        self.Vc = torch.empty_like(self.Kc)
        self.Kh = torch.empty((ctx // self.m_h, d), dtype=torch.bfloat16, device=device)
        self.Vh = torch.empty_like(self.Kh)
        lc.csa_compress(c["K"][: self.q0], c["V"][: self.q0], c["G"], m=self.m_c,
                        Kc=self.Kc[: self.q0 // self.m_c], Vc=self.Vc[: self.q0 // self.m_c])
        lc.hca_compress(h["K"][: self.q0], h["V"][: self.q0], h["G"], m=self.m_h,
                        Kc=self.Kh[: self.q0 // self.m_h], Vc=self.Vh[: self.q0 // self.m_h])
        self.b_csa = lc.DeviceBatch.from_workload(c["batch"], device=device)
        self.b_hca = lc.DeviceBatch.from_workload(h["batch"], device=device)
        self.ws = torch.empty(lc.workspace_size(lc.LC_OP_LIGHTNING_INDEX, self.b_csa,
                                                HI=c["HI"], dI=c["dI"], k=self.k),
                              dtype=torch.uint8, device=device)
        self.sel = torch.empty((chunk, self.k), dtype=torch.int32, device=device)
        self.O_csa = torch.empty_like(c["Q"])
        self.O_hca = torch.empty_like(h["Q"])
        self.lse_csa = torch.empty((chunk, self.H), dtype=torch.float32, device=device)
        self.lse_hca = torch.empty_like(self.lse_csa)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

    # algorithmic work of one step (causal counts), for the roofline
    def work(self):
        t = np.arange(self.q0, self.ctx, dtype=np.int64)
        nwin = _n_window(t, self.W)
        nv_c = (t + 1) // self.m_c
        nv_h = (t + 1) // self.m_h
        c = self.P["csa"]
        HI, dI = c["HI"], c["dI"]
        keys_csa = np.minimum(nv_c, self.k) + nwin
        keys_hca = nv_h + nwin
        return {
            "index_flop": float(2 * HI * dI * nv_c.sum()),
            "csa_attn_flop": float(4 * self.d * self.H * keys_csa.sum()),
            "hca_attn_flop": float(4 * self.d * self.H * keys_hca.sum()),
            "csa_keys": int(keys_csa.sum()),
        }

    def stage_extra(self, stage_ms, peaks):
        return gather_bound(self.work()["csa_keys"], self.d, self.chunk, self.H, self.k,
                            stage_ms[self.STAGES.index("sparse_mqa_attn")], peaks)

    def step(self, events=None):
        lc, c, h = self.lc, self.P["csa"], self.P["hca"]
        ev = events
        if ev:
            ev[0].record()
        lc.csa_compress(c["K"][self.q0:], c["V"][self.q0:], c["G"], m=self.m_c,
                        Kc=self.Kc[self.q0 // self.m_c:], Vc=self.Vc[self.q0 // self.m_c:])
        if ev:
            ev[1].record()
        lc.lightning_index(c["qI"], c["w"], c["kI"], self.b_csa, self.m_c, scores=False,
                           k=self.k, topk=self.sel, ws=self.ws, dev_err=self.err)
        if ev:
            ev[2].record()
        lc.sparse_mqa_attn(c["Q"], self.Kc, self.Vc, self.sel, c["K"], c["V"], self.b_csa,
                           self.m_c, self.W, c["scale"], O=self.O_csa, lse=self.lse_csa,
                           dev_err=self.err)
        if ev:
            ev[3].record()
        lc.hca_compress(h["K"][self.q0:], h["V"][self.q0:], h["G"], m=self.m_h,
                        Kc=self.Kh[self.q0 // self.m_h:], Vc=self.Vh[self.q0 // self.m_h:])
        if ev:
            ev[4].record()
        lc.hca_dense_attn(h["Q"], self.Kh, self.Vh, h["K"], h["V"], self.b_hca, self.m_h, self.W,
                          h["scale"], O=self.O_hca, lse=self.lse_hca, dev_err=self.err)
        if ev:
            ev[5].record()

    def config(self, world):
        return layer_pair_config(self.ctx, self.chunk, self.H, self.d, world)

    def roofline(self, stage_ms, peaks, region_ms, step_ms):
        w = self.work()
        flops_of = {"lightning_index+topk": w["index_flop"], "sparse_mqa_attn": w["csa_attn_flop"],
                    "hca_dense_attn": w["hca_attn_flop"]}
        key = "layer_pair_1m" if self.ctx == 1 << 20 else None
        return tensor_roofline(self.STAGES, stage_ms, flops_of, peaks, region_ms, key)

    def path_tflops(self, ms_step):
        w = self.work()
        return (w["index_flop"] + w["csa_attn_flop"] + w["hca_attn_flop"]) / (ms_step / 1e3) / 1e12

    def cpu_baseline(self, budget_s):
        return layer_pair_cpu_baseline(self, budget_s=budget_s)

    # per-step host inputs / outputs of the end-to-end measurement
    def host_io(self):
        c, h = self.P["csa"], self.P["hca"]
        n_new = self.chunk // self.m_c
        ins = {
            "Q_csa": c["Q"], "Q_hca": h["Q"], "qI": c["qI"], "w": c["w"],
            "kI_new": c["kI"][-n_new:],
            "K_csa_chunk": c["K"][self.q0:], "V_csa_chunk": c["V"][self.q0:],
            "K_hca_chunk": h["K"][self.q0:], "V_hca_chunk": h["V"][self.q0:],
        }
        outs = {"O_csa": self.O_csa, "O_hca": self.O_hca}
        return ins, outs


class Decode:
    """Device buffers and the step of the batch-64 CSA decode workload."""

    STAGES = ["lightning_index+topk", "sparse_mqa_attn"]

    def __init__(self, lc, device, seed=3):
        self.lc = lc
        D = decode_config(device)
        assert D["seed"] == seed
        self.D = D
        self.chunk = D["B"]  # query tokens per step
        self.m, self.k, self.W, self.H, self.d = D["m"], D["k"], D["W"], D["H"], D["d"]
        self.b = lc.DeviceBatch.from_workload(D["batch"], device=device)
        self.ws = torch.empty(lc.workspace_size(lc.LC_OP_LIGHTNING_INDEX, self.b, HI=D["HI"],
                                                dI=D["dI"], k=self.k),
                              dtype=torch.uint8, device=device)
        self.sel = torch.empty((D["B"], self.k), dtype=torch.int32, device=device)
        self.O = torch.empty_like(D["Q"])
        self.lse = torch.empty((D["B"], self.H), dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

    def work(self):
        """Algorithmic bytes of one step: every visible indexer key once, the
        query's indexer q and head weights, the selected indices written and
        read, every gathered K/V row (selected entries and window) once, Q
        read and O written."""
        D = self.D
        ctx = np.array(D["ctx"], dtype=np.int64)
        nv = ctx // self.m
        keys = np.minimum(nv, self.k) + _n_window(ctx - 1, self.W)
        idx_bytes = float(nv.sum() * D["HI"] * D["dI"] * 2 + D["B"] * D["HI"] * (D["dI"] * 2 + 4)
                          + D["B"] * self.k * 4)
        attn_bytes = float(keys.sum() * self.d * 2 * 2 + 2 * D["B"] * self.H * self.d * 2
                           + D["B"] * self.k * 4)
        return {"index_bytes": idx_bytes, "attn_bytes": attn_bytes,
                "step_bytes": idx_bytes + attn_bytes,
                "attn_flop": float(4 * self.d * self.H * keys.sum())}

    def step(self, events=None):
        lc, D = self.lc, self.D
        ev = events
        if ev:
            ev[0].record()
        lc.lightning_index(D["qI"], D["w"], D["kI"], self.b, self.m, scores=False, k=self.k,
                           topk=self.sel, ws=self.ws, dev_err=self.err)
        if ev:
            ev[1].record()
        lc.sparse_mqa_attn(D["Q"], D["Kc"], D["Vc"], self.sel, D["Kraw"], D["Vraw"], self.b,
                           self.m, self.W, D["scale"], O=self.O, lse=self.lse, dev_err=self.err)
        if ev:
            ev[2].record()

    def host_io(self):
        D = self.D
        ins = {"Q": D["Q"], "qI": D["qI"], "w": D["w"]}
        return ins, {"O": self.O}

    def config(self, world):
        lo, hi = DECODE_CTX or (65536, 262144)
        return {"workload": "csa_decode: 64 sequences, one query token each at its last "
                            f"position, contexts ~U[{lo}, {hi}] (seed 3), CSA m=4, indexer "
                            "8x64, top-k 1024, window 128, Q [64,128,128]",
                "batch": self.D["B"], "heads": self.H, "head_dim": self.d,
                "context_mean": float(np.mean(self.D["ctx"])),
                "parallelism": f"replicas x{world}",
                "l2": "inputs larger than L2 (indexer keys 2.7 GB, compressed K/V 1.3 GB)"}

    def path_tflops(self, ms_step):
        return self.work()["attn_flop"] / (ms_step / 1e3) / 1e12

    def cpu_baseline(self, budget_s):
        return decode_cpu_baseline(self, budget_s=budget_s)

    def roofline(self, stage_ms, peaks, region_ms, step_ms):
        """HBM roofline of the whole step: its algorithmic bytes over the
        timed step (a graph replay of its kernels, or the eager calls)."""
        w = self.work()
        gbs = w["step_bytes"] / (step_ms / 1e3) / 1e9
        return {"bound": "hbm", "kernel": "whole step (lightning_index+topk, sparse_mqa_attn)",
                "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"],
                "traffic": NCU_STAGE_TRAFFIC.get(("csa_decode", "step")),
                "traffic_unit": "DRAM bytes per step of the step's kernels (ncu)",
                "algorithmic_bytes": w["step_bytes"], "peak_source": peaks["source"]}


class DecodeMX(Decode):
    """The batch-64 decode step with the low-precision indexer: the indexer
    keys are stored MX-quantized (quantized once, outside the step, as the
    layer's indexer-key cache would be), each step quantizes the step's q_I,
    scores every visible entry on the MX values, selects the top-k of those
    scores and runs the bf16 CSA attention.  `recall` is the fraction of the
    exact (bf16 indexer) selection that the quantized selection keeps."""

    STAGES = ["mx_quantize(q)+lightning_index_mx+topk", "sparse_mqa_attn"]

    def __init__(self, lc, device, fmt):
        super().__init__(lc, device)
        self.fmt = fmt
        D = self.D
        self.kc, self.ks = lc.mx_quantize(D["kI"], fmt)
        self.qc, self.qs = lc.mx_quantize(D["qI"], fmt)
        torch.cuda.synchronize()

    @property
    def DTYPE(self):
        return f"mxfp{self.fmt} indexer, bf16 attention"

    def work(self):
        w = super().work()
        D = self.D
        nv = np.array(D["ctx"], dtype=np.int64) // self.m
        per_entry = D["HI"] * (D["dI"] * self.fmt // 8 + D["dI"] // 32)
        q_bytes = D["B"] * D["HI"] * (D["dI"] * 2 + D["dI"] * self.fmt // 8 + D["dI"] // 32 + 4)
        w["index_bytes"] = float(nv.sum() * per_entry + q_bytes + D["B"] * self.k * 4)
        w["step_bytes"] = w["index_bytes"] + w["attn_bytes"]
        return w

    def step(self, events=None):
        lc, D = self.lc, self.D
        ev = events
        if ev:
            ev[0].record()
        lc.mx_quantize(D["qI"], self.fmt, codes=self.qc, scales=self.qs)
        lc.lightning_index_mx(self.fmt, self.qc, self.qs, D["w"], self.kc, self.ks, self.b,
                              self.m, scores=False, k=self.k, topk=self.sel, ws=self.ws,
                              dev_err=self.err)
        if ev:
            ev[1].record()
        lc.sparse_mqa_attn(D["Q"], D["Kc"], D["Vc"], self.sel, D["Kraw"], D["Vraw"], self.b,
                           self.m, self.W, D["scale"], O=self.O, lse=self.lse, dev_err=self.err)
        if ev:
            ev[2].record()

    def config(self, world):
        c = super().config(world)
        c["workload"] = (f"csa_decode_mxfp{self.fmt}: " + c["workload"].split(": ", 1)[1] +
                         f"; indexer q/k in MXFP{self.fmt} (OCP MX, 32-value blocks)")
        return c

    def roofline(self, stage_ms, peaks, region_ms, step_ms):
        r = super().roofline(stage_ms, peaks, region_ms, step_ms)
        r["traffic"] = None
        return r

    def extra(self):
        """Recall of the quantized selection against the exact selection of
        the bf16 indexer (the fused exact path, parity-tested on its own)."""
        D = self.D
        exact = torch.empty_like(self.sel)
        self.lc.lightning_index(D["qI"], D["w"], D["kI"], self.b, self.m, scores=False, k=self.k,
                                topk=exact, ws=self.ws)
        torch.cuda.synchronize()
        a, b = exact.cpu().numpy(), self.sel.cpu().numpy()
        rec = [len(np.intersect1d(a[i][a[i] >= 0], b[i][b[i] >= 0])) / max(1, (a[i] >= 0).sum())
               for i in range(a.shape[0])]
        return {"recall": {"mean": float(np.mean(rec)), "min": float(np.min(rec)),
                           "against": "exact top-k of the bf16 indexer on the same inputs"}}

    def cpu_baseline(self, budget_s):
        return decode_cpu_baseline(self, budget_s=budget_s, fmt=self.fmt)


class DecodeMXFP4(DecodeMX):
    def __init__(self, lc, device):
        super().__init__(lc, device, 4)


class DecodeMXFP8(DecodeMX):
    def __init__(self, lc, device):
        super().__init__(lc, device, 8)


class DecodeIncremental:
    """Token-by-token decode of the batch-64 CSA setting through the decode
    state: each step appends one new token per request (ring, open block and,
    every fourth token, the block's compressed entry), then runs the fused
    index + top-k over the request's classical cache and the sparse attention
    with the window read from the ring.  The state starts from the decode
    setting's caches (contexts ~U[65536, 262144], seed 3), copied into each
    request's fixed-capacity region."""

    STAGES = ["decode_append", "lightning_index+topk", "sparse_mqa_attn"]

    def __init__(self, lc, device, seed=3):
        self.lc = lc
        D = decode_config(device)
        assert D["seed"] == seed
        self.ctx0 = list(D["ctx"])
        B, d, HI, dI, m, W = D["B"], D["d"], D["HI"], D["dI"], D["m"], D["W"]
        self.B, self.m, self.k, self.W, self.H, self.d = B, m, D["k"], W, D["H"], d
        self.HI, self.dI = HI, dI
        self.chunk = B
        cap = max(self.ctx0) // m + 64
        L = lc.DecodeLayer(B, W, d, m, cap, HI, dI, device=device)
        bt = D["batch"]
        for b in range(B):
            c0, c1, r0, r1 = bt.cu_c[b], bt.cu_c[b + 1], bt.cu_raw[b], bt.cu_raw[b + 1]
            L.Kc[b * cap:b * cap + (c1 - c0)] = D["Kc"][c0:c1]
            L.Vc[b * cap:b * cap + (c1 - c0)] = D["Vc"][c0:c1]
            L.kI[b * cap:b * cap + (c1 - c0)] = D["kI"][c0:c1]
            # the ring holds the last W positions: p0 .. ctx-1
            p0 = bt.raw_pos0[b]
            rows = torch.arange(p0, p0 + (r1 - r0), device=device) % W + b * 2 * W
            for off in (0, W):
                L.Kring[rows + off] = D["Kraw"][r0:r1]
                L.Vring[rows + off] = D["Vraw"][r0:r1]
        L.n_tok.copy_(torch.tensor(self.ctx0, dtype=torch.int64, device=device))
        self.L = L
        g = wl._gen(seed + 500, device)
        self.K_new = wl.normal(g, (B, d), "bf16", device)
        self.V_new = wl.normal(g, (B, d), "bf16", device)
        self.kI_new = wl.normal(g, (B, HI, dI), "bf16", device)
        self.G = wl.normal(g, (m, d), "f32", device)
        self.GI = wl.normal(g, (m, HI * dI), "f32", device)
        self.Q, self.qI, self.w, self.scale = D["Q"], D["qI"], D["w"], D["scale"]
        self.ws = torch.empty(lc.workspace_size(lc.LC_OP_LIGHTNING_INDEX, L.batch, HI=HI, dI=dI,
                                                k=self.k), dtype=torch.uint8, device=device)
        self.sel = torch.empty((B, self.k), dtype=torch.int32, device=device)
        self.O = torch.empty_like(self.Q)
        self.lse = torch.empty((B, self.H), dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        del D
        torch.cuda.synchronize()

    def step(self, events=None):
        lc, L = self.lc, self.L
        ev = events
        if ev:
            ev[0].record()
        lc.decode_append(L, self.K_new, self.V_new, self.G, kI_new=self.kI_new, G_I=self.GI,
                         dev_err=self.err)
        if ev:
            ev[1].record()
        lc.lightning_index(self.qI, self.w, L.kI, L.batch, self.m, scores=False, k=self.k,
                           topk=self.sel, ws=self.ws, dev_err=self.err)
        if ev:
            ev[2].record()
        lc.sparse_mqa_attn(self.Q, L.Kc, L.Vc, self.sel, L.Kring, L.Vring, L.batch, self.m,
                           self.W, self.scale, O=self.O, lse=self.lse, dev_err=self.err)
        if ev:
            ev[3].record()

    def work(self):
        """Algorithmic bytes of one step at the starting contexts: the append
        (the new token's K, V, indexer keys into the ring, a quarter of the
        requests writing an entry), then as for the decode setting."""
        ctx = np.array(self.ctx0, dtype=np.int64) + 1
        nv = ctx // self.m
        keys = np.minimum(nv, self.k) + np.minimum(ctx, self.W)
        B, d, dk = self.B, self.d, self.HI * self.dI
        append = B * (2 * d * 2 * 3 + dk * 2 * 2) + B / self.m * (2 * d * 2 + dk * 2) * 2
        idx = nv.sum() * dk * 2 + B * self.HI * (self.dI * 2 + 4) + B * self.k * 4
        attn = keys.sum() * d * 2 * 2 + 2 * B * self.H * d * 2 + B * self.k * 4
        return {"step_bytes": float(append + idx + attn),
                "attn_flop": float(4 * d * self.H * keys.sum())}

    def host_io(self):
        return ({"K_new": self.K_new, "V_new": self.V_new, "kI_new": self.kI_new, "Q": self.Q,
                 "qI": self.qI, "w": self.w}, {"O": self.O})

    def config(self, world):
        return {"workload": "csa_decode_incremental: 64 requests, contexts ~U[65536, 262144] "
                            "(seed 3), one new token each per step through the decode state "
                            "(append, index + top-k 1024, CSA attention with window 128)",
                "batch": self.B, "heads": self.H, "head_dim": self.d,
                "context_mean": float(np.mean(self.ctx0)), "parallelism": f"replicas x{world}",
                "l2": "inputs larger than L2 (indexer keys 2.7 GB)"}

    def roofline(self, stage_ms, peaks, region_ms, step_ms):
        w = self.work()
        gbs = w["step_bytes"] / (step_ms / 1e3) / 1e9
        return {"bound": "hbm", "kernel": "whole step (decode_append, lightning_index+topk, "
                                          "sparse_mqa_attn)",
                "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                "traffic_unit": "DRAM bytes per step of the step's kernels (ncu)",
                "algorithmic_bytes": w["step_bytes"], "peak_source": peaks["source"]}

    def path_tflops(self, ms_step):
        return self.work()["attn_flop"] / (ms_step / 1e3) / 1e12

    def cpu_baseline(self, budget_s):
        return None


class CsaPrefill:
    """A 32,768-token CSA prefill: compress -> index + top-k (k=512) ->
    sparse attention, 64 heads."""

    STAGES = ["csa_compress", "lightning_index+topk", "sparse_mqa_attn"]

    def __init__(self, lc, device):
        self.lc = lc
        L = wl.CONFIGS["csa_prefill"](device=device)
        self.L = L
        self.T, self.m, self.k, self.W, self.H, self.d = (L["T"], L["m"], L["k"], L["W"], L["H"],
                                                          L["d"])
        self.chunk = self.T
        self.b = lc.DeviceBatch.from_workload(L["batch"], device=device)
        self.Kc = torch.empty((self.T // self.m, self.d), dtype=torch.bfloat16, device=device)
        self.Vc = torch.empty_like(self.Kc)
        self.ws = torch.empty(lc.workspace_size(lc.LC_OP_LIGHTNING_INDEX, self.b, HI=L["HI"],
                                                dI=L["dI"], k=self.k),
                              dtype=torch.uint8, device=device)
        self.sel = torch.empty((self.T, self.k), dtype=torch.int32, device=device)
        self.O = torch.empty_like(L["Q"])
        self.lse = torch.empty((self.T, self.H), dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

    def work(self):
        L = self.L
        t = np.arange(self.T, dtype=np.int64)
        nv = (t + 1) // self.m
        keys = np.minimum(nv, self.k) + _n_window(t, self.W)
        return {"index_flop": float(2 * L["HI"] * L["dI"] * nv.sum()),
                "attn_flop": float(4 * self.d * self.H * keys.sum()), "keys": int(keys.sum())}

    def stage_extra(self, stage_ms, peaks):
        return gather_bound(self.work()["keys"], self.d, self.T, self.H, self.k,
                            stage_ms[self.STAGES.index("sparse_mqa_attn")], peaks)

    def step(self, events=None):
        lc, L = self.lc, self.L
        ev = events
        if ev:
            ev[0].record()
        lc.csa_compress(L["K"], L["V"], L["G"], m=self.m, Kc=self.Kc, Vc=self.Vc)
        if ev:
            ev[1].record()
        lc.lightning_index(L["qI"], L["w"], L["kI"], self.b, self.m, scores=False, k=self.k,
                           topk=self.sel, ws=self.ws, dev_err=self.err)
        if ev:
            ev[2].record()
        lc.sparse_mqa_attn(L["Q"], self.Kc, self.Vc, self.sel, L["K"], L["V"], self.b, self.m,
                           self.W, L["scale"], O=self.O, lse=self.lse, dev_err=self.err)
        if ev:
            ev[3].record()

    def host_io(self):
        L = self.L
        return ({"Q": L["Q"], "K": L["K"], "V": L["V"], "qI": L["qI"], "kI": L["kI"],
                 "w": L["w"]}, {"O": self.O})

    def config(self, world):
        return {"workload": "csa_prefill: one 32,768-token sequence, every position queried, "
                            "Q [32768,64,128], K,V [32768,128], CSA m=4 (8192 entries), "
                            "indexer 8x64, top-k 512, window 128 (seed 1)",
                "seq_len": self.T, "heads": self.H, "head_dim": self.d,
                "parallelism": f"replicas x{world}",
                "l2": "inputs larger than L2 (Q 512 MiB)"}

    def roofline(self, stage_ms, peaks, region_ms, step_ms):
        w = self.work()
        return tensor_roofline(self.STAGES, stage_ms,
                               {"lightning_index+topk": w["index_flop"],
                                "sparse_mqa_attn": w["attn_flop"]}, peaks, region_ms,
                               "csa_prefill")

    def path_tflops(self, ms_step):
        w = self.work()
        return (w["index_flop"] + w["attn_flop"]) / (ms_step / 1e3) / 1e12

    def cpu_baseline(self, budget_s):
        import oracle
        L = _cpu(self.L)
        Kc = oracle.compress(L["K"], L["G"], self.m)
        Vc = oracle.compress(L["V"], L["G"], self.m)
        Kc = torch.from_numpy(Kc).to(torch.bfloat16).double().numpy()
        Vc = torch.from_numpy(Vc).to(torch.bfloat16).double().numpy()
        kI = L["kI"].double().numpy()

        def run(rows):
            t = rows.astype(np.int64)
            I = oracle.index(L["qI"][rows], L["w"][rows], kI, t, self.m)
            sel = oracle.topk(I, (t + 1) // self.m, self.k)
            oracle.sparse_attn(L["Q"][rows], Kc, Vc, sel, L["K"], L["V"], 0, t, self.W,
                               L["scale"])
        return sampled_rows_baseline(run, self.T, budget_s,
                                     "query rows of the 32,768-token CSA prefill (index over "
                                     "the visible entries, top-k 512, CSA attention, fp64); "
                                     "compressed entries built untimed")


class HcaPrefill:
    """A 131,072-token HCA prefill: compress -> dense attention, 64 heads."""

    STAGES = ["hca_compress", "hca_dense_attn"]

    def __init__(self, lc, device):
        self.lc = lc
        L = wl.CONFIGS["hca_prefill"](device=device)
        self.L = L
        self.T, self.m, self.W, self.H, self.d = L["T"], L["m"], L["W"], L["H"], L["d"]
        self.chunk = self.T
        self.b = lc.DeviceBatch.from_workload(L["batch"], device=device)
        self.Kc = torch.empty((self.T // self.m, self.d), dtype=torch.bfloat16, device=device)
        self.Vc = torch.empty_like(self.Kc)
        self.O = torch.empty_like(L["Q"])
        self.lse = torch.empty((self.T, self.H), dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

    def work(self):
        t = np.arange(self.T, dtype=np.int64)
        keys = (t + 1) // self.m + _n_window(t, self.W)
        return {"attn_flop": float(4 * self.d * self.H * keys.sum())}

    def step(self, events=None):
        lc, L = self.lc, self.L
        ev = events
        if ev:
            ev[0].record()
        lc.hca_compress(L["K"], L["V"], L["G"], m=self.m, Kc=self.Kc, Vc=self.Vc)
        if ev:
            ev[1].record()
        lc.hca_dense_attn(L["Q"], self.Kc, self.Vc, L["K"], L["V"], self.b, self.m, self.W,
                          L["scale"], O=self.O, lse=self.lse, dev_err=self.err)
        if ev:
            ev[2].record()

    def host_io(self):
        L = self.L
        return {"Q": L["Q"], "K": L["K"], "V": L["V"]}, {"O": self.O}

    def config(self, world):
        return {"workload": "hca_prefill: one 131,072-token sequence, every position queried, "
                            "Q [131072,64,128], K,V [131072,128], HCA m'=128 (1024 entries), "
                            "window 128 (seed 2)",
                "seq_len": self.T, "heads": self.H, "head_dim": self.d,
                "parallelism": f"replicas x{world}",
                "l2": "inputs larger than L2 (Q 2 GiB)"}

    def roofline(self, stage_ms, peaks, region_ms, step_ms):
        return tensor_roofline(self.STAGES, stage_ms, {"hca_dense_attn": self.work()["attn_flop"]},
                               peaks, region_ms, "hca_prefill")

    def path_tflops(self, ms_step):
        return self.work()["attn_flop"] / (ms_step / 1e3) / 1e12

    def cpu_baseline(self, budget_s):
        import oracle
        L = _cpu(self.L)
        Kc = torch.from_numpy(oracle.compress(L["K"], L["G"], self.m)).to(torch.bfloat16)
        Vc = torch.from_numpy(oracle.compress(L["V"], L["G"], self.m)).to(torch.bfloat16)
        Kc, Vc = Kc.double().numpy(), Vc.double().numpy()

        def run(rows):
            oracle.hca_attn(L["Q"][rows], Kc, Vc, self.m, L["K"], L["V"], 0,
                            rows.astype(np.int64), self.W, L["scale"])
        return sampled_rows_baseline(run, self.T, budget_s,
                                     "query rows of the 131,072-token HCA prefill (dense "
                                     "attention over the visible entries and the window, "
                                     "fp64); compressed entries built untimed")


WORKLOADS = {"layer_pair_1m": LayerPair, "csa_decode": Decode,
             "csa_decode_incremental": DecodeIncremental, "csa_decode_mxfp4": DecodeMXFP4,
             "csa_decode_mxfp8": DecodeMXFP8, "csa_prefill": CsaPrefill,
             "hca_prefill": HcaPrefill}
SUB_RECORDS = {"csa_decode": "decode", "csa_decode_incremental": "decode_incremental",
               "csa_decode_mxfp4": "decode_mxfp4", "csa_decode_mxfp8": "decode_mxfp8",
               "csa_prefill": "csa_prefill", "hca_prefill": "hca_prefill"}


# ---------------------------------------------------------------- ranks

def max_over_ranks(dist, x: float, device) -> float:
    """The largest x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, ms_per_step: float) -> float:
    """Units all ranks processed per second: every rank runs one replica of
    the step, so the job does world x units_per_rank per (slowest) step."""
    return units_per_rank * world / (ms_per_step / 1e3)


# ---------------------------------------------------------------- our arm

def measure(wk, args, dist, device, peaks, world, rank, cpu_budget):
    """Device-timed region, end-to-end region and CPU baseline of one workload.
    Returns the record (the fields of the JSON line)."""
    lc = wk.lc
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        wk.step()
    torch.cuda.synchronize()

    # ---- the step as a CUDA graph: its C-ABI calls captured once, before the
    # timed region (no kernel runs during capture), so that each timed step is
    # one replay of the same kernels on the same buffers without per-launch
    # host gaps; --eager times the calls themselves
    graph, launch_mode, per_step = None, "eager calls", None
    if not args.eager:
        try:
            l0 = lc.launch_count()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                wk.step()
            per_step = lc.launch_count() - l0
            g.replay()
            torch.cuda.synchronize()
            graph, launch_mode = g, "one CUDA-graph replay per step (the step's calls captured once)"
        except RuntimeError as e:  # capture refused: time the calls
            print(f"graph capture unavailable ({e}); timing eager calls", file=sys.stderr)
            torch.cuda.synchronize()

    # ---- device-timed region
    nst = len(wk.STAGES)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    for _ in range(2):  # the clocks back up after the sampler's start-up wait
        wk.step()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    l0 = lc.launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            wk.step(ev[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = lc.launch_count() - l0 if graph is None else per_step * args.steps
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(dist, t_start.elapsed_time(t_end), device)
    if graph is not None:
        # per-stage times from as many eager steps with events between the stages
        for s in range(args.steps):
            wk.step(ev[s])
        torch.cuda.synchronize()
        del graph
    stage_ms = [statistics.mean(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps))
                for i in range(nst)]
    err = int(wk.err.item())

    # ---- end-to-end region: pinned host inputs -> device -> step -> host
    # outputs, every step.  Pipelined as a serving loop runs it: uploads on one
    # copy stream, downloads on another, device staging double-buffered, so
    # step i+1's upload and step i-1's download overlap step i's kernels.  The
    # step itself takes its inputs from the staging buffer by a device copy
    # and leaves its outputs there the same way.
    ins, outs = wk.host_io()
    h_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v) for k, v in ins.items()}
    h_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = sum(v.numel() * v.element_size() for v in h_out.values())
    e2e_steps = max(4, min(args.steps, 10))
    st_in = [{k: torch.empty_like(v) for k, v in ins.items()} for _ in range(2)]
    st_out = [{k: torch.empty_like(v) for k, v in outs.items()} for _ in range(2)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    uploaded = [torch.cuda.Event() for _ in range(2)]  # st_in[j] holds a step's inputs
    consumed = [torch.cuda.Event() for _ in range(2)]  # the step has copied st_in[j] in
    produced = [torch.cuda.Event() for _ in range(2)]  # st_out[j] holds a step's outputs
    drained = [torch.cuda.Event() for _ in range(2)]   # st_out[j] is on the host

    def upload(i):
        j = i % 2
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(consumed[j])
            for k_, v in h_in.items():
                st_in[j][k_].copy_(v, non_blocking=True)
            uploaded[j].record(up)

    def run(i):
        j = i % 2
        stream.wait_event(uploaded[j])
        for k_, v in ins.items():
            v.copy_(st_in[j][k_], non_blocking=True)
        consumed[j].record(stream)
        wk.step()
        if i >= 2:
            stream.wait_event(drained[j])
        for k_, v in outs.items():
            st_out[j][k_].copy_(v, non_blocking=True)
        produced[j].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(produced[j])
            for k_, v in h_out.items():
                v.copy_(st_out[j][k_], non_blocking=True)
            drained[j].record(down)

    def pipeline(n):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            run(i)
        torch.cuda.synchronize()

    pipeline(2)
    if dist:
        dist.barrier()
    e0 = time.perf_counter()
    pipeline(e2e_steps)
    e2e_s = max_over_ranks(dist, (time.perf_counter() - e0) / e2e_steps, device)
    del h_in, h_out, st_in, st_out

    ms_step = ms / args.steps
    rec = {
        "metric": METRIC, "value": whole_job_rate(wk.chunk, world, ms_step), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": getattr(wk, "DTYPE", "bf16"),
        "data": "synthetic",
        "config": wk.config(world),
        "roofline": wk.roofline(stage_ms, peaks, ms, ms_step),
        "stages_ms": dict(zip(wk.STAGES, stage_ms)),
        "path_tflops": wk.path_tflops(ms_step),
        "e2e": {"value": whole_job_rate(wk.chunk, world, e2e_s * 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "overlap": "uploads and downloads on two copy streams, double-buffered device "
                           "staging: step i+1's upload and step i-1's download run during step "
                           "i"},
        "gpu_launches": int(launches),
        "launch": launch_mode,
        "dev_err": err,
        "clocks": clocks,
    }
    if hasattr(wk, "stage_extra"):
        rec.update(wk.stage_extra(stage_ms, peaks))
    if hasattr(wk, "extra"):
        rec.update(wk.extra())
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = wk.cpu_baseline(cpu_budget)
        if cb is not None:
            rec["cpu_baseline"] = cb
    return rec


def run_ours(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    names = ["layer_pair_1m", "csa_decode", "csa_decode_incremental", "csa_decode_mxfp4",
             "csa_decode_mxfp8", "csa_prefill", "hca_prefill"] \
        if args.workload == "all" else [args.workload]
    recs = {}
    if len(names) > 1 and world == 1:
        # one process per workload: run in one process after the others, the
        # decode steps measured up to 7x slower in places (the random gathers
        # of the CSA attention most), a state of the device that a pause did
        # not clear and a fresh process does not have
        for name in names:
            budget = args.cpu_budget if name == names[0] else args.cpu_budget / 2
            cmd = [sys.executable, os.path.abspath(__file__), "--workload", name,
                   "--steps", str(args.steps), "--warmup", str(args.warmup),
                   "--cpu-budget", str(budget), "--ctx", str(args.ctx)]
            if args.no_cpu_baseline:
                cmd.append("--no-cpu-baseline")
            if args.eager:
                cmd.append("--eager")
            if args.decode_ctx:
                cmd += ["--decode-ctx", args.decode_ctx]
            res = subprocess.run(cmd, stdout=subprocess.PIPE, text=True)
            if res.returncode != 0:
                raise SystemExit(f"bench.py: workload {name} failed ({res.returncode})")
            lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
            recs[name] = json.loads(lines[-1])
        out = recs[names[0]]
        for name in names[1:]:
            out[SUB_RECORDS[name]] = recs[name]
        print(json.dumps(out), flush=True)
        return
    import long_context_compressed_13_b300 as lc
    lc.load_library()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(device))
    peaks = load_peaks()

    for name in names:
        if name == "layer_pair_1m":
            wk = LayerPair(lc, device, ctx=args.ctx)
        else:
            wk = WORKLOADS[name](lc, device)
        budget = args.cpu_budget if name == names[0] else args.cpu_budget / 2
        recs[name] = measure(wk, args, dist, device, peaks, world, rank, budget)
        del wk
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    out = recs[names[0]]
    for name in names[1:]:
        out[SUB_RECORDS[name]] = recs[name]
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------- oracle arm

def _oracle_rows_step(P, rows, q0, ctx, m_c, m_h, k, W, Kc64, Vc64, Kh64, Vh64, Kraw, kI64):
    """Oracle pipeline for a sample of query rows of the layer pair: index,
    top-k, CSA attention, HCA attention (compressed caches precomputed)."""
    import oracle
    c, h = P["csa"], P["hca"]
    t = np.array([q0 + r for r in rows], dtype=np.int64)
    I = oracle.index(c["qI"][rows], c["w"][rows], kI64, t, m_c)
    sel = oracle.topk(I, (t + 1) // m_c, k)
    oracle.sparse_attn(c["Q"][rows], Kc64, Vc64, sel, Kraw["csa_K"], Kraw["csa_V"],
                       Kraw["pos0"], t, W, c["scale"])
    oracle.hca_attn(h["Q"][rows], Kh64, Vh64, m_h, Kraw["hca_K"], Kraw["hca_V"], Kraw["pos0"], t,
                    W, h["scale"])


def _oracle_state(P, q0, ctx, m_c, m_h, W):
    """fp64 host copies the oracle needs: compressed caches (the oracle's own
    compression of the raw prefix and chunk) and the raw window region."""
    import oracle
    c, h = P["csa"], P["hca"]
    out = {}
    for name, L, m in (("c", c, m_c), ("h", h, m_h)):
        Ks, Vs = [], []
        step = 1 << 16
        for s in range(0, ctx, step):
            Ks.append(oracle.compress(L["K"][s:s + step].cpu(), L["G"].cpu(), m))
            Vs.append(oracle.compress(L["V"][s:s + step].cpu(), L["G"].cpu(), m))
        out["K" + name] = np.concatenate(Ks)
        out["V" + name] = np.concatenate(Vs)
    lo = q0 - W
    raw = {"pos0": lo, "csa_K": c["K"][lo:].cpu().double().numpy(),
           "csa_V": c["V"][lo:].cpu().double().numpy(),
           "hca_K": h["K"][lo:].cpu().double().numpy(),
           "hca_V": h["V"][lo:].cpu().double().numpy()}
    kI64 = c["kI"].cpu().double().numpy()
    return out, raw, kI64


def sampled_rows_baseline(run, n_rows, budget_s, what):
    """Times run(rows) on a seeded sample of query rows sized to about
    budget_s seconds (calibrated on a small first sample)."""
    import oracle
    nt = oracle.num_threads()
    rng = np.random.default_rng(0)
    perm = rng.permutation(n_rows)
    cal = np.sort(perm[:nt])
    t0 = time.perf_counter()
    run(cal)
    one = max((time.perf_counter() - t0) / len(cal), 1e-6)
    n = int(min(n_rows, max(nt, budget_s / one)))
    rows = np.sort(perm[:n])
    t0 = time.perf_counter()
    run(rows)
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": nt, "kind": "oracle",
            "sample": f"{n} of the {n_rows} {what}", "seconds": dt}


def layer_pair_cpu_baseline(wk, budget_s=20.0):
    P = wk.P
    Pc = {"csa": _cpu(P["csa"]), "hca": _cpu(P["hca"])}
    st, raw, kI64 = _oracle_state(Pc, wk.q0, wk.ctx, wk.m_c, wk.m_h, wk.W)

    def run(rows):
        _oracle_rows_step(Pc, rows, wk.q0, wk.ctx, wk.m_c, wk.m_h, wk.k, wk.W, st["Kc"],
                          st["Vc"], st["Kh"], st["Vh"], raw, kI64)
    return sampled_rows_baseline(run, wk.chunk, budget_s,
                                 "query rows of the layer pair (index over all 262144 entries, "
                                 "top-k 1024, CSA and HCA attention, fp64); compressed caches "
                                 "built untimed")


def decode_cpu_baseline(wk, budget_s=20.0, fmt=None):
    """The oracle on whole sequences of the decode batch (index over every
    visible entry, top-k, CSA attention), as many as fit the time budget;
    with fmt, the indexer runs on MX-quantized q_I and k_I."""
    import oracle
    D = wk.D
    B = D["B"]
    cu_c, cu_raw = D["batch"].cu_c, D["batch"].cu_raw
    host = {k: D[k].cpu() for k in ("Q", "Kc", "Vc", "Kraw", "Vraw", "qI", "kI", "w")}
    done, t_used = 0, 0.0
    for b in range(B):
        c0, c1, r0, r1 = cu_c[b], cu_c[b + 1], cu_raw[b], cu_raw[b + 1]
        t = np.array([D["ctx"][b] - 1], dtype=np.int64)
        kI = host["kI"][c0:c1].double().numpy()
        Kc = host["Kc"][c0:c1].double().numpy()
        Vc = host["Vc"][c0:c1].double().numpy()
        t0 = time.perf_counter()
        if fmt is None:
            I = oracle.index(host["qI"][b:b + 1], host["w"][b:b + 1], kI, t, wk.m)
        else:
            I = oracle.index_mx(host["qI"][b:b + 1], host["w"][b:b + 1], kI, t, wk.m, fmt)
        sel = oracle.topk(I, (t + 1) // wk.m, wk.k)
        oracle.sparse_attn(host["Q"][b:b + 1], Kc, Vc, sel, host["Kraw"][r0:r1],
                           host["Vraw"][r0:r1], D["batch"].raw_pos0[b], t, wk.W, D["scale"])
        t_used += time.perf_counter() - t0
        done += 1
        if t_used > budget_s:
            break
    return {"value": done / t_used, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{done} of the 64 decode sequences (whole sequences: index over every "
                      f"visible entry" + (f" on MXFP{fmt} q/k" if fmt else "") +
                      ", top-k 1024, CSA attention, fp64)", "seconds": t_used}


def run_reference(args):
    """The CPU oracle on the layer-pair workload: each step runs the whole
    path (index, top-k, CSA and HCA attention) for a seeded sample of the
    chunk's query rows; ms_per_step is the measured time of that sample."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    P = wl.layer_pair(seed=4, device="cpu")
    q0, ctx, chunk = P["ctx"] - P["chunk"], P["ctx"], P["chunk"]
    c, h = P["csa"], P["hca"]
    st, raw, kI64 = _oracle_state(P, q0, ctx, c["m"], h["m"], c["W"])
    rng = np.random.default_rng(1)
    n = max(oracle.num_threads(), 8)
    times = []
    for s in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(chunk, n, replace=False))
        t0 = time.perf_counter()
        _oracle_rows_step(P, rows, q0, ctx, c["m"], h["m"], c["k"], c["W"], st["Kc"], st["Vc"],
                          st["Kh"], st["Vh"], raw, kI64)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    step_s = sum(times) / len(times)
    value = n / step_s
    sample = (f"{n} seeded query rows per step of the {chunk}-row chunk (the whole path for "
              f"each row, fp64); ms_per_step is the measured time of those rows")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": layer_pair_config(ctx, chunk, c["H"], c["d"], world),
           "sample": sample,
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="time the step's calls as launched, not a CUDA-graph replay of them")
    # a shorter context keeps the same kernels on a smaller case (profiler
    # captures); the measured workload is the default 1,048,576 tokens
    ap.add_argument("--ctx", type=int, default=1 << 20)
    ap.add_argument("--decode-ctx", default=None,
                    help="LO,HI: decode contexts ~U[LO, HI] (profiler captures)")
    ap.add_argument("--workload", default="all", choices=["all", *WORKLOADS])
    args = ap.parse_args()
    if args.decode_ctx:
        global DECODE_CTX
        DECODE_CTX = tuple(int(x) for x in args.decode_ctx.split(","))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
