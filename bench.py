#!/usr/bin/env python3
"""Benchmark of the 4-bit groupwise-affine MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill4096|prefill512|canvas|tiny|decode3b|decode2b|
                                prefill512b3|prefill512b2|sweep] [--no-secondary]

Prints ONE JSON line.  Headline workload: batch-1 decode through 40 distinct
chained MoE layers (T=1, d=2048, E=256, top-8 + shared expert, I=512); a step
is the 40-layer pass, captured in a CUDA graph.  The line also carries the
T=4096 long prefill (four chunks of 1024 tokens, Zipf-skewed routing) measured
the same way.  `value` is tokens per second through one MoE layer: layer
invocations x tokens / time.  The low-bit workloads (decode3b, decode2b,
prefill512b3, prefill512b2) are the same layers with 3- and 2-bit expert codes;
`--workload sweep` prints the rows-per-expert and canvas-batching tables.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the layer has no exchange step on one node); value sums the ranks' tokens
over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from bit_moe_expert_gb300 import synth  # noqa: E402

TILE_ROWS = 128  # rows per tensor-core tile (moe_route block_rows) on the prefill path

METRIC = "MoE layer tokens/s at T=1 decode (40 distinct chained layers); T=4096 prefill reported alongside"


# ----------------------------------------------------------------------------- distributed plumbing

class Dist:
    def __init__(self):
        import torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend)
            self.dist = dist

    def barrier(self):
        import torch
        if torch.cuda.is_available():
            torch.cuda.synchronize()
        if self.dist is not None:
            self.dist.barrier()
        if torch.cuda.is_available():
            torch.cuda.synchronize()

    def reduce(self, x: float, op: str) -> float:
        if self.dist is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX if op == "max" else self.dist.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


# ----------------------------------------------------------------------------- clocks (NVML via ctypes)

class ClockSampler:
    """Samples SM clock, max clock, power and throttle reasons every few ms while
    active.  Uses the driver's NVML library directly; falls back to nvidia-smi."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle",
               0x2: "applications_clocks_setting", 0x100: "display_clock_setting"}

    def __init__(self, gpu_index: int, period_s: float = 0.005):
        self.period = period_s
        self.samples = []
        self.nvml = None
        self.handle = None
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(h)) == 0:
                    self.nvml, self.handle = nv, h
                    m = ctypes.c_uint()
                    if nv.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(m)) == 0:  # 1 = SM
                        self.max_mhz = m.value
        except OSError:
            self.nvml = None

    def _sample(self):
        nv, h = self.nvml, self.handle
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        nv.nvmlDeviceGetClockInfo(h, ctypes.c_int(1), ctypes.byref(clk))
        nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
        nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs))
        self.samples.append((clk.value, pw.value / 1000.0, rs.value))

    def _loop(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def start(self):
        self.samples = []
        self._stop.clear()
        if self.nvml is not None:
            self._sample()
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()

    def stop(self) -> dict:
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            self._sample()
        return self.summary()

    def summary(self) -> dict:
        if not self.samples:
            return self._smi_snapshot()
        mhz = [s[0] for s in self.samples]
        reasons = 0
        for s in self.samples:
            reasons |= s[2]
        names = sorted({n for bit, n in self.REASONS.items() if reasons & bit})
        return {"sm_mhz": statistics.median(mhz), "sm_min_mhz": min(mhz), "sm_max_mhz": self.max_mhz,
                "power_w_max": max(s[1] for s in self.samples), "reasons": names,
                "samples": len(self.samples), "source": "nvml"}

    def _smi_snapshot(self) -> dict:
        import subprocess
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            out = subprocess.run(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits"],
                                 capture_output=True, text=True, timeout=20).stdout.strip().splitlines()[0]
            f = [x.strip() for x in out.split(",")]
            names = [n for n, v in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                        "sw_power_cap"], f[3:]) if v.lower() == "active"]
            return {"sm_mhz": float(f[0]), "sm_max_mhz": float(f[1]), "reasons": names, "samples": 1,
                    "source": "nvidia-smi after the timed region"}
        except Exception as e:  # pragma: no cover - diagnostic only
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": f"unavailable: {e}"}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- workloads

class Workload:
    """One benchmark workload on one GPU (our arm)."""
    name = ""
    tokens_per_step = 0        # token-layer invocations per step
    dtype = ""

    def step(self):
        raise NotImplementedError

    def e2e_step(self):
        raise NotImplementedError


def _dev_layer(cfg, layer, dev, with_shared=True):
    import bit_moe_expert_gb300 as bm
    rex = synth.draw_experts_torch(cfg, layer, dev)
    sex = synth.draw_experts_torch(cfg, layer, dev, E=1, I=cfg.I_shared, tag=20) if (cfg.I_shared and with_shared) \
        else None
    routed = bm.prepare_experts(rex, dev)
    shared = bm.prepare_experts(sex, dev) if sex is not None else None
    return rex, sex, routed, shared


class DecodeWorkload(Workload):
    dtype = "f32"
    api_desc = "moe_layer"

    def __init__(self, dev, layers=None, name="decode"):
        import torch
        import bit_moe_expert_gb300 as bm
        self.bm = bm
        self.name = name
        self.cfg = cfg = synth.CONFIGS[name]
        self.L = layers or cfg.layers
        self.T = cfg.T
        self.dev = dev
        self.raw, self.routed, self.shared, self.X, self.logits = [], [], [], [], []
        self.X_host, self.logits_host = [], []
        for l in range(self.L):
            rex, sex, routed, shared = _dev_layer(cfg, l, dev)
            self.raw.append((rex, sex))
            self.routed.append(routed)
            self.shared.append(shared)
            xh = synth.draw_x(cfg, self.T, l)
            lh = synth.draw_logits(cfg, self.T, l)
            self.X_host.append(xh)
            self.logits_host.append(lh)
            self.X.append(torch.from_numpy(xh.view(np.int16)).to(dev))
            self.logits.append(torch.from_numpy(lh).to(dev))
        self.block_rows = TILE_ROWS
        self.r = bm.Routing.empty(self.T, cfg.E, cfg.k, self.block_rows, dev)
        self.ws = bm.workspace(bm.moe_layer_workspace_bytes(self.T, cfg.d, cfg.I, cfg.E, cfg.k, cfg.I_shared), dev)
        self.Y = torch.empty((self.L, self.T, cfg.d), dtype=torch.int16, device=dev)
        self.tokens_per_step = self.L * self.T
        # pinned host buffers for the end-to-end measurement: the step's inputs (every layer's X and
        # logits) and its result (every layer's Y), each moved in one copy per step
        self.X_pin = torch.from_numpy(np.stack([x.view(np.int16) for x in self.X_host])).pin_memory()
        self.lg_pin = torch.from_numpy(np.stack(self.logits_host)).pin_memory()
        self.Y_pin = torch.empty((self.L, self.T, cfg.d), dtype=torch.int16).pin_memory()
        self.X_e2e = torch.empty(self.X_pin.shape, dtype=torch.int16, device=dev)
        self.lg_e2e = torch.empty(self.lg_pin.shape, dtype=torch.float32, device=dev)
        self.X_e2e_l = [self.X_e2e[l] for l in range(self.L)]
        self.lg_e2e_l = [self.lg_e2e[l] for l in range(self.L)]
        self.Y_l = [self.Y[l] for l in range(self.L)]
        self.h2d_bytes = self.L * (self.X_host[0].nbytes + self.logits_host[0].nbytes)
        self.d2h_bytes = self.L * self.T * cfg.d * 2

    def launches_per_step(self):
        return self.L  # moe_layer at T=1: one decode kernel that also routes

    def step(self):
        bm, cfg = self.bm, self.cfg
        for l in range(self.L):
            bm.moe_layer(self.logits[l], self.X[l], self.routed[l], self.shared[l], cfg.k, self.block_rows, self.r,
                         self.Y_l[l], self.ws)

    def e2e_step(self):
        bm, cfg = self.bm, self.cfg
        self.X_e2e.copy_(self.X_pin, non_blocking=True)
        self.lg_e2e.copy_(self.lg_pin, non_blocking=True)
        for l in range(self.L):
            bm.moe_layer(self.lg_e2e_l[l], self.X_e2e_l[l], self.routed[l], self.shared[l], cfg.k, self.block_rows,
                         self.r, self.Y_l[l], self.ws)
        self.Y_pin.copy_(self.Y, non_blocking=True)

    # algorithmic work
    def bytes_per_step(self):
        cfg = self.cfg
        return self.L * (cfg.k * synth.ffn_bytes(cfg.d, cfg.I, cfg.bits) + synth.ffn_bytes(cfg.d, cfg.I_shared, cfg.bits))

    def dominant(self, peaks):
        cfg = self.cfg
        per_launch = cfg.k * synth.ffn_bytes(cfg.d, cfg.I, cfg.bits) + synth.ffn_bytes(cfg.d, cfg.I_shared, cfg.bits)
        return "decode", "hbm", per_launch, (
            f"({cfg.k} routed + 1 shared) experts x (gate+up+down) {cfg.bits}-bit codes and bf16 scale/bias "
            f"= {per_launch} B per launch")

    def workload_desc(self):
        c = self.cfg
        return (f"{self.name}: T={c.T}, d={c.d}, E={c.E}, top-{c.k} + shared expert, I={c.I}; {self.L} distinct "
                f"chained layers per step (CUDA graph); {c.bits}-bit codes + bf16 scale/bias per 64")

    def cpu_sample(self, budget_s):
        """Oracle (routing + layer) on the host for the first layers until the budget is spent."""
        import oracle
        done, t_used = 0, 0.0
        while t_used < budget_s and done < self.L:
            routed, shared, ids, w = self._host_subset(done)
            t0 = time.perf_counter()
            r = oracle.route(self.logits_host[done], self.cfg.k, self.block_rows)
            oracle.forward(self.X_host[done], routed, shared, self._remap(r["ids"], ids), r["w"])
            t_used += time.perf_counter() - t0
            done += 1
        return done * self.T, t_used, f"{done} decode layer(s) of 1 token (routing + layer), single-threaded oracle"

    def _host_subset(self, l):
        """Host copies of the experts layer l's token selects (the oracle reads only those)."""
        import oracle
        r = oracle.route(self.logits_host[l], self.cfg.k, self.block_rows)
        sel = sorted(set(int(e) for e in r["ids"].reshape(-1)))
        rex, sex = self.raw[l]
        idx = __import__("torch").tensor(sel, device=self.dev)

        def host(ex, index=None):
            out = {}
            for m, (q, s, b) in ex.items():
                if index is not None:
                    q, s, b = q.index_select(0, index), s.index_select(0, index), b.index_select(0, index)
                out[m] = (q.cpu().numpy().view(np.uint32), s.cpu().numpy().view(np.uint16),
                          b.cpu().numpy().view(np.uint16))
            return out
        return host(rex, idx), host(sex) if sex is not None else None, sel, r["w"]

    @staticmethod
    def _remap(ids, sel):
        lut = {e: i for i, e in enumerate(sel)}
        return np.vectorize(lambda e: lut[int(e)])(ids).astype(np.int32)


class PrefillWorkload(Workload):
    """Chunked prefill: T tokens as chunks, each chunk through a different weight set."""
    dtype = "f16 MMA, f32 accumulate"
    api_desc = "moe_route + moe_forward"

    def __init__(self, dev, name="prefill4096", sets=None):
        import torch
        import bit_moe_expert_gb300 as bm
        self.bm = bm
        self.name = name
        self.cfg = cfg = synth.CONFIGS[name]
        self.dev = dev
        self.chunk = cfg.tokens_per_call
        self.nchunks = cfg.T // self.chunk
        self.sets = sets or max(self.nchunks, 4)
        self.raw, self.routed, self.shared = [], [], []
        for l in range(self.sets):
            rex, sex, routed, shared = _dev_layer(cfg, l, dev)
            self.raw.append((rex, sex))
            self.routed.append(routed)
            self.shared.append(shared)
        # one prompt: X and logits for all T tokens (logits per weight set, as a real layer would produce)
        self.X_host = synth.draw_x(cfg, cfg.T, 0)
        self.logits_host = [synth.draw_logits(cfg, cfg.T, l) for l in range(self.sets)]
        self.X = torch.from_numpy(self.X_host.view(np.int16)).to(dev)
        self.logits = [torch.from_numpy(x).to(dev) for x in self.logits_host]
        self.block_rows = TILE_ROWS
        C = self.chunk
        self.r = bm.Routing.empty(C, cfg.E, cfg.k, self.block_rows, dev)
        self.ws_r = bm.workspace(bm.moe_route_workspace_bytes(C, cfg.E, cfg.k), dev)
        self.ws_f = bm.workspace(bm.moe_forward_workspace_bytes(C, cfg.d, cfg.I, cfg.E, cfg.k, cfg.I_shared), dev)
        self.Y = torch.empty((cfg.T, cfg.d), dtype=torch.int16, device=dev)
        self.tokens_per_step = cfg.T
        # pinned host buffers for the end-to-end measurement: the prompt's X and each chunk's logits (from
        # the chunk's weight set) in one copy each per step, Y in one copy
        self.X_pin = torch.from_numpy(self.X_host.view(np.int16)).pin_memory()
        self.lg_pin = torch.from_numpy(np.concatenate(
            [self.logits_host[self._set(c)][c * C:(c + 1) * C] for c in range(self.nchunks)])).pin_memory()
        self.Y_pin = torch.empty((cfg.T, cfg.d), dtype=torch.int16).pin_memory()
        self.X_e2e = torch.empty((cfg.T, cfg.d), dtype=torch.int16, device=dev)
        self.lg_e2e = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device=dev)
        # copies run on their own stream, overlapped with the chunks' kernels: chunk c's inputs land
        # while earlier chunks compute, and its Y leaves while later chunks compute
        self.copy_stream = torch.cuda.Stream(device=dev)
        self.ev_step = torch.cuda.Event()
        self.ev_lg = [torch.cuda.Event() for _ in range(self.nchunks)]  # chunk c's logits landed (routing may start)
        self.ev_in = [torch.cuda.Event() for _ in range(self.nchunks)]  # and its X
        self.ev_out = [torch.cuda.Event() for _ in range(self.nchunks)]
        self.ev_done = torch.cuda.Event()
        self.h2d_bytes = self.X_host.nbytes + self.nchunks * C * cfg.E * 4
        self.d2h_bytes = cfg.T * cfg.d * 2
        self._flops = None

    def launches_per_step(self):
        return self.nchunks * 5  # route, X->fp16, gate/up GEMM, down GEMM, combine

    def _set(self, c):
        return c % self.sets

    def step(self):
        bm, cfg, C = self.bm, self.cfg, self.chunk
        for c in range(self.nchunks):
            s = self._set(c)
            bm.moe_route(self.logits[s][c * C:(c + 1) * C], cfg.k, self.block_rows, self.r, self.ws_r)
            bm.moe_forward(self.X[c * C:(c + 1) * C], self.routed[s], self.shared[s], self.r,
                           self.Y[c * C:(c + 1) * C], self.ws_f)

    def e2e_step(self):
        import torch
        bm, cfg, C = self.bm, self.cfg, self.chunk
        main, cs = torch.cuda.current_stream(), self.copy_stream
        self.ev_step.record(main)  # the previous step's kernels are done with the input buffers
        cs.wait_event(self.ev_step)
        with torch.cuda.stream(cs):
            for c in range(self.nchunks):
                rows = slice(c * C, (c + 1) * C)
                self.lg_e2e[rows].copy_(self.lg_pin[rows], non_blocking=True)
                self.ev_lg[c].record(cs)
                self.X_e2e[rows].copy_(self.X_pin[rows], non_blocking=True)
                self.ev_in[c].record(cs)
        for c in range(self.nchunks):
            s, rows = self._set(c), slice(c * C, (c + 1) * C)
            # the first chunk's routing starts once its logits have landed, its expert kernels once its X
            # has; the later chunks' inputs land while the first computes, so one wait after it covers them
            # and leaves their kernels chained
            if c == 0:
                main.wait_event(self.ev_lg[0])
            bm.moe_route(self.lg_e2e[rows], cfg.k, self.block_rows, self.r, self.ws_r)
            if c == 0:
                main.wait_event(self.ev_in[0])
            bm.moe_forward(self.X_e2e[rows], self.routed[s], self.shared[s], self.r, self.Y[rows], self.ws_f)
            if c == 0 and self.nchunks > 1:
                main.wait_event(self.ev_in[self.nchunks - 1])
            self.ev_out[c].record(main)
            cs.wait_event(self.ev_out[c])
            with torch.cuda.stream(cs):
                self.Y_pin[rows].copy_(self.Y[rows], non_blocking=True)
        self.ev_done.record(cs)
        main.wait_event(self.ev_done)  # the step ends when its last Y has reached the host buffer

    def flops_per_step(self):
        cfg = self.cfg
        per_tok_expert = 6 * cfg.d * cfg.I
        shared = 6 * cfg.d * cfg.I_shared
        return cfg.T * (cfg.k * per_tok_expert + shared)

    def active_experts(self):
        """Experts that chunk 0 routes to (every chunk of a workload has the same statistics)."""
        cfg, C = self.cfg, self.chunk
        self.bm.moe_route(self.logits[0][0:C], cfg.k, self.block_rows, self.r, self.ws_r)
        return int((self.r.counts.cpu().numpy() > 0).sum())

    def dominant(self, peaks):
        """The gate/up GEMM, against the tensor-core peak when its arithmetic intensity (FLOPs per streamed
        weight byte) is above the ridge point of the measured peaks, else against HBM on the weight bytes."""
        cfg = self.cfg
        flops = self.chunk * (cfg.k * 4 * cfg.d * cfg.I + 4 * cfg.d * cfg.I_shared)
        n_act = self.active_experts()
        # gate and up are two of the three equally sized matrices of an expert
        nbytes = (2 * n_act * synth.ffn_bytes(cfg.d, cfg.I, cfg.bits)
                  + 2 * synth.ffn_bytes(cfg.d, cfg.I_shared, cfg.bits)) // 3
        ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        if flops / nbytes > ridge:
            return "gemm_gateup", "tensor", flops, (
                f"{self.chunk} tokens x ({cfg.k} routed + shared) x 2 matrices x 2*{cfg.d}*{cfg.I} FLOP "
                f"= {flops / 1e9:.2f} GFLOP per launch ({flops / nbytes:.0f} FLOP per weight byte, "
                f"ridge {ridge:.0f})")
        return "gemm_gateup", "hbm", nbytes, (
            f"gate and up matrices of the {n_act} active experts{' + shared' if cfg.I_shared else ''} "
            f"({cfg.bits}-bit codes, bf16 scale/bias) = {nbytes} B per launch ({flops / nbytes:.0f} FLOP per weight byte, "
            f"ridge {ridge:.0f})")

    def workload_desc(self):
        c = self.cfg
        return (f"{self.name}: T={c.T} as {self.nchunks} chunk(s) of {self.chunk}, d={c.d}, E={c.E}, top-{c.k}"
                f"{' + shared' if c.I_shared else ''}, I={c.I}{', Zipf-skewed routing' if c.zipf else ''}; "
                f"chunk c uses weight set c ({self.sets} sets x "
                f"{(c.E * synth.ffn_bytes(c.d, c.I, c.bits)) / 1e6:.0f} MB, {c.bits}-bit codes)")

    def cpu_sample(self, budget_s):
        import oracle
        cfg, C = self.cfg, self.chunk
        lg = self.logits_host[0][:C]
        r = oracle.route(lg, cfg.k, self.block_rows)
        rex, sex = self.raw[0]
        routed = {m: (q.cpu().numpy().view(np.uint32), s.cpu().numpy().view(np.uint16), b.cpu().numpy().view(np.uint16))
                  for m, (q, s, b) in rex.items()}
        shared = ({m: (q.cpu().numpy().view(np.uint32), s.cpu().numpy().view(np.uint16),
                       b.cpu().numpy().view(np.uint16)) for m, (q, s, b) in sex.items()} if sex else None)
        X = self.X_host[:C]
        done, t_used = 0, 0.0
        while t_used < budget_s and done < C:
            t0 = time.perf_counter()
            oracle.forward(X, routed, shared, r["ids"], r["w"], done, done + 1)
            t_used += time.perf_counter() - t0
            done += 1
        return done, t_used, f"{done} token(s) of chunk 0 through the layer, single-threaded oracle"


# ----------------------------------------------------------------------------- timing

def time_graph(wl, steps, warmup, dist, clocks=None):
    import torch
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            wl.step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        wl.step()
    torch.cuda.synchronize()
    for _ in range(max(warmup, 3)):
        g.replay()
    dist.barrier()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    if clocks:
        clocks.start()
    start.record()
    for _ in range(steps):
        g.replay()
    stop.record()
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    dist.barrier()
    ms = start.elapsed_time(stop)
    return ms, clk


def time_e2e(wl, steps, warmup, dist):
    import torch
    for _ in range(max(warmup, 3)):
        wl.e2e_step()
    dist.barrier()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        wl.e2e_step()
    stop.record()
    torch.cuda.synchronize()
    dist.barrier()
    return start.elapsed_time(stop)


def time_kernels(wl, steps):
    """Per-kernel device time: the library brackets each launch with events on
    its own stream (a separate pass; events between kernels remove overlap)."""
    import torch
    bm = wl.bm
    bm.moe_profile_reset()
    bm.moe_profile_enable(True)
    try:
        for _ in range(steps):
            wl.step()
        torch.cuda.synchronize()
        return bm.moe_profile_read()
    finally:
        bm.moe_profile_enable(False)
        bm.moe_profile_reset()


def run_workload(wl, args, dist, peaks, clocks):
    ms, clk = time_graph(wl, args.steps, args.warmup, dist, clocks)
    ms = dist.reduce(ms, "max")
    tok = dist.reduce(float(wl.tokens_per_step * args.steps), "sum")
    value = tok / (ms / 1e3)
    ms_e2e = dist.reduce(time_e2e(wl, args.steps, args.warmup, dist), "max")
    e2e = {"value": tok / (ms_e2e / 1e3), "unit": "tok/s", "h2d_bytes_per_step": wl.h2d_bytes,
           "d2h_bytes_per_step": wl.d2h_bytes, "ms_per_step": ms_e2e / args.steps,
           "note": f"public API per call ({wl.api_desc}); every step copies its inputs from pinned host memory "
                   "(one copy per input tensor) and its Y back (one copy), no CUDA graph"}
    kt = time_kernels(wl, min(args.steps, 200))
    kname, bound, work, work_desc = wl.dominant(peaks)
    kms, kn = kt[kname]
    avg_s = (kms / max(kn, 1)) / 1e3
    avg_method = "separate pass with events around every launch (no overlap between kernels)"
    if isinstance(wl, DecodeWorkload):
        # the decode kernel is the only kernel of the step: its average launch
        # duration is the timed region over its launches
        avg_s = (ms / args.steps) / wl.L / 1e3
        avg_method = "timed region (CUDA graph of the chained layers) / launches; the only kernel of the step"
    if bound == "hbm":
        achieved = work / avg_s / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    else:
        achieved = work / avg_s / 1e12
        peak = peaks["bf16_tflops"]  # fp16 dense rate = bf16 dense rate (nominal ratio 1)
        unit = "TFLOP/s"
    total_k = sum(v[0] for v in kt.values())
    shares = {k: {"launches": v[1], "avg_us": (v[0] / max(v[1], 1)) * 1e3,
                  "share": (v[0] / total_k if total_k else 0.0)} for k, v in kt.items() if v[1]}
    roof = {"bound": bound, "kernel": kname, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": profiled_traffic(wl.name, kname), "traffic_unit": "B per launch",
            "algorithmic_work_per_launch": work_desc,
            "avg_launch_us": avg_s * 1e6, "avg_launch_method": avg_method, "peak_source": peaks["source"] + (
                " copy bandwidth" if bound == "hbm" else " cuBLAS bf16 GEMM (burst); fp16 MMA has the same rate")}
    out = {"value": value, "ms_per_step": ms / args.steps, "e2e": e2e, "roofline": roof, "kernels": shares,
           "clocks": clk, "dtype": wl.dtype}
    if isinstance(wl, DecodeWorkload):
        t_layer = (ms / args.steps) / wl.L / 1e3
        gbs = wl.bytes_per_step() / wl.L / t_layer / 1e9
        out["layer_roofline"] = {"bound": "hbm", "active_bytes_per_layer": wl.bytes_per_step() // wl.L,
                                 "us_per_layer": t_layer * 1e6, "achieved": gbs, "peak": peaks["hbm_gbs"],
                                 "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                                 "note": "whole layer (moe_layer: routing and both projections in one launch) inside the 40-layer graph"}
    else:
        t_step = (ms / args.steps) / 1e3
        fl = wl.flops_per_step() / t_step / 1e12
        out["step_roofline"] = {"bound": "tensor", "flops_per_step": wl.flops_per_step(), "achieved": fl,
                                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": fl / peaks["bf16_tflops"],
                                "note": "whole step (routing, conversion, both GEMMs, combine), algorithmic FLOPs"}
        if bound == "hbm":
            cfg = wl.cfg
            n_act = wl.active_experts()
            wbytes = wl.nchunks * (n_act * synth.ffn_bytes(cfg.d, cfg.I, cfg.bits)
                                   + synth.ffn_bytes(cfg.d, cfg.I_shared, cfg.bits))
            gbs = wbytes / t_step / 1e9
            out["step_roofline"] = {"bound": "hbm", "weight_bytes_per_step": wbytes, "achieved": gbs,
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                                    "flops_per_step": wl.flops_per_step(), "tflops": fl,
                                    "note": f"whole step; the {n_act} active experts' three matrices"
                                            f"{' and the shared expert' if cfg.I_shared else ''} streamed once per chunk"}
    return out


# DRAM bytes (read + write) per launch of each dominant kernel, from the ncu
# captures summarised under profiles/, with a hash of the sources the kernel is
# built from at the time of the capture.  A kernel whose sources changed since
# reports null.
_CSRC = os.path.join(ROOT, "bit_moe_expert_gb300", "csrc")
PROFILED_TRAFFIC = {
    # ncu dram__bytes of the first two gate/up launches of the long-prefill chunks (chunks 0 and 1, eager warm-up
    # step): 86,159,360 + 2,473,984 and 88,521,984 + 116,736 B; the mean.  Cold-cache (ncu flushes the caches
    # before each launch): the gathered X, 37.7 MB, comes back from DRAM there; in the timed step it is in L2
    "prefill4096/gemm_gateup": (88_636_032, ("gemm.cu", "ptx.cuh", "kernels.h", "status.h"), "b332703e66d1bfeb"),
    # ncu dram__bytes of five decode launches inside the 40-layer step: median 16,034,048 B read, 0 written (the
    # hash is of the sources after a change to the file's header comment alone, the kernel code as captured)
    "decode/decode": (16_034_048, ("decode.cu", "topk.cuh", "ptx.cuh", "kernels.h", "status.h"), "b71ce80da2e12c36"),
}


def profiled_traffic(workload, kname):
    ent = PROFILED_TRAFFIC.get(f"{workload}/{kname}")
    if ent is None:
        return None
    nbytes, files, sha = ent
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(_CSRC, f), "rb") as fh:
            h.update(fh.read())
    return float(nbytes) if h.hexdigest()[:16] == sha else None


def router_measure(dev, peaks):
    """The router projection (moe_router_logits) at one decode token and at one 1024-token prefill chunk:
    200 calls on 200 distinct 1 MB routers (beyond L2) in a CUDA graph, timed with events."""
    import torch
    import bit_moe_expert_gb300 as bm
    cfg = synth.CONFIGS["decode"]
    nw = 200
    W = torch.empty((nw, cfg.E, cfg.d), dtype=torch.int16, device=dev)
    for i in range(0, nw, 50):  # seeded synthetic routers, N(0, 1/d)
        W[i] = torch.from_numpy(synth.draw_router(cfg, i).view(np.int16)).to(dev)
    for i in range(nw):
        if i % 50:
            W[i] = W[i - i % 50]
    out = {}
    s = torch.cuda.Stream(device=dev)
    # (tokens, key, MOE_ROUTER_TC): the default kernels, and at 1024 tokens the
    # warp-MMA kernel the tensor-core one replaces
    for T, key, tc in ((1, "T1", None), (1024, "T1024", None), (4096, "T4096", None),
                       (1024, "T1024_warp_mma", "0")):
        X = torch.from_numpy(synth.draw_x(cfg, T, 0).view(np.int16)).to(dev)
        lg = torch.empty((T, cfg.E), dtype=torch.float32, device=dev)
        old_tc = os.environ.get("MOE_ROUTER_TC")
        if tc is not None:
            os.environ["MOE_ROUTER_TC"] = tc
        with torch.cuda.stream(s):
            for i in range(3):
                bm.moe_router_logits(X, W[i], lg)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(nw):
                    bm.moe_router_logits(X, W[i], lg)
            g.replay()
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            e1.synchronize()
        if tc is not None:
            if old_tc is None:
                del os.environ["MOE_ROUTER_TC"]
            else:
                os.environ["MOE_ROUTER_TC"] = old_tc
        us = e0.elapsed_time(e1) / nw * 1e3
        nbytes = cfg.E * cfg.d * 2 + T * cfg.d * 2 + T * cfg.E * 4
        flops = 2 * T * cfg.E * cfg.d
        ent = {"us_per_call": us, "bytes": nbytes, "gbs": nbytes / us / 1e3, "tflops": flops / us / 1e6}
        if T == 1:
            ent.update(bound="hbm", frac=ent["gbs"] / peaks["hbm_gbs"], peak=peaks["hbm_gbs"], unit="GB/s")
        else:
            ent.update(bound="tensor", frac=ent["tflops"] / peaks["bf16_tflops"], peak=peaks["bf16_tflops"],
                       unit="TFLOP/s")
        ent["kernel"] = ("router_rows_kernel (CUDA cores)" if T <= 32 else
                         "router_smem_kernel (mma.sync)" if tc == "0" else
                         "router_tc_kernel (tcgen05, TMA, 4-CTA cluster split-K)")
        out[key] = ent
    out["note"] = (f"logits = X W_r^T, d={cfg.d}, E={cfg.E}, bf16 in, fp32 out; 200 calls on distinct routers "
                   "in one CUDA graph")
    del W
    torch.cuda.empty_cache()
    out["T1_in_decode_step"] = decode_router_measure(dev)
    return out


def decode_router_measure(dev, reps=20):
    """The one-token projection inside the chained decode step: 40 distinct layers of moe_layer_x (projection,
    then the one-launch layer) against moe_layer on precomputed logits, each step one CUDA graph."""
    import torch
    import bit_moe_expert_gb300 as bm
    wl = DecodeWorkload(dev)
    cfg = wl.cfg
    Wr = [torch.from_numpy(synth.draw_router(cfg, l).view(np.int16)).to(dev) for l in range(wl.L)]
    lg = [torch.empty((wl.T, cfg.E), dtype=torch.float32, device=dev) for _ in range(wl.L)]

    def step_x():
        for l in range(wl.L):
            bm.moe_layer_x(wl.X[l], Wr[l], wl.routed[l], wl.shared[l], cfg.k, wl.block_rows, lg[l], wl.r,
                           wl.Y_l[l], wl.ws)

    s = torch.cuda.Stream(device=dev)
    res = {}
    for key, fn in (("moe_layer", wl.step), ("moe_layer_x", step_x)):
        with torch.cuda.stream(s):
            for _ in range(3):
                fn()
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                fn()
            for _ in range(3):
                g.replay()
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(reps):
                g.replay()
            e1.record(s)
            e1.synchronize()
        res[key] = e0.elapsed_time(e1) / reps / wl.L * 1e3
    out = {"us_per_layer_moe_layer": res["moe_layer"], "us_per_layer_moe_layer_x": res["moe_layer_x"],
           "router_us_per_layer": res["moe_layer_x"] - res["moe_layer"],
           "note": "40 distinct decode layers chained in one CUDA graph (PDL); moe_layer_x adds the router "
                   "projection (router_rows_kernel) ahead of each layer's decode kernel"}
    del wl, Wr, lg
    torch.cuda.empty_cache()
    return out


def uniform_logits(T, E, k):
    """Logits that route token t to experts (k t + j) mod E, j = 0..k-1, in that order: over T = M E / k tokens
    every expert receives exactly M rows."""
    lg = np.full((T, E), -10.0, np.float32)
    for t in range(T):
        for j in range(k):
            lg[t, (k * t + j) % E] = 10.0 - j
    return lg


def run_sweep(dev, peaks, args):
    """Rows per expert (M) against the weight-streaming rate, at fixed weights (the decode layer's experts,
    every expert active); then the canvas layer at B canvases of 256 tokens per call.  Each point is a CUDA
    graph of `steps` calls rotating over 4 weight sets (1.8 GB, beyond L2), timed with events."""
    import torch
    import bit_moe_expert_gb300 as bm

    def point(cfg, T, logits_np, sets, steps):
        C = T
        r = bm.Routing.empty(C, cfg.E, cfg.k, TILE_ROWS, dev)
        ws_r = bm.workspace(bm.moe_route_workspace_bytes(C, cfg.E, cfg.k), dev)
        ws_f = bm.workspace(bm.moe_forward_workspace_bytes(C, cfg.d, cfg.I, cfg.E, cfg.k, cfg.I_shared), dev)
        X = torch.from_numpy(synth.draw_x(cfg, C, 0).view(np.int16)).to(dev)
        lg = torch.from_numpy(logits_np).to(dev)
        Y = torch.empty((C, cfg.d), dtype=torch.int16, device=dev)

        def call(i):
            bm.moe_route(lg, cfg.k, TILE_ROWS, r, ws_r)
            bm.moe_forward(X, sets[i % len(sets)][0], sets[i % len(sets)][1], r, Y, ws_f)

        s = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(s):
            for i in range(3):
                call(i)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(steps):
                    call(i)
            g.replay()
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            e1.synchronize()
        assert bm.moe_check_status(ws_f) == 0 and bm.moe_check_status(ws_r) == 0
        t_call = e0.elapsed_time(e1) / steps / 1e3
        counts = r.counts.cpu().numpy()
        n_act = int((counts > 0).sum())
        wbytes = n_act * synth.ffn_bytes(cfg.d, cfg.I, cfg.bits) + (synth.ffn_bytes(cfg.d, cfg.I_shared, cfg.bits)
                                                                     if cfg.I_shared else 0)
        flops = 6 * T * cfg.d * (cfg.k * cfg.I + cfg.I_shared)
        return {"T": T, "active_experts": n_act, "rows_per_expert_max": int(counts.max()),
                "us_per_call": t_call * 1e6, "weight_bytes": wbytes, "gbs": wbytes / t_call / 1e9,
                "hbm_frac": wbytes / t_call / 1e9 / peaks["hbm_gbs"], "tok_s": T / t_call,
                "tflops": flops / t_call / 1e12}

    steps = max(4, min(args.steps, 40))
    cfg = synth.CONFIGS["decode"]
    sets = [_dev_layer(cfg, l, dev)[2:] for l in range(4)]
    sweep = []
    for M in (1, 2, 4, 8, 16, 32, 64, 128):
        T = M * cfg.E // cfg.k
        pt = point(cfg, T, uniform_logits(T, cfg.E, cfg.k), sets, steps)
        pt["M"] = M
        sweep.append(pt)
    del sets
    torch.cuda.empty_cache()
    ccfg = synth.CONFIGS["canvas"]
    csets = [_dev_layer(ccfg, l, dev)[2:] for l in range(4)]
    batching = []
    for B in (1, 2, 4):
        T = 256 * B
        lg = np.concatenate([synth.draw_logits(ccfg, 256, b) for b in range(B)])
        pt = point(ccfg, T, lg, csets, steps)
        pt["B"] = B
        batching.append(pt)
    return {"metric": "4-bit expert weight-streaming rate against rows per expert; canvas tokens/s against canvases "
                      "per call", "unit": "GB/s", "n_gpus": 1, "steps": steps,
            "config": {"workload": f"sweep: decode layer dims (d={cfg.d}, E={cfg.E}, k={cfg.k}, I={cfg.I}, "
                                   f"shared {cfg.I_shared}), T = M E / k tokens routed so that every expert gets "
                                   f"exactly M rows, moe_route + moe_forward per call; canvas layer "
                                   f"(d={ccfg.d}, E={ccfg.E}, I={ccfg.I}) at B x 256 tokens",
                       "l2": "4 weight sets per point, rotated (beyond L2)"},
            "data": "synthetic (seeded)", "sweep": sweep, "canvas_batching": batching,
            "peak_hbm_gbs": peaks["hbm_gbs"], "clocks": None}


def topk_wide_measure(dev, peaks):
    """The exact wide top-K (moe_topk_wide) at the canvas sampler's shape: 256 positions x 262,144 logits, K = 64
    (268 MB of logits, beyond L2); 20 calls in a CUDA graph, timed with events."""
    import torch
    import bit_moe_expert_gb300 as bm
    T, V, K = 256, 262144, 64
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    x = torch.randn((T, V), generator=gen, device=dev, dtype=torch.float32)
    vals = torch.empty((T, K), device=dev, dtype=torch.float32)
    idx = torch.empty((T, K), device=dev, dtype=torch.int32)
    s = torch.cuda.Stream(device=dev)
    n = 20
    with torch.cuda.stream(s):
        for _ in range(3):
            bm.moe_topk_wide(x, K, vals, idx)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(n):
                bm.moe_topk_wide(x, K, vals, idx)
        g.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        g.replay()
        e1.record(s)
        e1.synchronize()
    us = e0.elapsed_time(e1) / n * 1e3
    nbytes = T * V * 4 + T * K * 8
    del x
    return {"T": T, "V": V, "K": K, "us_per_call": us, "positions_per_s": T / (us * 1e-6), "bound": "hbm",
            "achieved": nbytes / us / 1e3, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": nbytes / us / 1e3 / peaks["hbm_gbs"], "bytes_per_call": nbytes,
            "note": "logits N(0,1) fp32 from a seeded device generator; one launch per call"}


def host_cpu():
    """The host's logical CPU count and model (from /proc/cpuinfo where present)."""
    import platform
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "cpu model"):
            for line in info.splitlines():
                if line.split(":")[0].strip() == key and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
            if model:
                break
        if not model:  # Arm: implementer and part numbers
            impl = [l.split(":", 1)[1].strip() for l in info.splitlines() if l.startswith("CPU implementer")]
            part = [l.split(":", 1)[1].strip() for l in info.splitlines() if l.startswith("CPU part")]
            if impl and part:
                model = f"{platform.machine()} implementer {impl[0]} part {part[0]}"
    except OSError:
        pass
    return {"host_nproc": os.cpu_count(), "host_cpu": model or platform.machine()}


def ablations_measure(dev, peaks, calls=20):
    """The pages' two ablations on the 512-token prefill layer ([Lily-M5] "Prefill: keep routing on the GPU,
    dequantize in flight": +77.4% from dequantising inside the GEMM, +89% from GPU-resident routing, both at a
    512-token prompt), as GB300 counterparts, every arm computing the same layer on the same 4 weight sets:
      fused        the product path: moe_route + moe_forward (dequantisation inside the tensor-core GEMM);
      unfused      moe_route, then the weights expanded to fp16 in HBM (moe_dequant_experts, all three matrices
                   of every expert and of the shared expert), then cuBLAS batched GEMMs over experts padded to
                   the most rows an expert has, SwiGLU and the weighted combine in torch;
      host_routing the top-k on the GPU (moe_route; its own grouping outputs are then overwritten), then the
                   histogram, scan, scatter and block map on the host behind a device-to-host copy and a
                   synchronisation, copied back, then moe_forward."""
    import torch
    import torch.nn.functional as F
    import bit_moe_expert_gb300 as bm
    cfg = synth.CONFIGS["prefill512"]
    T, E, k, d, I, Ish = cfg.T, cfg.E, cfg.k, cfg.d, cfg.I, cfg.I_shared
    nsets = 4
    sets = [_dev_layer(cfg, l, dev)[2:] for l in range(nsets)]
    X = torch.from_numpy(synth.draw_x(cfg, T, 0).view(np.int16)).to(dev)
    lg = torch.from_numpy(synth.draw_logits(cfg, T, 0)).to(dev)
    r = bm.Routing.empty(T, E, k, TILE_ROWS, dev)
    ws_r = bm.workspace(bm.moe_route_workspace_bytes(T, E, k), dev)
    ws_f = bm.workspace(bm.moe_forward_workspace_bytes(T, d, I, E, k, Ish), dev)
    Y = torch.empty((T, d), dtype=torch.int16, device=dev)
    s = torch.cuda.Stream(device=dev)

    def timed_graph(fn):
        with torch.cuda.stream(s):
            for i in range(3):
                fn(i)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(calls):
                    fn(i)
            g.replay()
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            e1.synchronize()
        return e0.elapsed_time(e1) / calls * 1e3  # us per call

    def fused(i):
        bm.moe_route(lg, k, TILE_ROWS, r, ws_r)
        bm.moe_forward(X, sets[i % nsets][0], sets[i % nsets][1], r, Y, ws_f)

    t_fused = timed_graph(fused)
    fused(0)  # the reference output: weight set 0, as the checks below use
    torch.cuda.synchronize()
    Y_fused = Y.clone()

    # unfused: static padding layout from this layer's routing (the same every call)
    bm.moe_route(lg, k, TILE_ROWS, r, ws_r)
    torch.cuda.synchronize()
    counts = r.counts.cpu().numpy()
    Mmax = int(counts.max())
    perm = r.perm.long()
    offsets = r.offsets.long()
    expert_of_row = torch.repeat_interleave(torch.arange(E, device=dev), r.counts.long())
    slot_of_row = torch.arange(T * k, device=dev) - offsets[expert_of_row]
    pad_index = expert_of_row * Mmax + slot_of_row  # permuted row -> padded row
    W16 = {m: torch.empty((E, *(getattr(sets[0][0], m).sb.shape[2:3]), getattr(sets[0][0], m).sb.shape[1] * 64),
                          dtype=torch.int16, device=dev) for m in ("gate", "up", "down")}
    Ws16 = {m: torch.empty((1, getattr(sets[0][1], m).sb.shape[2], getattr(sets[0][1], m).sb.shape[1] * 64),
                           dtype=torch.int16, device=dev) for m in ("gate", "up", "down")}
    Xf = X.view(torch.bfloat16).to(torch.float16)
    Xpad = torch.zeros((E * Mmax, d), dtype=torch.float16, device=dev)
    Yun = torch.empty((T, d), dtype=torch.float32, device=dev)

    def unfused(i):
        routed, shared = sets[i % nsets]
        bm.moe_route(lg, k, TILE_ROWS, r, ws_r)
        for m in ("gate", "up", "down"):
            bm.moe_dequant_experts(getattr(routed, m), routed.bits, W16[m])
            bm.moe_dequant_experts(getattr(shared, m), shared.bits, Ws16[m])
        Xpad.index_copy_(0, pad_index, Xf.index_select(0, perm // k))
        xp = Xpad.view(E, Mmax, d)
        g = torch.bmm(xp, W16["gate"].view(torch.float16).transpose(1, 2))
        u = torch.bmm(xp, W16["up"].view(torch.float16).transpose(1, 2))
        h = (F.silu(g.float()) * u.float()).to(torch.float16)
        ye = torch.bmm(h, W16["down"].view(torch.float16).transpose(1, 2)).view(E * Mmax, d)
        rows = ye.index_select(0, pad_index).float()  # permuted row order
        wv = r.w.view(-1)
        contrib = rows.index_select(0, r.inv_perm.long()) * wv.unsqueeze(1)  # assignment order t*k + j
        Yun.copy_(contrib.view(T, k, d).sum(1))
        gs = Xf @ Ws16["gate"][0].view(torch.float16).t()
        us = Xf @ Ws16["up"][0].view(torch.float16).t()
        hs = (F.silu(gs.float()) * us.float()).to(torch.float16)
        Yun.add_(hs @ Ws16["down"][0].view(torch.float16).t())

    t_unfused = timed_graph(unfused)
    torch.cuda.synchronize()
    unfused(0)
    torch.cuda.synchronize()
    yf = Y_fused.view(torch.bfloat16).float()
    rel = float(torch.linalg.norm(Yun - yf) / torch.linalg.norm(yf))
    del W16, Ws16, Xpad

    # host routing: top-k on the device, the grouping on the host behind a synchronisation
    ids_h = torch.empty((T, k), dtype=torch.int32).pin_memory()
    bufs = {n: torch.empty(sz, dtype=torch.int32).pin_memory()
            for n, sz in (("counts", E), ("offsets", E + 1), ("perm", T * k), ("inv_perm", T * k),
                          ("block_map", r.block_map.numel()), ("num_blocks", 1))}

    def host_routing(i):
        routed, shared = sets[i % nsets]
        bm.moe_route(lg, k, TILE_ROWS, r, ws_r)  # its top-k (ids, w) is what the host receives
        ids_h.copy_(r.ids, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        ids = ids_h.numpy().reshape(-1)
        cnt = np.bincount(ids, minlength=E).astype(np.int32)
        off = np.zeros(E + 1, np.int32)
        np.cumsum(cnt, out=off[1:])
        order = np.argsort(ids, kind="stable").astype(np.int32)
        inv = np.empty_like(order)
        inv[order] = np.arange(order.size, dtype=np.int32)
        bmap = []
        for e in np.nonzero(cnt)[0]:
            for r0 in range(0, int(cnt[e]), TILE_ROWS):
                bmap += [int(e), int(off[e]) + r0, min(TILE_ROWS, int(cnt[e]) - r0)]
        bufs["counts"].numpy()[:] = cnt
        bufs["offsets"].numpy()[:] = off
        bufs["perm"].numpy()[:] = order
        bufs["inv_perm"].numpy()[:] = inv
        bufs["block_map"].numpy()[:len(bmap)] = bmap
        bufs["num_blocks"].numpy()[0] = len(bmap) // 3
        for n in bufs:
            getattr(r, n).view(-1)[:bufs[n].numel()].copy_(bufs[n], non_blocking=True)
        bm.moe_forward(X, routed, shared, r, Y, ws_f)

    with torch.cuda.stream(s):
        for i in range(3):
            host_routing(i)
        s.synchronize()
        t0 = time.perf_counter()
        for i in range(calls):
            host_routing(i)
        s.synchronize()
        t_host = (time.perf_counter() - t0) / calls * 1e6
    fused(0)
    torch.cuda.synchronize()
    Y0 = Y.clone()
    host_routing(0)
    torch.cuda.synchronize()
    same = bool(torch.equal(Y, Y0))
    assert bm.moe_check_status(ws_f) == 0 and bm.moe_check_status(ws_r) == 0
    del sets
    torch.cuda.empty_cache()
    return {"workload": f"prefill512 layer (T={T}, d={d}, E={E}, top-{k} + shared, I={I}), 4 weight sets rotated",
            "fused_us": t_fused, "unfused_dequant_us": t_unfused, "host_routing_us": t_host,
            "fused_dequant_speedup": t_unfused / t_fused, "gpu_routing_speedup": t_host / t_fused,
            "pages": {"fused_dequant_gain": "+77.4% end-to-end prefill at 512 tokens (M5)",
                      "gpu_routing_gain": "+89% end-to-end prefill at 512 tokens (M5)"},
            "unfused_rel_l2_vs_fused": rel, "host_routing_output_identical": same,
            "note": "MoE layer alone (the pages' gains are whole-model prefill); fused and unfused timed as CUDA "
                    "graphs of 20 calls, host routing by wall clock over 20 calls (it synchronises every call)"}


def cpu_baseline(wl, budget_s):
    tokens, secs, desc = wl.cpu_sample(budget_s)
    out = {"value": tokens / secs, "unit": "tok/s", "cores": 1, "kind": "oracle", "sample": desc,
           "seconds": secs}
    out.update(host_cpu())
    return out


# ----------------------------------------------------------------------------- reference arm (the oracle)

def _host_experts(ex, index=None):
    out = {}
    for m, (q, sc, bi) in ex.items():
        if index is not None:
            q, sc, bi = q.index_select(0, index), sc.index_select(0, index), bi.index_select(0, index)
        out[m] = (q.cpu().numpy().view(np.uint32), sc.cpu().numpy().view(np.uint16), bi.cpu().numpy().view(np.uint16))
    return out


def reference_arm(args, dist):
    """The oracle, as it stands, timed on the host cores: each step one bounded
    sample of the headline workload (routing + layer for the decode token of
    each sampled layer).  The device only draws the synthetic weights (torch's
    generator, the same bytes as the GPU arm); nothing of the CUDA library runs."""
    if dist.rank != 0:
        return None
    if args.workload != "decode":
        return {"impl": "reference", "unavailable": "reference arm is defined for the decode headline workload"}
    import torch
    import oracle
    dev = torch.device("cuda", dist.local_rank) if torch.cuda.is_available() else torch.device("cpu")
    cfg = synth.CONFIGS["decode"]
    n_layers = 8
    layers = []
    for l in range(n_layers):
        logits = synth.draw_logits(cfg, cfg.T, l)
        X = synth.draw_x(cfg, cfg.T, l)
        ids, _ = oracle.topk(logits, cfg.k)
        sel = sorted(set(int(e) for e in ids.reshape(-1)))
        rex = synth.draw_experts_torch(cfg, l, dev)
        sex = synth.draw_experts_torch(cfg, l, dev, E=1, I=cfg.I_shared, tag=20)
        routed = _host_experts(rex, torch.tensor(sel, device=dev))
        shared = _host_experts(sex)
        del rex, sex
        lut = {e: i for i, e in enumerate(sel)}
        layers.append((logits, X, routed, shared, lut))

    def one_layer(l):
        logits, X, routed, shared, lut = layers[l]
        r = oracle.route(logits, cfg.k, 128)
        ids = np.vectorize(lambda e: lut[int(e)])(r["ids"]).astype(np.int32)
        oracle.forward(X, routed, shared, ids, r["w"])

    t0 = time.perf_counter()
    one_layer(0)
    t_layer = time.perf_counter() - t0
    budget = 120.0  # seconds for the whole --steps/--warmup run
    per_step = max(1, min(n_layers, int(budget / max(args.steps + args.warmup, 1) / t_layer)))

    def step():
        for l in range(per_step):
            one_layer(l)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = time.perf_counter() - t0
    value = per_step * cfg.T * args.steps / secs
    sample = f"{per_step} decode layer(s) of 1 token per step (routing + layer)"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": f"decode: T={cfg.T}, d={cfg.d}, E={cfg.E}, top-{cfg.k} + shared expert, "
                                   f"I={cfg.I}; CPU oracle", "reference_sample": sample},
            "cpu_baseline": dict({"value": value, "unit": "tok/s", "cores": 1, "kind": "oracle", "sample": sample},
                                 **host_cpu()),
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode",
                    choices=sorted(synth.CONFIGS) + ["sweep", "router", "topk_wide", "ablations"],
                    help="sweep: rows-per-expert and canvas-batching measurements; router, topk_wide, ablations: "
                         "those measurements of the default run alone (one JSON line each)")
    ap.add_argument("--no-secondary", action="store_true", help="skip the T=4096 prefill object")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--layers", type=int, default=0,
                    help="decode: layers per step; prefill: weight sets (default: the workload's own)")
    ap.add_argument("--only-graph", action="store_true",
                    help="time the graph only (no end-to-end pass, kernel-timing pass or CPU baseline): "
                         "a small, quick case for profilers")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    dist = Dist()
    if args.impl == "reference":
        res = reference_arm(args, dist)
        if res is not None:
            print(json.dumps(res), flush=True)
        dist.close()
        return

    import torch
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    peaks = measured_peaks()
    clocks = ClockSampler(dist.local_rank)

    if args.workload in ("sweep", "router", "topk_wide", "ablations"):
        clocks.start()
        if args.workload == "sweep":
            res = run_sweep(dev, peaks, args)
        elif args.workload == "router":
            res = router_measure(dev, peaks)
        elif args.workload == "topk_wide":
            res = topk_wide_measure(dev, peaks)
        else:
            res = ablations_measure(dev, peaks)
        res["clocks"] = clocks.stop()
        if dist.rank == 0:
            print(json.dumps(res), flush=True)
        dist.close()
        return
    if args.workload in ("decode", "decode3b", "decode2b"):
        wl = DecodeWorkload(dev, layers=args.layers or None, name=args.workload)
    else:
        wl = PrefillWorkload(dev, args.workload, sets=args.layers or None)
    if args.only_graph:
        ms, clk = time_graph(wl, args.steps, args.warmup, dist, clocks)
        if dist.rank == 0:
            print(json.dumps({"workload": wl.workload_desc(), "ms_per_step": ms / args.steps,
                              "value": wl.tokens_per_step * args.steps / (ms / 1e3), "unit": "tok/s",
                              "clocks": clk, "only_graph": True}), flush=True)
        dist.close()
        return
    main_res = run_workload(wl, args, dist, peaks, clocks)
    cpu = cpu_baseline(wl, args.cpu_budget) if dist.rank == 0 else None
    desc = wl.workload_desc()
    launches = wl.launches_per_step() * args.steps
    del wl
    torch.cuda.empty_cache()

    def secondary_run(name, budget):
        wl2 = PrefillWorkload(dev, name)
        steps2 = max(3, min(args.steps, 200))
        a2 = argparse.Namespace(**vars(args))
        a2.steps = steps2
        r2 = run_workload(wl2, a2, dist, peaks, ClockSampler(dist.local_rank))
        r2["cpu_baseline"] = cpu_baseline(wl2, budget) if dist.rank == 0 else None
        r2["workload"] = wl2.workload_desc()
        r2["steps"] = steps2
        r2["gpu_launches"] = wl2.launches_per_step() * steps2
        r2["tok_s"] = r2["value"]
        if name == "canvas":
            # the block-diffusion canvas step runs the layer once per each of its 30 layers
            cfg2 = wl2.cfg
            per_layer = cfg2.E * synth.ffn_bytes(cfg2.d, cfg2.I, cfg2.bits)  # every expert active
            n_act = wl2.active_experts()
            r2["canvas_step"] = {"layers": cfg2.layers, "active_experts_per_layer": n_act,
                                 "expert_bytes_per_layer": per_layer,
                                 "gb_per_step": cfg2.layers * n_act * synth.ffn_bytes(cfg2.d, cfg2.I, cfg2.bits) / 1e9,
                                 "ms_per_step": cfg2.layers * r2["ms_per_step"],
                                 "canvases_per_s": 1e3 / (cfg2.layers * r2["ms_per_step"]),
                                 "note": "30 distinct layers of the canvas layer per denoising step; each layer "
                                         "timed on its own weight set (4 sets rotated, beyond L2)"}
        del wl2
        torch.cuda.empty_cache()
        return r2

    secondary = None
    extra = {}
    if args.workload == "decode" and not args.no_secondary:
        secondary = secondary_run("prefill4096", args.cpu_budget)
        extra["prefill512"] = secondary_run("prefill512", args.cpu_budget / 2)
        extra["canvas"] = secondary_run("canvas", args.cpu_budget / 2)
        sw = run_sweep(dev, peaks, args)
        extra["sweep"] = {k: sw[k] for k in ("sweep", "canvas_batching", "steps", "config", "peak_hbm_gbs")}
        torch.cuda.empty_cache()
    if args.workload == "decode" and not args.no_secondary:
        extra["ablations"] = ablations_measure(dev, peaks)
    router = router_measure(dev, peaks) if (args.workload == "decode" and not args.no_secondary) else None
    wide = topk_wide_measure(dev, peaks) if (args.workload == "decode" and not args.no_secondary) else None

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": main_res["value"], "unit": "tok/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main_res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": main_res["dtype"],
            "data": "synthetic (seeded; random 4-bit codes, bf16 scale/bias, N(0,1) X and logits)",
            "config": {"workload": desc, "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "1 GPU",
                       "l2": "inputs larger than L2 (decode: 40 distinct layers, 18.2 GB of weights; prefill: "
                             "each chunk on its own 455 MB weight set)"},
            "e2e": main_res["e2e"], "roofline": main_res["roofline"], "cpu_baseline": cpu,
            "clocks": main_res["clocks"], "gpu_launches": launches, "kernels": main_res["kernels"],
        }
        for key in ("layer_roofline", "step_roofline"):
            if key in main_res:
                line[key] = main_res[key]
        if secondary is not None:
            line["prefill4096"] = secondary
        line.update(extra)
        if router is not None:
            line["router_projection"] = router
        if wide is not None:
            line["topk_wide"] = wide
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
