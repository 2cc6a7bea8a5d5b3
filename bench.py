#!/usr/bin/env python3
"""Benchmark of the GGUF Q4_0 / Q8_0 decode DMMV on GB300.

Workload (default): the dense Q4_0 4096 x 4096 decode DMMV, batch 1. One STEP is
LAYERS launches over LAYERS distinct weight matrices of that shape, each with its
own fp32 activation (per layer: quantize the activation to Q8_0, then the DMMV,
fused in one launch), ordered in one stream so that each launch waits for the
previous grid before it reads its inputs, as the layers of a decode token do;
every step streams LAYERS x 9.44 MB of weights. The stack (605 MB at 64 layers)
is larger than 4x the 129 MB L2, so no layer's weights are L2-resident when it
runs. Inputs are resident in HBM before the timed region; the step is captured
once in a CUDA graph and replayed (decode chains are replayed as graphs: "RTX
5090: Batched Prefill & CUDA Graphs in ZINC", "CUDA graphs -- the structural
answer to launch latency").

Printed: one JSON line (rank 0) with value = algorithmic GB/s over the whole job
(weights read once + Q8_0 activation blocks + fp32 outputs), the
roofline of the step's kernel (the fused quantize + DMMV; the DMMV over
pre-quantized blocks beside it) against the measured HBM copy bandwidth, the CPU oracle as baseline, the end-to-end number through the
host-buffer C-ABI call, clocks sampled during the timed region, and per-workload
measurements of the other four decode workloads.

--impl reference times the CPU oracle on the same workload and metric: with no
upstream code to run, the oracle is the reference implementation of the method.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q4_0/Q8_0 DMMV achieved HBM GB/s and % of GB300 peak; rows/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["zdmmv", "reference"], default="zdmmv")
    p.add_argument("--layers", type=int, default=64, help="distinct weight matrices per step")
    p.add_argument("--no-extra", action="store_true", help="skip the other four workloads")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--eager", action="store_true", help="launch eagerly instead of graph replay")
    p.add_argument("--profile", default=None, metavar="WORKLOAD",
                   help="no timing: a few launches of one workload (for ncu captures)")
    return p.parse_args()


# --------------------------------------------------------------------- helpers
def peaks():
    try:
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the sources that define the dense pipelined DMMV kernel (its code and arguments)
DENSE_KERNEL_SOURCES = ("zdmmv_device.cuh", "zdmmv_internal.h", "zdmmv_tma.cuh", "zdmmv_tma_q4.cu")


def kernel_sources_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gguf_block_quant_gb300", "csrc")
    for f in DENSE_KERNEL_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu summary,
    or None if there is none or the kernel sources changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d[workload]
        if e.get("src_sha") != kernel_sources_sha():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.proc = None
        self.gpu = gpu_index
        self.interval = interval_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device) -> float:
    """Max of a per-rank scalar over all ranks (timing only; no data-path collective)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ CPU oracle
def cpu_baseline_dense(cfg, layers_budget_s: float = 12.0):
    """Time the oracle (as it stands, single thread) on a bounded sample of the
    dense workload: whole layers (quantize + DMMV of one 4096 x 4096 matrix)
    until about layers_budget_s of CPU work."""
    import oracle
    from gguf_block_quant_gb300 import synth
    w = synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)
    x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale)
    oracle.lib()
    done = 0
    t0 = time.perf_counter()
    while True:
        xq = oracle.quantize_q8_0(x)
        oracle.dmmv(cfg.fmt, w, cfg.rows, cfg.cols, xq)
        done += 1
        el = time.perf_counter() - t0
        if el >= layers_budget_s or done >= 2000:
            break
    gbs = done * cfg.algorithmic_bytes() / el / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} layers ({cfg.name}: quantize + DMMV each) in {el:.1f} s, single-threaded C",
            "rows_per_s": done * cfg.rows / el}


# The oracle over row ranges in worker processes (spawned, never forked: the
# parent may already hold a CUDA context). Each worker gets the whole matrix once.
_ORACLE_W = None


def _oracle_worker_init(fmt, w_bytes, rows, cols):
    global _ORACLE_W
    import numpy as np
    import oracle
    oracle.lib()
    _ORACLE_W = (fmt, np.frombuffer(w_bytes, dtype=np.uint8).reshape(rows, -1), cols)


def _oracle_worker_rows(task):
    import oracle
    r0, r1, xq = task
    fmt, w, cols = _ORACLE_W
    y, _ = oracle.dmmv(fmt, w[r0:r1].reshape(-1), r1 - r0, cols, xq)
    return r0, y


def cpu_baseline_parallel(cfg, budget_s: float = 12.0):
    """The same oracle, unchanged, on every core this process may use: each layer's
    rows are split over a pool of spawned worker processes (the per-row arithmetic
    is unchanged, so the result is bit-identical to the single-threaded run)."""
    import multiprocessing as mp
    import numpy as np
    import oracle
    from gguf_block_quant_gb300 import synth
    w = synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)
    x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale)
    cores = len(os.sched_getaffinity(0))
    bounds = [cfg.rows * i // cores for i in range(cores + 1)]
    with mp.get_context("spawn").Pool(cores, initializer=_oracle_worker_init,
                                      initargs=(cfg.fmt, w.tobytes(), cfg.rows, cfg.cols)) as pool:
        def layer():
            xq = oracle.quantize_q8_0(x)
            y = np.empty(cfg.rows)
            for r0, part in pool.map(_oracle_worker_rows, [(bounds[i], bounds[i + 1], xq) for i in range(cores)]):
                y[r0:r0 + len(part)] = part
            return y, xq
        y, xq = layer()  # workers started and warm
        y1, _ = oracle.dmmv(cfg.fmt, w, cfg.rows, cfg.cols, xq)
        if not np.array_equal(y, y1):
            raise RuntimeError("parallel oracle disagrees with the single-threaded oracle")
        done = 0
        t0 = time.perf_counter()
        while True:
            layer()
            done += 1
            el = time.perf_counter() - t0
            if el >= budget_s or done >= 20000:
                break
    return {"value": done * cfg.algorithmic_bytes() / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} layers ({cfg.name}: quantize + DMMV each) in {el:.1f} s, rows split over {cores} "
                      f"worker processes", "rows_per_s": done * cfg.rows / el}


# ----------------------------------------------------------------- GPU arm
def graph_or_eager(fn, eager: bool):
    import torch
    if eager:
        return fn
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g.replay


def time_fn(run, steps: int, warmup: int, world: int, device, sampler=None):
    import torch
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.start()
        time.sleep(0.05)
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier(world)
    ms = e0.elapsed_time(e1)
    return reduce_max(ms, world, device), clocks


class DensePool:
    """LAYERS distinct copies of one dense workload's tensors, resident in HBM
    (weights in the GGUF layout, or repacked once when layout == REPACKED)."""

    def __init__(self, cfg, layers: int, layout: int = 0):
        import numpy as np
        import torch
        from gguf_block_quant_gb300 import synth
        from gguf_block_quant_gb300 import zdmmv as Z
        self.cfg, self.layers = cfg, layers
        w = torch.from_numpy(synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)).cuda()
        if layout == Z.REPACKED:
            w = Z.repack(cfg.fmt, w, cfg.rows, cfg.cols)
        self.layout = layout
        self.w = [w] + [w.clone() for _ in range(layers - 1)]
        x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale, batch=max(cfg.batch, 1))
        x = torch.from_numpy(np.ascontiguousarray(x).reshape(-1)).cuda()
        self.x = [x] + [x.clone() for _ in range(layers - 1)]
        nq = cfg.batch * cfg.nb * 34
        self.xq = [torch.empty(nq, dtype=torch.uint8, device="cuda") for _ in range(layers)]
        self.y = [torch.empty(cfg.batch * cfg.rows, dtype=torch.float32, device="cuda") for _ in range(layers)]
        self.Z = Z
        self.step_unfused()   # activations quantized once so the DMMV-only pass reads valid blocks
        torch.cuda.synchronize()

    def step(self):
        """One decode token: per layer the fused quantize + DMMV (one launch)."""
        Z, c = self.Z, self.cfg
        for l in range(self.layers):
            Z.dmmv_f32(c.fmt, self.w[l], c.rows, c.cols, self.x[l], batch=c.batch, y=self.y[l], layout=self.layout)

    def step_unfused(self):
        """The same token with the two-kernel chain: quantize, then DMMV."""
        Z, c = self.Z, self.cfg
        for l in range(self.layers):
            Z.quantize_act_q8_0(self.x[l], self.xq[l])
            if c.batch == 1:
                Z.dmmv(c.fmt, self.w[l], c.rows, c.cols, self.xq[l], y=self.y[l], layout=self.layout)
            else:
                Z.dmmv_batched(c.fmt, self.w[l], c.rows, c.cols, self.xq[l], c.batch, y=self.y[l],
                               layout=self.layout)

    def dmmv_only(self):
        Z, c = self.Z, self.cfg
        for l in range(self.layers):
            if c.batch == 1:
                Z.dmmv(c.fmt, self.w[l], c.rows, c.cols, self.xq[l], y=self.y[l], layout=self.layout)
            else:
                Z.dmmv_batched(c.fmt, self.w[l], c.rows, c.cols, self.xq[l], c.batch, y=self.y[l],
                               layout=self.layout)


def layers_for(cfg, l2_bytes: int, min_layers: int = 2) -> int:
    per = cfg.weight_bytes
    return max(min_layers, -(-4 * l2_bytes // per))


def measure_dense(cfg, layers, steps, warmup, world, device, eager, layout=0):
    import torch
    pool = DensePool(cfg, layers, layout)
    run = graph_or_eager(pool.dmmv_only, eager)
    pool_step = graph_or_eager(pool.step, eager)
    pool_step2 = graph_or_eager(pool.step_unfused, eager)
    ms_dmmv, _ = time_fn(run, steps, warmup, world, device)
    ms_step, _ = time_fn(pool_step, steps, warmup, world, device)
    ms_step2, _ = time_fn(pool_step2, steps, warmup, world, device)
    per_launch_s = ms_dmmv / 1e3 / (steps * layers)
    per_step_s = ms_step / 1e3 / steps
    nbytes = cfg.algorithmic_bytes()
    del pool
    torch.cuda.empty_cache()
    return {"layers": layers, "dmmv_us": per_launch_s * 1e6, "dmmv_gbs": nbytes / per_launch_s / 1e9,
            "fused_step_gbs": layers * nbytes / per_step_s / 1e9,
            "fused_us_per_layer": per_step_s / layers * 1e6,
            "two_kernel_step_gbs": layers * nbytes / (ms_step2 / 1e3 / steps) / 1e9,
            "rows_per_s": cfg.batch * cfg.rows / per_launch_s, "algorithmic_bytes": nbytes}


def measure_xf32(cfg, layers, steps, warmup, world, device, eager):
    """The DMMV with the fp32 activation taken as is (no quantization), back to
    back over the layer stack; algorithmic bytes = weights + fp32 x + fp32 y."""
    import torch
    pool = DensePool(cfg, layers)
    Z, c = pool.Z, cfg

    def run_all():
        for l in range(layers):
            Z.dmmv_xf32(c.fmt, pool.w[l], c.rows, c.cols, pool.x[l], batch=c.batch, y=pool.y[l])

    run = graph_or_eager(run_all, eager)
    ms, _ = time_fn(run, steps, warmup, world, device)
    per = ms / 1e3 / (steps * layers)
    nbytes = cfg.weight_bytes + c.batch * (4 * c.cols + 4 * c.rows)
    del pool
    torch.cuda.empty_cache()
    return {"us": per * 1e6, "gbs": nbytes / per / 1e9, "algorithmic_bytes": nbytes,
            "note": "fp32 activation, no quantization: one fp32 fma per weight (ALU-heavy)"}


def measure_grouped(cfg, layers, steps, warmup, world, device, eager):
    """The same dense DMMV over LAYERS distinct matrices issued as ONE launch
    (the expert-gather entry point over a stack, index k -> matrix k, each slot
    its own activation): the kernel's streaming rate on this shape once the
    per-launch latency is amortized. Not a decode chain: the matrices are
    independent problems."""
    import numpy as np
    import torch
    from gguf_block_quant_gb300 import synth
    from gguf_block_quant_gb300 import zdmmv as Z
    w = torch.from_numpy(synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)).cuda()
    stack = w.repeat(layers)
    per = w.numel()
    idx = torch.arange(layers, dtype=torch.int32, device="cuda")
    x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale, batch=layers)
    xq = Z.quantize_act_q8_0(torch.from_numpy(np.ascontiguousarray(x).reshape(-1)).cuda())
    y = torch.empty(layers, cfg.rows, dtype=torch.float32, device="cuda")

    def run_all():
        Z.expert_gather(cfg.fmt, stack, per, cfg.rows, cfg.cols, idx, layers, xq, cfg.nb * 34, y=y)

    run = graph_or_eager(run_all, eager)
    ms, _ = time_fn(run, steps, warmup, world, device)
    per_matrix = ms / 1e3 / (steps * layers)
    nbytes = cfg.algorithmic_bytes() + 4
    del stack, w, run
    torch.cuda.empty_cache()
    return {"matrices_per_launch": layers, "us_per_matrix": per_matrix * 1e6, "gbs": nbytes / per_matrix / 1e9,
            "note": "independent matrices in one launch (expert-gather entry point); not a decode chain"}


def measure_argmax(cfg, layers, steps, warmup, world, device, eager):
    """The LM head with the fused argmax epilogue (no logits written), back to back."""
    import torch
    pool = DensePool(cfg, layers)
    Z = pool.Z
    ws = [torch.empty(Z.ARGMAX_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda") for _ in range(layers)]
    out = [torch.empty(1, dtype=torch.int32, device="cuda") for _ in range(layers)]

    def run_all():
        for l in range(layers):
            Z.dmmv_argmax(cfg.fmt, pool.w[l], cfg.rows, cfg.cols, pool.xq[l], workspace=ws[l], out=out[l])

    run = graph_or_eager(run_all, eager)
    ms, _ = time_fn(run, steps, warmup, world, device)
    per = ms / 1e3 / (steps * layers)
    nbytes = cfg.weight_bytes + cfg.nb * 34 + 4
    del pool
    torch.cuda.empty_cache()
    return {"us": per * 1e6, "gbs": nbytes / per / 1e9, "algorithmic_bytes": nbytes,
            "launches": 2, "note": "DMMV with per-CTA (max, row) partials + one-CTA reduce; logits never written"}


def measure_moe(steps, warmup, world, device, eager, l2_bytes):
    """Config: 9 selected experts (8 routed + shared) of a 129-slot stack; one
    step = gate, up (Q4_0 512x2048) and down (Q8_0 2048x512) gathers, each ONE
    launch; stacks rotated over copies so that > 4x L2 is touched per pass."""
    import numpy as np
    import torch
    from gguf_block_quant_gb300 import synth
    from gguf_block_quant_gb300 import zdmmv as Z
    m = synth.MOE
    gate = torch.from_numpy(synth.weight_blocks(synth.Q4_0, m.n_slots * m.ffn, m.hidden, seed=m.seed)).cuda()
    up = torch.from_numpy(synth.weight_blocks(synth.Q4_0, m.n_slots * m.ffn, m.hidden, seed=m.seed,
                                              stream=synth.S_WEIGHT2)).cuda()
    down = torch.from_numpy(synth.weight_blocks(synth.Q8_0, m.n_slots * m.hidden, m.ffn, seed=m.seed,
                                                stream=synth.S_WEIGHT3)).cuda()
    # different routing per layer so touched experts differ; stacks are 296 MB per layer set
    n_sets = 2
    stacks = [(gate, up, down)] + [(gate.clone(), up.clone(), down.clone()) for _ in range(n_sets - 1)]
    idxs = [torch.from_numpy(synth.expert_indices(m.seed + 100 * i, m.n_routed, m.top_k)).cuda()
            for i in range(8)]
    x = torch.from_numpy(synth.activations(m.hidden, seed=m.seed)).cuda()
    xd = torch.from_numpy(np.ascontiguousarray(
        synth.activations(m.ffn, seed=m.seed, stream=synth.S_ACT2, batch=m.n_sel)).reshape(-1)).cuda()
    xq = Z.quantize_act_q8_0(x)
    xqd = Z.quantize_act_q8_0(xd)
    yg = torch.empty(m.n_sel, m.ffn, device="cuda")
    yu = torch.empty(m.n_sel, m.ffn, device="cuda")
    yd = torch.empty(m.n_sel, m.hidden, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gu, dn = m.gate_up_bytes(), m.down_bytes()
    layers = 16

    def step3():
        for l in range(layers):
            g, u, d = stacks[l % n_sets]
            idx = idxs[l % len(idxs)]
            Z.expert_gather(Z.Q4_0, g, gu, m.ffn, m.hidden, idx, m.n_slots, xq, 0, y=yg, status=st)
            Z.expert_gather(Z.Q4_0, u, gu, m.ffn, m.hidden, idx, m.n_slots, xq, 0, y=yu, status=st)
            Z.expert_gather(Z.Q8_0, d, dn, m.hidden, m.ffn, idx, m.n_slots, xqd, (m.ffn // 32) * 34, y=yd,
                            status=st)

    def step2():
        for l in range(layers):
            g, u, d = stacks[l % n_sets]
            idx = idxs[l % len(idxs)]
            Z.expert_gather2(Z.Q4_0, g, u, gu, m.ffn, m.hidden, idx, m.n_slots, xq, 0, y_a=yg, y_b=yu, status=st)
            Z.expert_gather(Z.Q8_0, d, dn, m.hidden, m.ffn, idx, m.n_slots, xqd, (m.ffn // 32) * 34, y=yd,
                            status=st)

    h = torch.empty(m.n_sel, m.ffn, device="cuda")

    def step_swiglu():
        for l in range(layers):
            g, u, d = stacks[l % n_sets]
            idx = idxs[l % len(idxs)]
            Z.expert_swiglu(Z.Q4_0, g, u, m.ffn, m.hidden, xq, idx=idx, expert_stride=gu, n_experts=m.n_slots,
                            h=h, status=st)
            Z.expert_gather(Z.Q8_0, d, dn, m.hidden, m.ffn, idx, m.n_slots, xqd, (m.ffn // 32) * 34, y=yd,
                            status=st)

    hq = torch.empty(m.n_sel * (m.ffn // 32) * 34, dtype=torch.uint8, device="cuda")

    def step_chain():
        # the same FFN through separate launches: SwiGLU, quantize h, down gather of h
        for l in range(layers):
            g, u, d = stacks[l % n_sets]
            idx = idxs[l % len(idxs)]
            Z.expert_swiglu(Z.Q4_0, g, u, m.ffn, m.hidden, xq, idx=idx, expert_stride=gu, n_experts=m.n_slots,
                            h=h, status=st)
            Z.quantize_act_q8_0(h.reshape(-1), hq)
            Z.expert_gather(Z.Q8_0, d, dn, m.hidden, m.ffn, idx, m.n_slots, hq, (m.ffn // 32) * 34, y=yd,
                            status=st)

    ws = Z.expert_ffn_workspace(m.n_sel, m.ffn)

    def step_ffn():
        for l in range(layers):
            g, u, d = stacks[l % n_sets]
            idx = idxs[l % len(idxs)]
            Z.expert_ffn(Z.Q4_0, g, u, gu, Z.Q8_0, d, dn, m.hidden, m.ffn, idx, m.n_slots, xq, y=yd,
                         workspace=ws, status=st)

    nbytes = m.algorithmic_bytes()
    # the SwiGLU epilogue writes h instead of the gate and up outputs
    nbytes_swiglu = nbytes - m.n_sel * m.ffn * 4
    out = {"layers": layers, "algorithmic_bytes": nbytes,
           "note": "touched experts differ per layer; stack copies alternate (some L2 reuse possible)"}
    for name, fn, launches, nb_ in (("three_launch", step3, 3, nbytes), ("gate_up_fused", step2, 2, nbytes),
                                    ("gate_up_swiglu", step_swiglu, 2, nbytes_swiglu),
                                    ("ffn_chained_three_launch", step_chain, 3, nbytes_swiglu),
                                    ("ffn_one_launch", step_ffn, 1, nbytes_swiglu)):
        run = graph_or_eager(fn, eager)
        ms, _ = time_fn(run, steps, warmup, world, device)
        per_layer = ms / 1e3 / (steps * layers)
        out[name] = {"us_per_token_layer": per_layer * 1e6, "gbs": nb_ / per_layer / 1e9,
                     "algorithmic_bytes": nb_,
                     "rows_per_s": m.n_sel * (2 * m.ffn + m.hidden) / per_layer, "launches_per_layer": launches}
    out["ffn_one_launch"]["note"] = ("gate/up + SwiGLU and the down DMMV of the quantized SwiGLU output in one "
                                     "launch (the down input is h, not the independent activation)")
    out["ffn_chained_three_launch"]["note"] = "the same chained FFN as SwiGLU, quantize h, down gather"
    out["gbs"] = max(out[k]["gbs"] for k in ("three_launch", "gate_up_fused", "gate_up_swiglu", "ffn_one_launch"))
    return out


def e2e_dense(cfg, layers, steps, warmup, world, device, eager=False):
    """End to end through the public API: every step uploads the step's fp32
    activations (one per layer) from pinned host memory, runs the fused
    quantize + DMMV of every layer, and reads every layer's output back into
    pinned host memory; copies and kernels are replayed as one graph (the pages
    fold the token's upload and readback into the graph as copy nodes)."""
    import numpy as np
    import torch
    from gguf_block_quant_gb300 import synth
    from gguf_block_quant_gb300 import zdmmv as Z
    w = torch.from_numpy(synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)).cuda()
    ws_ = [w] + [w.clone() for _ in range(layers - 1)]
    x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale)
    xh = torch.from_numpy(np.ascontiguousarray(np.tile(x, (layers, 1)))).pin_memory()
    yh = torch.empty(layers, cfg.rows, dtype=torch.float32).pin_memory()
    xd = torch.empty(layers, cfg.cols, dtype=torch.float32, device="cuda")
    yd = torch.empty(layers, cfg.rows, dtype=torch.float32, device="cuda")

    def step():
        xd.copy_(xh, non_blocking=True)
        for l in range(layers):
            Z.dmmv_f32(cfg.fmt, ws_[l], cfg.rows, cfg.cols, xd[l], y=yd[l])
        yh.copy_(yd, non_blocking=True)

    run = graph_or_eager(step, eager)
    ms, _ = time_fn(run, steps, warmup, world, device)
    per_step = ms / 1e3 / steps
    return {"value": layers * cfg.algorithmic_bytes() * world / per_step / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": xh.numel() * 4, "d2h_bytes_per_step": yh.numel() * 4,
            "ms_per_step": ms / steps,
            "launch": ("eager" if eager else "cuda_graph replay") +
                      ": pinned H2D of the step's activations, fused quantize + DMMV per layer, pinned D2H of the outputs"}


def e2e_host_step(cfg, layers, steps, warmup, world, device, eager=False):
    """End to end through the host-buffer C-ABI call: one zdmmv_host_step per
    layer. The buffers are page-locked, so the call moves the data without copy
    calls: its quantizer reads the layer's fp32 activation from host memory and
    its DMMV stores the layer's output into host memory."""
    import numpy as np
    import torch
    from gguf_block_quant_gb300 import synth
    from gguf_block_quant_gb300 import zdmmv as Z
    w = torch.from_numpy(synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)).cuda()
    ws_ = [w] + [w.clone() for _ in range(layers - 1)]
    x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale)
    xh = torch.from_numpy(np.ascontiguousarray(np.tile(x, (layers, 1)))).pin_memory()
    yh = torch.empty(layers, cfg.rows, dtype=torch.float32).pin_memory()
    wsb = Z.host_step_workspace_bytes(cfg.rows, cfg.cols)
    work = [torch.empty(wsb, dtype=torch.uint8, device="cuda") for _ in range(layers)]

    def step():
        for l in range(layers):
            Z.host_step(cfg.fmt, ws_[l], cfg.rows, cfg.cols, xh[l], yh[l], work[l])

    run = graph_or_eager(step, eager)
    ms, _ = time_fn(run, steps, warmup, world, device)
    per_step = ms / 1e3 / steps
    return {"value": layers * cfg.algorithmic_bytes() * world / per_step / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": xh.numel() * 4, "d2h_bytes_per_step": yh.numel() * 4,
            "ms_per_step": ms / steps,
            "launch": ("eager" if eager else "cuda_graph replay") +
                      ": zdmmv_host_step per layer (quantizer reading the layer's activation from page-locked host "
                      "memory, DMMV storing its output into page-locked host memory: host<->device traffic over the "
                      "chip-to-chip link inside the kernels, no copy calls)"}


def gpu_arm(args):
    import torch
    world, rank, local = dist_setup(args)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from gguf_block_quant_gb300 import synth
    from gguf_block_quant_gb300 import zdmmv as Z
    Z.lib()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    cfg = synth.DENSE_Q4_0
    layers = max(args.layers, layers_for(cfg, l2))
    pool = DensePool(cfg, layers)
    hbm_peak, peak_kind = peaks()

    # the DMMV kernel alone (activations pre-quantized): its average launch duration
    run_dmmv = graph_or_eager(pool.dmmv_only, args.eager)
    ms_dmmv, _ = time_fn(run_dmmv, args.steps, args.warmup, world, device)
    per_launch = ms_dmmv / 1e3 / (args.steps * layers)
    nbytes = cfg.algorithmic_bytes()
    achieved = nbytes / per_launch / 1e9

    # the two-kernel chain (quantize kernel, then DMMV kernel, per layer)
    run_unfused = graph_or_eager(pool.step_unfused, args.eager)
    ms_unfused, _ = time_fn(run_unfused, args.steps, args.warmup, world, device)

    # the headline: whole steps (fused quantize + DMMV per layer), clocks sampled meanwhile
    run_step = graph_or_eager(pool.step, args.eager)
    sampler = ClockSampler(local)
    ms, clocks = time_fn(run_step, args.steps, args.warmup, world, device, sampler)
    ms_per_step = ms / args.steps
    value = world * layers * nbytes / (ms_per_step / 1e3) / 1e9
    rows_per_s = world * layers * cfg.rows / (ms_per_step / 1e3)
    unfused_gbs = world * layers * nbytes / (ms_unfused / args.steps / 1e3) / 1e9
    del pool, run_dmmv, run_step, run_unfused
    torch.cuda.empty_cache()

    # end to end through the host-buffer C-ABI call, once per layer
    e2e = e2e_host_step(cfg, min(layers, 64), max(3, args.steps // 4), args.warmup, world, device, args.eager)
    # the same step with one bulk upload and one bulk readback around the device calls
    e2e["bulk_copies"] = e2e_dense(cfg, min(layers, 64), max(3, args.steps // 4), args.warmup, world, device,
                                   args.eager)

    workloads = {}
    if not args.no_extra:
        for c in (synth.SSM_ALPHA_BETA, synth.LM_HEAD_Q4_0, *synth.BATCHED_Q8_0.values()):
            workloads[c.name] = measure_dense(c, layers_for(c, l2), max(5, args.steps // 4), args.warmup,
                                              world, device, args.eager)
            workloads[c.name]["pct_of_peak"] = 100 * workloads[c.name]["dmmv_gbs"] / hbm_peak
            rp = measure_dense(c, layers_for(c, l2), max(5, args.steps // 4), args.warmup, world, device,
                               args.eager, layout=1)
            workloads[c.name]["repacked_layout"] = {"dmmv_gbs": rp["dmmv_gbs"], "dmmv_us": rp["dmmv_us"],
                                                    "pct_of_peak": 100 * rp["dmmv_gbs"] / hbm_peak}
        for c in (synth.DENSE_Q4_0, synth.LM_HEAD_Q4_0, synth.BATCHED_Q8_0[1]):
            xf = measure_xf32(c, layers_for(c, l2), max(5, args.steps // 4), args.warmup, world, device,
                              args.eager)
            xf["pct_of_peak"] = 100 * xf["gbs"] / hbm_peak
            workloads.setdefault(c.name, {})["xf32_activation"] = xf
        gr = measure_grouped(synth.DENSE_Q4_0, layers, max(5, args.steps // 4), args.warmup, world, device,
                             args.eager)
        gr["pct_of_peak"] = 100 * gr["gbs"] / hbm_peak
        workloads.setdefault(synth.DENSE_Q4_0.name, {})["grouped_launch"] = gr
        workloads["lm_head_q4_0_248320x2048"]["argmax_epilogue"] = measure_argmax(
            synth.LM_HEAD_Q4_0, layers_for(synth.LM_HEAD_Q4_0, l2), max(5, args.steps // 4), args.warmup, world,
            device, args.eager)
        workloads["moe_experts_top8_plus_shared"] = measure_moe(max(5, args.steps // 4), args.warmup, world,
                                                                device, args.eager, l2)

    out = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            # the oracle on all the host cores this process may use; the single-threaded run beside it
            cpu = cpu_baseline_parallel(cfg)
            cpu["single_thread"] = cpu_baseline_dense(cfg)
        traffic = recorded_traffic(cfg.name)
        traffic_dmmv = recorded_traffic(cfg.name + ":dmmv_only")
        # the step's only kernel is the fused quantize + DMMV: its average launch
        # duration inside the timed region
        per_launch_fused = ms_per_step / 1e3 / layers
        achieved_fused = nbytes / per_launch_fused / 1e9
        out = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {"workload": cfg.name, "rows": cfg.rows, "cols": cfg.cols, "format": "Q4_0", "batch": 1,
                       "layers_per_step": layers,
                       "step": "per layer: fp32 activation -> Q8_0 quantization + DMMV (fused, one launch)",
                       "l2": f"inputs larger than L2: {layers} distinct weight matrices "
                             f"({layers * cfg.weight_bytes / 1e6:.0f} MB) per step, L2 {l2 / 1e6:.0f} MB",
                       "launch": "eager" if args.eager else "cuda_graph replay", "parallelism": f"replicas x{world}"},
            "pct_of_peak": round(100 * value / world / hbm_peak, 2),
            "rows_per_s": rows_per_s,
            "roofline": {"bound": "hbm", "achieved": round(achieved_fused, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(achieved_fused / hbm_peak, 4), "traffic": traffic,
                         "kernel": "dmmv_tma_kernel with the fused Q8_0 activation quantization (Q4_0, GGUF layout)",
                         "algorithmic_bytes_per_launch": nbytes,
                         "us_per_launch": round(per_launch_fused * 1e6, 3),
                         # ncu's DRAM bytes per launch over the live launch time
                         "dram_gbs": round(traffic / per_launch_fused / 1e9, 1) if traffic else None,
                         "peak_kind": f"{peak_kind} HBM copy bandwidth",
                         "dmmv_only_chain": {
                             "kernel": "dmmv_tma_kernel over pre-quantized activation blocks",
                             "achieved": round(achieved, 1), "frac": round(achieved / hbm_peak, 4),
                             "us_per_launch": round(per_launch * 1e6, 3), "traffic": traffic_dmmv,
                             "dram_gbs": round(traffic_dmmv / per_launch / 1e9, 1) if traffic_dmmv else None}},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "two_kernel_chain_gbs": round(unfused_gbs, 2),
            "gpu_launches": layers * args.steps,
            "clocks": clocks,
            "workloads": workloads,
        }
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


# ------------------------------------------------------------ reference arm
def reference_arm(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    import multiprocessing as mp
    import numpy as np
    import oracle
    from gguf_block_quant_gb300 import synth
    cfg = synth.DENSE_Q4_0
    w = synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)
    x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale)
    oracle.lib()
    layers_per_step = 8   # a bounded sample of the 64-layer step, so K steps finish in minutes
    cores = len(os.sched_getaffinity(0))
    bounds = [cfg.rows * i // cores for i in range(cores + 1)]
    with mp.get_context("spawn").Pool(cores, initializer=_oracle_worker_init,
                                      initargs=(cfg.fmt, w.tobytes(), cfg.rows, cfg.cols)) as pool:
        def step():
            for _ in range(layers_per_step):
                xq = oracle.quantize_q8_0(x)
                y = np.empty(cfg.rows)
                for r0, part in pool.map(_oracle_worker_rows,
                                         [(bounds[i], bounds[i + 1], xq) for i in range(cores)]):
                    y[r0:r0 + len(part)] = part

        for _ in range(max(1, args.warmup)):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        el = time.perf_counter() - t0
    ms_per_step = el * 1e3 / args.steps
    value = layers_per_step * cfg.algorithmic_bytes() / (el / args.steps) / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": cfg.name, "rows": cfg.rows, "cols": cfg.cols, "format": "Q4_0", "batch": 1,
                   "layers_per_step": layers_per_step, "step": "quantize_act_q8_0 + DMMV per layer"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{layers_per_step} layers per step of {cfg.name}, C oracle with the rows "
                                   f"split over {cores} worker processes"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def profile_mode(name: str):
    """A handful of untimed launches on a small pool (4 layers): the two-kernel
    chain once to fill the activation blocks, then 3 x (fused step, two-kernel
    step). Meant to run under ncu with a kernel filter and a launch count."""
    import torch
    from gguf_block_quant_gb300 import synth
    from gguf_block_quant_gb300 import zdmmv as Z
    Z.lib()
    if name == synth.MOE.name:
        # the MoE step three ways, 3 times: gate/up+SwiGLU, quantize h, down gather; then the one-launch FFN
        m = synth.MOE
        gate = torch.from_numpy(synth.weight_blocks(synth.Q4_0, m.n_slots * m.ffn, m.hidden, seed=m.seed)).cuda()
        up = torch.from_numpy(synth.weight_blocks(synth.Q4_0, m.n_slots * m.ffn, m.hidden, seed=m.seed,
                                                  stream=synth.S_WEIGHT2)).cuda()
        down = torch.from_numpy(synth.weight_blocks(synth.Q8_0, m.n_slots * m.hidden, m.ffn, seed=m.seed,
                                                    stream=synth.S_WEIGHT3)).cuda()
        idx = torch.from_numpy(synth.expert_indices(m.seed, m.n_routed, m.top_k)).cuda()
        xq = Z.quantize_act_q8_0(torch.from_numpy(synth.activations(m.hidden, seed=m.seed)).cuda())
        gu, dn = m.gate_up_bytes(), m.down_bytes()
        ws = Z.expert_ffn_workspace(m.n_sel, m.ffn)
        for _ in range(3):
            h = Z.expert_swiglu(Z.Q4_0, gate, up, m.ffn, m.hidden, xq, idx=idx, expert_stride=gu,
                                n_experts=m.n_slots)
            hq = Z.quantize_act_q8_0(h.reshape(-1))
            Z.expert_gather(Z.Q8_0, down, dn, m.hidden, m.ffn, idx, m.n_slots, hq, (m.ffn // 32) * 34)
            Z.expert_ffn(Z.Q4_0, gate, up, gu, Z.Q8_0, down, dn, m.hidden, m.ffn, idx, m.n_slots, xq, workspace=ws)
        torch.cuda.synchronize()
        print(json.dumps({"profile": name, "fault": Z.device_status()}))
        return
    workloads = {c.name: c for c in (synth.SSM_ALPHA_BETA, synth.DENSE_Q4_0, synth.LM_HEAD_Q4_0,
                                     *synth.BATCHED_Q8_0.values())}
    # "<workload>:xf32": the DMMV with the fp32 activation taken as is, 3 x 4 layers
    xf32 = name.endswith(":xf32")
    cfg = workloads[name[: -len(":xf32")] if xf32 else name]
    pool = DensePool(cfg, 4)
    for _ in range(3):
        if xf32:
            for l in range(4):
                Z.dmmv_xf32(cfg.fmt, pool.w[l], cfg.rows, cfg.cols, pool.x[l], batch=cfg.batch, y=pool.y[l])
        else:
            pool.step()
            pool.step_unfused()
    torch.cuda.synchronize()
    print(json.dumps({"profile": name, "layers": 4, "fault": Z.device_status()}))


def main():
    args = parse()
    if args.profile:
        profile_mode(args.profile)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
