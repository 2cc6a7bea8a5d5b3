#!/usr/bin/env python3
"""Benchmark of the GGUF Q4_0 / Q8_0 decode DMMV on GB300.

Headline workload: the LM head (vocab projection), Q4_0 248320 x 2048 (286 MB of
weights), batch 1. One STEP is one decode token's projection: the token's fp32
activation is quantized to Q8_0 and multiplied by the matrix (fused in one
launch), producing 248320 fp32 logits. Steps alternate over LM_HEAD_COPIES
distinct copies of the matrix (together more than 4x the 129 MB L2), so every
step streams its weights from HBM. Inputs are resident in HBM before the timed
region; the K timed steps are captured once in a CUDA graph and replayed (decode
chains are replayed as graphs: "RTX 5090: Batched Prefill & CUDA Graphs in
ZINC", "CUDA graphs -- the structural answer to launch latency"). The vocab
projection is the pages' bandwidth showcase (habr ZINC article, "Утилизация
полосы памяти по операциям").

Printed: ONE compact JSON line on stdout (rank 0): value = algorithmic GB/s
over the whole job (weights read once + Q8_0 activation blocks + fp32 logits),
the roofline of the step's kernel against the measured HBM copy bandwidth, the
CPU oracle as baseline, the end-to-end number through the host-buffer C-ABI
call, clocks sampled during the timed region, and a `summary` of every other
workload ([microseconds, % of the copy peak] per variant). The full per-workload
detail goes to stderr as one more JSON line prefixed "detail: ".

--impl reference times the CPU oracle on the same workload, config and metric:
with no upstream code to run, the oracle is the reference implementation of the
method.
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
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["zdmmv", "reference"], default="zdmmv")
    p.add_argument("--layers", type=int, default=64, help="distinct weight matrices per step of the dense chain")
    p.add_argument("--no-extra", action="store_true", help="skip the other workloads")
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
# The oracle over row ranges in worker processes (spawned, never forked: the
# parent may already hold a CUDA context). The matrix lives once in a shared
# memory segment that every worker maps.
_ORACLE_W = None


def _oracle_worker_init(fmt, shm_name, rows, row_bytes, cols):
    global _ORACLE_W
    from multiprocessing import shared_memory
    import numpy as np
    import oracle
    oracle.lib()
    shm = shared_memory.SharedMemory(name=shm_name)
    _ORACLE_W = (fmt, np.ndarray((rows, row_bytes), dtype=np.uint8, buffer=shm.buf), cols, shm)


def _oracle_worker_rows(task):
    import oracle
    r0, r1, xq = task
    fmt, w, cols, _ = _ORACLE_W
    y, _ = oracle.dmmv(fmt, w[r0:r1], r1 - r0, cols, xq)
    return r0, y


class OracleStep:
    """One step of a Dense workload on the CPU oracle, unchanged: quantize the
    activation (oracle.quantize_q8_0), then the oracle DMMV with the rows split
    over `workers` spawned processes (1: in this process). The per-row arithmetic
    does not depend on the split, so every split gives the same bits."""

    def __init__(self, cfg, workers: int):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        import numpy as np
        import oracle
        from gguf_block_quant_gb300 import synth
        oracle.lib()
        self.cfg, self.workers = cfg, workers
        w = synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)
        self.x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale)
        self.pool = None
        if workers == 1:
            self.w = w
            return
        row_bytes = cfg.nb * synth.BLOCK_BYTES[cfg.fmt]
        self.shm = shared_memory.SharedMemory(create=True, size=w.nbytes)
        self.w = np.ndarray(w.shape, dtype=np.uint8, buffer=self.shm.buf)
        self.w[:] = w
        del w
        self.bounds = [cfg.rows * i // workers for i in range(workers + 1)]
        self.pool = mp.get_context("spawn").Pool(workers, initializer=_oracle_worker_init,
                                                 initargs=(cfg.fmt, self.shm.name, cfg.rows, row_bytes, cfg.cols))

    def __call__(self):
        import numpy as np
        import oracle
        c = self.cfg
        xq = oracle.quantize_q8_0(self.x)
        if self.pool is None:
            y, _ = oracle.dmmv(c.fmt, self.w, c.rows, c.cols, xq)
            return y
        y = np.empty(c.rows)
        tasks = [(self.bounds[i], self.bounds[i + 1], xq) for i in range(self.workers)]
        for r0, part in self.pool.map(_oracle_worker_rows, tasks):
            y[r0:r0 + len(part)] = part
        return y

    def close(self):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()
            self.w = None
            self.shm.close()
            self.shm.unlink()
            self.pool = None


def cpu_baseline(cfg, budget_s: float = 12.0):
    """Time the oracle (as it stands) on a bounded sample of the workload: whole
    steps (quantize + DMMV of the full matrix) until about budget_s of CPU time,
    with the rows split over one spawned worker per core this process may use;
    the same on one thread beside it. The parallel result is checked bit for bit
    against the single-threaded one."""
    import numpy as np
    cores = len(os.sched_getaffinity(0))
    out = {}
    for workers in dict.fromkeys((cores, 1)):
        step = OracleStep(cfg, workers)
        try:
            y = step()   # workers started and warm
            if "y" in out and not np.array_equal(y, out["y"]):
                raise RuntimeError("parallel oracle disagrees with the single-threaded oracle")
            out["y"] = y
            done, t0 = 0, time.perf_counter()
            while True:
                step()
                done += 1
                el = time.perf_counter() - t0
                if el >= budget_s or done >= 20000:
                    break
        finally:
            step.close()
        out[workers] = {"value": round(done * cfg.algorithmic_bytes() / el / 1e9, 3), "unit": "GB/s",
                        "cores": workers, "kind": "oracle",
                        "sample": f"{done} whole steps (quantize + DMMV) in {el:.1f} s"
                                  + (f", rows over {workers} processes" if workers > 1 else ", one thread"),
                        "rows_per_s": round(done * cfg.rows / el)}
    res = out[cores]
    res["single_thread"] = out[1]
    return res


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


MOE_LAYERS = 40   # the pages' 35B-A3B model: 40 layers, each with its own experts


def measure_moe(steps, warmup, world, device, eager, l2_bytes):
    """Config: 9 selected experts (8 routed + shared) of a 129-slot stack; one
    step = gate, up (Q4_0 512x2048) and down (Q8_0 2048x512) gathers over
    MOE_LAYERS layers, each layer with its OWN stacks (296 MB per layer) and its
    own routing, like a decode token. Between two reads of any expert (the shared
    slot included) the step touches every other layer's experts, MOE_LAYERS x
    20.6 MB, more than 4x L2, so every read comes from HBM."""
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
    layers = MOE_LAYERS
    stacks = [(gate, up, down)] + [(gate.clone(), up.clone(), down.clone()) for _ in range(layers - 1)]
    idxs = [torch.from_numpy(synth.expert_indices(m.seed + 100 * l, m.n_routed, m.top_k)).cuda()
            for l in range(layers)]
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
    touched = m.n_sel * (2 * gu + dn)

    # The first call of a layer reads the layer's index list after its dependency
    # wait (the router would write it just before); later calls of the same
    # selection read it at once (zdmmv_expert_gather_ready) and stream their
    # weights during the previous launch.
    def step3():
        for l in range(layers):
            g, u, d = stacks[l]
            idx = idxs[l]
            Z.expert_gather(Z.Q4_0, g, gu, m.ffn, m.hidden, idx, m.n_slots, xq, 0, y=yg, status=st)
            Z.expert_gather(Z.Q4_0, u, gu, m.ffn, m.hidden, idx, m.n_slots, xq, 0, y=yu, status=st,
                            idx_ready=True)
            Z.expert_gather(Z.Q8_0, d, dn, m.hidden, m.ffn, idx, m.n_slots, xqd, (m.ffn // 32) * 34, y=yd,
                            status=st, idx_ready=True)

    def step2():
        for l in range(layers):
            g, u, d = stacks[l]
            idx = idxs[l]
            Z.expert_gather2(Z.Q4_0, g, u, gu, m.ffn, m.hidden, idx, m.n_slots, xq, 0, y_a=yg, y_b=yu, status=st)
            Z.expert_gather(Z.Q8_0, d, dn, m.hidden, m.ffn, idx, m.n_slots, xqd, (m.ffn // 32) * 34, y=yd,
                            status=st, idx_ready=True)

    h = torch.empty(m.n_sel, m.ffn, device="cuda")

    def step_swiglu():
        for l in range(layers):
            g, u, d = stacks[l]
            idx = idxs[l]
            Z.expert_swiglu(Z.Q4_0, g, u, m.ffn, m.hidden, xq, idx=idx, expert_stride=gu, n_experts=m.n_slots,
                            h=h, status=st)
            Z.expert_gather(Z.Q8_0, d, dn, m.hidden, m.ffn, idx, m.n_slots, xqd, (m.ffn // 32) * 34, y=yd,
                            status=st, idx_ready=True)

    hq = torch.empty(m.n_sel * (m.ffn // 32) * 34, dtype=torch.uint8, device="cuda")

    def step_chain():
        # the same FFN through separate launches: SwiGLU, quantize h, down gather of h
        # (the down gather waits for its indices: behind the quantizer the ready
        # gather measured no faster, 9.31 against 9.32 us per token-layer)
        for l in range(layers):
            g, u, d = stacks[l]
            idx = idxs[l]
            Z.expert_swiglu(Z.Q4_0, g, u, m.ffn, m.hidden, xq, idx=idx, expert_stride=gu, n_experts=m.n_slots,
                            h=h, status=st)
            Z.quantize_act_q8_0(h.reshape(-1), hq)
            Z.expert_gather(Z.Q8_0, d, dn, m.hidden, m.ffn, idx, m.n_slots, hq, (m.ffn // 32) * 34, y=yd,
                            status=st)

    def step_ffn2():
        # the same FFN in two launches: SwiGLU, then the down gather of h (fp32,
        # quantized in the gather's prologue), which reads its indices at once
        for l in range(layers):
            g, u, d = stacks[l]
            idx = idxs[l]
            Z.expert_swiglu(Z.Q4_0, g, u, m.ffn, m.hidden, xq, idx=idx, expert_stride=gu, n_experts=m.n_slots,
                            h=h, status=st)
            Z.expert_gather_f32(Z.Q8_0, d, dn, m.hidden, m.ffn, idx, m.n_slots, h, m.ffn, y=yd, status=st,
                                idx_ready=True)

    ws = Z.expert_ffn_workspace(m.n_sel, m.ffn)

    def step_ffn():
        for l in range(layers):
            g, u, d = stacks[l]
            Z.expert_ffn(Z.Q4_0, g, u, gu, Z.Q8_0, d, dn, m.hidden, m.ffn, idxs[l], m.n_slots, xq, y=yd,
                         workspace=ws, status=st)

    nbytes = m.algorithmic_bytes()
    # the SwiGLU epilogue writes h instead of the gate and up outputs
    nbytes_swiglu = nbytes - m.n_sel * m.ffn * 4
    out = {"layers": layers, "algorithmic_bytes": nbytes,
           "reuse_distance_bytes": layers * touched, "l2_bytes": l2_bytes,
           "note": f"{layers} layers, each with its own 129-slot stacks and routing: "
                   f"{layers * touched / 1e6:.0f} MB touched between two reads of any expert"}
    for name, fn, launches, nb_ in (("three_launch", step3, 3, nbytes), ("gate_up_fused", step2, 2, nbytes),
                                    ("gate_up_swiglu", step_swiglu, 2, nbytes_swiglu),
                                    ("ffn_chained_three_launch", step_chain, 3, nbytes_swiglu),
                                    ("ffn_chained_two_launch", step_ffn2, 2, nbytes_swiglu),
                                    ("ffn_one_launch", step_ffn, 1, nbytes_swiglu)):
        run = graph_or_eager(fn, eager)
        ms, _ = time_fn(run, steps, warmup, world, device)
        per_layer = ms / 1e3 / (steps * layers)
        out[name] = {"us_per_token_layer": per_layer * 1e6, "gbs": nb_ / per_layer / 1e9,
                     "algorithmic_bytes": nb_,
                     "rows_per_s": m.n_sel * (2 * m.ffn + m.hidden) / per_layer, "launches_per_layer": launches}
        del run
    out["ffn_one_launch"]["note"] = ("gate/up + SwiGLU and the down DMMV of the quantized SwiGLU output in one "
                                     "launch (the down input is h, not the independent activation)")
    out["ffn_chained_three_launch"]["note"] = "the same chained FFN as SwiGLU, quantize h, down gather"
    out["ffn_chained_two_launch"]["note"] = ("the same chained FFN as SwiGLU, then the down gather of the fp32 h "
                                             "(quantized in its prologue; indices read at once)")
    for k in ("three_launch", "gate_up_fused", "gate_up_swiglu"):
        out[k]["note"] = ("the calls after a layer's first read its index list at once "
                          "(zdmmv_expert_gather_ready) and stream their weights during the previous launch")
    if Z.device_status() != 0 or int(st.item()) != 0:
        raise RuntimeError("MoE measurement: the device reported a fault or a bad expert index")
    del stacks, gate, up, down
    torch.cuda.empty_cache()
    return out


def run_step_sequence(step_fn, k: int, w: int, world: int, device, eager: bool, sampler=None):
    """Time EXACTLY k steps: step_fn(i) issues step i on the current stream.
    The w warm-up steps and the k timed steps are each captured in one CUDA
    graph (or issued eagerly with eager=True); the timed region, bracketed by a
    barrier and a synchronize on both sides, is one replay of the k-step graph,
    timed with CUDA events on the launching stream. Returns (ms, clocks), ms the
    max over ranks."""
    import torch

    def seq(n, base):
        def f():
            for i in range(n):
                step_fn(base + i)
        return f

    warm = graph_or_eager(seq(max(w, 1), 0), eager)
    timed = graph_or_eager(seq(k, max(w, 1)), eager)
    warm()
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
    timed()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier(world)
    return reduce_max(e0.elapsed_time(e1), world, device), clocks


LM_HEAD_COPIES = 3   # 3 x 286 MB = 859 MB of distinct weights, more than 4x the 129 MB L2


def headline_config(cfg, copies: int) -> dict:
    """The headline workload's config, identical in both arms."""
    return {"workload": cfg.name, "rows": cfg.rows, "cols": cfg.cols, "format": "Q4_0", "batch": 1,
            "step": "one decode token's vocab projection: fp32 activation -> Q8_0 quantization + DMMV "
                    "(one fused launch) -> fp32 logits",
            "l2": f"inputs larger than L2: each step streams a {cfg.weight_bytes / 1e6:.0f} MB matrix; steps "
                  f"alternate over {copies} distinct copies ({copies * cfg.weight_bytes / 1e6:.0f} MB, more than "
                  f"4x the 129 MB L2)",
            "parallelism": "replicas (one independent problem per GPU)"}


def e2e_host_step(cfg, copies, k, w, world, device, eager=False):
    """End to end through the host-buffer C-ABI call, one zdmmv_host_step per
    step (step i on copy i % copies). The host buffers are page-locked, so the
    call moves the data without copy calls: its quantizer reads the step's fp32
    activation from host memory and its DMMV stores the step's output into host
    memory."""
    import numpy as np
    import torch
    from gguf_block_quant_gb300 import synth
    from gguf_block_quant_gb300 import zdmmv as Z
    wt = torch.from_numpy(synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)).cuda()
    ws_ = [wt] + [wt.clone() for _ in range(copies - 1)]
    x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale)
    xh = torch.from_numpy(np.ascontiguousarray(np.tile(x, (copies, 1)))).pin_memory()
    yh = torch.empty(copies, cfg.rows, dtype=torch.float32).pin_memory()
    wsb = Z.host_step_workspace_bytes(cfg.rows, cfg.cols)
    work = [torch.empty(wsb, dtype=torch.uint8, device="cuda") for _ in range(copies)]

    def step(i):
        c = i % copies
        Z.host_step(cfg.fmt, ws_[c], cfg.rows, cfg.cols, xh[c], yh[c], work[c])

    ms, _ = run_step_sequence(step, k, w, world, device, eager)
    per_step = ms / 1e3 / k
    out = {"value": round(cfg.algorithmic_bytes() * world / per_step / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": cfg.cols * 4, "d2h_bytes_per_step": cfg.rows * 4,
           "ms_per_step": round(ms / k, 5),
           "launch": ("eager" if eager else "graph") +
                     " of zdmmv_host_step calls; page-locked x and y read/written by the kernels"}
    del ws_, wt, work
    torch.cuda.empty_cache()
    return out


def e2e_bulk_copies(cfg, copies, k, w, world, device, eager=False):
    """The same step with explicit copies: a pinned H2D copy of the step's fp32
    activation, the fused quantize + DMMV, a pinned D2H copy of the outputs."""
    import numpy as np
    import torch
    from gguf_block_quant_gb300 import synth
    from gguf_block_quant_gb300 import zdmmv as Z
    wt = torch.from_numpy(synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)).cuda()
    ws_ = [wt] + [wt.clone() for _ in range(copies - 1)]
    x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale)
    xh = torch.from_numpy(np.ascontiguousarray(np.tile(x, (copies, 1)))).pin_memory()
    yh = torch.empty(copies, cfg.rows, dtype=torch.float32).pin_memory()
    xd = torch.empty(copies, cfg.cols, dtype=torch.float32, device="cuda")
    yd = torch.empty(copies, cfg.rows, dtype=torch.float32, device="cuda")

    def step(i):
        c = i % copies
        xd[c].copy_(xh[c], non_blocking=True)
        Z.dmmv_f32(cfg.fmt, ws_[c], cfg.rows, cfg.cols, xd[c], y=yd[c])
        yh[c].copy_(yd[c], non_blocking=True)

    ms, _ = run_step_sequence(step, k, w, world, device, eager)
    per_step = ms / 1e3 / k
    del ws_, wt
    torch.cuda.empty_cache()
    return {"value": round(cfg.algorithmic_bytes() * world / per_step / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms / k, 5)}


def pair(us: float, gbs: float, peak: float):
    """[microseconds, % of the copy peak] for the compact summary."""
    return [round(us, 2), round(100 * gbs / peak, 1)]


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
    hbm_peak, peak_kind = peaks()
    cfg = synth.LM_HEAD_Q4_0
    copies = max(LM_HEAD_COPIES, layers_for(cfg, l2))
    nbytes = cfg.algorithmic_bytes()
    K, W = args.steps, max(args.warmup, 1)

    # ------------------------------------------------ the headline: LM-head tokens
    pool = DensePool(cfg, copies)

    def fused_step(i):
        c = i % copies
        Z.dmmv_f32(cfg.fmt, pool.w[c], cfg.rows, cfg.cols, pool.x[c], y=pool.y[c])

    def dmmv_step(i):
        c = i % copies
        Z.dmmv(cfg.fmt, pool.w[c], cfg.rows, cfg.cols, pool.xq[c], y=pool.y[c])

    def two_kernel_step(i):
        c = i % copies
        Z.quantize_act_q8_0(pool.x[c], pool.xq[c])
        Z.dmmv(cfg.fmt, pool.w[c], cfg.rows, cfg.cols, pool.xq[c], y=pool.y[c])

    sampler = ClockSampler(local)
    ms, clocks = run_step_sequence(fused_step, K, W, world, device, args.eager, sampler)
    ms_dmmv, _ = run_step_sequence(dmmv_step, K, W, world, device, args.eager)
    ms_two, _ = run_step_sequence(two_kernel_step, K, W, world, device, args.eager)
    if Z.device_status() != 0:
        raise RuntimeError("the device reported a fault during the headline")
    del pool
    torch.cuda.empty_cache()
    ms_per_step = ms / K
    per_launch = ms_per_step / 1e3          # one launch per step
    achieved = nbytes / per_launch / 1e9
    value = world * nbytes / per_launch / 1e9
    detail = {"headline": {"fused_us": per_launch * 1e6, "dmmv_only_us": ms_dmmv / K * 1e3,
                           "two_kernel_us_per_step": ms_two / K * 1e3, "copies": copies, "l2_bytes": l2}}

    # ------------------------------------ end to end through the host-buffer call
    e2e = e2e_host_step(cfg, copies, K, W, world, device, args.eager)
    bulk = e2e_bulk_copies(cfg, copies, K, W, world, device, args.eager)
    e2e["bulk_copies_gbs"] = bulk["value"]

    # ------------------------------------------------------------ other workloads
    summary = {"unit": "[us (MoE: per token-layer), % of copy peak]",
               cfg.name: {"fused": pair(per_launch * 1e6, achieved, hbm_peak),
                          "dmmv": pair(ms_dmmv / K * 1e3, nbytes / (ms_dmmv / K / 1e3) / 1e9, hbm_peak),
                          "two_kernel": pair(ms_two / K * 1e3, nbytes / (ms_two / K / 1e3) / 1e9, hbm_peak)}}
    if not args.no_extra:
        ns = max(5, K // 4)
        lm = summary[cfg.name]
        rp = measure_dense(cfg, copies, ns, W, world, device, args.eager, layout=1)
        lm["repacked"] = pair(rp["dmmv_us"], rp["dmmv_gbs"], hbm_peak)
        am = measure_argmax(cfg, copies, ns, W, world, device, args.eager)
        lm["argmax"] = pair(am["us"], am["gbs"], hbm_peak)
        xf = measure_xf32(cfg, copies, ns, W, world, device, args.eager)
        lm["xf32"] = pair(xf["us"], xf["gbs"], hbm_peak)
        detail[cfg.name] = {"repacked_layout": rp, "argmax_epilogue": am, "xf32_activation": xf}

        d = synth.DENSE_Q4_0
        dl = max(args.layers, layers_for(d, l2))
        dn = measure_dense(d, dl, ns, W, world, device, args.eager)
        gr = measure_grouped(d, dl, ns, W, world, device, args.eager)
        dx = measure_xf32(d, dl, ns, W, world, device, args.eager)
        summary[d.name] = {"fused_chain": pair(dn["fused_us_per_layer"], dn["fused_step_gbs"], hbm_peak),
                           "dmmv_chain": pair(dn["dmmv_us"], dn["dmmv_gbs"], hbm_peak),
                           "two_kernel_chain": pair(d.algorithmic_bytes() / dn["two_kernel_step_gbs"] / 1e3,
                                                    dn["two_kernel_step_gbs"], hbm_peak),
                           f"grouped_{dl}": pair(gr["us_per_matrix"], gr["gbs"], hbm_peak),
                           "xf32_chain": pair(dx["us"], dx["gbs"], hbm_peak)}
        detail[d.name] = {"chain": dn, "grouped_launch": gr, "xf32_activation": dx}

        c = synth.SSM_ALPHA_BETA
        sm = measure_dense(c, layers_for(c, l2), ns, W, world, device, args.eager)
        summary[c.name] = {"dmmv_chain": pair(sm["dmmv_us"], sm["dmmv_gbs"], hbm_peak),
                           "fused_chain": pair(sm["fused_us_per_layer"], sm["fused_step_gbs"], hbm_peak)}
        detail[c.name] = sm

        bsum, bdet = {}, {}
        for b, c in synth.BATCHED_Q8_0.items():
            r = measure_dense(c, layers_for(c, l2), ns, W, world, device, args.eager)
            rp = measure_dense(c, layers_for(c, l2), ns, W, world, device, args.eager, layout=1)
            bsum[f"b{b}"] = pair(r["dmmv_us"], r["dmmv_gbs"], hbm_peak)
            bsum[f"b{b}_repacked"] = pair(rp["dmmv_us"], rp["dmmv_gbs"], hbm_peak)
            bsum[f"b{b}_fused"] = pair(r["fused_us_per_layer"], r["fused_step_gbs"], hbm_peak)
            bdet[c.name] = {"gguf": r, "repacked": rp}
        c = synth.BATCHED_Q8_0[1]
        bx = measure_xf32(c, layers_for(c, l2), ns, W, world, device, args.eager)
        bsum["b1_xf32"] = pair(bx["us"], bx["gbs"], hbm_peak)
        bdet["xf32_b1"] = bx
        summary["batched_q8_0_14336x4096"] = bsum
        detail["batched_q8_0_14336x4096"] = bdet

        moe = measure_moe(ns, W, world, device, args.eager, l2)
        summary["moe_experts_top8_plus_shared"] = {
            k: pair(moe[k]["us_per_token_layer"], moe[k]["gbs"], hbm_peak)
            for k in ("three_launch", "gate_up_fused", "gate_up_swiglu", "ffn_chained_three_launch",
                      "ffn_chained_two_launch", "ffn_one_launch")}
        detail["moe_experts_top8_plus_shared"] = moe
    if Z.device_status() != 0:
        raise RuntimeError("the device reported a fault during the measurements")

    out = None
    if rank == 0:
        cpu = None if args.no_cpu_baseline else cpu_baseline(cfg)
        if cpu is not None:
            cpu.pop("y", None)
        traffic = recorded_traffic(cfg.name)
        out = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": headline_config(cfg, copies),
            "pct_of_peak": round(100 * achieved / hbm_peak, 2),
            "rows_per_s": round(world * cfg.rows / per_launch),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                         "kernel": "dmmv_tma_kernel (fused Q8_0 quantization)",
                         "algorithmic_bytes_per_launch": nbytes, "us_per_launch": round(per_launch * 1e6, 3),
                         "dram_gbs": round(traffic / per_launch / 1e9, 1) if traffic else None,
                         "peak_kind": f"{peak_kind} HBM copy bandwidth"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": K,
            "clocks": clocks,
            "summary": summary,
        }
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if out is not None:
        print("detail: " + json.dumps(detail), file=sys.stderr, flush=True)
        print(json.dumps(out, separators=(",", ":")), flush=True)


# ------------------------------------------------------------ reference arm
def reference_arm(args):
    """The CPU oracle on the headline's workload and config: each step is one
    whole LM-head token (quantize + DMMV over all 248320 rows), rows split over
    one spawned worker per host core. Rank 0 only."""
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    from gguf_block_quant_gb300 import synth
    cfg = synth.LM_HEAD_Q4_0
    cores = len(os.sched_getaffinity(0))
    step = OracleStep(cfg, cores)
    try:
        for _ in range(max(1, args.warmup)):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        el = time.perf_counter() - t0
    finally:
        step.close()
    ms_per_step = el * 1e3 / args.steps
    value = cfg.algorithmic_bytes() / (el / args.steps) / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": headline_config(cfg, LM_HEAD_COPIES),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} whole steps of {cfg.name} (quantize + DMMV), C oracle with the "
                                   f"rows split over {cores} worker processes"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }, separators=(",", ":")), flush=True)


def profile_mode(name: str):
    """A handful of untimed launches on a small pool (4 layers): the two-kernel
    chain once to fill the activation blocks, then 3 x (fused step, two-kernel
    step). Meant to run under ncu with a kernel filter and a launch count."""
    import torch
    from gguf_block_quant_gb300 import synth
    from gguf_block_quant_gb300 import zdmmv as Z
    Z.lib()
    if name == synth.MOE.name:
        # the MoE FFN three ways, 3 times: gate/up+SwiGLU, quantize h, down gather; the one-launch FFN;
        # gate/up+SwiGLU, then the down gather of the fp32 h (indices read at once)
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
            h2 = Z.expert_swiglu(Z.Q4_0, gate, up, m.ffn, m.hidden, xq, idx=idx, expert_stride=gu,
                                 n_experts=m.n_slots)
            Z.expert_gather_f32(Z.Q8_0, down, dn, m.hidden, m.ffn, idx, m.n_slots, h2, m.ffn, idx_ready=True)
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
