"""Seeded synthetic inputs for the GGUF Q8_0 / Q4_0 decode DMMV.

This module only DRAWS inputs: random quantized weight blocks, random fp32
activations, random pre-quantized activation blocks and expert indices. It holds
none of the method's arithmetic (no quantization, no dot products, no scaling),
so the CUDA path and the CPU oracle can both be fed from it without sharing any
computation. numpy only; no torch, no CUDA.

Workloads (shapes and distributions of the pages' decode workload; model weights
are not available, so every tensor is synthetic):
  * ssm_alpha_beta_q8_0   Q8_0 64 x 2048, batch 1 (32 alpha + 32 beta rows),
                          int8 U[-127,127], fp16 scales U[1e-3,1e-2], x ~ N(0,1)
  * dense_q4_0            Q4_0 4096 x 4096, batch 1, nibbles U{0..15}, same scales
  * lm_head_q4_0          Q4_0 248320 x 2048 (vocab projection), batch 1, x ~ 0.1*N(0,1)
  * moe_experts           128 routed experts + 1 shared: gate/up Q4_0 512 x 2048,
                          down Q8_0 2048 x 512; 8 distinct routed indices + the shared one
  * batched_q8_0          Q8_0 14336 x 4096 with 1, 2, 4 or 8 activation vectors
Seeds: workload i uses seed i with one PCG64 sub-stream per tensor.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

QK = 32
Q4_0 = 2
Q8_0 = 8
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34}

# sub-stream ids (one per tensor kind) so that tensors of one workload are independent
S_WEIGHT, S_ACT, S_ACT_BLOCKS, S_INDEX, S_WEIGHT2, S_WEIGHT3, S_ACT2 = range(7)


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def _scales_f16(g: np.random.Generator, n: int, lo: float, hi: float) -> np.ndarray:
    return g.uniform(lo, hi, size=n).astype(np.float16)


def weight_blocks(fmt: int, rows: int, cols: int, seed: int, stream: int = S_WEIGHT,
                  scale_lo: float = 1e-3, scale_hi: float = 1e-2) -> np.ndarray:
    """Random GGUF-layout weight matrix [rows][cols/32 blocks] as flat uint8 bytes.

    Q8_0: quants int8 uniform in [-127, 127]; Q4_0: every 4-bit value uniform in
    {0..15} (so every quant byte is uniform in 0..255); scales fp16 uniform in
    [scale_lo, scale_hi]."""
    if cols % QK:
        raise ValueError("cols must be a multiple of 32")
    g = rng(seed, stream)
    n = rows * (cols // QK)
    if fmt == Q8_0:
        dt = np.dtype([("d", "<f2"), ("qs", "i1", (32,))])
        blk = np.empty(n, dtype=dt)
        blk["d"] = _scales_f16(g, n, scale_lo, scale_hi)
        blk["qs"] = g.integers(-127, 127, size=(n, 32), dtype=np.int8, endpoint=True)
    elif fmt == Q4_0:
        dt = np.dtype([("d", "<f2"), ("qs", "u1", (16,))])
        blk = np.empty(n, dtype=dt)
        blk["d"] = _scales_f16(g, n, scale_lo, scale_hi)
        blk["qs"] = g.integers(0, 255, size=(n, 16), dtype=np.uint8, endpoint=True)
    else:
        raise ValueError(f"unknown format {fmt}")
    assert dt.itemsize == BLOCK_BYTES[fmt]
    return blk.view(np.uint8).reshape(-1)


def weight_blocks_small(fmt: int, rows: int, cols: int, seed: int, qmax: int,
                        scale: float = 1.0, stream: int = S_WEIGHT) -> np.ndarray:
    """Weight blocks with small integer values and one fixed scale, for tests in
    which every fp32 partial sum of the DMMV is an exact integer. Q8_0 quants are
    uniform in [-qmax, qmax]; Q4_0 4-bit values are uniform in [8-qmax, 8+qmax-1]
    clipped to {0..15}."""
    g = rng(seed, stream)
    n = rows * (cols // QK)
    if fmt == Q8_0:
        dt = np.dtype([("d", "<f2"), ("qs", "i1", (32,))])
        blk = np.empty(n, dtype=dt)
        blk["d"] = np.float16(scale)
        blk["qs"] = g.integers(-qmax, qmax + 1, size=(n, 32)).astype(np.int8)
    elif fmt == Q4_0:
        dt = np.dtype([("d", "<f2"), ("qs", "u1", (16,))])
        blk = np.empty(n, dtype=dt)
        blk["d"] = np.float16(scale)
        lo = g.integers(max(0, 8 - qmax), min(16, 8 + qmax), size=(n, 16))
        hi = g.integers(max(0, 8 - qmax), min(16, 8 + qmax), size=(n, 16))
        blk["qs"] = (lo | (hi << 4)).astype(np.uint8)
    else:
        raise ValueError(f"unknown format {fmt}")
    return blk.view(np.uint8).reshape(-1)


def activations(k: int, seed: int, stream: int = S_ACT, scale: float = 1.0,
                batch: int = 1) -> np.ndarray:
    """fp32 activations ~ scale * N(0, 1), shape [batch, k] (or [k] for batch 1)."""
    g = rng(seed, stream)
    x = (g.standard_normal(size=(batch, k)) * scale).astype(np.float32)
    return x[0] if batch == 1 else x


def activation_blocks(nblocks: int, seed: int, stream: int = S_ACT_BLOCKS,
                      qmax: int = 127, scale_lo: float = 1e-3,
                      scale_hi: float = 1e-2, fixed_scale: float | None = None) -> np.ndarray:
    """Random pre-quantized Q8_0 activation blocks (flat uint8), drawn directly
    (not produced by any quantizer): int8 uniform in [-qmax, qmax], fp16 scale
    uniform in [scale_lo, scale_hi] or equal to fixed_scale."""
    g = rng(seed, stream)
    dt = np.dtype([("d", "<f2"), ("qs", "i1", (32,))])
    blk = np.empty(nblocks, dtype=dt)
    if fixed_scale is None:
        blk["d"] = _scales_f16(g, nblocks, scale_lo, scale_hi)
    else:
        blk["d"] = np.float16(fixed_scale)
    blk["qs"] = g.integers(-qmax, qmax + 1, size=(nblocks, 32)).astype(np.int8)
    return blk.view(np.uint8).reshape(-1)


def extreme_code_blocks(fmt: int, nblocks: int, seed: int, stream: int = S_ACT_BLOCKS) -> np.ndarray:
    """Blocks whose codes take only their format's extreme values, scale 1.0:
    Q8_0 codes in {-128, 127}, Q4_0 4-bit values in {0, 15}. With few blocks per
    row every fp32 partial sum of a DMMV is still an exact integer, while every
    product is as large as the format allows."""
    g = rng(seed, stream)
    if fmt == Q8_0:
        blk = np.empty(nblocks, dtype=np.dtype([("d", "<f2"), ("qs", "i1", (32,))]))
        blk["qs"] = np.where(g.integers(0, 2, size=(nblocks, 32)) == 1, 127, -128).astype(np.int8)
    elif fmt == Q4_0:
        blk = np.empty(nblocks, dtype=np.dtype([("d", "<f2"), ("qs", "u1", (16,))]))
        lo = np.where(g.integers(0, 2, size=(nblocks, 16)) == 1, 15, 0)
        hi = np.where(g.integers(0, 2, size=(nblocks, 16)) == 1, 15, 0)
        blk["qs"] = (lo | (hi << 4)).astype(np.uint8)
    else:
        raise ValueError(f"unknown format {fmt}")
    blk["d"] = np.float16(1.0)
    return blk.view(np.uint8).reshape(-1)


def expert_indices(seed: int, n_routed: int = 128, top_k: int = 8,
                   with_shared: bool = True) -> np.ndarray:
    """top_k distinct routed expert ids from a seeded permutation of 0..n_routed-1,
    followed by the always-on shared expert, stored as slot n_routed."""
    g = rng(seed, S_INDEX)
    sel = g.permutation(n_routed)[:top_k].astype(np.int32)
    if with_shared:
        sel = np.concatenate([sel, np.array([n_routed], dtype=np.int32)])
    return sel


@dataclass(frozen=True)
class Dense:
    name: str
    fmt: int
    rows: int
    cols: int
    seed: int
    x_scale: float = 1.0
    batch: int = 1

    @property
    def nb(self) -> int:
        return self.cols // QK

    @property
    def weight_bytes(self) -> int:
        return self.rows * self.nb * BLOCK_BYTES[self.fmt]

    def algorithmic_bytes(self) -> int:
        """Weights read once + the Q8_0 activation blocks + fp32 outputs."""
        return self.weight_bytes + self.batch * (self.nb * 34 + self.rows * 4)


@dataclass(frozen=True)
class Moe:
    name: str = "moe_experts"
    n_routed: int = 128
    top_k: int = 8
    hidden: int = 2048
    ffn: int = 512
    seed: int = 3

    @property
    def n_slots(self) -> int:
        return self.n_routed + 1

    @property
    def n_sel(self) -> int:
        return self.top_k + 1

    def gate_up_bytes(self) -> int:
        return self.ffn * (self.hidden // QK) * BLOCK_BYTES[Q4_0]

    def down_bytes(self) -> int:
        return self.hidden * (self.ffn // QK) * BLOCK_BYTES[Q8_0]

    def algorithmic_bytes(self) -> int:
        n = self.n_sel
        w = n * (2 * self.gate_up_bytes() + self.down_bytes())
        x = (self.hidden // QK) * 34 + n * (self.ffn // QK) * 34
        idx = 4 * n
        y = n * (2 * self.ffn + self.hidden) * 4
        return w + x + idx + y


SSM_ALPHA_BETA = Dense("ssm_alpha_beta_q8_0_64x2048", Q8_0, 64, 2048, seed=0)
DENSE_Q4_0 = Dense("dense_q4_0_4096x4096", Q4_0, 4096, 4096, seed=1)
LM_HEAD_Q4_0 = Dense("lm_head_q4_0_248320x2048", Q4_0, 248320, 2048, seed=2, x_scale=0.1)
MOE = Moe()
BATCHED_Q8_0 = {b: Dense(f"batched_q8_0_14336x4096_b{b}", Q8_0, 14336, 4096, seed=4, batch=b)
                for b in (1, 2, 4, 8)}
