"""Seeded synthetic workloads for the denoising step (inputs only).

This module draws the tensors a denoising step consumes -- canvas queries,
cached and canvas keys/values, canvas hidden states and the vocabulary
projection -- with numpy's PCG64 generator, and rounds them to bf16 bit
patterns (``uint16``).  It holds none of the method's arithmetic: the random
numbers the method itself draws (Gumbel noise, renoise, canvas init) come
from Philox inside each implementation.  Both the CUDA path and the oracle
consume what this module returns, so one seed gives both the same bytes.

Large tensors are drawn in fixed row chunks, each from its own child of one
``SeedSequence``, so the values do not depend on the number of threads used.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class StepConfig:
    """Shapes and value distributions of one synthetic denoising step."""
    name: str
    B: int = 1                 # independent canvases
    L: int = 256               # canvas length
    Hq: int = 4                # query heads
    Hkv: int = 1               # key/value heads
    D: int = 128               # head dim
    P: int = 256               # cached prefix length
    d: int = 1024              # hidden size
    V: int = 16384             # vocabulary
    w_std: float = 0.05        # W ~ N(0, w_std^2)
    row_scale: Optional[tuple] = None   # hidden row i scaled by U(lo, hi)
    temperature: float = 0.8
    entropy_bound: float = 0.1
    stop_threshold: float = 0.005
    max_steps: int = 48
    t_start: float = 0.8
    t_end: float = 0.4
    seed: int = 0

    @property
    def M(self) -> int:
        return self.B * self.L


# The five workloads.  Numbers in N(0, s) for W are standard deviations; the
# block loop's N(0, 1/d) noise is a variance (std 1/sqrt(d)).
CONFIGS = {
    # single step, batch 1, small LM head
    "step_small": StepConfig("step_small"),
    # full-width single step: 16q/8kv heads, head_dim 256, 4096 cached keys,
    # LM head 2816 x 262144, per-row logit scale U(0.5, 8)
    "step_full": StepConfig("step_full", Hq=16, Hkv=8, D=256, P=4096, d=2816, V=262144,
                            w_std=0.02, row_scale=(0.5, 8.0)),
    # batch sweep of the small step with 2048 cached keys
    "batch1": StepConfig("batch1", B=1, P=2048),
    "batch4": StepConfig("batch4", B=4, P=2048),
    "batch16": StepConfig("batch16", B=16, P=2048),
    # long context: 32768 cached keys
    "long_context": StepConfig("long_context", P=32768),
    # full block loop (hidden states built per step, see block_hidden)
    "block_full": StepConfig("block_full", d=2816, V=262144, w_std=0.02, P=0, Hq=4, Hkv=1),
    # encoder cache append after a committed block (causal attention over
    # [cache ; block]) at the full-width step's attention shapes
    "encoder_full": StepConfig("encoder_full", Hq=16, Hkv=8, D=256, P=4096),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the raw bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(seed_seq: np.random.SeedSequence, shape, std: float = 1.0,
                 chunk_rows: int = 64, threads: Optional[int] = None) -> np.ndarray:
    """bf16 bits of N(0, std^2) draws; rows (first axis) drawn in fixed chunks."""
    shape = tuple(int(s) for s in shape)
    rows = shape[0] if shape else 1
    inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    out = np.empty((rows, inner), dtype=np.uint16)
    n_chunks = max(1, (rows + chunk_rows - 1) // chunk_rows)
    children = seed_seq.spawn(n_chunks)

    def work(c):
        r0, r1 = c * chunk_rows, min(rows, (c + 1) * chunk_rows)
        g = np.random.Generator(np.random.PCG64(children[c]))
        x = g.standard_normal((r1 - r0, inner), dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[r0:r1] = f32_to_bf16_bits(x)

    nthreads = threads or min(16, os.cpu_count() or 1)
    if n_chunks == 1 or nthreads == 1:
        for c in range(n_chunks):
            work(c)
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(work, range(n_chunks)))
    return out.reshape(shape)


def _ss(seed: int, tag: int) -> np.random.SeedSequence:
    return np.random.SeedSequence([int(seed), int(tag)])


def attention_inputs(cfg: StepConfig, seed: Optional[int] = None) -> dict:
    """Q [B,L,Hq,D], K/V prefix [B,P,Hkv,D], K/V canvas [B,L,Hkv,D], all ~N(0,1), bf16 bits."""
    s = cfg.seed if seed is None else seed
    B, L, P, Hq, Hkv, D = cfg.B, cfg.L, cfg.P, cfg.Hq, cfg.Hkv, cfg.D
    return dict(
        q=_normal_bf16(_ss(s, 1), (B, L, Hq, D)),
        kp=_normal_bf16(_ss(s, 2), (B, P, Hkv, D)),
        vp=_normal_bf16(_ss(s, 3), (B, P, Hkv, D)),
        kc=_normal_bf16(_ss(s, 4), (B, L, Hkv, D)),
        vc=_normal_bf16(_ss(s, 5), (B, L, Hkv, D)),
    )


def lm_weight(cfg: StepConfig, seed: Optional[int] = None) -> np.ndarray:
    """Vocabulary projection W [d, V] ~ N(0, w_std^2), bf16 bits."""
    s = cfg.seed if seed is None else seed
    return _normal_bf16(_ss(s, 6), (cfg.d, cfg.V), std=cfg.w_std, chunk_rows=16)


def lm_hidden(cfg: StepConfig, seed: Optional[int] = None) -> np.ndarray:
    """Canvas hidden states X [B*L, d]: rows ~N(0,1), times U(lo,hi) per row if configured."""
    s = cfg.seed if seed is None else seed
    if cfg.row_scale is None:
        return _normal_bf16(_ss(s, 7), (cfg.M, cfg.d))
    g = np.random.Generator(np.random.PCG64(_ss(s, 8)))
    x = g.standard_normal((cfg.M, cfg.d), dtype=np.float32)
    sc = g.uniform(cfg.row_scale[0], cfg.row_scale[1], size=(cfg.M, 1)).astype(np.float32)
    return f32_to_bf16_bits(x * sc)


def block_targets(cfg: StepConfig, seed: Optional[int] = None) -> dict:
    """Per-position target token t ~ U(V) and confidence c ~ U(0,1) of the block loop."""
    s = cfg.seed if seed is None else seed
    g = np.random.Generator(np.random.PCG64(_ss(s, 9)))
    t = g.integers(0, cfg.V, size=cfg.M, dtype=np.int64)
    c = g.uniform(0.0, 1.0, size=cfg.M)
    return dict(t=t, c=c)


def block_hidden(cfg: StepConfig, w_bits: np.ndarray, targets: dict, k: int,
                 seed: Optional[int] = None) -> np.ndarray:
    """Hidden states of step k: h_i = g_k(c_i) W[:,t_i]/||W[:,t_i]|| + N(0, 1/d),
    g_k(c) = (2 + 6c)(1 + k/4); built in fp64, rounded to bf16 bits."""
    s = cfg.seed if seed is None else seed
    cols = bf16_bits_to_f32(w_bits[:, targets["t"]]).astype(np.float64).T   # [M, d]
    cols /= np.linalg.norm(cols, axis=1, keepdims=True)
    gk = (2.0 + 6.0 * targets["c"]) * (1.0 + k / 4.0)
    g = np.random.Generator(np.random.PCG64(_ss(s, 100 + k)))
    noise = g.standard_normal((cfg.M, cfg.d)) / np.sqrt(cfg.d)
    return f32_to_bf16_bits((gk[:, None] * cols + noise).astype(np.float32))


@dataclasses.dataclass(frozen=True)
class MoeConfig:
    """Shapes and value distributions of one synthetic MoE FFN layer over a canvas."""
    name: str
    M: int = 256               # canvas rows (B * L)
    d: int = 2816              # hidden size
    f: int = 768               # FFN width of every expert
    E: int = 128               # routed experts (plus one shared)
    top_k: int = 8
    alpha: float = 1.2         # weight of the canvas-wide component of the hidden rows
    seed: int = 0


# The MoE workload: 128 experts, top-8 plus one shared expert (the pages'
# routing); d as the full-width step; f = 768 per expert (the pages give no
# expert shapes).  The hidden rows share a canvas-wide component, which makes
# the router's choices overlap: about 84 distinct experts per canvas, the
# count the pages report for a canvas forward.
MOE_CONFIGS = {
    "moe_full": MoeConfig("moe_full"),
}


def moe_inputs(cfg: MoeConfig, seed: Optional[int] = None) -> dict:
    """x [M, d] = (alpha c + n) / sqrt(1 + alpha^2) with one canvas vector c and
    per-row noise n (both N(0, 1)); router wr [E, d] ~ N(0, 1/d); gate / up
    [E+1, f, d] ~ N(0, 1/d); down [E+1, d, f] ~ N(0, 1/f); all bf16 bits."""
    s = cfg.seed if seed is None else seed
    g = np.random.Generator(np.random.PCG64(_ss(s, 200)))
    c = g.standard_normal(cfg.d)
    n = g.standard_normal((cfg.M, cfg.d))
    x = (cfg.alpha * c[None, :] + n) / np.sqrt(1.0 + cfg.alpha ** 2)
    return dict(
        x=f32_to_bf16_bits(x.astype(np.float32)),
        wr=_normal_bf16(_ss(s, 201), (cfg.E, cfg.d), std=cfg.d ** -0.5),
        wg=_normal_bf16(_ss(s, 202), (cfg.E + 1, cfg.f, cfg.d), std=cfg.d ** -0.5, chunk_rows=4),
        wu=_normal_bf16(_ss(s, 203), (cfg.E + 1, cfg.f, cfg.d), std=cfg.d ** -0.5, chunk_rows=4),
        wd=_normal_bf16(_ss(s, 204), (cfg.E + 1, cfg.d, cfg.f), std=cfg.f ** -0.5, chunk_rows=4),
    )
