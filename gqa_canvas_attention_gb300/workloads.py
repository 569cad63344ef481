"""Seeded synthetic inputs for the canvas attention block.

This module holds no arithmetic of the method: it only draws random tensors in a fixed order,
so that the CUDA library and the CPU oracle see the same bytes.

Every tensor is fp32 ~N(0, 1) (norm weights are 1 + 0.1 * N(0, 1)), drawn on the CPU from
``torch.Generator().manual_seed(seed)`` in the order
``q, k_canvas, v_canvas, k_cache, v_cache, q_norm_w, k_norm_w`` (weights only when enabled,
the cache only when ctx > 0).  The cache is treated as already normed and roped.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

EPS = 1e-6
ROPE_THETA = 10000.0


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    ctx: int
    nh: int
    nkv: int
    hd: int
    seed: int
    weighted: bool
    steps: int = 1           # denoising steps sharing one cache
    canvases: int = 1        # independent canvases (each its own seed)
    seeds: tuple = field(default_factory=tuple)
    theta: float = ROPE_THETA
    pos0: int | None = None  # position of canvas row 0 (None: ctx, the cache length)

    @property
    def S(self) -> int:
        return self.ctx + self.T

    def flops_per_forward(self) -> int:
        """Useful attention FLOPs of one forward: 4 * T * nh * (ctx + T) * hd."""
        return 4 * self.T * self.nh * self.S * self.hd

    def forwards(self) -> int:
        return self.steps * self.canvases


WORKLOADS = {
    "tiny": Workload("tiny", T=16, ctx=32, nh=4, nkv=2, hd=64, seed=0, weighted=True),
    "gqa_hd256_ctx1k": Workload("gqa_hd256_ctx1k", T=256, ctx=1024, nh=8, nkv=4, hd=256, seed=1,
                                weighted=True),
    "gqa_hd128_ctx4k": Workload("gqa_hd128_ctx4k", T=256, ctx=4096, nh=16, nkv=8, hd=128, seed=2,
                                weighted=True),
    "denoise48_ctx8k": Workload("denoise48_ctx8k", T=512, ctx=8192, nh=8, nkv=4, hd=256, seed=3,
                                weighted=False, steps=48),
    "mha_canvas4k_x4": Workload("mha_canvas4k_x4", T=4096, ctx=0, nh=16, nkv=16, hd=64, seed=10,
                                weighted=False, canvases=4, seeds=(10, 11, 12, 13)),
    # The two layer types of the decoder: a sliding-window layer, whose cache holds the last
    # 1024 positions of an 8192-long sequence (canvas positions continue at 8192), and a global
    # layer with its own kv-head count and rope base.
    "sliding_w1k": Workload("sliding_w1k", T=512, ctx=1024, nh=8, nkv=4, hd=256, seed=20,
                            weighted=True, pos0=8192),
    "global_kv2_theta1m": Workload("global_kv2_theta1m", T=512, ctx=8192, nh=8, nkv=2, hd=256,
                                   seed=21, weighted=True, theta=1.0e6),
}


def _randn(g: torch.Generator, *shape) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32)


def make_inputs(T: int, ctx: int, nh: int, nkv: int, hd: int, seed: int,
                weighted: bool = True, draw_cache: bool = True) -> dict:
    """One forward's inputs as CPU fp32 tensors (cache None when ctx == 0 or not drawn)."""
    g = torch.Generator().manual_seed(int(seed))
    d = {
        "q": _randn(g, T, nh * hd),
        "k_canvas": _randn(g, T, nkv * hd),
        "v_canvas": _randn(g, T, nkv * hd),
        "k_cache": None,
        "v_cache": None,
        "q_norm_w": None,
        "k_norm_w": None,
    }
    if ctx > 0 and draw_cache:
        d["k_cache"] = _randn(g, nkv, ctx, hd)
        d["v_cache"] = _randn(g, nkv, ctx, hd)
    if weighted:
        d["q_norm_w"] = 1.0 + 0.1 * _randn(g, hd)
        d["k_norm_w"] = 1.0 + 0.1 * _randn(g, hd)
    return d


def workload_inputs(w: Workload, step: int = 0, canvas: int = 0) -> dict:
    """Inputs of one forward of a named workload.

    Denoising loops: step 0 draws the canvas then the shared cache from ``seed``; step s > 0
    draws a fresh canvas from ``seed + s`` (its cache is step 0's).  Canvas batches: canvas c
    uses ``seeds[c]``."""
    if w.canvases > 1:
        return make_inputs(w.T, w.ctx, w.nh, w.nkv, w.hd, w.seeds[canvas], w.weighted)
    if step == 0:
        return make_inputs(w.T, w.ctx, w.nh, w.nkv, w.hd, w.seed, w.weighted)
    d = make_inputs(w.T, w.ctx, w.nh, w.nkv, w.hd, w.seed + step, w.weighted, draw_cache=False)
    return d


def shared_cache(w: Workload) -> tuple:
    """The (k_cache, v_cache) a denoising loop shares across its steps (step 0's draw)."""
    d = make_inputs(w.T, w.ctx, w.nh, w.nkv, w.hd, w.seed, w.weighted)
    return d["k_cache"], d["v_cache"]
