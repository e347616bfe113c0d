"""Seeded synthetic inputs for the attention workloads (shared by tests, bench and smoke).

This module only draws random tensors: it holds none of the attention or quantization
arithmetic, and it imports neither the oracle nor the CUDA package. Every tensor is drawn
from ``torch.Generator('cpu').manual_seed(seed)`` in the order Q, K, V, then extras, computed
in float32 and cast once to bf16 (round to nearest even). The layout is [B, S, H, 128].

The pages measure on trained video models with real prompts (Wan 2.2, HunyuanVideo 1.5,
Cosmos 3 in "SAGE + Skip-Softmax -- API Design & Test Plan", Part 2). Those are not
available here, so these generators stand in for them with the shapes and value
structure of DiT self-attention:

* ``iid``      Q, K, V ~ N(0, 1).
* ``koffset``  Q, V ~ N(0, 1); K = N(0, 1) + c[kv head, channel], c ~ N(0, 2^2) shared by
               all tokens (a per-channel K bias, the thing K-smoothing removes).
* ``outlier``  Q, K, V ~ N(0, 1); round(1% of the Hkv*128 (kv head, channel) pairs), chosen
               without replacement, scaled by 8 in K for every token and batch.
* ``video``    tokens on a (t, h, w) grid in raster order (token = t*H*W + h*W + w);
               Q = x + 3 f(p), K = y + 3 f(p) with x, y ~ N(0, 0.5^2), V ~ N(0, 1), and
               f(p) = [cos(w_k . p), sin(w_k . p)] for 64 frequency vectors w_k in R^3 whose
               components are ~ N(0, 0.15^2). Scores then decay with grid distance.
"""

from __future__ import annotations

import dataclasses
import math

import torch

HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    kind: str = "iid"            # iid | koffset | outlier | video
    mode: str = "dense"          # dense | sage | qk16pv8 (V per tensor) | mxfp8, nvfp4 (V per channel)
    qk_dtype: str = "bf16"       # bf16 | int8 | fp8_e4m3 | mxfp8 | nvfp4
    q_block: int = 1
    k_block: int = 16
    factors: tuple = ()          # Skip-Softmax threshold_scale_factor values (empty: no skip)
    grid: tuple = ()             # (T, H, W) for kind == 'video'

    @property
    def dense_equiv_flop(self) -> float:
        """4 * B * Hq * Sq * Skv * d: the two matrix products, counted as if dense."""
        return 4.0 * self.B * self.Hq * self.Sq * self.Skv * HEAD_DIM

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


VIDEO_GRID = (21, 45, 80)

# The five workloads the measurements are quoted on, plus the QK16PV8 recipe (BF16 Q/K, FP8 V
# with one tensor-wide scale) and the MXFP8 and NVFP4 Q/K + FP8 V recipes (per-channel V) on the DiT inputs.
WORKLOADS = {
    "tiny_dense_256": Workload("tiny_dense_256", 1, 2, 2, 256, 256),
    "dit_dense_32k": Workload("dit_dense_32k", 1, 40, 40, 32768, 32768, kind="koffset"),
    "dit_sage_int8_32k": Workload("dit_sage_int8_32k", 1, 40, 40, 32768, 32768, kind="koffset", mode="sage",
                                  qk_dtype="int8", q_block=1, k_block=16),
    "gqa_sage_fp8_16k": Workload("gqa_sage_fp8_16k", 2, 32, 8, 16384, 16384, kind="outlier", mode="sage",
                                 qk_dtype="fp8_e4m3", q_block=1, k_block=4),
    "dit_qk16pv8_32k": Workload("dit_qk16pv8_32k", 1, 40, 40, 32768, 32768, kind="koffset", mode="qk16pv8",
                                qk_dtype="bf16", q_block=0, k_block=0),
    "dit_mxfp8_32k": Workload("dit_mxfp8_32k", 1, 40, 40, 32768, 32768, kind="koffset", mode="mxfp8",
                              qk_dtype="mxfp8", q_block=0, k_block=0),
    "dit_nvfp4_32k": Workload("dit_nvfp4_32k", 1, 40, 40, 32768, 32768, kind="koffset", mode="nvfp4",
                              qk_dtype="nvfp4", q_block=0, k_block=0),
    "video_skip_int8_75600": Workload("video_skip_int8_75600", 1, 40, 40, 75600, 75600, kind="video", mode="sage",
                                      qk_dtype="int8", q_block=1, k_block=16,
                                      factors=(0.0, 1.0, 2.0, 5.0, 20.0, 50.0, 200.0, 800.0, 3200.0),
                                      grid=VIDEO_GRID),
}


def _randn(gen: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32, device=gen.device)
    return x * std if std != 1.0 else x


def video_embedding(gen: torch.Generator, grid, n_freq: int = 64, std: float = 0.15) -> torch.Tensor:
    """The fixed random Fourier embedding f(p) of the grid coordinates: [T*H*W, 2*n_freq]."""
    T, H, W = grid
    omega = _randn(gen, (n_freq, 3), std).double()
    dev = gen.device
    t = torch.arange(T, dtype=torch.float64, device=dev)
    h = torch.arange(H, dtype=torch.float64, device=dev)
    w = torch.arange(W, dtype=torch.float64, device=dev)
    p = torch.stack(torch.meshgrid(t, h, w, indexing="ij"), dim=-1).reshape(-1, 3)  # raster order
    ang = p @ omega.T
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).float()


def generate(w: Workload, seed: int = 0, device: str = "cpu"):
    """(q, k, v) as bf16 tensors of shape [B, Sq, Hq, 128] / [B, Skv, Hkv, 128].

    The CPU generator is the canonical one (parity tests and the oracle use it). With
    device='cuda' the same recipe is drawn by the device generator: a different random stream
    with the same distribution, used where only timing matters.
    """
    gen = torch.Generator(device).manual_seed(seed)
    D = HEAD_DIM
    if w.kind == "video":
        assert w.Sq == w.Skv == math.prod(w.grid), "video workloads are self-attention over the grid"
        x = _randn(gen, (w.B, w.Sq, w.Hq, D), 0.5)
        y = _randn(gen, (w.B, w.Skv, w.Hkv, D), 0.5)
        v = _randn(gen, (w.B, w.Skv, w.Hkv, D))
        f = video_embedding(gen, w.grid)[None, :, None, :]
        q = x.add_(f, alpha=3.0)
        k = y.add_(f, alpha=3.0)
        return q.bfloat16(), k.bfloat16(), v.bfloat16()
    q = _randn(gen, (w.B, w.Sq, w.Hq, D))
    k = _randn(gen, (w.B, w.Skv, w.Hkv, D))
    v = _randn(gen, (w.B, w.Skv, w.Hkv, D))
    if w.kind == "koffset":
        c = _randn(gen, (w.Hkv, D), 2.0)
        k.add_(c[None, None])
    elif w.kind == "outlier":
        n = round(0.01 * w.Hkv * D)
        pick = torch.randperm(w.Hkv * D, generator=gen, device=gen.device)[:n]
        kv = k.view(w.B, w.Skv, w.Hkv * D)
        kv[:, :, pick] *= 8.0
    elif w.kind != "iid":
        raise ValueError(f"unknown workload kind {w.kind!r}")
    return q.bfloat16(), k.bfloat16(), v.bfloat16()


def to_f32_numpy(t: torch.Tensor):
    """bf16 tensor -> float32 numpy array holding the same values (exact)."""
    return t.float().numpy()
