"""Seeded synthetic video-shaped KV tensors and the workload recipes.

This module only makes inputs.  It holds none of the compression method's arithmetic,
and both the CUDA path and the CPU oracle receive the very same bytes from it.

The pages measure on the KV caches of real video diffusion models (LongCat-Video-13B,
HY-WorldPlay-8B, Self-Forcing-Wan-1.3B) driven by the MovieGen prompt suite; none of that
exists here, so this generator stands in for it.  What the pages fix is the structure:
tokens sit on a (frame, row, column) grid, neighbouring tokens in space and time are
numerically close, keys reach |x| ~ 1e2 and values |x| ~ 1e3 through a few outlier
channels.  The field below has exactly that structure:

  z_k(f, y, x) = sqrt(2/M) * sum_m a_km cos(w_m . (f/lt, y/ls, x/ls) + phi_km)

with M = 32 random Fourier features of a squared-exponential kernel (w ~ N(0, I3),
a ~ N(0, 1), phi ~ U[0, 2pi)), so every channel is marginally close to N(0, 1) and
correlated over ls = 6 tokens in space and lt = 8 latent frames in time (a slowly
changing scene: consecutive 3-frame chunks are about 0.93 correlated).  Every element
gets iid N(0, 0.1^2) noise from a counter-based hash of (seed, tensor, token, channel), so
a chunk of frames is the same slice of the same field whichever call produces it.  Four
channels per tensor (chosen by the seed) are outliers: A_k + 10 z_k with
A_k = +-U(60, 90), clipped to |x| <= 100.  Value tensors are the same construction
scaled by 10 (clip 1000).  The result is cast to fp16 / bf16 with round-to-nearest-even.

Tensor ids: (layer, head, K/V) -> 2 * (layer * heads + head) + kv; even ids are keys.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Sequence

import numpy as np
import torch

M_FEATURES = 32
LEN_SPACE = 6.0
LEN_TIME = 8.0
D_HEAD = 128
N_OUTLIERS = 4


def tensor_id(layer: int, head: int, kv: int, heads: int) -> int:
    return 2 * (layer * heads + head) + kv


def _params(seed: int, tid: int):
    rng = np.random.default_rng([int(seed), int(tid), 0x51D])
    omega = rng.standard_normal((M_FEATURES, 3))
    a = rng.standard_normal((D_HEAD, M_FEATURES))
    phi = rng.uniform(0.0, 2.0 * math.pi, (D_HEAD, M_FEATURES))
    out_ch = rng.choice(D_HEAD, N_OUTLIERS, replace=False)
    amp = rng.uniform(60.0, 90.0, N_OUTLIERS) * rng.choice([-1.0, 1.0], N_OUTLIERS)
    w = math.sqrt(2.0 / M_FEATURES) * np.concatenate([(a * np.cos(phi)).T,
                                                      (-a * np.sin(phi)).T], axis=0)
    return omega, w, out_ch, amp


_MASK31 = (1 << 31) - 1
_MASK24 = (1 << 24) - 1


def _mix(h: torch.Tensor) -> torch.Tensor:
    # Integer mixing (wrapping int64 arithmetic); only used to draw the noise term.
    h = h ^ ((h >> 29) & ((1 << 35) - 1))
    h = h * 0x5851F42D4C957F2D
    h = h ^ ((h >> 32) & 0xFFFFFFFF)
    h = h * 0x14057B7EF767814F
    h = h ^ ((h >> 29) & ((1 << 35) - 1))
    return h


def _noise(seed: int, tids: Sequence[int], gtok: torch.Tensor) -> torch.Tensor:
    """iid N(0,1) per (tensor, token, channel) from a counter hash; gtok is [N] global token
    ids.  Returns [len(tids)][N][128]."""
    k = torch.arange(D_HEAD, device=gtok.device, dtype=torch.int64)
    key = ((gtok[:, None] * D_HEAD + k[None, :]) * 2)[None]
    base = torch.tensor([(int(seed) * 0x9E3779B1 + int(t) * 0x85EBCA77) & ((1 << 62) - 1)
                         for t in tids], device=gtok.device, dtype=torch.int64)[:, None, None]
    h1 = _mix(key + base)
    h2 = _mix(key + 1 + base)
    u1 = (((h1 >> 8) & _MASK24).to(torch.float32) + 0.5) / float(1 << 24)
    u2 = ((h2 >> 8) & _MASK24).to(torch.float32) / float(1 << 24)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)


def kv_tensor(seed: int, tids: Sequence[int], f0: int, nf: int, gh: int, gw: int,
              dtype=torch.bfloat16, device="cpu", batch: int = 32) -> torch.Tensor:
    """[len(tids)][nf*gh*gw][128] tensor of frames [f0, f0+nf) of the field, raster order.
    Tensors are generated `batch` at a time; each tensor's values depend only on (seed, its
    id, the token), not on the batching."""
    dev = torch.device(device)
    f = torch.arange(f0, f0 + nf, device=dev, dtype=torch.float32)
    y = torch.arange(gh, device=dev, dtype=torch.float32)
    x = torch.arange(gw, device=dev, dtype=torch.float32)
    ff, yy, xx = torch.meshgrid(f, y, x, indexing="ij")
    pos = torch.stack([ff.reshape(-1) / LEN_TIME, yy.reshape(-1) / LEN_SPACE,
                       xx.reshape(-1) / LEN_SPACE], dim=1)
    gtok = torch.arange(f0 * gh * gw, (f0 + nf) * gh * gw, device=dev, dtype=torch.int64)
    tids = list(tids)
    out = torch.empty((len(tids), pos.shape[0], D_HEAD), dtype=dtype, device=dev)
    for b0 in range(0, len(tids), batch):
        bt = tids[b0:b0 + batch]
        prm = [_params(seed, t) for t in bt]
        omega = torch.as_tensor(np.stack([q[0] for q in prm]), dtype=torch.float32, device=dev)
        w = torch.as_tensor(np.stack([q[1] for q in prm]), dtype=torch.float32, device=dev)
        theta = torch.matmul(pos[None], omega.transpose(1, 2))          # [G][N][M]
        feats = torch.cat([torch.cos(theta), torch.sin(theta)], dim=2)  # [G][N][2M]
        v = torch.matmul(feats, w) + 0.1 * _noise(seed, bt, gtok)       # [G][N][128]
        for g, q in enumerate(prm):
            oc = torch.as_tensor(q[2], device=dev, dtype=torch.int64)
            v[g, :, oc] = torch.as_tensor(q[3], dtype=torch.float32, device=dev) + 10.0 * v[g, :, oc]
        v = v.clamp(-100.0, 100.0)
        vk = torch.tensor([t % 2 == 1 for t in bt], device=dev)[:, None, None]
        v = torch.where(vk, v * 10.0, v)
        out[b0:b0 + len(bt)] = v.to(dtype)
    return out


# ---------------------------------------------------------------------------------------
# Workload recipes.  Sizes follow the five configurations the method is measured on here.
# ---------------------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    seed: int
    layers: int
    heads: int
    kinds: Sequence[int]      # 0 = K, 1 = V
    frames: int
    gh: int
    gw: int
    dtype: torch.dtype
    C: int
    T: int
    bits: int
    group: int
    iters: int
    chunk_frames: int = 0     # streaming: frames per chunk (0 = no streaming)
    warm_iters: int = 2
    extra: dict = field(default_factory=dict)

    @property
    def tids(self):
        return [tensor_id(l, h, kv, self.heads) for l in range(self.layers)
                for h in range(self.heads) for kv in self.kinds]

    @property
    def H(self):
        return len(self.tids)

    @property
    def N(self):
        return self.frames * self.gh * self.gw

    @property
    def tokens_per_frame(self):
        return self.gh * self.gw

    def make(self, device="cpu", f0: int = 0, nf: int | None = None, tids=None):
        nf = self.frames if nf is None else nf
        return kv_tensor(self.seed, self.tids if tids is None else tids, f0, nf, self.gh,
                         self.gw, self.dtype, device)


def workload(name: str) -> Workload:
    """Named workloads:
    single_head_4x32x32   one fp16 key tensor, 4 frames of 32x32, C=64, T=1, 10 iters, INT2 B32
    layer_1p3b_32760      12 heads K+V, 21 frames of 30x52 (32760 tokens), C=256, T=2, INT2 B32
    dit13b_65536          32 heads K+V, 16 frames of 64x64 (65536 tokens), C=256, T=4, 8 iters
    stream_30x12_60chunk  30 layers x 12 heads K+V, 60 chunks of 3 frames of 30x52, C=256, T=2,
                          chunk 0 cold (10 iters), later chunks warm-started (2 iters)
    """
    if name == "single_head_4x32x32":
        return Workload(name, 1, 1, 1, [0], 4, 32, 32, torch.float16, 64, 1, 2, 32, 10)
    if name == "layer_1p3b_32760":
        return Workload(name, 2, 1, 12, [0, 1], 21, 30, 52, torch.bfloat16, 256, 2, 2, 32, 10)
    if name == "dit13b_65536":
        return Workload(name, 3, 1, 32, [0, 1], 16, 64, 64, torch.bfloat16, 256, 4, 2, 32, 8)
    if name == "stream_30x12_60chunk":
        return Workload(name, 5, 30, 12, [0, 1], 180, 30, 52, torch.bfloat16, 256, 2, 2, 32,
                        10, chunk_frames=3, warm_iters=2)
    raise KeyError(name)


# Precision sweep on the layer_1p3b_32760 shapes.
SWEEP_PRECISIONS = [(4, 64), (2, 16)]
SWEEP_C = [64, 128, 256]
SWEEP_T = [0, 1, 2, 3]
