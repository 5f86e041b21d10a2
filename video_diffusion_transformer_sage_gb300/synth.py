"""Seeded synthetic Q/K/V inputs for the packed video-DiT attention workloads.

This module holds only random-number generation and buffer layout; none of the
attention or quantisation arithmetic lives here, so both the CUDA path and the
CPU oracle can consume the same bf16 bytes.

Workloads (token counts, heads, head dim and layouts follow the attention call
profiled in "gb10-sage2-p0-interleave-softmax-latency.json", keys `q_shape`
and `metadata.segments`, and the strided-NHD dataflow of
"gb10-sage-strided-nhd-summary-...json", key `dataflow.qkv_input`):

  tiny      N=1024,  H=2,  D=128  contiguous NHD; Q,K,V ~ N(0,1); per-(h,c) K bias ~ N(0, var 2)
  tails     N=4100,  H=8,  D=128  contiguous NHD; K bias ~ N(0, var 4); 4 outlier channels/head x20 in Q,K
  strided64 N=16384, H=24, D=64   strided views of one token-major [N, 3*H*D] buffer; K bias ~ N(0, var 4)
  video     N=37810 (100 text + 414 conditioning + 37296 video), H=56, D=128, strided views of [N, 21504];
            per-(token, head) RMS-normalised Q,K rows; K bias ~ N(0, var 4); 3 outlier channels/head x20
  sweep     N in {8192, 18905, 37810, 75620}, H=56, D=128, as `video`; plus an HND-contiguous copy

Draw order (one CPU generator per workload): K bias, outlier channels (per head), then
Q, K and V in full, each in token order.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_tokens: int
    n_heads: int
    head_dim: int
    layout: str            # "nhd" (contiguous [N,H,D]), "qkv" (views of [N,3HD]), "hnd" ([H,N,D] contiguous)
    k_bias_var: float      # variance of the per-(head, channel) K bias shared by all tokens
    n_outlier: int         # outlier channels per head (same channels in Q and K)
    outlier_mult: float
    rms_norm: bool         # RMS-normalise each (token, head) row of Q and K before outliers / bias
    seed: int

    @property
    def flops(self) -> float:
        """Attention FLOPs per call, 4*N^2*H*D (two N x N x D contractions)."""
        return 4.0 * self.n_tokens ** 2 * self.n_heads * self.head_dim


# Segment layout of the packed sequence: [start, end, type] with 1 = text,
# 2 = conditioning, 0 = video (metadata.segments of the block-24 attention call).
VIDEO_SEGMENTS = ((0, 100, 1), (100, 514, 2), (514, 37810, 0))

WORKLOADS = {
    "tiny": Workload("tiny", 1024, 2, 128, "nhd", 2.0, 0, 1.0, False, 0),
    "tails": Workload("tails", 4100, 8, 128, "nhd", 4.0, 4, 20.0, False, 1),
    "strided64": Workload("strided64", 16384, 24, 64, "qkv", 4.0, 0, 1.0, False, 2),
    "video": Workload("video", 37810, 56, 128, "qkv", 4.0, 3, 20.0, True, 440420),
}
for _n in (8192, 18905, 37810, 75620):
    WORKLOADS[f"sweep{_n}"] = Workload(f"sweep{_n}", _n, 56, 128, "qkv", 4.0, 3, 20.0, True, 3)
WORKLOADS["sweep37810_hnd"] = Workload("sweep37810_hnd", 37810, 56, 128, "hnd", 4.0, 3, 20.0, True, 3)


def custom(n_tokens: int, n_heads: int, head_dim: int, layout: str = "qkv", seed: int = 0,
           k_bias_var: float = 4.0, n_outlier: int = 0, outlier_mult: float = 20.0,
           rms_norm: bool = False) -> Workload:
    return Workload(f"custom_{n_tokens}x{n_heads}x{head_dim}_{layout}", n_tokens, n_heads, head_dim,
                    layout, k_bias_var, n_outlier, outlier_mult, rms_norm, seed)


@dataclasses.dataclass
class Inputs:
    """bf16 CPU tensors.  q, k, v are [N, H, D] views (possibly strided) of `storage`."""
    workload: Workload
    storage: torch.Tensor
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor


def _rms_rows(x: torch.Tensor) -> torch.Tensor:
    return x / torch.sqrt(torch.mean(x * x, dim=-1, keepdim=True))


def _aux(w: Workload, g: torch.Generator):
    """K bias and outlier-channel multipliers (drawn first, before the bulk Q, K, V)."""
    h, d = w.n_heads, w.head_dim
    bias = torch.randn((h, d), generator=g) * math.sqrt(w.k_bias_var)
    mult = torch.ones((h, d))
    for hh in range(h):
        idx = torch.randperm(d, generator=g)[: w.n_outlier]
        mult[hh, idx] = w.outlier_mult
    return bias, mult


def make_inputs(w: Workload | str, chunk_tokens: int = 4096) -> Inputs:
    if isinstance(w, str):
        w = WORKLOADS[w]
    n, h, d = w.n_tokens, w.n_heads, w.head_dim
    g = torch.Generator("cpu").manual_seed(w.seed)
    bias, mult = _aux(w, g)
    if w.layout == "qkv":
        storage = torch.empty((n, 3 * h * d), dtype=torch.bfloat16)
        views = [storage[:, i * h * d:(i + 1) * h * d].view(n, h, d) for i in range(3)]
    elif w.layout == "nhd":
        storage = torch.empty((3, n, h, d), dtype=torch.bfloat16)
        views = [storage[i] for i in range(3)]
    elif w.layout == "hnd":
        storage = torch.empty((3, h, n, d), dtype=torch.bfloat16)
        views = [storage[i].transpose(0, 1) for i in range(3)]
    else:
        raise ValueError(w.layout)
    for which in range(3):  # 0 = Q, 1 = K, 2 = V
        t0 = 0
        while t0 < n:
            t1 = min(n, t0 + chunk_tokens)
            x = torch.randn((t1 - t0, h, d), generator=g)
            if which < 2:
                if w.rms_norm:
                    x = _rms_rows(x)
                x = x * mult
                if which == 1:
                    x = x + bias
            views[which][t0:t1].copy_(x.to(torch.bfloat16))
            t0 = t1
    return Inputs(w, storage, views[0], views[1], views[2])


def to_hnd(inp: Inputs) -> Inputs:
    """Same values as `inp`, re-laid out as HND-contiguous [H, N, D] buffers (viewed as [N, H, D])."""
    w = dataclasses.replace(inp.workload, layout="hnd", name=inp.workload.name + "_hnd")
    storage = torch.empty((3, w.n_heads, w.n_tokens, w.head_dim), dtype=torch.bfloat16)
    views = [storage[i].transpose(0, 1) for i in range(3)]
    for dst, src in zip(views, (inp.q, inp.k, inp.v)):
        dst.copy_(src)
    return Inputs(w, storage, views[0], views[1], views[2])


def with_v_offset(inp: Inputs, std: float = 8.0, seed: int = 17) -> Inputs:
    """A copy of `inp` (same layout and strides) whose V carries a per-(head, channel) offset
    ~ N(0, std^2) shared by all tokens, drawn from its own generator: the input that V
    smoothing is for.  Q and K are unchanged."""
    storage = inp.storage.clone()

    def view(t: torch.Tensor) -> torch.Tensor:
        return storage.as_strided(t.shape, t.stride(), t.storage_offset())

    q, k, v = view(inp.q), view(inp.k), view(inp.v)
    g = torch.Generator("cpu").manual_seed(seed)
    off = torch.randn((inp.v.shape[1], inp.v.shape[2]), generator=g) * std
    v.copy_((inp.v.float() + off).to(torch.bfloat16))
    w = dataclasses.replace(inp.workload, name=inp.workload.name + "_voff")
    return Inputs(w, storage, q, k, v)


def sample_rows(n_tokens: int, count: int, seed: int) -> list:
    """Seeded query-row sample that always includes both ends, the last 128-row tile and,
    where present, the text / conditioning / video segment borders (99/100, 513/514)."""
    must = {0, n_tokens - 1}
    must |= {b for b in (99, 100, 513, 514) if b < n_tokens}
    tail0 = ((n_tokens - 1) // 128) * 128
    must |= {r for r in (tail0, tail0 + 1) if r < n_tokens}
    g = torch.Generator("cpu").manual_seed(seed)
    out = list(must)
    for r in torch.randperm(n_tokens, generator=g).tolist():
        if len(out) >= count:
            break
        if r not in must:
            out.append(r)
    return sorted(out)


# ---------------------------------------------------------------------------------------
# Inputs of the qk_transform stage ("in-place ... RMSNorm and RoPE on strided views",
# gb10-sage-strided-nhd-summary key dataflow.qk_transform).  The pages give neither the norm
# weights nor the rotary table, so both are inputs made here; the norm and the rotation that
# use them live in the CUDA kernel and in the oracle only.
#   gamma: per-channel norm weights ~ N(1, 0.1^2), one vector for Q and one for K.
#   positions: the 514 text / conditioning tokens get the 1-D position (t, t, t); the 37296
#     video tokens a (frame, row, column) position on a 37 x 24 x 42 latent grid, in
#     frame-major order (37 * 24 * 42 = 37296).
#   table: D/2 channel pairs split into three bands (frame, row, column; the frame band takes
#     the remainder), pair i of a band of size nb turning at base^(-i/nb) radians per
#     position step; cos and sin of the angles computed in fp64, stored as fp32 [N, D/2].
VIDEO_GRID = (37, 24, 42)


def qk_norm_weights(head_dim: int, seed: int = 7):
    g = torch.Generator("cpu").manual_seed(seed)
    gq = (1.0 + 0.1 * torch.randn(head_dim, generator=g)).float()
    gk = (1.0 + 0.1 * torch.randn(head_dim, generator=g)).float()
    return gq, gk


def rope_positions(n_tokens: int, n_text: int = 514, grid=VIDEO_GRID) -> torch.Tensor:
    """[N, 3] int64 (frame, row, column) positions of the packed sequence."""
    t = torch.arange(n_tokens, dtype=torch.int64)
    v = (t - n_text).clamp(min=0)
    _, gy, gx = grid
    pos = torch.stack([v // (gy * gx), (v // gx) % gy, v % gx], dim=1)
    text = t < n_text
    pos[text] = t[text, None].expand(-1, 3)
    return pos


def rope_table(positions: torch.Tensor, head_dim: int, base: float = 10000.0):
    """cos, sin fp32 [N, D/2] of the rotary angles of `positions` ([N, 3])."""
    half = head_dim // 2
    nb_y = nb_x = half // 3
    nb_f = half - nb_y - nb_x
    ang = torch.empty((positions.shape[0], half), dtype=torch.float64)
    off = 0
    for axis, nb in enumerate((nb_f, nb_y, nb_x)):
        freq = base ** (-torch.arange(nb, dtype=torch.float64) / nb)
        ang[:, off:off + nb] = positions[:, axis:axis + 1].double() * freq[None, :]
        off += nb
    return torch.cos(ang).float().contiguous(), torch.sin(ang).float().contiguous()
