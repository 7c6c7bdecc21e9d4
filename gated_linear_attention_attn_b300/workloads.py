"""Workload shapes and seeded synthetic inputs: the linear-attention layer, the
gated-softmax anchor layer and the AttnRes aggregation.

This module holds no arithmetic of the layers themselves: it only names the
shapes and draws the random inputs, so both the CUDA path and the fp64 oracle
can be fed the same values.

Shapes come from the latent token grids of SANA-Video 2.0 (NVlabs/Sana
docs/sana_video2.md, "Architecture": 20 heads x 128 for 5B, 32 heads x 128 for
14B; (1, 1, 1) latent patches over an LTX 2.3 latent with (8, 32, 32)
temporal/spatial strides, so N = T * (height/32) * (width/32) with
T = (frames - 1)/8 + 1).

Input recipe: one CPU ``torch.Generator`` seeded with ``seed`` draws q, k, v, g
in that order as float32 N(0, 1) tensors of shape [B, H, N, d]; k is then
scaled by ``k_scale``; all four are cast to the workload dtype.  Values are
i.i.d., so no dataset is needed.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    grid: Tuple[int, int, int]          # (T, Hs, Ws) latent token grid
    d: int = 128
    dtype: torch.dtype = torch.bfloat16
    rope: bool = False
    split: Tuple[int, int, int] = (44, 42, 42)   # head-dim bands for t, h, w
    base: float = 10000.0
    eps: float = 1e-6
    k_scale: float = 1.0
    tol: float = 1e-2                   # max|err| / max|ref| bound for parity
    description: str = ""
    block_frames: int = 0               # > 0: block-causal form, blocks of this many frames
    layer: str = "linear"               # "linear", "anchor" (gated-softmax, d = 256) or
                                        # "attnres" (H = number of sources, d = hidden size)

    @property
    def N(self) -> int:
        T, Hs, Ws = self.grid
        return T * Hs * Ws

    @property
    def block_tokens(self) -> int:
        """Tokens per block of the block-causal form (0 for the bidirectional layer)."""
        T, Hs, Ws = self.grid
        return self.block_frames * Hs * Ws

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.N

    @property
    def elem_size(self) -> int:
        return torch.empty((), dtype=self.dtype).element_size()

    @property
    def tokens(self) -> int:
        return self.B * self.N

    @property
    def algorithmic_bytes(self) -> int:
        """Attention layers: reads of q, k, v, g and the write of o, 5 * B*H*N*d
        elements.  AttnRes: the H source rows read and one row written per token."""
        if self.layer == "attnres":
            return (self.H + 1) * self.tokens * self.d * self.elem_size
        return 5 * self.B * self.H * self.N * self.d * self.elem_size

    @property
    def algorithmic_flops(self) -> int:
        """Linear layer: two d x d contractions per token, 4 * B*H*N*d^2.  Anchor
        layer: the N x N scores and their product with v, 4 * B*H*N^2*d."""
        if self.layer == "anchor":
            return 4 * self.B * self.H * self.N * self.N * self.d
        return 4 * self.B * self.H * self.N * self.d * self.d

    def with_(self, **kw) -> "Workload":
        fields = dict(self.__dict__)
        fields.update(kw)
        return Workload(**fields)


WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", B=1, H=2, grid=(4, 8, 8), dtype=torch.float32, tol=1e-5,
        description="oracle-size check: B=1 H=2 N=256 (4x8x8) fp32, no RoPE"),
    "5b_480p": Workload(
        "5b_480p", B=2, H=20, grid=(11, 15, 26),
        description="5B shape, 480p/81 frames: B=2 H=20 N=4290 (11x15x26) bf16, no RoPE"),
    "5b_720p": Workload(
        "5b_720p", B=2, H=20, grid=(25, 22, 40), rope=True,
        description="5B shape, 720p/193 frames: B=2 H=20 N=22000 (25x22x40) bf16, 3D RoPE 44/42/42"),
    "14b_480p": Workload(
        "14b_480p", B=2, H=32, grid=(11, 15, 26), rope=True,
        description="14B shape, 480p/81 frames: B=2 H=32 N=4290 bf16, 3D RoPE 44/42/42"),
    "5b_720p_60s": Workload(
        "5b_720p_60s", B=1, H=20, grid=(181, 22, 40), rope=True, k_scale=0.5,
        description="long clip, 720p/60 s: B=1 H=20 N=159280 (181x22x40) bf16, 3D RoPE, k x 0.5"),
    "5b_720p_736": Workload(
        "5b_720p_736", B=2, H=20, grid=(25, 23, 40), rope=True,
        description="5B shape, 720p/193 frames in the 736x1280 bucket: B=2 H=20 "
                    "N=23000 (25x23x40) bf16, 3D RoPE 44/42/42"),
    "5b_720p_block5": Workload(
        "5b_720p_block5", B=2, H=20, grid=(25, 22, 40), rope=True, block_frames=5,
        description="block-causal form of the 720p shape: 5 blocks of 5 latent frames "
                    "(4400 tokens), carried state in and out"),
    # gated-softmax anchor layers: 10 heads x 256 (5B), 16 heads x 256 (14B),
    # Wan 3D RoPE with the 88/84/84 split of d = 256
    "anchor_5b_480p": Workload(
        "anchor_5b_480p", B=2, H=10, grid=(11, 15, 26), d=256, rope=True, split=(88, 84, 84),
        layer="anchor",
        description="5B softmax anchor, 480p/81 frames: B=2 H=10 N=4290 d=256 bf16, 3D RoPE"),
    "anchor_5b_720p": Workload(
        "anchor_5b_720p", B=2, H=10, grid=(25, 22, 40), d=256, rope=True, split=(88, 84, 84),
        layer="anchor",
        description="5B softmax anchor, 720p/193 frames: B=2 H=10 N=22000 d=256 bf16, 3D RoPE"),
    "anchor_14b_480p": Workload(
        "anchor_14b_480p", B=2, H=16, grid=(11, 15, 26), d=256, rope=True, split=(88, 84, 84),
        layer="anchor",
        description="14B softmax anchor, 480p/81 frames: B=2 H=16 N=4290 d=256 bf16, 3D RoPE"),
    # AttnRes aggregation: the last block of each model reads every earlier
    # block's summary plus its own running one (5B: 32 layers in blocks of 8,
    # 4 sources, hidden 2560; 14B: 40 layers, 5 sources, hidden 4096)
    "attnres_5b_720p": Workload(
        "attnres_5b_720p", B=2, H=4, grid=(25, 22, 40), d=2560, layer="attnres",
        description="AttnRes, 5B at 720p/193 frames: 4 sources of [44000, 2560] bf16"),
    "attnres_14b_480p": Workload(
        "attnres_14b_480p", B=2, H=5, grid=(11, 15, 26), d=4096, layer="attnres",
        description="AttnRes, 14B at 480p/81 frames: 5 sources of [8580, 4096] bf16"),
}

# The workload the throughput metric is quoted on (5B shape at 720p).
HEADLINE = "5b_720p"


def make_inputs(wl: Workload, seed: int = 0, device: Optional[str] = None):
    """Draw (q, k, v, g) for ``wl``: see the module docstring for the recipe."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    shape = (wl.B, wl.H, wl.N, wl.d)
    out = []
    for name in ("q", "k", "v", "g"):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        if name == "k" and wl.k_scale != 1.0:
            x.mul_(wl.k_scale)
        x = x.to(wl.dtype)
        if device is not None:
            x = x.to(device)
        out.append(x)
    return tuple(out)


def make_attnres_inputs(wl: Workload, seed: int = 0, device: Optional[str] = None):
    """Draw (sources [M, T, C] bf16, w [C] fp32) for an AttnRes workload: one CPU
    generator seeded with ``seed`` draws the sources as N(0, 1) scaled by 1 + n
    for source n (summaries of growing magnitude), then w as N(0, 1) * 3 / sqrt(C)
    (scores of a few units)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    M, T, C = wl.H, wl.tokens, wl.d
    s = torch.randn((M, T, C), generator=gen, dtype=torch.float32)
    s.mul_(torch.arange(1, M + 1, dtype=torch.float32).view(M, 1, 1))
    w = torch.randn((C,), generator=gen, dtype=torch.float32) * (3.0 / C ** 0.5)
    s = s.to(torch.bfloat16)
    if device is not None:
        s, w = s.to(device), w.to(device)
    return s, w


def sample_rows(N: int, count: int, seed: int = 1):
    """Token rows to check at full size: the first, the last, and a seeded spread."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    picks = torch.randint(0, N, (max(count - 2, 0),), generator=gen).tolist()
    rows = sorted(set([0, N - 1] + picks))
    return rows
