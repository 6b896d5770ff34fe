"""Seeded synthetic workloads for the segmented delta-rule forward.

This module holds no arithmetic of the method: it only draws inputs.  The
CUDA path and the CPU oracle both consume what it returns, so it is the one
piece of code they share.

Workloads follow the shapes and value distributions of the article's test
matrix and of the five workload descriptions this library is measured on
(the article, "flash-linear-attention 上下文并行CP ...", §5.1, gives the
CP2/CP4/CP8 cut patterns; no dataset is involved anywhere):

* q, k ~ N(0, 1), L2-normalised per (token, head) in fp32, then rounded to
  the input dtype; v ~ N(0, 1); beta = sigmoid(N(mu_b, s_b)).
* Gates are fp32 natural-log gates g = log(alpha):
  GDN (scalar) alpha = sigmoid(N(mu, s)) per (token, head);
  KDA (per key dim) alpha = sigmoid(N(mu, s)) per (token, head, dim);
  "slow" alpha = 1 - 1e-3 u, u ~ U(0, 1) (the merge-sensitive workload).
* Draw order: (varlen lengths,) q, k, v, beta, gate -- from one generator
  seeded with ``seed`` (default 1000 + workload index).  With grouped query
  heads q is drawn with Hq heads.  Tokens are drawn i.i.d., so a draw serves
  as sequence-ordered input or, unchanged, as zigzag-ordered memory alike.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch
import torch.nn.functional as F


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    gate: str                  # "gdn" (scalar) or "kda" (per key dim)
    dtype: str                 # "fp32" or "bf16" for q, k, v, beta (and o)
    B: int
    T: int                     # tokens per row; total tokens when packed
    H: int
    d: int                     # dk == dv
    R: int                     # contiguous segments (virtual context ranks)
    gate_dist: tuple = ("sigmoid", 2.0, 1.0)
    beta_dist: tuple = (0.0, 1.0)
    num_seqs: int = 0          # > 0: packed varlen batch of that many sequences
    len_range: tuple = (1024, 12288)
    lengths: Optional[tuple] = None  # explicit packed lengths (overrides the draw)
    seed: int = 0
    Hq: int = 0                # > 0: query heads of q and o (grouped query heads, a multiple of H)
    layout: str = "contiguous"  # token layout: "contiguous" or "zigzag"
    state_v_first: bool = False  # dk x dv states stored [dv, dk]
    op: str = "delta"          # "delta" (the delta-rule path) or "conv1d" (causal conv1d only)
    conv_width: int = 0        # conv1d: kernel size W
    conv_channels: int = 0     # conv1d: channels C of x [B, T, C]

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    @property
    def tokens(self) -> int:
        return self.B * self.T


# The five measured workloads (index = seed offset) and the added cases.
WORKLOADS = {
    "gdn_fp32_t1024_h2_d64_r4": Workload("gdn_fp32_t1024_h2_d64_r4", "gdn", "fp32", 1, 1024, 2, 64, 4,
                                         seed=1000),
    "gdn_bf16_b2_t8192_h16_d128_r8": Workload("gdn_bf16_b2_t8192_h16_d128_r8", "gdn", "bf16", 2, 8192, 16,
                                              128, 8, seed=1001),
    "kda_bf16_t32768_h32_d128_r16": Workload("kda_bf16_t32768_h32_d128_r16", "kda", "bf16", 1, 32768, 32,
                                             128, 16, gate_dist=("sigmoid", 3.0, 1.0), seed=1002),
    "gdn_bf16_varlen65536_n12_h16_d128_r32": Workload("gdn_bf16_varlen65536_n12_h16_d128_r32", "gdn", "bf16",
                                                      1, 65536, 16, 128, 32, num_seqs=12, seed=1003),
    "gdn_bf16_t262144_h16_d128_r64": Workload("gdn_bf16_t262144_h16_d128_r64", "gdn", "bf16", 1, 262144, 16,
                                              128, 64, gate_dist=("sigmoid", 4.0, 0.5), seed=1004),
    # merge-sensitive: slow decay so that cross-segment state dominates
    "merge_fp32_t16384_h4_d128_r16": Workload("merge_fp32_t16384_h4_d128_r16", "gdn", "fp32", 1, 16384, 4, 128,
                                              16, gate_dist=("slow",), beta_dist=(-3.0, 1.0), seed=1005),
    "merge_bf16_t16384_h4_d128_r16": Workload("merge_bf16_t16384_h4_d128_r16", "gdn", "bf16", 1, 16384, 4, 128,
                                              16, gate_dist=("slow",), beta_dist=(-3.0, 1.0), seed=1006),
}
# layout variants of the headline shape: zigzag token order, [dv, dk]
# states, and two query heads per state head
WORKLOADS.update({
    "gdn_bf16_t262144_h16_d128_r64_zigzag": Workload("gdn_bf16_t262144_h16_d128_r64_zigzag", "gdn", "bf16", 1,
                                                     262144, 16, 128, 64, gate_dist=("sigmoid", 4.0, 0.5),
                                                     seed=1004, layout="zigzag"),
    "gdn_bf16_t262144_h16_d128_r64_vfirst": Workload("gdn_bf16_t262144_h16_d128_r64_vfirst", "gdn", "bf16", 1,
                                                     262144, 16, 128, 64, gate_dist=("sigmoid", 4.0, 0.5),
                                                     seed=1004, state_v_first=True),
    "gdn_bf16_t262144_h16_hq32_d128_r64": Workload("gdn_bf16_t262144_h16_hq32_d128_r64", "gdn", "bf16", 1,
                                                   262144, 16, 128, 64, gate_dist=("sigmoid", 4.0, 0.5),
                                                   seed=1004, Hq=32),
})
# causal conv1d of the q, k, v projections (3 H d channels) at the headline shape
WORKLOADS.update({
    "conv_bf16_t262144_c6144_w4_r64": Workload("conv_bf16_t262144_c6144_w4_r64", "gdn", "bf16", 1, 262144, 16,
                                               128, 64, seed=1010, op="conv1d", conv_width=4, conv_channels=6144),
})
WORKLOAD_ORDER = list(WORKLOADS)[:5]
HEADLINE = "gdn_bf16_t262144_h16_d128_r64"


def varlen_lengths(total: int, n: int, lo: int, hi: int, seed: int) -> list:
    """n lengths summing to ``total``, each in [lo, hi].

    Draw n uniform lengths in [lo, hi], rescale by total/sum, floor, and give
    the remainder to the last one; redraw with seed+1, seed+2, ... until every
    length lies in [lo, hi].
    """
    for attempt in range(1000):
        g = torch.Generator().manual_seed(seed + attempt)
        raw = lo + (hi - lo) * torch.rand(n, generator=g, dtype=torch.float64)
        scaled = [int(math.floor(float(x) * total / float(raw.sum()))) for x in raw]
        scaled[-1] += total - sum(scaled)
        if all(lo <= x <= hi for x in scaled):
            return scaled
    raise RuntimeError("could not draw varlen lengths")


def cu_from_lengths(lengths: Sequence[int]) -> torch.Tensor:
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + int(x))
    return torch.tensor(cu, dtype=torch.int64)


def _gate(w: Workload, shape, gen, device):
    kind = w.gate_dist[0]
    if kind == "sigmoid":
        mu, s = w.gate_dist[1], w.gate_dist[2]
        return F.logsigmoid(mu + s * torch.randn(shape, generator=gen, device=device, dtype=torch.float32))
    if kind == "slow":
        u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
        return torch.log1p(-1e-3 * u)
    raise ValueError(kind)


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None, T: Optional[int] = None,
                B: Optional[int] = None, H: Optional[int] = None, lengths: Optional[Sequence[int]] = None,
                Hq: Optional[int] = None):
    """Draw one batch for workload ``w`` (optionally with shapes overridden).

    Returns a dict with q, k, v, beta (input dtype), g (fp32), cu_seqlens
    (int64 CPU tensor or None) and the shapes used.
    """
    seed = w.seed if seed is None else seed
    B = w.B if B is None else B
    T = w.T if T is None else T
    H = w.H if H is None else H
    if Hq is None:   # keep the workload's query heads per state head
        Hq = H * (w.Hq // w.H) if w.Hq else H
    d = w.d
    cu = None
    if lengths is None and w.lengths is not None:
        lengths = w.lengths
    if lengths is None and w.num_seqs:
        lengths = varlen_lengths(T, w.num_seqs, w.len_range[0], w.len_range[1], seed)
    if lengths is not None:
        cu = cu_from_lengths(lengths)
        B, T = 1, int(cu[-1])
    gen = torch.Generator(device=device).manual_seed(seed)
    dt = w.torch_dtype

    def unit(shape):
        x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        return (x / x.norm(dim=-1, keepdim=True)).to(dt)

    q = unit((B, T, Hq, d))
    k = unit((B, T, H, d))
    v = torch.randn((B, T, H, d), generator=gen, device=device, dtype=torch.float32).to(dt)
    mb, sb = w.beta_dist
    beta = torch.sigmoid(mb + sb * torch.randn((B, T, H), generator=gen, device=device,
                                               dtype=torch.float32)).to(dt)
    gshape = (B, T, H) if w.gate == "gdn" else (B, T, H, d)
    g = _gate(w, gshape, gen, device)
    return dict(q=q, k=k, v=v, beta=beta, g=g, cu_seqlens=cu, B=B, T=T, H=H, d=d, R=w.R,
                gate=w.gate, dtype=w.dtype, Hq=Hq, layout=w.layout, state_v_first=w.state_v_first)


def make_conv_inputs(w: Workload, device="cpu", seed: Optional[int] = None, T: Optional[int] = None,
                     B: Optional[int] = None, C: Optional[int] = None, lengths: Optional[Sequence[int]] = None):
    """Draw x [B, T, C] ~ N(0, 1) in the input dtype, weight [C, W] ~ N(0, 1/W)
    and bias [C] ~ N(0, 0.1^2) in fp32 (draw order: lengths, x, weight, bias)."""
    seed = w.seed if seed is None else seed
    B = w.B if B is None else B
    T = w.T if T is None else T
    C = w.conv_channels if C is None else C
    W = w.conv_width
    cu = None
    if lengths is None and w.lengths is not None:
        lengths = w.lengths
    if lengths is None and w.num_seqs:
        lengths = varlen_lengths(T, w.num_seqs, w.len_range[0], w.len_range[1], seed)
    if lengths is not None:
        cu = cu_from_lengths(lengths)
        B, T = 1, int(cu[-1])
    gen = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn((B, T, C), generator=gen, device=device, dtype=torch.float32).to(w.torch_dtype)
    weight = torch.randn((C, W), generator=gen, device=device, dtype=torch.float32) / math.sqrt(W)
    bias = 0.1 * torch.randn((C,), generator=gen, device=device, dtype=torch.float32)
    return dict(x=x, weight=weight, bias=bias, cu_seqlens=cu, B=B, T=T, C=C, W=W, R=w.R, dtype=w.dtype,
                layout=w.layout)
