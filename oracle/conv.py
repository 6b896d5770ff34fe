"""fp64 oracle of the causal depthwise conv1d that precedes the delta rule.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle``: the tests and the
benchmark's CPU-baseline leg call it; the CUDA library shares nothing with it.

Source: the article "flash-linear-attention 上下文并行CP 从 CP2TP、Ring CP 到
True CP 的设计取舍与源码实现" ([FLA-CP]).  §2.4: the conv looks only at the
W - 1 tokens before each token, so in context parallelism a rank fetches the
tail of the previous rank's tokens (zero for the first rank); §3.2-§3.3: the
context carries conv1d_kernel_size and pre_num_conv_tokens, the number of
tokens the local interval's first sequence extends before it.  The pages
give no formula for the conv itself; the reading here is the usual causal
depthwise one, zero before each sequence start,

    y[t, c] = act(bias[c] + sum_{i=0}^{W-1} weight[c, i] * x[t - (W-1) + i, c]),

act = identity or SiLU z * sigmoid(z).  Everything is in sequence order
(the zigzag memory order is undone by the caller with ``oracle.layout``).
"""
from __future__ import annotations

import numpy as np


def _as64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float64)


def causal_conv1d(x, weight, bias=None, cu_seqlens=None, activation="silu"):
    """x [B, T, C] (sequence order), weight [C, W], bias [C] or None.

    With ``cu_seqlens`` (N+1 offsets) the batch is packed (B == 1) and every
    sequence is convolved on its own.  Returns y [B, T, C] in fp64.
    """
    x = _as64(x)
    w = _as64(weight)
    B, T, C = x.shape
    W = w.shape[1]
    b = np.zeros(C) if bias is None else _as64(bias)
    if cu_seqlens is None:
        bounds = [(bb, 0, T) for bb in range(B)]
    else:
        cu = [int(v) for v in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
        bounds = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    y = np.zeros_like(x)
    for bb, s, e in bounds:
        for t in range(s, e):
            acc = b.copy()
            for i in range(W):
                src = t - (W - 1) + i
                if src >= s:
                    acc += w[:, i] * x[bb, src]
            y[bb, t] = acc
    if activation == "silu":
        y = y / (1.0 + np.exp(-y))
    elif activation not in (None, "none"):
        raise ValueError(activation)
    return y


def pre_num_conv_tokens(cu_seqlens, total, R, W, zigzag=False):
    """Per segment (sequence order; 2R parts with zigzag): how many of the
    W - 1 tokens before its start belong to the sequence it starts in."""
    cu = [int(v) for v in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    parts = 2 * R if zigzag else R
    L = total // parts
    out = []
    for r in range(parts):
        s0 = r * L
        # the sequence that holds token s0
        n = next(i for i in range(len(cu) - 1) if cu[i] <= s0 < cu[i + 1])
        out.append(min(W - 1, s0 - cu[n]))
    return out
