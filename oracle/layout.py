"""Token and state layouts of the segmented scheme, written out as index maps.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle``): the tests use these
maps to lay inputs out the way a caller would and to bring results back to
sequence order before comparing them with the oracle.  The CUDA library has
its own planner and shares nothing with this file.

Source: the article "flash-linear-attention 上下文并行CP 从 CP2TP、Ring CP 到
True CP 的设计取舍与源码实现" ([FLA-CP]):

* §3.2 zigzag layout: the token range is cut into 2W equal parts; rank r
  holds part r followed by part 2W-1-r, and its local input is that
  concatenation [front; back].  Laying the W ranks' local inputs side by side
  (rank 0 first) gives the order the tokens have in memory.  On one device
  every part is a segment of its own, so the exchange buffers are indexed by
  part in sequence order, 2W entries.
* §5.1 ``state_v_first``: a state is stored [V, K] instead of [K, V].
"""
from __future__ import annotations

import numpy as np


def zigzag_positions(total: int, W: int) -> np.ndarray:
    """pos[s] = sequence position of the token at memory position s.

    ``total`` tokens (a row, or a packed batch) in the zigzag layout of W
    ranks.  Raises ValueError unless total >= 2W and 2W divides it (the cut
    rule of [FLA-CP] §3.3 for zigzag).
    """
    parts = 2 * W
    if W < 1 or total < parts or total % parts:
        raise ValueError(f"zigzag needs total >= 2W and divisible by 2W (total={total}, W={W})")
    P = total // parts
    order = []
    for r in range(W):
        order += [r, parts - 1 - r]   # rank r: [front part r; back part 2W-1-r]
    return np.concatenate([np.arange(p * P, (p + 1) * P) for p in order]).astype(np.int64)


def to_zigzag(x, W: int, axis: int = 1):
    """Gather a sequence-ordered array into zigzag memory order along ``axis``."""
    pos = zigzag_positions(x.shape[axis], W)
    return _take(x, pos, axis)


def from_zigzag(x, W: int, axis: int = 1):
    """Inverse of ``to_zigzag``: memory order back to sequence order."""
    pos = zigzag_positions(x.shape[axis], W)
    inv = np.empty_like(pos)
    inv[pos] = np.arange(len(pos))
    return _take(x, inv, axis)


def v_first(S):
    """A [..., K, V] state in the ``state_v_first`` layout [..., V, K]."""
    return S.swapaxes(-1, -2)


def _take(x, idx, axis):
    if hasattr(x, "index_select"):   # torch tensor
        import torch
        return x.index_select(axis, torch.as_tensor(idx, device=x.device))
    return np.take(x, idx, axis=axis)
