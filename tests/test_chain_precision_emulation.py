"""Why the transfer-matrix chain and the merge need split operands (CPU).

The article ("flash-linear-attention 上下文并行CP ...", [FLA-CP] §2.2) requires
the chain M <- M_[t] M, M_[t] = Diag(gamma^C) - (Gamma ⊙ K)^T W, to stay at
fp32 accuracy (§3.2 names the tf32x3 dot as the way to get there on tensor
cores).  The tensor-core kernels take every operand that carries a rounded
quantity -- T'' = T diag(beta gamma), W, M and Delta diag(Gamma) -- as a bf16
hi/lo pair and form each product as hi*hi + lo*hi + hi*lo with fp32
accumulation (the bf16x3 analogue of tf32x3); the merge S <- M_j S + S_ext,j
does the same with M_j and S.

This module emulates those rounding points in numpy on the merge-sensitive
workload (slow decay, so the transfer matrices stay O(1) over a whole
segment) and checks, against the fp64 oracle's M and S_init:

* with every operand split, the error is far inside the 1e-4 bound that
  the GPU tests (tests/test_gpu_chain_precision.py) put on the kernels;
* a single-pass bf16 chain -- and a chain that drops the lo half of any one
  of the four rounded operands -- exceeds that bound, so each GPU test would
  fail on such a regression; likewise a single-pass merge.

The emulation products run in float32 (fp32 accumulation, as the tensor
cores' TMEM accumulators); the WY inverse is taken in fp64 and rounded to
fp32, as the kernel's fp32 block solve delivers it.
"""
import numpy as np
import pytest
import torch

import oracle
from context_merge_gb300 import inputs

BOUND = 1e-4
OPERANDS = ("T", "W", "M", "D")


def bf16(x):
    """Round to bf16 (round to nearest even) and return float32."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def pair(x, split):
    """(hi, lo) bf16 pair of x; lo is zero for a single-pass operand."""
    hi = bf16(x)
    lo = bf16(np.asarray(x, np.float32) - hi) if split else np.zeros_like(hi)
    return hi, lo


def mm(a, b):
    """hi*hi + lo*hi + hi*lo in float32 (the lo*lo term is dropped, as on the GPU)."""
    (ah, al), (bh, bl) = a, b
    return (ah @ bh + al @ bh + ah @ bl).astype(np.float32)


def m_chain(k, beta, g, split, C=64):
    """Transfer matrix of one fragment from M_0 = I with the kernel's rounding
    points; ``split`` maps each rounded operand ("T", "W", "M", "D") to True
    (hi/lo pair) or False (single bf16)."""
    d = k.shape[1]
    Mx = np.eye(d, dtype=np.float32)
    for c0 in range(0, k.shape[0], C):
        K = k[c0:c0 + C].astype(np.float32)           # exact bf16 values
        b = beta[c0:c0 + C].astype(np.float64)
        G = np.cumsum(g[c0:c0 + C].astype(np.float64))
        n = K.shape[0]
        Kd = K.astype(np.float64)
        A = np.tril(b[:, None] * (Kd @ Kd.T) * np.exp(G[:, None] - G[None, :]), -1)
        T = np.linalg.inv(np.eye(n) + A).astype(np.float32)
        T2 = (T * (b * np.exp(G))[None, :]).astype(np.float32)       # T'' = T diag(beta gamma)
        W = mm(pair(T2, split["T"]), (K, np.zeros_like(K)))           # W = T'' K
        # Delta = -W M  (as -M^T W^T in the kernel: both orders give the same sums)
        Dl = -mm(pair(W, split["W"]), pair(Mx, split["M"]))
        Gam = np.exp(G[-1] - G).astype(np.float32)
        DG = (Dl * Gam[:, None]).astype(np.float32)
        PS = mm((K.T.copy(), np.zeros_like(K.T)), pair(DG, split["D"]))   # (Gamma ⊙ K)^T Delta
        Mx = (np.float32(np.exp(G[-1])) * Mx + PS).astype(np.float32)
    return Mx


def rel(x, ref):
    return float(np.linalg.norm(np.asarray(x, np.float64) - ref) / np.linalg.norm(ref))


@pytest.fixture(scope="module")
def merge_case():
    """merge_bf16_t16384_h4_d128_r16, head 0 (16 chunks per segment)."""
    w = inputs.WORKLOADS["merge_bf16_t16384_h4_d128_r16"]
    inp = inputs.make_inputs(w, device="cpu", H=1)
    ref = oracle.Problem(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"]).segmented(w.R)
    arr = {x: inp[x][0, :, 0].float().numpy() for x in ("k", "beta", "g")}
    return w, inp, ref, arr


def chain_errors(merge_case, split, segs=(0, 7, 14)):
    w, inp, ref, a = merge_case
    L = inp["T"] // w.R
    out = []
    for r in segs:
        sl = slice(r * L, (r + 1) * L)
        out.append(rel(m_chain(a["k"][sl], a["beta"][sl], a["g"][sl], split), ref["M"][r, 0, 0]))
    return max(out)


def test_transfer_matrices_are_order_one(merge_case):
    """The workload keeps M far from underflow, so relative errors are meaningful."""
    _, _, ref, _ = merge_case
    norms = [np.linalg.norm(ref["M"][r, 0, 0]) for r in range(ref["M"].shape[0] - 1)]
    assert min(norms) > 1.0 and max(norms) < 20.0


def test_split_chain_meets_bound(merge_case):
    e = chain_errors(merge_case, {o: True for o in OPERANDS})
    assert e < BOUND / 10, e


def test_single_pass_chain_fails_bound(merge_case):
    e = chain_errors(merge_case, {o: False for o in OPERANDS})
    assert e > 3 * BOUND, e


@pytest.mark.parametrize("dropped", OPERANDS)
def test_dropping_any_lo_half_fails_bound(merge_case, dropped):
    split = {o: o != dropped for o in OPERANDS}
    e = chain_errors(merge_case, split)
    assert e > BOUND, (dropped, e)


def merge_scan(S_ext, M, split):
    """S_init[r] for r >= 1 of one (row, head): S <- M_j S + S_ext,j with the
    tensor-core merge's rounding points (fp32 inputs, as in HBM)."""
    R = S_ext.shape[0]
    S = np.zeros_like(S_ext[0], dtype=np.float32)
    out = [S.copy()]
    for j in range(R - 1):
        S = (mm(pair(M[j].astype(np.float32), split), pair(S, split)) + S_ext[j].astype(np.float32)).astype(np.float32)
        out.append(S.copy())
    return out


def test_merge_split_meets_bound_and_single_pass_fails(merge_case):
    _, _, ref, _ = merge_case
    S_ext, M = ref["S_ext"][:, 0, 0], ref["M"][:, 0, 0]
    for split, ok in ((True, True), (False, False)):
        got = merge_scan(S_ext, M, split)
        e = max(rel(got[r], ref["S_init"][r, 0, 0]) for r in range(1, len(got)))
        if ok:
            assert e < BOUND / 10, e
        else:
            assert e > 3 * BOUND, e
