"""GPU parity of the causal conv1d (cpdr_conv1d_fwd) against the fp64 oracle
(oracle/conv.py), on the context's segments: the article's cut patterns,
fixed-length rows, the zigzag layout (inputs gathered into zigzag memory
order, outputs brought back), every supported width, both activations and
both dtypes, tiny and ragged cases, and the benchmarked shape on sampled
channels.  [FLA-CP] §2.4, §3.2-§3.3 of "flash-linear-attention 上下文并行CP ...".

Bars: fp32 max|y - ref| <= 1e-5 max|ref|; bf16 elementwise
|y - ref| <= 2^-8 |ref| + 1e-5 max|ref| (one rounding of an fp32 sum).
"""
import dataclasses

import numpy as np
import pytest
import torch

from context_merge_gb300 import cpdr, inputs
from oracle import conv as oconv
from oracle import layout as olayout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(cpdr_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)


def check(y, ref, dtype):
    y = np.asarray(y.float().numpy() if hasattr(y, "float") else y, np.float64)
    assert np.isfinite(y).all()
    m = np.abs(ref).max()
    if dtype == "fp32":
        assert np.abs(y - ref).max() <= 1e-5 * m, np.abs(y - ref).max() / m
    else:
        bad = np.abs(y - ref) > 2.0 ** -8 * np.abs(ref) + 1e-5 * m
        assert not bad.any(), (int(bad.sum()), np.abs(y - ref)[bad].max())


def run(inp, activation, channels=None):
    """Device run through the C-ABI; y in sequence order, on CPU."""
    B, T, C, R = inp["B"], inp["T"], inp["C"], inp["R"]
    zig = inp["layout"] == "zigzag"
    ctx = cpdr.Context(B, T, 1, 64, R, gate="gdn", dtype=inp["dtype"], cu_seqlens=inp["cu_seqlens"],
                       layout=inp["layout"], conv_width=inp["W"])
    x = (olayout.to_zigzag(inp["x"], R) if zig else inp["x"]).contiguous().cuda()
    y = torch.full_like(x, float("nan"))
    bias = inp["bias"].cuda() if inp["bias"] is not None else None
    ctx.conv1d_fwd(x, inp["weight"].cuda(), bias, y, activation=activation)
    torch.cuda.synchronize()
    y = y.cpu()
    return olayout.from_zigzag(y, R) if zig else y


def workload(dtype, W, R, C, layout="contiguous", seed=41, B=1, T=1024):
    return inputs.Workload("conv", "gdn", dtype, B, T, 1, 64, R, seed=seed, op="conv1d", conv_width=W,
                           conv_channels=C, layout=layout)


CUTS = [([3000, 4000, 3240], 2), ([7000, 3240], 4), ([400, 624], 2), ([5118, 5122], 2), ([10240], 8)]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
@pytest.mark.parametrize("cut", CUTS, ids=[f"R{r}-{'-'.join(map(str, l))}" for l, r in CUTS])
def test_cut_patterns(cut, layout, dtype):
    lengths, R = cut
    inp = inputs.make_conv_inputs(workload(dtype, 4, R, 264, layout), lengths=lengths)
    ref = oconv.causal_conv1d(inp["x"], inp["weight"], inp["bias"], cu_seqlens=inp["cu_seqlens"])
    check(run(inp, "silu"), ref, dtype)


@pytest.mark.parametrize("act", ["silu", None])
@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 6, 7, 8])
def test_widths(W, act):
    inp = inputs.make_conv_inputs(workload("bf16", W, 4, 1032, seed=43), lengths=[100, 1, 3, 700, 220])
    ref = oconv.causal_conv1d(inp["x"], inp["weight"], inp["bias"], cu_seqlens=inp["cu_seqlens"], activation=act)
    check(run(inp, act), ref, "bf16")


TINY = [
    # (B, T, lengths, R, layout, W)
    (1, 1, None, 1, "contiguous", 4),
    (1, 2, None, 1, "zigzag", 4),
    (1, 16, [1] * 16, 8, "zigzag", 8),     # one-token parts: the halo spans several parts
    (1, 16, [16], 8, "zigzag", 8),
    (3, 96, None, 4, "zigzag", 4),
    (2, 130, None, 2, "contiguous", 3),
    (1, 200, [1, 63, 0, 64, 71, 1], 2, "zigzag", 5),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("case", TINY, ids=[str(i) for i in range(len(TINY))])
def test_tiny_and_ragged(case, dtype):
    B, T, lengths, R, layout, W = case
    w = dataclasses.replace(workload(dtype, W, R, 8, layout, seed=45), B=B, T=T)
    inp = inputs.make_conv_inputs(w, lengths=lengths)
    ref = oconv.causal_conv1d(inp["x"], inp["weight"], inp["bias"], cu_seqlens=inp["cu_seqlens"])
    check(run(inp, "silu"), ref, dtype)


def test_no_bias():
    inp = inputs.make_conv_inputs(workload("fp32", 4, 2, 64, seed=47), lengths=[300, 724])
    inp["bias"] = None
    ref = oconv.causal_conv1d(inp["x"], inp["weight"], None, cu_seqlens=inp["cu_seqlens"])
    check(run(inp, "silu"), ref, "fp32")


def test_benchmarked_shape_sampled_channels():
    """The benchmark's workload in its launch configuration; the oracle checks
    three 8-channel groups (channels are independent)."""
    w = inputs.WORKLOADS["conv_bf16_t262144_c6144_w4_r64"]
    inp = inputs.make_conv_inputs(w, device="cuda")
    ctx = cpdr.Context(inp["B"], inp["T"], 1, 64, inp["R"], gate="gdn", dtype="bf16", conv_width=inp["W"])
    y = torch.full_like(inp["x"], float("nan"))
    ctx.conv1d_fwd(inp["x"], inp["weight"], inp["bias"], y)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    for c0 in (0, 3000, inp["C"] - 8):
        sl = slice(c0, c0 + 8)
        ref = oconv.causal_conv1d(inp["x"][:, :, sl].cpu(), inp["weight"][sl].cpu(), inp["bias"][sl].cpu())
        check(y[:, :, sl].cpu(), ref, "bf16")
