"""GPU parity of the backward (cpdr_bwd) against the fp64 backward oracle
(the reverse of the per-token scan, pinned by finite differences): the
article's cut patterns at R = 2/4/8, fixed rows, packed batches with short
and empty sequences, the zigzag layout, both gates and both dtypes, with and
without a final-state gradient, and longer chains on the headline's and the
merge-sensitive gate distributions, grouped query heads (G = 2, 3) on both
gates with [dv, dk] states and the zigzag layout.  The forward path (WY build,
pre-process, merge) runs first through the C-ABI and its S_init and M feed
the backward.

Bars, per gradient tensor and per (sequence, head), ||x - ref|| / ||ref||:
fp32 inputs 1e-4 (the fp32 CUDA-core path, forward included); bf16 inputs
5e-3, the article's gradient acceptance line ([FLA-CP] §5.2).  For bf16,
d = 128 and the scalar gate the backward runs on the tensor cores (the
recomputed states and the state-gradient chain with bf16 operands, the
input gradients with tf32 products); its errors sit near 1e-3 to 2.6e-3."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from context_merge_gb300 import cpdr, inputs
from oracle import layout as olayout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(cpdr_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)


def run_case(w, lengths=None, with_dht=True, seed=7, whole_tensor=False, **kw):
    inp = inputs.make_inputs(w, device="cpu", lengths=lengths, **kw)
    B, T, H, d, R = inp["B"], inp["T"], inp["H"], inp["d"], inp["R"]
    Hq = inp["Hq"]
    gen = torch.Generator().manual_seed(seed)
    do = torch.randn((B, T, Hq, d), generator=gen).to(w.torch_dtype)
    N = B if inp["cu_seqlens"] is None else len(inp["cu_seqlens"]) - 1
    dht = torch.randn((N, H, d, d), generator=gen) if with_dht else None
    zig = w.layout == "zigzag"
    vf = bool(w.state_v_first)
    ctx = cpdr.Context(B, T, H, d, R, gate=w.gate, dtype=w.dtype, cu_seqlens=inp["cu_seqlens"], layout=w.layout,
                       state_v_first=vf, Hq=Hq)
    place = (lambda x: olayout.to_zigzag(x, R)) if zig else (lambda x: x)
    dev = {k: place(inp[k]).contiguous().cuda() for k in ("q", "k", "v", "beta", "g")}
    o, bufs = ctx.run(dev["q"], dev["k"], dev["v"], dev["beta"], dev["g"])
    dht_dev = None
    if dht is not None:   # [dv, dk] states take dht transposed
        dht_dev = (dht.transpose(-1, -2) if vf else dht).contiguous().cuda()
    grads = ctx.backward(dev["q"], dev["k"], dev["v"], dev["beta"], dev["g"], place(do).contiguous().cuda(),
                         bufs["S_init"], bufs["M"], dht=dht_dev)
    torch.cuda.synchronize()
    ctx.check_device_status()
    unplace = (lambda x: olayout.from_zigzag(x, R)) if zig else (lambda x: x)
    got = {k: unplace(v.cpu()).double().numpy() for k, v in grads.items()}
    ref = oracle.Problem(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], cu_seqlens=inp["cu_seqlens"]).backward(
        do, dht=dht.double().numpy() if dht is not None else None)
    cu = [int(x) for x in inp["cu_seqlens"]] if inp["cu_seqlens"] is not None else None
    errs = {}
    # whole_tensor: the norm ratio over each gradient tensor, as the article's
    # acceptance test compares them ([FLA-CP] §5.2); a tensor whose reference
    # is zero (the gate gradient of one-token sequences from a zero state) is
    # measured against 1e-3 of the largest gradient norm of the problem
    scale_all = max(np.linalg.norm(ref[k]) for k in ("dq", "dk", "dv", "dbeta", "dg"))
    for key in ("dq", "dk", "dv", "dbeta", "dg"):
        worst = 0.0
        if whole_tensor:
            den = max(np.linalg.norm(ref[key]), 1e-3 * scale_all)
            errs[key] = float(np.linalg.norm(got[key] - ref[key]) / den)
            continue
        spans = [(b, 0, T) for b in range(B)] if cu is None else [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
        for b, s, e in spans:
            if e == s:
                continue
            for h in range(Hq if key == "dq" else H):
                x, r = got[key][b, s:e, h], ref[key][b, s:e, h]
                den = np.linalg.norm(r)
                num = np.linalg.norm(x - r)
                worst = max(worst, float(num / den) if den > 0 else float(num > 0) * np.inf)
        errs[key] = worst
    tol = 1e-4 if w.dtype == "fp32" else 5e-3
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"over tolerance: {bad} (all: {errs})"
    return errs


CUTS = [([3000, 4000, 3240], 2), ([7000, 3240], 4), ([400, 624], 2), ([2048], 8), ([300, 0, 17, 700, 7], 4)]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("gate", ["gdn", "kda"])
@pytest.mark.parametrize("cut", CUTS, ids=[f"R{r}-{'-'.join(map(str, l))}" for l, r in CUTS])
def test_backward_cut_patterns(cut, gate, dtype):
    lengths, R = cut
    base = inputs.WORKLOADS["kda_bf16_t32768_h32_d128_r16" if gate == "kda" else "gdn_bf16_b2_t8192_h16_d128_r8"]
    w = inputs.Workload("bwd", gate, dtype, 1, sum(lengths), 2, 128, R, gate_dist=base.gate_dist, seed=41)
    print(cut, gate, dtype, run_case(w, lengths=lengths))


@pytest.mark.parametrize("case", [
    dict(B=2, T=1024, R=4, d=128, layout="contiguous", dht=True),
    dict(B=3, T=192, R=3, d=64, layout="contiguous", dht=False),
    dict(B=1, T=1024, R=2, d=128, layout="zigzag", dht=True),
    dict(B=1, T=130, R=1, d=64, layout="contiguous", dht=True),
])
def test_backward_rows_and_layouts(case):
    w = inputs.Workload("bwd", "gdn", "bf16", case["B"], case["T"], 2, case["d"], case["R"], seed=43,
                        layout=case["layout"])
    print(case, run_case(w, with_dht=case["dht"]))


@pytest.mark.parametrize("name,kw", [
    ("gdn_bf16_t262144_h16_d128_r64", dict(T=16384, H=2, R=16)),    # headline gate, 16-chunk fragments
    ("merge_bf16_t16384_h4_d128_r16", dict(T=8192, H=2, R=8)),      # slow decay: cross-segment gradients matter
], ids=["headline-gate", "merge-sensitive"])
def test_backward_long_chains(name, kw):
    kw = dict(kw)
    w = dataclasses.replace(inputs.WORKLOADS[name], R=kw.pop("R"))
    print(name, run_case(w, **kw))


@pytest.mark.parametrize("case", [
    dict(T=4096, H=2, R=8, gate_dist=None),                       # the per-dim workload's gates, 8-chunk fragments
    dict(T=2048, H=2, R=4, gate_dist=("sigmoid", -3.0, 0.5)),     # steep per-dim decay: the exact branch
    dict(T=2048, H=2, R=4, gate_dist=("sigmoid", 1.0, 2.5)),      # a wide spread of per-dim decays
], ids=["kda-gates", "kda-steep", "kda-spread"])
def test_backward_per_dim_gate(case):
    """Per-dim gate on the tensor cores (bf16, d = 128): the preparation's T,
    the recomputed forward and the state-gradient chain on the unit's
    pre-gated tiles, the input gradients with the per-dim factors folded into
    the operands (exact per-term exponentials for steep units)."""
    base = inputs.WORKLOADS["kda_bf16_t32768_h32_d128_r16"]
    w = dataclasses.replace(base, R=case["R"], gate_dist=case["gate_dist"] or base.gate_dist)
    print(case, run_case(w, T=case["T"], H=case["H"], lengths=[case["T"] // 3, case["T"] - case["T"] // 3]))


@pytest.mark.parametrize("gate", ["gdn", "kda"])
@pytest.mark.parametrize("lengths,R", [
    ([1], 1), ([63], 1), ([66], 2), ([64, 1, 0, 129], 2), ([3, 61, 2], 3), ([203], 7),
], ids=["t1", "t63", "t65-r2", "mixed-empty", "short-r3", "t200-r7"])
def test_backward_tiny_and_ragged(gate, lengths, R):
    """The tensor-core backward (bf16, d = 128) on one-token fragments, partial
    chunks, sequences shorter than a chunk, an empty sequence, and more
    segments than chunks.  The bar applies to whole gradient tensors: per
    (sequence, head) of a one- to three-token sequence, dbeta is one to three
    scalars, whose relative error is that of a single dot product."""
    base = inputs.WORKLOADS["kda_bf16_t32768_h32_d128_r16" if gate == "kda" else "gdn_bf16_b2_t8192_h16_d128_r8"]
    w = inputs.Workload("bwd", gate, "bf16", 1, sum(lengths), 2, 128, R, gate_dist=base.gate_dist, seed=49)
    print(gate, lengths, R, run_case(w, lengths=lengths, whole_tensor=True))


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp32", 64)])
def test_backward_state_v_first(dtype, d):
    """[dv, dk] states ([FLA-CP] §5.1 runs its gradient tests with state_v_first)."""
    w = inputs.Workload("bwd", "gdn", dtype, 1, 2048, 2, d, 4, seed=45, state_v_first=True)
    print(dtype, d, run_case(w, lengths=[700, 1348]))


@pytest.mark.parametrize("case", [
    dict(gate="gdn", dtype="bf16", G=2, lengths=[700, 1348], R=4),
    dict(gate="kda", dtype="bf16", G=2, lengths=[1000, 0, 1048], R=2),
    dict(gate="gdn", dtype="fp32", G=3, lengths=[517, 1531], R=4, d=64),
    dict(gate="kda", dtype="fp32", G=2, lengths=[2048], R=8),
    dict(gate="gdn", dtype="bf16", G=2, lengths=[2048], R=4, vfirst=True, layout="zigzag"),
    dict(gate="gdn", dtype="bf16", G=3, lengths=[1500, 0, 548], R=4),
    dict(gate="gdn", dtype="bf16", G=2, lengths=[8192], R=8, workload="merge_bf16_t16384_h4_d128_r16"),
    dict(gate="kda", dtype="bf16", G=3, lengths=[1500, 548], R=4),
    dict(gate="kda", dtype="bf16", G=2, lengths=[2048], R=4, vfirst=True, layout="zigzag"),
], ids=["gdn-bf16-g2", "kda-bf16-g2", "gdn-fp32-g3-d64", "kda-fp32-g2", "gdn-bf16-g2-vfirst-zigzag",
        "gdn-bf16-g3", "gdn-bf16-g2-merge-sensitive", "kda-bf16-g3", "kda-bf16-g2-vfirst-zigzag"])
def test_backward_grouped_query_heads(case):
    """G query heads per state ([FLA-CP] §5.1): each state's chain takes the
    scale q do^T of all of its query heads, each query head its own dq (bf16,
    d = 128: the tensor-core backward with a state-gradient chain pass per
    query head, both gates; fp32 and d = 64 on the CUDA-core chain)."""
    base = inputs.WORKLOADS[case.get("workload") or
                            ("kda_bf16_t32768_h32_d128_r16" if case["gate"] == "kda" else "gdn_bf16_b2_t8192_h16_d128_r8")]
    H = 2
    w = inputs.Workload("bwd", case["gate"], case["dtype"], 1, sum(case["lengths"]), H, case.get("d", 128), case["R"],
                        gate_dist=base.gate_dist, seed=47, Hq=H * case["G"], layout=case.get("layout", "contiguous"),
                        state_v_first=case.get("vfirst", False))
    lengths = case["lengths"] if case.get("layout", "contiguous") == "contiguous" else None
    print(case, run_case(w, lengths=lengths))
