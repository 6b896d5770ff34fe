"""The allocation-free entry point (cpdr_forward_noalloc).

It serves callers that cannot allocate device memory (code inside a runtime
that owns all device memory through its own pool or static memory plan):
the library keeps its exchange buffers, plan tables and status word in one
fixed device array instead.  Here its outputs are checked, through the C
ABI, on two calls in a row, against the regular entry points (preprocess ->
merge -> fwd with caller-owned buffers) and against the fp64 oracle, with
the tolerances the parity tests use, on the tensor-core path (scalar and
per-dim gate, fixed-length and packed) and on the CUDA-core path.  The
context is created host-only, so the library allocates no device memory at
all; after every call the array's status word must read clear.
This file is collected last.
"""
import pytest
import torch

from context_merge_gb300 import cpdr, inputs
from _parity import compare, run_oracle

pytestmark = pytest.mark.gpu

CASES = [
    # (workload, overrides, tolerance kind)
    ("gdn_bf16_b2_t8192_h16_d128_r8", dict(B=1, T=2048, H=4), "bf16"),     # tcgen05 kernels
    ("gdn_bf16_b2_t8192_h16_d128_r8", dict(B=1, T=2048, H=4, Hq=8), "bf16"),  # two query heads per chain
    ("gdn_bf16_varlen65536_n12_h16_d128_r32", dict(lengths=[700, 1100, 248]), "bf16"),
    ("kda_bf16_t32768_h32_d128_r16", dict(T=2048, H=2, R=4), "bf16"),       # per-dim gate
    ("kda_bf16_t32768_h32_d128_r16", dict(T=2048, H=2, R=4, Hq=4), "bf16"),  # and grouped query heads
    ("gdn_fp32_t1024_h2_d64_r4", {}, "fp32"),                                # CUDA-core kernels
]


def rel_err(x, ref, kind):
    x, ref = x.double(), ref.double()
    if kind == "fp32":
        return float((x - ref).abs().max() / ref.abs().max())
    return float((x - ref).norm() / ref.norm())


@pytest.mark.parametrize("name,kw,kind", CASES, ids=[c[0] + ("-gqa" if "Hq" in c[1] else "") for c in CASES])
def test_noalloc_matches_regular_entry_points(cpdr_lib, name, kw, kind):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    w = inputs.WORKLOADS[name]
    kw = dict(kw)
    lengths = kw.pop("lengths", None)
    R = kw.pop("R", w.R if lengths is None else 2)
    inp = inputs.make_inputs(w, device="cuda", lengths=lengths, **kw)
    q, k, v, beta, g = (inp[x] for x in ("q", "k", "v", "beta", "g"))
    args = (inp["B"], inp["T"], inp["H"], inp["d"], R)
    Hq = inp["Hq"]
    ref_ctx = cpdr.Context(*args, gate=w.gate, dtype=w.dtype, cu_seqlens=inp["cu_seqlens"], Hq=Hq)
    o_ref, bufs = ref_ctx.run(q, k, v, beta, g)
    torch.cuda.synchronize()
    ctx = cpdr.Context(*args, gate=w.gate, dtype=w.dtype, cu_seqlens=inp["cu_seqlens"], host_only=True, Hq=Hq)
    tol = 1e-4 if kind == "fp32" else 2e-2
    cpu = {x: inp[x].cpu() for x in ("q", "k", "v", "beta", "g")}
    ref = run_oracle(dict(inp, **cpu, R=R))
    for _ in range(2):   # two calls in a row share (and must clear) the static scratch
        o = torch.full_like(o_ref, float("nan"))
        fs = torch.full_like(bufs["final_state"], float("nan"))
        ctx.forward_noalloc(q, k, v, beta, g, o, fs)
        torch.cuda.synchronize()
        ctx.check_device_status()      # the array's status word: no wait gave up
        assert torch.isfinite(o.float()).all() and torch.isfinite(fs).all()
        assert rel_err(o, o_ref, kind) <= tol
        assert rel_err(fs, bufs["final_state"], kind) <= tol
        compare(dict(o=o.cpu(), final_state=fs.cpu()), ref, dict(inp, R=R), check_exchange=False)


def test_noalloc_rejects_problems_beyond_its_scratch(cpdr_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    # T = 262144, H = 16, R = 64: 3 x 64 x 16 x 64 KiB of exchange buffers and
    # 4096 x 16 x 24 KiB of WY tiles >> 32 MiB
    ctx = cpdr.Context(1, 262144, 16, 128, 64, gate="gdn", dtype="bf16", host_only=True)
    x = torch.zeros(16, device="cuda")
    with pytest.raises(cpdr.CpdrError) as ei:
        cpdr_lib_call = ctx._lib.cpdr_forward_noalloc
        cpdr._check(cpdr_lib_call(ctx._h, *[cpdr._ptr(x)] * 7, cpdr._stream(None)))
    assert ei.value.status == cpdr.ERR_WORKSPACE
    assert b"33554432" in cpdr_lib.cpdr_last_error()
