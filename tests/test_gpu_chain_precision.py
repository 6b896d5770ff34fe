"""fp32-level accuracy of the tensor-core transfer-matrix chain and merge (GPU).

The article ("flash-linear-attention 上下文并行CP ...", [FLA-CP] §2.2) requires
the transfer-matrix chain to stay at fp32 accuracy; the tensor-core kernels
meet it with bf16 hi/lo operand pairs.  The parity tests' bf16 tolerance
(2e-2 relative to the norm) cannot tell a split chain from a single-pass one
(about 1e-3, tests/test_chain_precision_emulation.py), so these tests hold the
kernels to 1e-4 relative Frobenius error against the fp64 oracle:

* M from the pre-process (every input an exact bf16 value, so the oracle's M
  is the exact answer) on the merge-sensitive workload at 16 and 64 chunks
  per segment (64 is the headline's segment length) and on the headline's
  gate distribution at reduced length;
* S_init from the tensor-core merge fed with the oracle's own S_ext and M
  (rounded to fp32), on 16 and 64 segments -- so that the merge is judged on
  its arithmetic alone.

S_ext, S_init from the full path and the outputs keep the bf16 tolerance:
their chain is the single-pass bf16 state chain of the article's kernels.
"""
import numpy as np
import pytest
import torch

from context_merge_gb300 import cpdr, inputs
from _parity import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

BOUND = 1e-4
W = inputs.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _cuda(cpdr_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)


def rel_fro(x, ref):
    x = np.asarray(x, np.float64)
    return float(np.linalg.norm(x - ref) / np.linalg.norm(ref))


CHAIN_CASES = [
    # (workload, overrides): 16 chunks per segment, 64 chunks per segment,
    # the headline gate (sigmoid(N(4, 0.5))) over 1024-token segments
    ("merge_bf16_t16384_h4_d128_r16", {}),
    ("merge_bf16_t16384_h4_d128_r16", dict(T=65536, H=2)),
    ("gdn_bf16_t262144_h16_d128_r64", dict(T=16384, H=4, R=16)),
]


@pytest.mark.parametrize("name,kw", CHAIN_CASES, ids=["16chunks", "64chunks", "headline-gate"])
def test_transfer_matrix_chain_fp32_accuracy(name, kw):
    kw = dict(kw)
    R = kw.pop("R", W[name].R)
    inp = inputs.make_inputs(W[name], device="cpu", **kw)
    inp["R"] = R
    gpu = run_gpu(inp)
    assert gpu["counts"]["tc"] == 1, "the tensor-core kernels must run"
    ref = run_oracle(inp)
    errs = compare(gpu, ref, inp)
    M, Mref = gpu["M"].double().numpy(), ref["M"]
    worst, checked = 0.0, 0
    for r in range(R - 1):           # the last segment has no continuing fragment
        for h in range(inp["H"]):
            mr = Mref[r, 0, h]
            assert np.linalg.norm(mr) > 1e-20, "M must not underflow in this case"
            worst = max(worst, rel_fro(M[r, 0, h], mr))
            checked += 1
    print(name, kw, "M rel. Frobenius error", worst, "over", checked, "matrices;", errs)
    assert worst <= BOUND, worst


MERGE_CASES = [
    ("merge_bf16_t16384_h4_d128_r16", {}, 16),
    ("merge_bf16_t16384_h4_d128_r16", {}, 64),   # 63 merge steps, as at the headline
]


@pytest.mark.parametrize("name,kw,R", MERGE_CASES, ids=["R16", "R64"])
def test_tensor_core_merge_fp32_accuracy(name, kw, R):
    inp = inputs.make_inputs(W[name], device="cpu", **kw)
    inp["R"] = R
    ref = run_oracle(inp)
    assert np.abs(ref["S_init"][-1]).max() > 1e-2, "cross-segment terms must matter"
    ctx = cpdr.Context(inp["B"], inp["T"], inp["H"], inp["d"], R, gate="gdn", dtype="bf16")
    assert ctx.counts()["tc"] == 1
    S_ext = torch.from_numpy(ref["S_ext"].astype(np.float32)).cuda()
    M = torch.from_numpy(ref["M"].astype(np.float32)).cuda()
    S_init = torch.full_like(S_ext, float("nan"))
    ctx.merge(S_ext, M, S_init)
    torch.cuda.synchronize()
    ctx.check_device_status()
    got = S_init.double().cpu().numpy()
    assert not got[0].any()
    worst = max(rel_fro(got[r, 0, h], ref["S_init"][r, 0, h]) for r in range(1, R) for h in range(inp["H"]))
    print(name, R, "S_init rel. Frobenius error", worst)
    assert worst <= BOUND, worst
