"""GPU parity of the layout variants against the fp64 oracle.

* zigzag token layout ([FLA-CP] §3.2): inputs are gathered into zigzag memory
  order with the oracle's index map, the path runs on them, and o comes back
  to sequence order; the oracle runs on sequence-ordered inputs over the 2R
  parts.
* state_v_first ([FLA-CP] §5.1): S_ext, S_init and final_state are [dv, dk]
  and are transposed back before comparison; M keeps [dk, dk].
* grouped query heads ([FLA-CP] §5.1, Hq > H): q and o have Hq = G H heads,
  query head hq reading the state of head hq // G.

[FLA-CP] is the article "flash-linear-attention 上下文并行CP 从 CP2TP、Ring CP
到 True CP 的设计取舍与源码实现".  Tolerances are those of tests/_parity.py.
"""
import dataclasses

import pytest
import torch

from context_merge_gb300 import inputs
from _parity import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

W = inputs.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _cuda(cpdr_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)


VARIANTS = {
    "zigzag": dict(layout="zigzag"),
    "vfirst": dict(state_v_first=True),
    "gqa2": dict(Hq=4),
    "gqa3-vfirst-zigzag": dict(Hq=6, layout="zigzag", state_v_first=True),
    "gqa4": dict(Hq=8),
}
CUTS = [
    ([3000, 4000, 3240], 2),
    ([7000, 3240], 4),
    ([400, 624], 2),
    ([10240], 4),
]


def workload(gate, dtype, B, T, H, d, R, seed, **variant):
    base = W["kda_bf16_t32768_h32_d128_r16"] if gate == "kda" else W["gdn_bf16_b2_t8192_h16_d128_r8"]
    return inputs.Workload("layout", gate, dtype, B, T, H, d, R, gate_dist=base.gate_dist, seed=seed, **variant)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("gate", ["gdn", "kda"])
@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("cut", CUTS, ids=[f"R{r}-{'-'.join(map(str, l))}" for l, r in CUTS])
def test_variant_cut_patterns(cut, variant, gate, dtype):
    lengths, R = cut
    w = workload(gate, dtype, 1, sum(lengths), 2, 128, R, 31, **VARIANTS[variant])
    inp = inputs.make_inputs(w, device="cpu", lengths=lengths)
    print(cut, variant, gate, dtype, compare(run_gpu(inp), run_oracle(inp), inp))


TINY = [
    # (B, T, lengths, R, d)
    (1, 2, None, 1, 128),
    (1, 130, None, 1, 128),
    (2, 264, None, 3, 128),
    (1, 200, [1, 63, 0, 64, 71, 1], 2, 128),
    (1, 128, [1] * 128, 32, 128),
    (1, 260, None, 2, 64),
    (3, 96, None, 4, 64),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("case", TINY, ids=[str(i) for i in range(len(TINY))])
def test_variant_tiny_and_ragged(case, variant, dtype):
    B, T, lengths, R, d = case
    w = workload("gdn", dtype, B, T, 3, d, R, 33, **VARIANTS[variant])
    inp = inputs.make_inputs(w, device="cpu", lengths=lengths)
    print(case, variant, compare(run_gpu(inp), run_oracle(inp), inp))


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_variant_fp32_cuda_core_cross_check(variant):
    w = workload("gdn", "bf16", 1, 4096, 4, 128, 4, 35, **VARIANTS[variant])
    inp = inputs.make_inputs(w, device="cpu")
    print(variant, compare(run_gpu(inp, force_simt=True), run_oracle(inp), inp))


@pytest.mark.parametrize("name", ["gdn_bf16_t262144_h16_d128_r64_zigzag", "gdn_bf16_t262144_h16_d128_r64_vfirst",
                                  "gdn_bf16_t262144_h16_hq32_d128_r64"])
def test_variant_workload(name):
    """The benchmarked variant workloads in their launch configuration, on a
    quarter of the tokens (T = 65536, R = 64 keeps 1024-token segments of
    16 chunks) so the oracle stays within seconds per head."""
    w = dataclasses.replace(W[name], T=65536)
    inp = inputs.make_inputs(w, device="cuda")
    for key in ("q", "k", "v", "beta", "g"):
        inp[key] = inp[key].cpu()
    gpu = run_gpu(inp)
    print(name, compare(gpu, run_oracle(inp), inp), gpu["counts"])
