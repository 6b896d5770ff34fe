"""GPU parity: preprocess -> merge -> fwd through the C-ABI against the fp64
oracle, element by element, on seeded inputs (tolerances in tests/_parity.py).

Cases: the five measured workloads at full size (in the launch configuration
the benchmark times), the article's cut patterns (§5.1, §5.2 of
"flash-linear-attention 上下文并行CP ...") at R = 2/4/8, tiny and ragged
shapes (partial chunks, one-token fragments, an empty sequence), the
merge-sensitive slow-decay workload, and the fp32 CUDA-core path as a
cross-check of the default path.
"""
import pytest
import torch

from context_merge_gb300 import inputs
from _parity import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

W = inputs.WORKLOADS


def gen(name, device="cuda", **kw):
    inp = inputs.make_inputs(W[name], device=device, **kw)
    for key in ("q", "k", "v", "beta", "g"):
        inp[key] = inp[key].cpu()
    return inp


@pytest.fixture(scope="module", autouse=True)
def _cuda(cpdr_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)


@pytest.mark.parametrize("name", inputs.WORKLOAD_ORDER)
def test_workload_full_size(name):
    inp = gen(name)
    gpu = run_gpu(inp)
    errs = compare(gpu, run_oracle(inp), inp)
    print(name, errs, gpu["counts"])


@pytest.mark.parametrize("name", ["merge_fp32_t16384_h4_d128_r16", "merge_bf16_t16384_h4_d128_r16"])
def test_merge_sensitive(name):
    inp = gen(name)
    gpu = run_gpu(inp)
    ref = run_oracle(inp)
    # the cross-segment terms matter here: S_init is far from zero
    assert abs(ref["S_init"][-1]).max() > 1e-2
    print(name, compare(gpu, ref, inp))


CUTS = [
    ([3000, 4000, 3240], 2),
    ([5120, 5120], 2),
    ([7000, 3240], 4),
    ([400, 624], 2),
    ([10240], 8),
    ([900, 1100, 700, 1300, 1500, 1240, 1500, 2000], 2),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("gate", ["gdn", "kda"])
@pytest.mark.parametrize("cut", CUTS, ids=[f"R{r}-{'-'.join(map(str, l))}" for l, r in CUTS])
def test_article_cut_patterns(cut, gate, dtype):
    lengths, R = cut
    base = W["kda_bf16_t32768_h32_d128_r16"] if gate == "kda" else W["gdn_bf16_b2_t8192_h16_d128_r8"]
    w = inputs.Workload("cut", gate, dtype, 1, sum(lengths), 2, 128, R, gate_dist=base.gate_dist, seed=7)
    inp = inputs.make_inputs(w, device="cpu", lengths=lengths)
    print(cut, gate, dtype, compare(run_gpu(inp), run_oracle(inp), inp))


TINY = [
    # (B, T, lengths, R, d)
    (1, 1, None, 1, 128),
    (1, 63, None, 1, 128),
    (1, 64, None, 1, 128),
    (1, 65, None, 1, 128),
    (2, 129, None, 3, 128),
    (1, 200, [1, 63, 0, 64, 71, 1], 2, 128),
    (1, 64, [1] * 64, 64, 128),
    (1, 130, None, 2, 64),
    (3, 96, None, 4, 64),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("gate", ["gdn", "kda"])
@pytest.mark.parametrize("case", TINY, ids=[str(i) for i in range(len(TINY))])
def test_tiny_and_ragged(case, gate, dtype):
    B, T, lengths, R, d = case
    w = inputs.Workload("tiny", gate, dtype, B, T, 3, d, R,
                        gate_dist=("sigmoid", 3.0, 1.0) if gate == "kda" else ("sigmoid", 2.0, 1.0), seed=11)
    inp = inputs.make_inputs(w, device="cpu", lengths=lengths)
    print(case, compare(run_gpu(inp), run_oracle(inp), inp))


@pytest.mark.parametrize("gate", ["gdn", "kda"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_steep_decay(dtype, gate):
    """alpha ~ sigmoid(N(-3, 0.5)) ~ 0.05 per token: the in-chunk decay spans
    far more than 2^100, which takes the exact-exponential branch."""
    w = inputs.Workload("steep", gate, dtype, 1, 2048, 4, 128, 4, gate_dist=("sigmoid", -3.0, 0.5), seed=21)
    inp = inputs.make_inputs(w, device="cpu")
    print(compare(run_gpu(inp), run_oracle(inp), inp))


def test_kda_steep_and_mild_units():
    """Per-dim gates where a few (chunk, head) units decay steeply in a few key
    dims and the rest mildly: both branches of the preparation (the tensor-core
    products and the exact per-term exponentials) in one call."""
    inp = gen("kda_bf16_t32768_h32_d128_r16", B=1, T=2048, H=4)
    g = inp["g"].clone()
    g[0, 64 * 3:64 * 4, 1, :3] = -6.0     # chunk 3, head 1: span about 280 in log2
    g[0, 64 * 17 + 40:64 * 18, 2, 100] = -12.0
    inp["g"] = g
    inp["R"] = 4
    print(compare(run_gpu(inp), run_oracle(inp), inp))


@pytest.mark.parametrize("name", ["gdn_bf16_b2_t8192_h16_d128_r8", "kda_bf16_t32768_h32_d128_r16"])
def test_fp32_cuda_core_path_cross_check(name):
    inp = gen(name, B=1, T=2048, H=4)
    print(name, compare(run_gpu(inp, force_simt=True), run_oracle(inp), inp))


def test_output_scale():
    inp = inputs.make_inputs(W["gdn_bf16_b2_t8192_h16_d128_r8"], device="cpu", B=1, T=512, H=2)
    inp["R"] = 2
    print(compare(run_gpu(inp, scale=0.125), run_oracle(inp, scale=0.125), inp))
