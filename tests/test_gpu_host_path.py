"""The whole path from host buffers (cpdr_forward_host): its copies run on
the context's copy stream and each stage waits for its own inputs, so the
results must be bit-identical to the device-buffer path on the same inputs,
for each path the library selects (tensor cores with the scalar and the
per-dim gate, CUDA cores)."""
import pytest
import torch

from context_merge_gb300 import cpdr, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(cpdr_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)


@pytest.mark.parametrize("name,T,H,Hq", [("gdn_bf16_b2_t8192_h16_d128_r8", 4096, 4, None),
                                         ("gdn_bf16_b2_t8192_h16_d128_r8", 4096, 4, 8),   # two query heads per chain
                                         ("kda_bf16_t32768_h32_d128_r16", 4096, 4, None),
                                         ("gdn_fp32_t1024_h2_d64_r4", 1024, 2, None),
                                         ("gdn_bf16_varlen65536_n12_h16_d128_r32", 65536, 2, None)])
def test_host_path_matches_device_path(name, T, H, Hq):
    w = inputs.WORKLOADS[name]
    inp = inputs.make_inputs(w, device="cpu", T=T, H=H, Hq=Hq)
    B, T, d, R = inp["B"], inp["T"], inp["d"], inp["R"]
    ctx = cpdr.Context(B, T, H, d, R, gate=w.gate, dtype=w.dtype, cu_seqlens=inp["cu_seqlens"], Hq=inp["Hq"])
    dev = {k: inp[k].cuda() for k in ("q", "k", "v", "beta", "g")}
    o_dev, bufs = ctx.run(dev["q"], dev["k"], dev["v"], dev["beta"], dev["g"])
    host = {k: inp[k].contiguous().pin_memory() for k in ("q", "k", "v", "beta", "g")}
    o_h = torch.full(o_dev.shape, float("nan"), dtype=o_dev.dtype).pin_memory()
    fs_h = torch.full(bufs["final_state"].shape, float("nan"), dtype=torch.float32).pin_memory()
    work = torch.empty(ctx.host_workspace_bytes(), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(2):   # twice: the second call reuses the workspace and events
        ctx.forward_host(host["q"], host["k"], host["v"], host["beta"], host["g"], o_h, fs_h, work, stream)
        torch.cuda.synchronize()
        ctx.check_device_status()
        assert torch.equal(o_h, o_dev.cpu())
        assert torch.equal(fs_h, bufs["final_state"].cpu())
