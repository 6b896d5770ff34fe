"""Failure detection on the GPU without a GPU fault.

Every mbarrier wait in the library's kernels is bounded; when one gives up
it records (code, site, block) in the context's device status word and the
kernel returns.  cpdr_selftest_wait_timeout makes one such wait run out on
purpose (an mbarrier phase nothing completes, a ~10 ms limit): the status
must come back as CPDR_ERR_TIMEOUT, be cleared by the read, and the same
context must then compute the same results as before.
"""
import pytest
import torch

from context_merge_gb300 import cpdr, inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_context_stays_usable(cpdr_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    w = inputs.WORKLOADS["gdn_bf16_b2_t8192_h16_d128_r8"]
    inp = inputs.make_inputs(w, device="cuda", B=1, T=1024, H=2)
    ctx = cpdr.Context(inp["B"], inp["T"], inp["H"], inp["d"], 4, gate=w.gate, dtype=w.dtype)
    args = [inp[k] for k in ("q", "k", "v", "beta", "g")]
    o1, b1 = ctx.run(*args)
    fs1 = b1["final_state"].clone()
    torch.cuda.synchronize()
    ctx.check_device_status()                      # clean before

    ctx.selftest_wait_timeout(20_000_000)          # about 10 ms of SM clock
    with pytest.raises(cpdr.CpdrError) as ei:
        ctx.check_device_status()
    assert ei.value.status == cpdr.ERR_TIMEOUT
    assert b"site 99" in cpdr_lib.cpdr_last_error()
    ctx.check_device_status()                      # the read cleared it

    o2, b2 = ctx.run(*args)                        # the context is still usable
    torch.cuda.synchronize()
    ctx.check_device_status()
    assert torch.equal(o1, o2)
    assert torch.equal(fs1, b2["final_state"])


def test_selftest_argument_validation(cpdr_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ctx = cpdr.Context(1, 256, 2, 64, 2, gate="gdn", dtype="fp32")
    for bad in (0, -5, 5_000_000_000):
        with pytest.raises(cpdr.CpdrError) as ei:
            ctx.selftest_wait_timeout(bad)
        assert ei.value.status == cpdr.ERR_INVALID
