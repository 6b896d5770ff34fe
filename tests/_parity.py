"""Helpers for the GPU-vs-oracle parity tests.

Tolerances (stated per (sequence, head) for o and final states, per
(segment, head) for S_init, S_ext and M):
* fp32 inputs: max|x - ref| / max|ref| <= 1e-4
* bf16 inputs: ||x - ref||_2 / ||ref||_2 <= 2e-2
* S_ext and M are only compared where ||ref||_F >= 1e-30; below that (fp32
  underflow of long decays) the GPU value must satisfy max|x| <= 1e-30.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from context_merge_gb300 import cpdr
from oracle import layout as oracle_layout

TOL = {"fp32": 1e-4, "bf16": 2e-2}


def _variant(inp):
    return inp.get("layout", "contiguous"), inp.get("Hq") or inp["H"], bool(inp.get("state_v_first", False))


def run_gpu(inp, force_simt=False, scale=1.0):
    """WY build -> preprocess -> merge -> fwd through the C-ABI on cuda:0; CPU results.

    Inputs are sequence-ordered; in the zigzag layout they are gathered into
    zigzag memory order first and o is brought back to sequence order, and
    [dv, dk] states are transposed back, so that results compare directly
    with the oracle."""
    B, T, H, d, R = inp["B"], inp["T"], inp["H"], inp["d"], inp["R"]
    lay, Hq, vf = _variant(inp)
    ctx = cpdr.Context(B, T, H, d, R, gate=inp["gate"], dtype=inp["dtype"], cu_seqlens=inp["cu_seqlens"],
                       scale=scale, force_simt=force_simt, layout=lay, Hq=Hq, state_v_first=vf)
    place = (lambda x: oracle_layout.to_zigzag(x, R)) if lay == "zigzag" else (lambda x: x)
    dev = {k: place(inp[k]).contiguous().cuda() for k in ("q", "k", "v", "beta", "g")}
    bufs = ctx.alloc_buffers("cuda")
    for t in bufs.values():            # poison: every element must be written
        if t is not None:              # (WY tiles: 0xffff is a bf16 NaN)
            t.fill_(255 if t.dtype == torch.uint8 else float("nan"))
    o = torch.full((B, T, Hq, d), float("nan"), dtype=dev["v"].dtype, device="cuda")
    ctx.run(dev["q"], dev["k"], dev["v"], dev["beta"], dev["g"], bufs=bufs, o=o)
    torch.cuda.synchronize()
    ctx.check_device_status()
    out = {k: v.cpu() for k, v in bufs.items() if k != "wy"}
    if vf:
        for k in ("S_ext", "S_init", "final_state"):
            out[k] = out[k].transpose(-1, -2).contiguous()
    out["o"] = oracle_layout.from_zigzag(o.cpu(), R) if lay == "zigzag" else o.cpu()
    out["counts"] = ctx.counts()
    return out


def run_oracle(inp, scale=1.0):
    """The oracle on the sequence-ordered inputs, over the segments the
    layout makes: R contiguous segments, or the 2R zigzag parts."""
    P = oracle.Problem(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], cu_seqlens=inp["cu_seqlens"],
                       scale=scale)
    lay, _, _ = _variant(inp)
    return P.segmented(2 * inp["R"] if lay == "zigzag" else inp["R"])


def _err(x, ref, kind):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    if not np.isfinite(x).all():
        return float("inf")
    if kind == "fp32":
        den = np.abs(ref).max()
        num = np.abs(x - ref).max()
    else:
        den = np.linalg.norm(ref)
        num = np.linalg.norm(x - ref)
    if den == 0:
        return 0.0 if num == 0 else float("inf")
    return float(num / den)


def compare(gpu, ref, inp, check_exchange=True):
    """Max relative errors per quantity; raises AssertionError over tolerance."""
    kind = inp["dtype"]
    tol = TOL[kind]
    B, T, H = inp["B"], inp["T"], inp["H"]
    o = gpu["o"].double().numpy()
    errs = {}
    # o per (sequence, head)
    cu = inp["cu_seqlens"]
    worst = 0.0
    Hq = o.shape[2]
    if cu is None:
        for b in range(B):
            for h in range(Hq):
                worst = max(worst, _err(o[b, :, h], ref["o"][b, :, h], kind))
    else:
        cu = [int(x) for x in cu]
        for n in range(len(cu) - 1):
            if cu[n + 1] == cu[n]:
                continue
            for h in range(Hq):
                worst = max(worst, _err(o[0, cu[n]:cu[n + 1], h], ref["o"][0, cu[n]:cu[n + 1], h], kind))
    errs["o"] = worst
    fs = gpu["final_state"].double().numpy()
    errs["final_state"] = max(_err(fs[n, h], ref["ht"][n, h], kind)
                              for n in range(fs.shape[0]) for h in range(H))
    if "S_init" in gpu:     # (the allocation-free entry point keeps it internal)
        si = gpu["S_init"].double().numpy()
        e = 0.0
        for r in range(si.shape[0]):
            for b in range(si.shape[1]):
                for h in range(H):
                    if not ref["S_init"][r, b, h].any():
                        e = max(e, 0.0 if not si[r, b, h].any() else float("inf"))
                    else:
                        e = max(e, _err(si[r, b, h], ref["S_init"][r, b, h], kind))
        errs["S_init"] = e
    if check_exchange:
        for key in ("S_ext", "M"):
            x = gpu[key].double().numpy()
            e = 0.0
            for r in range(x.shape[0]):
                for b in range(x.shape[1]):
                    for h in range(H):
                        rr = ref[key][r, b, h]
                        if np.linalg.norm(rr) >= 1e-30:
                            e = max(e, _err(x[r, b, h], rr, kind))
                        elif not (np.isfinite(x[r, b, h]).all() and np.abs(x[r, b, h]).max() <= 1e-30):
                            e = float("inf")
            errs[key] = e
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"over tolerance {tol}: {bad} (all: {errs})"
    return errs
