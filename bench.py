"""Throughput of the segmented delta-rule forward (preprocess + merge + fwd).

One step = one pass of the whole path over one batch of the workload with
inputs resident in HBM.  Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline] [--no-e2e]

Multi-GPU (torchrun, one rank per GPU): every rank runs an independent
replica of the workload (weak scaling, no collective on the data path);
value = tokens of all ranks / max-over-ranks time.

--impl reference times the fp64 CPU oracle (the reference arm of this
method, which has no other implementation) on bounded samples of the same
workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from context_merge_gb300 import inputs  # noqa: E402

METRIC = "tokens/sec (preprocess+merge+fwd, 1 GB300)"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=inputs.HEADLINE, choices=list(inputs.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-sample-heads", type=int, default=4)
    ap.add_argument("--force-simt", action="store_true")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward (gradients of the forward) instead of the forward")
    # profiling aids: shrink the workload (same shapes otherwise) for ncu captures
    ap.add_argument("--T", type=int, default=None, help="override tokens per row (profiling only)")
    ap.add_argument("--H", type=int, default=None, help="override heads (profiling only)")
    ap.add_argument("--Hq", type=int, default=None,
                    help="override query heads, a multiple of the heads (profiling only)")
    return ap.parse_args()


def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        except Exception:
            self.uuid = None

    def start(self):
        try:
            # raw samples go to CPDR_CLOCK_DIR (default: the temp directory);
            # the JSON line carries their summary
            out_dir = os.environ.get("CPDR_CLOCK_DIR") or tempfile.gettempdir()
            os.makedirs(out_dir, exist_ok=True)
            self.path = os.path.join(out_dir, f"clocks_{os.getpid()}.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid.replace("GPU-", "") not in parts[0]:
                continue
            rows.append(parts)
        if not rows:
            return None
        try:
            sm = [float(r[1]) for r in rows]
            mx = max(float(r[2]) for r in rows)
        except ValueError:
            return None
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for nm, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(rows)}


# ---------------------------------------------------------------- peaks
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return float(json.load(open(p))["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def stage_bytes(w, ctx, inp):
    """Algorithmic HBM bytes per launch of each stage (each tensor element
    read or written once)."""
    es = 4 if w.dtype == "fp32" else 2
    H, d, Hq = inp["H"], inp["d"], inp["Hq"]
    frags = ctx.fragments()
    gate_w = d if w.gate == "kda" else 1
    # q in and o out per query head; k, v, beta, g in per state head
    tok_bytes_fwd = Hq * 2 * d * es + H * (2 * d * es + es + gate_w * 4)
    tok_bytes_pre = H * (2 * d * es + es + gate_w * 4)               # k, v, beta, g in
    state = H * d * d * 4
    pre_tok = sum(f[1] for f in frags if f[4] & 2)
    n_pre = sum(1 for f in frags if f[4] & 2)
    n_cont = sum(1 for f in frags if f[4] & 1)
    n_end = sum(1 for f in frags if f[4] & 4)
    tokens = inp["B"] * inp["T"]
    c = ctx.counts()
    fwd = tokens * tok_bytes_fwd + n_cont * state + n_end * state
    pre = pre_tok * tok_bytes_pre + n_pre * 2 * state
    # merge: every chain step reads M_j and S_ext_j once and writes S_init
    merge = n_cont * 3 * state
    # WY build: k, beta and g of every token (the tiles it writes are an
    # intermediate of this implementation, not algorithmic bytes)
    wy = tokens * H * (d * es + es + gate_w * 4) if c["tc"] else 0
    return {"wy": wy, "pre": pre, "merge": merge, "fwd": fwd, "chains": c["chains"]}


def traffic_record(kernel_tag):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json),
    if it was taken on the current kernel sources (matched by hash); else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        rec = json.load(open(p)).get(kernel_tag)
        if not rec:
            return None
        h = hashlib.sha256()
        for src in rec["sources"]:
            h.update(open(os.path.join(ROOT, src), "rb").read())
        return rec["bytes_per_launch"] if h.hexdigest()[:16] == rec["source_sha"] else None
    except Exception:
        return None


def variant_keys(w, inp):
    """Config keys of a layout variant (absent for the default layout)."""
    out = {}
    if w.layout != "contiguous":
        out["layout"] = w.layout
    if w.Hq or (inp is not None and inp["Hq"] != inp["H"]):
        out["Hq"] = w.Hq if inp is None else inp["Hq"]
    if w.state_v_first:
        out["state_v_first"] = True
    return out


# ---------------------------------------------------------------- CPU oracle
def cpu_oracle_sample(inp_dev, w, heads):
    """Time the fp64 oracle (as it stands) on the first `heads` heads of the
    workload; returns (seconds, head-tokens processed, threads)."""
    import oracle
    from oracle import layout
    hs = min(heads, inp_dev["H"])
    G = inp_dev["Hq"] // inp_dev["H"]
    sub = {}
    for key in ("q", "k", "v", "beta", "g"):
        x = inp_dev[key][:, :, :hs * G if key == "q" else hs].contiguous().cpu()
        # the device tensors are in memory order; the oracle takes sequence order
        sub[key] = layout.from_zigzag(x, w.R) if w.layout == "zigzag" else x
    P = oracle.Problem(sub["q"], sub["k"], sub["v"], sub["beta"], sub["g"], cu_seqlens=inp_dev["cu_seqlens"])
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    P.segmented(2 * w.R if w.layout == "zigzag" else w.R, nthreads=threads)
    dt = time.perf_counter() - t0
    return dt, inp_dev["B"] * inp_dev["T"] * hs, threads


def run_reference(args, ws, rank):
    w = inputs.WORKLOADS[args.workload]
    if rank != 0:
        return
    import oracle
    oracle.build()
    hs = 1
    inp = inputs.make_inputs(w, device="cpu", H=hs)
    times = []
    for i in range(args.warmup + args.steps):
        dt, ht, threads = cpu_oracle_sample(inp, w, hs)
        if i >= args.warmup:
            times.append(dt)
    tokens_equiv = inp["B"] * inp["T"] * hs / w.H
    total = sum(times)
    value = tokens_equiv * len(times) / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict({"workload": w.name, "B": inp["B"], "T": inp["T"], "H": w.H, "d": w.d, "R": w.R,
                            "gate": w.gate, "in_dtype": w.dtype}, **variant_keys(w, None)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"fp64 segmented oracle on {hs} of {w.H} heads per step, full T; "
                                       f"tokens scaled by heads sampled / heads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- ours
def run_ours(args, ws, rank, local):
    from context_merge_gb300 import cpdr
    w = inputs.WORKLOADS[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = inputs.make_inputs(w, device=dev, seed=w.seed + 1000 * rank, T=args.T, H=args.H, Hq=args.Hq)
    B, T, H, d, R = inp["B"], inp["T"], inp["H"], inp["d"], inp["R"]
    ctx = cpdr.Context(B, T, H, d, R, gate=w.gate, dtype=w.dtype, cu_seqlens=inp["cu_seqlens"],
                       force_simt=args.force_simt, layout=w.layout, Hq=inp["Hq"], state_v_first=w.state_v_first)
    bufs = ctx.alloc_buffers(dev)
    o = torch.empty((B, T, inp["Hq"], d), dtype=inp["v"].dtype, device=dev)
    q, k, v, beta, g = (inp[x] for x in ("q", "k", "v", "beta", "g"))
    stream = torch.cuda.current_stream()

    wy = bufs["wy"]

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        ctx.wy_build(q, k, beta, g, wy, stream)
        if ev is not None:
            ev[1].record(stream)
        ctx.preprocess(k, v, beta, g, bufs["S_ext"], bufs["M"], wy=wy, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        ctx.merge(bufs["S_ext"], bufs["M"], bufs["S_init"], stream)
        if ev is not None:
            ev[3].record(stream)
        ctx.fwd(q, k, v, beta, g, bufs["S_init"], o, bufs["final_state"], wy=wy, stream=stream)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    ctx.check_device_status()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = ClockSampler() if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop() if clocks else None
    ctx.check_device_status()
    elapsed_ms = start.elapsed_time(end)
    stage_ms = {"wy": [], "pre": [], "merge": [], "fwd": []}
    for e in evs:
        for j, name in enumerate(stage_ms):
            stage_ms[name].append(e[j].elapsed_time(e[j + 1]))
    elapsed_ms = max_over_ranks(elapsed_ms, ws)
    tokens = B * T
    value = tokens * ws * args.steps / (elapsed_ms / 1e3)

    # ---- e2e through the host-buffer C-ABI call (H2D + path + D2H timed)
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hb, hg = (x.cpu().pin_memory() for x in (q, k, v, beta, g))
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hfs = torch.empty(bufs["final_state"].shape, dtype=torch.float32).pin_memory()
        ws_bytes = ctx.host_workspace_bytes()
        del bufs
        torch.cuda.empty_cache()
        work = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        ctx.forward_host(hq, hk, hv, hb, hg, ho, hfs, work, stream)
        torch.cuda.synchronize()
        k_e = max(3, min(20, args.steps))
        barrier(ws)
        s2 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        for _ in range(k_e):
            ctx.forward_host(hq, hk, hv, hb, hg, ho, hfs, work, stream)
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(s2.elapsed_time(e2), ws)
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hb, hg))
        d2h = ho.numel() * ho.element_size() + hfs.numel() * hfs.element_size()
        e2e = {"value": tokens * ws * k_e / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": k_e}
        del work

    if rank != 0:
        return
    # ---- roofline of the dominant stage (HBM-bound)
    nbytes = stage_bytes(w, ctx, inp)
    mean_ms = {s: statistics.mean(v) for s, v in stage_ms.items()}
    # the dominant kernel: one launch per stage is timed; on the tensor-core
    # path the pre-process is two kernels (S and M chains), each below the
    # forward chain in the ncu launch list, so the candidates are WY and fwd
    counts0 = ctx.counts()
    cands = ("wy", "fwd") if counts0["tc"] else ("pre", "fwd")
    dom = max(cands, key=lambda s: mean_ms[s])
    peak, peak_kind = hbm_peak()
    achieved = nbytes[dom] / (mean_ms[dom] / 1e3) / 1e9
    counts = ctx.counts()
    kernel_tag = f"{'tc' if counts['tc'] else 'simt'}_{dom}:{w.name}"
    traffic = traffic_record(kernel_tag)
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "kernel": kernel_tag, "peak_source": peak_kind,
            "algorithmic_bytes_per_launch": nbytes[dom], "ms_per_launch": mean_ms[dom]}
    # every stage against the same peak (the pre-process is two kernels on
    # two streams, timed together), and the whole path: the algorithmic
    # bytes per step over the step time -- the pre-process, merge and forward
    # passes (the WY build reads the same k, beta, g those passes read, so
    # the path counts them once)
    stages = {s: {"ms": mean_ms[s], "algorithmic_bytes": nbytes[s],
                  "achieved_gbs": nbytes[s] / (mean_ms[s] / 1e3) / 1e9 if mean_ms[s] > 0 else None,
                  "frac": nbytes[s] / (mean_ms[s] / 1e3) / 1e9 / peak if mean_ms[s] > 0 else None}
              for s in ("wy", "pre", "merge", "fwd")}
    path_bytes = sum(nbytes[s] for s in ("pre", "merge", "fwd"))
    ms_step = elapsed_ms / args.steps
    path = {"algorithmic_bytes_per_step": path_bytes, "ms_per_step": ms_step,
            "achieved_gbs": path_bytes / (ms_step / 1e3) / 1e9,
            "frac": path_bytes / (ms_step / 1e3) / 1e9 / peak, "peak": peak, "peak_source": peak_kind}
    cpu = None
    if not args.no_cpu_baseline:
        try:
            dt, ht, threads = cpu_oracle_sample(inp, w, args.cpu_sample_heads)
            cpu = {"value": ht / H / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
                   "sample": f"fp64 segmented oracle on {min(args.cpu_sample_heads, H)} of {H} heads, full T "
                             f"({dt:.1f} s wall); tokens scaled by heads sampled / heads"}
        except Exception as ex:  # pragma: no cover
            cpu = {"error": str(ex)}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": dict({"workload": w.name, "B": B, "T": T, "H": H, "d": d, "R": R, "gate": w.gate,
                        "in_dtype": w.dtype, "parallelism": f"replicas{ws}",
                        "l2": "inputs larger than L2 (no flush)" if tokens * H * d * 2 > 256e6 else "inputs fit L2"},
                       **variant_keys(w, inp)),
        "stage_ms": mean_ms,
        "roofline": roof,
        "stage_roofline": stages,
        "path_roofline": path,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": counts["launches"] * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- causal conv1d
CONV_METRIC = "tokens/sec (causal conv1d, 1 GB300)"


def conv_oracle_sample(inp, w, channels=8):
    """Time the fp64 conv oracle on the first `channels` channels, full T;
    returns (seconds, token-channels processed)."""
    from oracle import conv as oconv
    from oracle import layout
    x = inp["x"][:, :, :channels].cpu()
    if w.layout == "zigzag":
        x = layout.from_zigzag(x, w.R)
    t0 = time.perf_counter()
    oconv.causal_conv1d(x, inp["weight"][:channels].cpu(), inp["bias"][:channels].cpu(),
                        cu_seqlens=inp["cu_seqlens"])
    return time.perf_counter() - t0, inp["B"] * inp["T"] * channels


def conv_config(w, inp, ws):
    return dict({"workload": w.name, "op": "conv1d", "B": inp["B"], "T": inp["T"], "C": inp["C"],
                 "W": inp["W"], "R": w.R, "in_dtype": w.dtype, "activation": "silu",
                 "parallelism": f"replicas{ws}", "l2": "inputs larger than L2 (no flush)"},
                **variant_keys(w, None))


def run_conv_reference(args, ws, rank):
    w = inputs.WORKLOADS[args.workload]
    if rank != 0:
        return
    inp = inputs.make_conv_inputs(w, device="cpu")
    times = []
    for i in range(args.warmup + args.steps):
        dt, tc = conv_oracle_sample(inp, w)
        if i >= args.warmup:
            times.append(dt)
    value = tc / inp["C"] * len(times) / sum(times)
    line = {"impl": "reference", "metric": CONV_METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": conv_config(w, inp, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"fp64 conv oracle on 8 of {inp['C']} channels per step, full T; "
                                       f"tokens scaled by channels sampled / channels"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_conv(args, ws, rank):
    from context_merge_gb300 import cpdr
    w = inputs.WORKLOADS[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = inputs.make_conv_inputs(w, device=dev, seed=w.seed + 1000 * rank, T=args.T)
    B, T, C = inp["B"], inp["T"], inp["C"]
    ctx = cpdr.Context(B, T, 1, 64, w.R, gate="gdn", dtype=w.dtype, cu_seqlens=inp["cu_seqlens"],
                       layout=w.layout, conv_width=inp["W"])
    x, weight, bias = inp["x"], inp["weight"], inp["bias"]
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        ctx.conv1d_fwd(x, weight, bias, y, stream=stream)
    torch.cuda.synchronize()
    clocks = ClockSampler() if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        ctx.conv1d_fwd(x, weight, bias, y, stream=stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(start.elapsed_time(end), ws) / args.steps
    tokens = B * T
    value = tokens * ws / (ms / 1e3)
    e2e = None
    if not args.no_e2e:
        # host x in (pinned), conv, host y out, all inside the timed region
        hx = x.cpu().pin_memory()
        hy = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        k_e = max(3, min(10, args.steps))
        barrier(ws)
        s2 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        for _ in range(k_e):
            x.copy_(hx, non_blocking=True)
            ctx.conv1d_fwd(x, weight, bias, y, stream=stream)
            hy.copy_(y, non_blocking=True)
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(s2.elapsed_time(e2), ws)
        nb = hx.numel() * hx.element_size()
        e2e = {"value": tokens * ws * k_e / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": nb,
               "d2h_bytes_per_step": nb, "steps": k_e}
    if rank != 0:
        return
    es = 2 if w.dtype == "bf16" else 4
    nbytes = 2 * tokens * C * es + C * (inp["W"] + 1) * 4      # x in, y out, weights
    peak, peak_kind = hbm_peak()
    achieved = nbytes / (ms / 1e3) / 1e9
    tag = f"conv1d:{w.name}"
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic_record(tag), "kernel": tag, "peak_source": peak_kind,
            "algorithmic_bytes_per_launch": nbytes, "ms_per_launch": ms}
    cpu = None
    if not args.no_cpu_baseline:
        dt, tc = conv_oracle_sample(inp, w)
        cpu = {"value": tc / C / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"fp64 conv oracle on 8 of {C} channels, full T ({dt:.1f} s wall); "
                         f"tokens scaled by channels sampled / channels"}
    line = {"metric": CONV_METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": conv_config(w, inp, ws), "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps, "clocks": clk}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- backward
BWD_METRIC = "tokens/sec (backward: gradients of q, k, v, beta, gate; 1 GB300)"


def bwd_oracle_sample(inp, w, heads=1):
    """Time the fp64 backward oracle on the first `heads` heads, full T."""
    import oracle
    hs = min(heads, inp["H"])
    G = inp["Hq"] // inp["H"]
    sub = {k: inp[k][:, :, :hs * (G if k == "q" else 1)].contiguous().cpu() for k in ("q", "k", "v", "beta", "g")}
    do = torch.randn(sub["q"].shape[:3] + sub["v"].shape[3:],
                     generator=torch.Generator().manual_seed(5)).to(sub["v"].dtype)
    P = oracle.Problem(sub["q"], sub["k"], sub["v"], sub["beta"], sub["g"], cu_seqlens=inp["cu_seqlens"])
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    P.backward(do, nthreads=threads)
    return time.perf_counter() - t0, inp["B"] * inp["T"] * hs, threads


def run_backward(args, ws, rank):
    from context_merge_gb300 import cpdr
    w = inputs.WORKLOADS[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = inputs.make_inputs(w, device=dev, seed=w.seed + 1000 * rank, T=args.T, H=args.H, Hq=args.Hq)
    B, T, H, d, R = inp["B"], inp["T"], inp["H"], inp["d"], inp["R"]
    Hq = inp["Hq"]
    ctx = cpdr.Context(B, T, H, d, R, gate=w.gate, dtype=w.dtype, cu_seqlens=inp["cu_seqlens"],
                       force_simt=args.force_simt, layout=w.layout, Hq=Hq, state_v_first=w.state_v_first)
    q, k, v, beta, g = (inp[x] for x in ("q", "k", "v", "beta", "g"))
    o, bufs = ctx.run(q, k, v, beta, g)
    do = torch.randn(o.shape, device=dev, dtype=torch.float32).to(v.dtype)
    dht = torch.randn(bufs["final_state"].shape, device=dev)
    work = torch.empty(ctx.bwd_workspace_bytes(), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    step = lambda: ctx.backward(q, k, v, beta, g, do, bufs["S_init"], bufs["M"], dht=dht, workspace=work,
                                stream=stream)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    ctx.check_device_status()
    clocks = ClockSampler() if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(start.elapsed_time(end), ws) / args.steps
    if rank != 0:
        return
    tokens = B * T
    cpu = None
    if not args.no_cpu_baseline:
        dt, ht, threads = bwd_oracle_sample(inp, w)
        cpu = {"value": ht / H / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"fp64 backward oracle on 1 of {H} heads, full T ({dt:.1f} s wall); tokens scaled by heads"}
    # algorithmic bytes of one backward: per (token, head) k, v, beta, g in
    # and dk, dv (fp32), dbeta, dg out; per (token, query head) q, do in and
    # dq (fp32) out; per (segment, head) the S_init and M states read.  The backward's launches are timed together, so its
    # line carries the whole backward's figure: on the tensor-core path (bf16,
    # d = 128, scalar gate) the WY build, the recomputed forward, the
    # state-gradient chains of the continuing fragments, the reverse merge,
    # the main chains and the input gradients; otherwise the CUDA-core
    # continuing-fragment pass, reverse merge and main pass.
    es = 4 if w.dtype == "fp32" else 2
    gate_w = d if w.gate == "kda" else 1
    counts = ctx.counts()
    tok_bytes = H * (2 * d * es + es + gate_w * 4 + 2 * d * 4 + 4 + gate_w * 4) + Hq * (2 * d * es + d * 4)
    state_bytes = R * B * H * d * d * 4 * 2
    nbytes = tokens * tok_bytes + state_bytes
    peak, peak_kind = hbm_peak()
    achieved = nbytes / (ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": None, "kernel": f"bwd(all launches):{w.name}", "peak_source": peak_kind,
            "algorithmic_bytes_per_launch": nbytes, "ms_per_launch": ms}
    # tensor-core path: WY build, recomputed forward, one main state-gradient
    # chain per query head of a state, input gradients; with cut sequences
    # also a pre-process chain per query head and the reverse merge
    G = Hq // H
    tc_bwd = bool(counts["tc"])
    if tc_bwd:   # the per-dim gate's preparation is two launches (preparation, solve)
        launches = (3 + G + ((G + 1) if counts["chains"] else 0) + (1 if w.gate == "kda" else 0)) * args.steps
    else:
        launches = (1 + (2 if counts["chains"] else 0)) * args.steps
    line = {"metric": BWD_METRIC, "value": tokens * ws / (ms / 1e3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict({"workload": w.name, "op": "backward", "B": B, "T": T, "H": H, "d": d, "R": R,
                            "gate": w.gate, "in_dtype": w.dtype, "parallelism": f"replicas{ws}"},
                           **variant_keys(w, inp)),
            "roofline": roof, "cpu_baseline": cpu, "e2e": None, "gpu_launches": launches, "clocks": clk}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, local = dist_setup(args)
    conv = inputs.WORKLOADS[args.workload].op == "conv1d"
    if args.impl == "reference":
        (run_conv_reference if conv else run_reference)(args, ws, rank)
    elif conv:
        run_conv(args, ws, rank)
    elif args.backward:
        run_backward(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
