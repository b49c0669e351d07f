#!/usr/bin/env python3
"""Benchmark of the dispatch + combine round trip on logical EP ranks.

One step = the whole hot path on one batch: routing (two kernels), the
dispatch row scatter, and the fused weighted combine with residual add and
RMSNorm (one kernel) -- four launches through the C ABI.  The default
workload is prefill: ep_size 8, 4096 tokens per rank, hidden 7168, 256
experts, top-8 with Zipf(1.2) expert popularity (contiguous placement).

Prints one JSON line.  `value` is tokens/s over all GPUs with inputs already
in HBM; `e2e` is the same metric with the step's inputs copied from pinned
host memory and its outputs copied back inside the timed region;
`roofline` is the dominant kernel (the fused combine) against the measured
HBM copy peak; `cpu_baseline` is the single-threaded C oracle on a bounded
sample of the same workload.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Under torchrun every rank runs its own replica (weak scaling: the ranks
share no data); rank 0 prints.
"""
import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and effective HBM GB/s (% of GB300 peak), 1 GPU"
# Sets of device input / output buffers the end-to-end leg rotates through.
E2E_BUFFERS = 3
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal: each phase also reports its fraction of it
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", default="prefill",
                    choices=["tiny", "decode", "prefill", "wide", "ladder", "moe_layer"])
    ap.add_argument("--tokens", type=int, default=None, help="tokens per rank (ladder rung)")
    ap.add_argument("--workspace-tokens", type=int, default=None,
                    help="size the workspace for this many tokens per rank (small profiling "
                         "cases); default: the workload's max_tokens_per_rank")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--e2e-buffers", type=int, default=E2E_BUFFERS,
                    help="input / output buffer sets the end-to-end leg rotates through")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layout", choices=["rank", "expert"], default=None,
                    help="receive layout: planes per (destination, source) rank (default), "
                         "or one row per (token, expert) in per-expert planes (the default "
                         "with --expert-gemm)")
    ap.add_argument("--l2-hot", action="store_true",
                    help="no L2 flush between steps even for small inputs (reports the "
                         "L2-hot figure beside the default flushed one; not a bench line)")
    ap.add_argument("--expert-gemm", action="store_true",
                    help="the expert-side product between dispatch and combine (random bf16 "
                         "weights W_e of H x H, output into the combine payload): one step is "
                         "a whole single-matrix MoE layer.  Expert layout by default; with "
                         "--layout rank the product runs on the rank planes and applies the "
                         "gates, and the combine is the unweighted rank sum; with --fp8 the "
                         "product takes the e4m3 receive rows and e4m3 weights")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 payloads: e4m3 dispatch rows with a per-token scale and an "
                         "e4m3 combine output with a per-token scale (needs hidden %% 16 == 0)")
    ap.add_argument("--graph", action="store_true",
                    help="time CUDA-graph replays of each phase's C-ABI call instead of "
                         "direct calls (measured no faster on GB300)")
    args = ap.parse_args()
    if args.expert_gemm:
        if args.graph:
            ap.error("--expert-gemm takes direct calls")
        if args.layout is None:
            args.layout = "expert"
    if args.layout is None:
        args.layout = "rank"
    return args


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def workload(args):
    from combine_topk_ids_rank_gb300 import synth
    w = synth.WORKLOADS[args.config]
    if args.tokens is not None:
        w = w.rung(args.tokens)
    if args.workspace_tokens is not None:
        from dataclasses import replace
        w = replace(w, max_tokens=max(args.workspace_tokens, w.runtime_max))
    return w


def measured_tensor_peak():
    """Sustained bf16 tensor throughput (the product runs inside a long step)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1700.0, "fallback"


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def phase_bytes(w, recv_rows, fp8=False):
    """Algorithmic payload bytes of one call of each phase: rows of 2H bytes
    (bf16), or H bytes plus a 4-byte scale (e4m3) for the received rows and
    the combine output in the FP8 variant."""
    N, row = w.tokens, 2 * w.hidden
    row8 = w.hidden + 4
    dispatch = N * row + recv_rows * (row8 if fp8 else row)
    combine = recv_rows * row + N * (row8 if fp8 else row)  # messages read, output written
    if w.fused:
        combine += 2 * N * row + row               # residual read, residual_out, gamma
    return dispatch, combine


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-i", str(device_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the oracle on a bounded sample (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

class OracleSample:
    """The C oracle (single-threaded, as it stands) on the first T_s tokens
    per rank of the workload: route + dispatch + combine, outputs
    preallocated outside the timed call."""

    def __init__(self, w, tokens_per_rank, seed):
        import numpy as np
        from combine_topk_ids_rank_gb300 import synth
        from oracle import oracle
        self.oracle = oracle
        self.w = w.rung(tokens_per_rank)
        ws = self.w
        R, T, H, K = ws.ep_size, ws.tokens_per_rank, ws.hidden, ws.top_k
        self.inp = synth.inputs(ws, seed)
        r = oracle.route(self.inp["topk_ids"], self.inp["topk_w"], ws.num_experts, T)
        self.eo = None
        if not ws.identity_experts:
            self.eo = synth.expert_out_planes(seed, R, T, H, r["recv_counts"])
        def touched(shape, dtype):
            a = np.empty(shape, dtype)
            a.fill(0)              # commit the pages outside the timed call
            return a
        self.recv = dict(recv_x=touched((R, R, T, H), np.uint16),
                         recv_ids=touched((R, R, T, K), np.int32),
                         recv_w=touched((R, R, T, K), np.float32))
        n = R * T
        self.outs = dict(acc=touched((n, H), np.float32), out=touched((n, H), np.uint16),
                         y=touched((n, H), np.float64))
        if ws.fused:
            self.outs["residual_out"] = touched((n, H), np.uint16)

    @property
    def tokens(self):
        return self.w.tokens

    def step(self) -> float:
        o, ws, inp = self.oracle, self.w, self.inp
        t0 = time.perf_counter()
        r = o.route(inp["topk_ids"], inp["topk_w"], ws.num_experts, ws.tokens_per_rank)
        d = o.dispatch(inp["topk_ids"], inp["topk_w"], inp["x"], ws.num_experts,
                       ws.tokens_per_rank, r, **self.recv)
        eo = d["recv_x"] if ws.identity_experts else self.eo
        o.combine(r, eo, ws.weighted, inp.get("residual"), inp.get("gamma"), ws.eps,
                  outputs=self.outs)
        return time.perf_counter() - t0


def oracle_seconds_per_token(w, seed):
    s = OracleSample(w, min(w.tokens_per_rank, 16), seed)
    s.step()
    return min(s.step() for _ in range(2)) / s.tokens


def host_cpu():
    """The host the oracle runs on: logical CPUs and the CPU model (from
    /proc/cpuinfo; Arm hosts give no model name, so the implementer / part
    numbers stand in), recorded beside the single core the oracle uses."""
    model = None
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" not in line:
                    continue
                k, v = (x.strip() for x in line.split(":", 1))
                if k in ("model name", "Model") and model is None and v:
                    model = v
                fields.setdefault(k, v)
    except OSError:
        pass
    if model is None and "CPU part" in fields:
        parts = {"0xd4f": "Neoverse-V2", "0xd40": "Neoverse-V1", "0xd0c": "Neoverse-N1",
                 "0xd49": "Neoverse-N2"}
        part = fields["CPU part"]
        model = "Arm %s (implementer %s, part %s)" % (
            parts.get(part.lower(), "core"), fields.get("CPU implementer", "?"), part)
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.processor() or "unknown",
            "machine": platform.machine(), "threads_used": 1}


def cpu_baseline(w, seed, target_seconds):
    per_tok = oracle_seconds_per_token(w, seed)
    T_s = int(max(1, min(w.tokens_per_rank, target_seconds / per_tok / w.ep_size)))
    sample = OracleSample(w, T_s, seed)
    # the whole batch when it takes less than the target: repeated passes
    # (at most 4) until the target is reached
    secs = [sample.step()]
    while sum(secs) < target_seconds and T_s == w.tokens_per_rank and len(secs) < 4:
        secs.append(sample.step())
    sec = sum(secs)
    return {"value": sample.tokens * len(secs) / sec, "unit": "tokens/s", "cores": 1,
            "kind": "oracle",
            "sample": "route+dispatch+combine of the first %d tokens per rank (%d tokens, "
                      "%s), %d pass(es), single-threaded C oracle, %.1f s" % (
                          T_s, sample.tokens, w.name, len(secs), sec),
            "host": host_cpu()}


def run_reference(args, w, rank):
    """The oracle as the reference arm: each step a bounded sample."""
    if rank != 0:
        return
    budget = 120.0 / max(1, args.steps + args.warmup)
    per_tok = oracle_seconds_per_token(w, args.seed)
    T_s = int(max(1, min(w.tokens_per_rank, budget / per_tok / w.ep_size)))
    sample = OracleSample(w, T_s, args.seed)
    for _ in range(args.warmup):
        sample.step()
    secs = [sample.step() for _ in range(args.steps)]
    total = sum(secs)
    value = sample.tokens * args.steps / total
    desc = ("route+dispatch+combine of the first %d tokens per rank (%d tokens of %s) "
            "per step, single-threaded C oracle" % (T_s, sample.tokens, w.name))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_dict(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": desc, "host": host_cpu()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(w, recv_rows=None):
    d = {"workload": w.name, "ep_size": w.ep_size, "tokens_per_rank": w.tokens_per_rank,
         "max_tokens_per_rank": w.max_tokens, "runtime_max_tokens_per_rank": w.runtime_max,
         "hidden": w.hidden, "num_experts": w.num_experts, "top_k": w.top_k,
         "routing": w.routing + ("(s=%.1f, contiguous placement)" % w.zipf_s
                                 if w.routing == "zipf" else ""),
         "combine": ("weighted" if w.weighted else "unweighted") +
                    (" + residual + RMSNorm" if w.fused else ""),
         "l2": "inputs larger than L2 (129 MB)" if w.tokens * w.hidden * 2 > 2 * 129e6
               else "L2 flushed (256 MB write + 256 MB read) before every step; "
                    "only the phases are timed"}
    if recv_rows is not None:
        d["recv_rows"] = int(recv_rows)
        d["mean_dest_ranks"] = recv_rows / w.tokens
    return d


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

def run_gpu(args, w, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist
    from combine_topk_ids_rank_gb300 import synth
    from combine_topk_ids_rank_gb300.moe_a2a import (MoeA2A, MOE_FORMAT_FP8_E4M3,
                                                     MOE_LAYOUT_EXPERT, MOE_LAYOUT_RANK)

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    R, T, H, E, K = w.ep_size, w.tokens_per_rank, w.hidden, w.num_experts, w.top_k
    N = w.tokens

    # ---- inputs: routing from the seeded generator, payloads N(0,1) bf16 ----
    ids_h = torch.from_numpy(synth.topk_ids(args.seed, R, T, E, K, w.routing, w.zipf_s))
    wts_h = torch.from_numpy(synth.topk_weights(args.seed, R, T, K))
    g = torch.Generator().manual_seed(args.seed)
    x_h = torch.randn((R, T, H), generator=g).to(torch.bfloat16)
    res_h = torch.randn((R, T, H), generator=g).to(torch.bfloat16) if w.fused else None
    gam_h = (1 + 0.1 * torch.randn((H,), generator=g)).to(torch.bfloat16)
    ids, wts, x = ids_h.to(dev), wts_h.to(dev), x_h.to(dev)
    res = res_h.to(dev) if w.fused else None
    gam = gam_h.to(dev)
    fp8 = args.fp8
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)
    rout = torch.empty_like(out) if w.fused else None
    out8 = torch.empty((R, T, H), dtype=torch.float8_e4m3fn, device=dev) if fp8 else None
    osc = torch.empty((R, T), dtype=torch.float32, device=dev) if fp8 else None
    identity = w.identity_experts and not fp8      # e4m3 rows are not a bf16 payload

    layout = MOE_LAYOUT_EXPERT if args.layout == "expert" else MOE_LAYOUT_RANK
    a2a = MoeA2A(R, w.max_tokens, H, E, K, dev, layout=layout)
    if fp8:
        a2a.set_recv_format(MOE_FORMAT_FP8_E4M3)
    view = a2a.dispatch(ids, wts, x, w.runtime_max)
    if not identity:
        gd = torch.Generator(device=dev).manual_seed(args.seed + 1)
        pay = a2a.combine_payload()
        pay.copy_(torch.randn(pay.shape, generator=gd, device=dev, dtype=torch.float32)
                  .to(torch.bfloat16))
    eo = view.recv_x if identity else None
    gemm = args.expert_gemm
    gemm_rank = gemm and args.layout == "rank"
    # the rank-plane product applies the gates; the combine is then the
    # pages' unweighted rank sum
    comb_weighted = False if gemm_rank else w.weighted
    if gemm:
        gw = torch.Generator(device=dev).manual_seed(args.seed + 2)
        w_exp = torch.randn((E, H, H), generator=gw, device=dev, dtype=torch.bfloat16)
        if fp8:
            # e4m3 weights of N(0,1) with a per-channel scale 1/sqrt(H)
            w8 = w_exp.to(torch.float8_e4m3fn)
            del w_exp
            w8_scale = torch.full((E, H), 1.0 / H ** 0.5, dtype=torch.float32, device=dev)
            if gemm_rank:
                a2a.expert_gemm_rank_fp8(w8, w8_scale, True)   # allocates its scratch, untimed

                def run_gemm():
                    a2a.expert_gemm_rank_fp8(w8, w8_scale, True)   # gated, into the payload
            else:
                def run_gemm():
                    a2a.expert_gemm_fp8(w8, w8_scale)   # into the combine payload
        elif gemm_rank:
            w_exp.mul_(1.0 / H ** 0.5)
            a2a.expert_gemm_rank(w_exp, True)   # allocates its scratch once, untimed

            def run_gemm():
                a2a.expert_gemm_rank(w_exp, True)   # gated, into the combine payload
        else:
            w_exp.mul_(1.0 / H ** 0.5)      # in place: E x H x H can be tens of GB

            def run_gemm():
                a2a.expert_gemm(w_exp)      # into the combine payload

    def combine_into(res_, outs):
        if fp8:
            a2a.combine_fp8(eo, comb_weighted, res_, gam, w.eps, outs[0], outs[1], outs[2])
        else:
            a2a.combine(eo, comb_weighted, res_, gam, w.eps, outs[0], outs[1])

    outs_main = [out8, osc, rout] if fp8 else [out, rout]
    combine_into(res, outs_main)
    torch.cuda.synchronize()
    recv_rows = int(view.recv_counts.sum().item())
    # rows the product multiplies: one per received row in the expert layout,
    # one per (row, local expert) pair on the rank planes
    gemm_rows = int(view.local_expert_counts.sum().item()) if gemm_rank else recv_rows
    st, flags = a2a.get_error()
    if st != 0:
        raise RuntimeError("device flag set: status %d flags %#x" % (st, flags))

    def run_dispatch():
        a2a.dispatch(ids, wts, x, w.runtime_max)

    def run_combine():
        combine_into(res, outs_main)

    if args.graph:
        # Capture each phase once (the same C-ABI calls, kernels only) and
        # replay it: the timed steps then carry no host launch overhead.
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for _ in range(3):
                run_dispatch()
                run_combine()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        g_disp, g_comb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_disp):
            run_dispatch()
        with torch.cuda.graph(g_comb):
            run_combine()
        torch.cuda.synchronize()
        phase_dispatch, phase_combine = g_disp.replay, g_comb.replay
    else:
        phase_dispatch, phase_combine = run_dispatch, run_combine

    phase_fns = [phase_dispatch] + ([run_gemm] if gemm else []) + [phase_combine]

    def step(stream_events=None):
        for j, fn in enumerate(phase_fns):
            if stream_events is not None:
                stream_events[j].record()
            fn()
        if stream_events is not None:
            stream_events[len(phase_fns)].record()

    flush = None
    cfg = config_dict(w, recv_rows)
    if args.layout == "expert":
        cfg["layout"] = ("expert-major: one row per (token, expert) in per-expert planes of "
                         "R*m rows; combine sums the top-k axis in problem order")
        cfg["mean_rows_per_token"] = cfg.pop("mean_dest_ranks")
    if fp8:
        cfg["payload"] = ("e4m3 dispatch rows + fp32 per-token scale; combine output e4m3 + "
                          "fp32 per-token scale (residual_out bf16)")
    if args.l2_hot:
        cfg["l2"] = "L2 hot: no flush between steps (small inputs may stay in L2)"
    if "flushed" in cfg["l2"]:
        # write a buffer twice the size of L2, then read another one, so the
        # timed kernels find L2 holding clean, unrelated lines
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        flush_read = torch.ones(64 << 20, dtype=torch.int32, device=dev)

        def do_flush(i):
            flush.fill_(i & 0xFF)
            flush_read.sum()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- timed region: inputs resident in HBM ----
    nev = len(phase_fns) + 1
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else local_rank)
    time.sleep(0.25)
    start.record()
    for i in range(args.steps):
        if flush is not None:
            do_flush(i)
        step(ev[i])
    stop.record()
    torch.cuda.synchronize()
    time.sleep(0.15)
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    total_ms = start.elapsed_time(stop)
    disp_ms = [e[0].elapsed_time(e[1]) for e in ev]
    comb_ms = [e[-2].elapsed_time(e[-1]) for e in ev]
    gemm_ms = [e[1].elapsed_time(e[2]) for e in ev] if gemm else []
    if flush is not None:       # time only the phases, not the flush
        total_ms = sum(disp_ms) + sum(comb_ms) + sum(gemm_ms)
    total_ms, ms_per_step, tokens_per_s = aggregate_over_ranks(total_ms, N, args.steps, world,
                                                               dev)
    st, flags = a2a.get_error()
    if st != 0:
        raise RuntimeError("device flag set during the timed region: %d %#x" % (st, flags))

    d_bytes, c_bytes = phase_bytes(w, recv_rows, fp8)
    peak, peak_kind = measured_peak()
    d_avg, c_avg = statistics.fmean(disp_ms), statistics.fmean(comb_ms)

    def pct(v, q):
        s = sorted(v)
        return s[min(len(s) - 1, int(q * len(s)))]

    phases = {
        "dispatch": {"ms_avg": d_avg, "ms_p50": pct(disp_ms, 0.5), "ms_p10": pct(disp_ms, 0.1),
                     "ms_p90": pct(disp_ms, 0.9), "bytes": d_bytes,
                     "gbs": d_bytes / d_avg / 1e6, "frac": d_bytes / d_avg / 1e6 / peak,
                     "frac_of_nominal": d_bytes / d_avg / 1e6 / NOMINAL_HBM_GBS,
                     "kernels": ([("dispatch_small_expert" if args.layout == "expert"
                                   else "dispatch_small") + ("_fp8" if fp8 else "")]
                                 if view.kernels == 1 else
                                 ["route_e_count", "route_e_scan"] if args.layout == "expert"
                                 else ["route_count", "route_scan"]) +
                                ([] if view.kernels == 1 else
                                 ["dispatch_fp8" if fp8 else "dispatch_rows"])},
        **({"expert_gemm": {
            "ms_avg": statistics.fmean(gemm_ms), "ms_p50": pct(gemm_ms, 0.5),
            "ms_p10": pct(gemm_ms, 0.1), "ms_p90": pct(gemm_ms, 0.9),
            "flops": 2.0 * gemm_rows * H * H, "weight_bytes": E * H * H * (1 if fp8 else 2),
            "tflops": 2.0 * gemm_rows * H * H / statistics.fmean(gemm_ms) / 1e9,
            "rows": gemm_rows,
            "kernels": (["rank_pairs", "expert_gemm (gathered rows)", "rank_aggregate"]
                        if gemm_rank else ["expert_gemm"])}} if gemm else {}),
        "combine": {"ms_avg": c_avg, "ms_p50": pct(comb_ms, 0.5), "ms_p10": pct(comb_ms, 0.1),
                    "ms_p90": pct(comb_ms, 0.9), "bytes": c_bytes,
                    "gbs": c_bytes / c_avg / 1e6, "frac": c_bytes / c_avg / 1e6 / peak,
                    "frac_of_nominal": c_bytes / c_avg / 1e6 / NOMINAL_HBM_GBS,
                    "kernels": ["combine_small" if N <= combine_small_max() and not fp8
                                else "combine"]},
    }
    eff_gbs = (d_bytes + c_bytes) / ms_per_step / 1e6

    # ---- end to end through the public API, host buffers ----
    # Every step copies its inputs (ids, weights, x, residual) from pinned
    # host memory and its outputs (y, residual_out) back, on three streams:
    # later steps' inputs go up and earlier steps' outputs come down while
    # step i runs dispatch + combine on the compute stream.  The steps rotate
    # through NB buffer sets, so a step's copies wait only for the step NB
    # before it.
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.pin_memory()
        hids, hw, hx = pin(ids_h), pin(wts_h), pin(x_h)
        hres = pin(res_h) if w.fused else None
        hin = [t for t in (hids, hw, hx, hres) if t is not None]
        specs = [((R, T, H), torch.float8_e4m3fn), ((R, T), torch.float32)] if fp8 else \
            [((R, T, H), torch.bfloat16)]
        if w.fused:
            specs.append(((R, T, H), torch.bfloat16))
        NB = max(2, args.e2e_buffers)
        hout = [[torch.empty(sh, dtype=dt).pin_memory() for sh, dt in specs] for _ in range(NB)]
        din = [[torch.empty_like(t, device=dev) for t in hin] for _ in range(NB)]
        dout = [[torch.empty(sh, dtype=dt, device=dev) for sh, dt in specs] for _ in range(NB)]
        h2d = sum(t.numel() * t.element_size() for t in hin)
        d2h = sum(t.numel() * t.element_size() for t in hout[0])
        compute = torch.cuda.current_stream(dev)
        up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()
        in_ready, in_free = [ev() for _ in range(NB)], [ev() for _ in range(NB)]
        out_ready, out_free = [ev() for _ in range(NB)], [ev() for _ in range(NB)]
        for b in range(NB):
            in_free[b].record(compute)
            out_free[b].record(compute)

        def e2e_step(i):
            b = i % NB
            with torch.cuda.stream(up):
                up.wait_event(in_free[b])
                for dst, src in zip(din[b], hin):
                    dst.copy_(src, non_blocking=True)
                in_ready[b].record(up)
            compute.wait_event(in_ready[b])
            compute.wait_event(out_free[b])
            d_ids, d_w, d_x = din[b][0], din[b][1], din[b][2]
            d_res = din[b][3] if w.fused else None
            a2a.dispatch(d_ids, d_w, d_x, w.runtime_max)
            if gemm:
                run_gemm()
            o = dout[b]
            combine_into(d_res, [o[0], o[1], o[2] if w.fused else None] if fp8
                         else [o[0], o[1] if w.fused else None])
            in_free[b].record(compute)
            out_ready[b].record(compute)
            with torch.cuda.stream(down):
                down.wait_event(out_ready[b])
                for dst, src in zip(hout[b], dout[b]):
                    dst.copy_(src, non_blocking=True)
                out_free[b].record(down)

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize()
        # The host link's throughput varies between and within runs on the
        # same machine (seen: 5.6 and 8.0 ms for the same step, copies alone
        # 5.5 and 11 ms), so both figures are taken in three trials: the
        # median trial for the end-to-end value, the fastest copy-only trial
        # as the link's bound.
        trials = []
        for _ in range(3):
            if world > 1:
                dist.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(compute)
            up.wait_event(e0)
            for i in range(args.e2e_steps):
                e2e_step(i)
            compute.wait_stream(down)
            e1.record(compute)
            torch.cuda.synchronize()
            trials.append(aggregate_over_ranks(e0.elapsed_time(e1), N, args.e2e_steps, world,
                                               dev))
        trials.sort(key=lambda r: r[0])
        e2e_ms, _, e2e_tps = trials[1]
        # The same copies with no kernels, up and down at once: the host
        # link's bound on this machine for the end-to-end step.
        copy_trials = []
        reps = max(4, args.e2e_steps // 4)
        for _ in range(3):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            c0.record(compute)
            up.wait_event(c0)
            down.wait_event(c0)
            for i in range(reps):
                b = i % NB
                with torch.cuda.stream(up):
                    for dst, src in zip(din[b], hin):
                        dst.copy_(src, non_blocking=True)
                with torch.cuda.stream(down):
                    for dst, src in zip(hout[b], dout[b]):
                        dst.copy_(src, non_blocking=True)
            compute.wait_stream(up)
            compute.wait_stream(down)
            c1.record(compute)
            torch.cuda.synchronize()
            copy_trials.append(c0.elapsed_time(c1) / reps)
        copy_ms = min(copy_trials)
        e2e = {"value": e2e_tps, "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.e2e_steps, "steps": args.e2e_steps,
               "trials_ms_per_step": [t[0] / args.e2e_steps for t in trials],
               "copy_only_ms_per_step": copy_ms,
               "copy_only_trials_ms": copy_trials,
               "link_gbs": (h2d + d2h) / copy_ms / 1e6,
               "frac_of_copy_bound": copy_ms / (e2e_ms / args.e2e_steps),
               "path": "pinned host -> device copies on a copy stream, moe_dispatch + "
                       "moe_combine on the compute stream, device -> pinned host copies on a "
                       "third stream; %d buffer sets in rotation so one step's inputs and another's "
                       "outputs move while a step computes" % NB}

    traffic = None
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    key = w.name + ("-expert" if args.layout == "expert" else "") + ("-fp8" if fp8 else "")
    if os.path.exists(prof):
        try:
            with open(prof) as f:
                tr = json.load(f)
            ent = tr.get(key, {}).get("combine")
            if ent and ent.get("sources_sha1") == sources_sha1(ent.get("sources", [])):
                traffic = ent["dram_bytes_per_launch"]
        except (OSError, ValueError, KeyError):
            traffic = None

    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded routing; N(0,1) bf16 payloads; random-init, no weights)",
        "config": cfg,
        "effective_gbs": eff_gbs, "hbm_frac": eff_gbs / peak,
        "phases": phases,
        "roofline": {"bound": "hbm", "kernel": "combine", "achieved": c_bytes / c_avg / 1e6,
                     "peak": peak, "unit": "GB/s", "frac": c_bytes / c_avg / 1e6 / peak,
                     "traffic": traffic, "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)"
                     % peak_kind if peak_kind == "measured" else "fallback 6.8 TB/s"},
        # the library's own kernels per step: what the dispatch reports it
        # queued (one launch for small batches, else three), the combine,
        # and the product's (three on the rank planes, one otherwise)
        "gpu_launches": (view.kernels + 1 + (3 if gemm_rank else 1 if gemm else 0)) * args.steps
                        if T > 0 else 0,
        "launch": "CUDA-graph replay of each phase's C-ABI call" if args.graph
                  else "direct C-ABI calls",
        "clocks": clk,
        "e2e": e2e,
    }
    if gemm:
        # the product dominates the step: report it against the tensor peak
        # (e4m3: the measured bf16 peak times the nominal fp8 / bf16 ratio, 2)
        tpk, tkind = measured_tensor_peak()
        if fp8:
            tpk, tkind = 2.0 * tpk, tkind + ", x2 for e4m3"
        tf = phases["expert_gemm"]["tflops"]
        gtraffic = None
        try:
            with open(prof) as f:
                ent = json.load(f).get(key, {}).get("expert_gemm")
            if ent and ent.get("sources_sha1") == sources_sha1(ent.get("sources", [])):
                gtraffic = ent["dram_bytes_per_launch"]
        except (OSError, ValueError, KeyError):
            gtraffic = None
        line["roofline"] = {"bound": "tensor", "kernel": "expert_gemm", "achieved": tf,
                            "peak": tpk, "unit": "TFLOP/s", "frac": tf / tpk,
                            "traffic": gtraffic,
                            "peak_source": "%s (MEASURED_PEAKS.json bf16_tflops_sustained)"
                            % tkind}
        line["roofline_combine"] = {"bound": "hbm", "achieved": c_bytes / c_avg / 1e6,
                                    "peak": peak, "unit": "GB/s",
                                    "frac": c_bytes / c_avg / 1e6 / peak}
        cfg["expert_gemm"] = ("W_e %s [%d][%d][%d], output into the combine payload" % (
            "e4m3 (per-channel scale 1/sqrt(H))" if fp8 else "bf16 N(0,1/H)", E, H, H))
        if gemm_rank:
            cfg["expert_gemm"] += ("; rank planes: each received row times each of its local "
                                   "experts (%d pairs), gated sum per row in ascending top-k "
                                   "order; combine unweighted (the rank sum)" % gemm_rows)
            line["roofline"]["achieved_over"] = ("the whole product call: pair lists, the "
                                                 "gathered tcgen05 product and the gated sum")
    return line


def aggregate_over_ranks(local_ms: float, tokens_per_rank_batch: int, steps: int, world: int,
                         device=None):
    """Whole-job timing of weak-scaled replicas: the slowest rank's elapsed
    time (all-reduce MAX) and the tokens all ranks processed per second.
    Returns (max_ms, ms_per_step, tokens_per_s)."""
    max_ms = float(local_ms)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([max_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        max_ms = float(t.item())
    ms_per_step = max_ms / steps
    return max_ms, ms_per_step, tokens_per_rank_batch * world / (ms_per_step / 1e3)


def combine_small_max():
    """Most tokens of a call the library combines on CTA clusters: its default (64)
    or the MOE_COMBINE_SMALL_MAX override (-1: never), for the phase's kernel label."""
    v = int(os.environ.get("MOE_COMBINE_SMALL_MAX", "0") or 0)
    return 64 if v == 0 else (0 if v < 0 else v)


def sources_sha1(names):
    """One sha1 over the listed kernel sources (csrc/), in order: the
    counters in profiles/traffic.json hold while it matches."""
    import hashlib
    h = hashlib.sha1()
    if not names:
        return None
    for name in names:
        path = os.path.join(ROOT, "combine_topk_ids_rank_gb300", "csrc", name)
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = workload(args)

    if args.impl == "reference":
        run_reference(args, w, rank)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    line = run_gpu(args, w, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, args.seed, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
