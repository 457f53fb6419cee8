#!/usr/bin/env python3
"""Benchmark of the KDA chunked prefill forward on GB300.

One step = one kda_fwd over the whole packed64 workload (64 packed sequences with
lengths ~ U{64..8192}, seed 4; H = 64; K = V = 128; fp32 initial/final state,
updated in place in one of two rotating pre-initialised state buffers), inputs
resident in HBM.  The inputs (~17 GB) are far larger than L2 (129 MB), so no L2
flush is needed between steps.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FLOP_PER_TOKEN_HEAD = 131072      # 6VK + 4CK + 4VC at C = 32, K = V = 128
BYTES_PER_TOKEN_HEAD = 1282       # q, k, v, g (4 x 256 B) + beta (2 B) + out (256 B)
WORKLOAD = "packed64"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "kda_fwd_tc_traffic.json")


def measured_traffic(workload_name: str):
    """DRAM bytes (read + write) of one forward launch from the committed ncu record, if the
    record is for this workload and the kernel sources are byte-identical to the measured ones."""
    import hashlib
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
        if rec.get("workload") != workload_name:
            return None
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        return float(rec["dram_bytes_per_launch"]) if h.hexdigest() == rec["sources_sha256"] else None
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank value across the job (identity for one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


METRIC = "KDA prefill tokens/s at 1 GB300 (TFLOP/s and roofline fractions alongside)"
# --kernel: the default kernel or one of the design alternatives (kda_fwd_ex's kernel field)
KERNELS = {"default": 0x000, "chunk16": 0x100, "register_state": 0x200, "bf16_state": 0x300, "smem_state": 0x400}


L2_BYTES = 129 * 1024 * 1024
# workloads whose algorithmic bytes are under this get an L2 flush between timed launches
FLUSH_BELOW = 4 * L2_BYTES
FLUSH_BYTES = 2 * L2_BYTES


def needs_flush(w) -> bool:
    return workload_totals(w)[2] < FLUSH_BELOW


def bench_config(w, world: int) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    name = lambda dt: {"float32": "fp32", "bfloat16": "bf16"}[str(dt).replace("torch.", "")]
    if w.init_dtype is not None:
        state = f"{name(w.init_dtype)} in, {name(w.final_dtype)} out, in place, 2 rotating buffers"
    else:
        state = f"zero initial state, {name(w.final_dtype)} final state, 2 rotating buffers"
    return {"workload": w.name, "tokens": w.total_tokens, "heads": w.H, "sequences": w.num_seqs,
            "head_dim": w.K, "chunk": 32, "state": state,
            "l2": (f"L2 flushed before each timed launch ({FLUSH_BYTES >> 20} MB write, outside the launch's events; "
                   "ms_per_step = sum of launch times / steps)") if needs_flush(w) else
                  "inputs larger than L2 (no flush)",
            "parallelism": f"replicas x{world}"}


def workload_totals(w):
    tokens = w.total_tokens
    th = tokens * w.H
    per_state = w.V * w.K
    state_bytes = w.units * per_state * (w.init_dtype.itemsize if w.init_dtype is not None else 0)
    state_bytes += w.units * per_state * w.final_dtype.itemsize
    return tokens, th, th * BYTES_PER_TOKEN_HEAD + state_bytes, th * FLOP_PER_TOKEN_HEAD


def oracle_sample(inp, budget_s: float, nthreads: int = 0):
    """Time the oracle on a bounded sample of whole (sequence, head) units.

    Units are taken in a fixed order (sequence 0.. , head 0..) until the estimated
    CPU time reaches ``budget_s``.  Returns (token-heads processed, seconds, threads, description)."""
    import torch
    from oracle import kda_oracle as O
    w = inp.w
    cu = [0] + list(torch.cumsum(torch.tensor(w.seq_lens), 0).tolist()) if w.packed else \
        [b * w.T for b in range(w.B + 1)]
    threads = nthreads or O.max_threads()
    cpu = lambda t: t.detach().cpu()
    flat = lambda t: t.reshape((w.B * w.T,) + tuple(t.shape[2:]))
    q, k, v, g, beta = (flat(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))

    def run(n, heads):
        b, e = cu[n], cu[n + 1]
        hi = torch.tensor(heads, device=q.device)
        sl = lambda t: cpu(t[b:e].index_select(1, hi)).unsqueeze(0)
        S0 = None if inp.initial_state is None else cpu(inp.initial_state[n].index_select(0, hi)).unsqueeze(0)
        args = (sl(q), sl(k), sl(v), sl(g), sl(beta), inp.scale, cpu(inp.A_log)[heads],
                cpu(inp.dt_bias)[heads], inp.lower_bound)
        t0 = time.perf_counter()
        O.kda_oracle_fwd(*args, initial_state=S0, nthreads=threads)
        return (e - b) * len(heads), time.perf_counter() - t0

    # calibrate on one head of sequence 0, then run whole sequences x `threads` heads
    th, dt = run(0, [0])
    rate_1core = th / max(dt, 1e-9)
    done_th, done_s, n = 0, 0.0, 0
    heads = list(range(min(threads, w.H)))
    while n < w.num_seqs:
        L = cu[n + 1] - cu[n]
        est = L * len(heads) / (rate_1core * len(heads)) if L else 0.0
        if done_s > 0 and done_s + est > budget_s:
            break
        if L:
            a, s = run(n, heads)
            done_th += a
            done_s += s
        n += 1
    desc = (f"oracle (fp64 C, OpenMP over units) on sequences 0..{n - 1} x heads 0..{len(heads) - 1} "
            f"of {w.name}: {done_th} token-heads in {done_s:.1f} s; tokens/s = token-heads/s / H")
    return done_th, done_s, threads, desc


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from gated_delta_rule_36_gb300.inputs import make_inputs, workload
    w = workload(args.workload)
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = make_inputs(w, dev)
    budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(inp, budget, args.oracle_threads)
    tot_th, tot_s, threads, desc = 0, 0.0, 1, ""
    for _ in range(args.steps):
        th, s, threads, desc = oracle_sample(inp, budget, args.oracle_threads)
        tot_th += th
        tot_s += s
    value = tot_th / w.H / tot_s
    line = {"impl": "reference", "metric": METRIC, "value": value,
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * tot_s / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(w, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import gated_delta_rule_36_gb300 as kda
    from gated_delta_rule_36_gb300.inputs import make_inputs, workload

    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.load()
    w = workload(args.workload)
    inp = make_inputs(w, dev)
    tokens, token_heads, alg_bytes, alg_flop = workload_totals(w)
    stream = torch.cuda.current_stream(dev)

    out = torch.empty_like(inp.q)
    states = [inp.initial_state.clone() for _ in range(2)] if inp.initial_state is not None else [None, None]
    finals = states if inp.initial_state is not None else \
        [torch.empty((w.num_seqs, w.H, w.V, w.K), dtype=w.final_dtype, device=dev) for _ in range(2)]
    ws = torch.empty(kda.kda_workspace_size(tokens, w.H, w.num_seqs), dtype=torch.uint8, device=dev)

    kflags = KERNELS[args.kernel]

    def step(i):
        kda.kda_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, out, inp.A_log, inp.dt_bias,
                    inp.lower_bound, initial_state=states[i % 2], final_state=finals[i % 2],
                    cu_seqlens=inp.cu_seqlens, workspace=ws, stream=stream, flags=kflags)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if kda.kda_read_device_status(ws) != 0:
        raise RuntimeError("device status error during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev) if needs_flush(w) else None
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(i)
            ev[i][0].record(stream)
            step(args.warmup + i)
            ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    per_launch_ms = [a.elapsed_time(b) for a, b in ev]
    # with a flush between launches the step time is the launches' own time, flushes excluded
    ms_total = sum(per_launch_ms) if flush is not None else t_start.elapsed_time(t_end)
    if kda.kda_read_device_status(ws) != 0:
        raise RuntimeError("device status error in the timed region")

    ms_step = max_over_ranks(ms_total / args.steps, world, dev)
    value = tokens * world / (ms_step / 1000.0)
    kernel_ms = statistics.mean(per_launch_ms)
    hbm_peak, tc_peak, tc_sus, peak_src = load_peaks()
    achieved_gbs = alg_bytes / (kernel_ms / 1000.0) / 1e9
    tflops = alg_flop / (kernel_ms / 1000.0) / 1e12
    clocks = clk.summary()

    # end to end through the public API: pinned host inputs -> device, forward, result -> host
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(kda, inp, w, dev, stream, args)

    line = {
        "metric": METRIC,
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": dict(bench_config(w, world), **({} if args.kernel == "default" else {"kernel": args.kernel})),
        "tflops": tflops,
        "tensor_frac": tflops / tc_peak,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved_gbs / hbm_peak,
                     "traffic": args.traffic if args.traffic is not None else measured_traffic(w.name),
                     "peak_source": peak_src,
                     "kernel_ms": kernel_ms, "algorithmic_bytes": alg_bytes},
        "clocks": clocks,
        "gpu_launches": (2 if w.packed else 1) * args.steps,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        th, s, threads, desc = oracle_sample(inp, args.cpu_budget, args.oracle_threads)
        line["cpu_baseline"] = {"value": th / w.H / s, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(kda, inp, w, dev, stream, args):
    """End to end through the host-buffer entry point kda_fwd_host: pinned host inputs
    in, forward, output and final state back to pinned host memory, every step."""
    import torch
    from gated_delta_rule_36_gb300 import binding as kb
    host = {n: getattr(inp, n).detach().cpu().pin_memory() for n in ("q", "k", "v", "g", "beta", "A_log", "dt_bias")}
    h_init = inp.initial_state.detach().cpu().pin_memory() if inp.initial_state is not None else None
    h_cu = inp.cu_seqlens.detach().cpu().pin_memory() if inp.cu_seqlens is not None else None
    h_out = torch.empty_like(host["q"]).pin_memory()
    h_final = torch.empty((w.num_seqs, w.H, w.V, w.K), dtype=w.final_dtype).pin_memory()
    nbytes = kb.kda_fwd_host_device_bytes(host["q"], cu_seqlens=h_cu, initial_state=h_init, final_state=h_final)
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    h2d += (h_init.numel() * h_init.element_size() if h_init is not None else 0)
    h2d += (h_cu.numel() * h_cu.element_size() if h_cu is not None else 0)
    d2h = h_out.numel() * h_out.element_size() + h_final.numel() * h_final.element_size()

    def step():
        kb.kda_fwd_host(host["q"], host["k"], host["v"], host["g"], host["beta"], inp.scale, h_out, host["A_log"],
                        host["dt_bias"], inp.lower_bound, initial_state=h_init, final_state=h_final,
                        cu_seqlens=h_cu, device_buffer=buf, groups=args.e2e_groups, stream=stream)

    step()
    torch.cuda.synchronize()
    n = args.e2e_steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    ev[0].record(stream)
    for i in range(n):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]
    ms = ev[0].elapsed_time(ev[n]) / n

    # the copies alone, for the bound: every input host -> device, then out and final_state back
    dev_in = {k: torch.empty_like(t, device=dev) for k, t in host.items()}
    d_init = torch.empty_like(h_init, device=dev) if h_init is not None else None
    d_out = torch.empty_like(h_out, device=dev)
    d_final = torch.empty_like(h_final, device=dev)

    def copies_in():
        for k, t in host.items():
            dev_in[k].copy_(t, non_blocking=True)
        if h_init is not None:
            d_init.copy_(h_init, non_blocking=True)

    def copies_out():
        h_out.copy_(d_out, non_blocking=True)
        h_final.copy_(d_final, non_blocking=True)

    def timed(fn, reps=3):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    h2d_ms, d2h_ms = timed(copies_in), timed(copies_out)
    del dev_in, d_init, d_out, d_final
    return {"value": w.total_tokens / (ms / 1000.0), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms, "ms_per_step_min": min(per),
            "ms_per_step_median": statistics.median(per), "steps": n, "groups": args.e2e_groups,
            "api": "kda_fwd_host",
            "copies_alone": {"h2d_ms": h2d_ms, "h2d_gbs": h2d / (h2d_ms / 1e3) / 1e9,
                             "d2h_ms": d2h_ms, "d2h_gbs": d2h / (d2h_ms / 1e3) / 1e9}}


def run_decode(args):
    """The single-token decode step (kda_decode), one line of its own: B sequences x H heads,
    each step one token per sequence with the fp32 state updated in place (268 MB at
    B = H = 64, larger than L2, so no flush).  Bound by the state's HBM traffic."""
    import torch
    import gated_delta_rule_36_gb300 as kda
    B, H = args.decode_batch, args.decode_heads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kda.load()
    gen = torch.Generator(device=dev).manual_seed(7)
    bf = lambda *s: torch.randn(*s, generator=gen, device=dev).to(torch.bfloat16)
    q, k, v, g = bf(B, H, 128), bf(B, H, 128), bf(B, H, 128), bf(B, H, 128)
    beta = torch.rand(B, H, generator=gen, device=dev).to(torch.bfloat16)
    A_log = torch.rand(H, generator=gen, device=dev)
    dt_bias = torch.rand(H, 128, generator=gen, device=dev)
    state = 0.1 * torch.randn(B, H, 128, 128, generator=gen, device=dev)
    out = torch.empty(B, H, 128, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = lambda: kda.kda_decode(q, k, v, g, beta, 128 ** -0.5, out, A_log, dt_bias, -5.0,
                                  initial_state=state, final_state=state, stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    alg = B * H * (2 * 128 * 128 * 4 + 4 * 128 * 2 + 128 * 2 + 2)   # state in + out, q k v g, out, beta
    hbm_peak, _, _, peak_src = load_peaks()
    gbs = alg / (ms / 1000.0) / 1e9
    print(json.dumps({
        "metric": "KDA decode tokens/s (one token per sequence per step)", "value": B / (ms / 1000.0),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "bf16 inputs, fp32 state", "data": "synthetic",
        "config": {"workload": f"decode B={B} H={H}", "state": "fp32, in place", "l2": "state larger than L2"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                     "peak_source": peak_src, "algorithmic_bytes": alg},
        "clocks": clk.summary(), "gpu_launches": args.steps}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--kernel", choices=tuple(KERNELS), default="default",
                    help="the default kernel or a design alternative (timed on the same workload)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-groups", type=int, default=8, help="sequence groups kda_fwd_host pipelines over")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--oracle-threads", type=int, default=0,
                    help="host threads of the oracle legs (cpu_baseline, --impl reference); 0 = all cores")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes (read+write) of one launch of the forward kernel; by default the "
                         "committed record in profiles/, used only while the kernel sources match it")
    ap.add_argument("--decode", action="store_true", help="time the single-token decode step instead")
    ap.add_argument("--decode-batch", type=int, default=64)
    ap.add_argument("--decode-heads", type=int, default=64)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)   # at least 3 untimed warm-up steps
    if args.decode:
        run_decode(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
