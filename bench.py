"""Benchmark of the DSpark verification hot path on one GB300 (or N replicas).

One step = the whole hot path on one batch: sv_schedule (survival products, tau cut,
budget check) then sv_verify (fused rejection-sampling verification) for B=64
requests x K=8 drafted tokens over a 151,936-entry vocabulary in bf16 at T=1 (draft
noise 1.0, full-length blocks: tau=0, budget=B*K). Inputs are synthetic and seeded.

Prints one JSON line (rank 0). `value` is verified draft tokens per second with the
inputs resident in HBM; `e2e` is the same metric through the public calls with the
inputs copied from pinned host memory every step and the results copied back.
`--impl reference` times the float64 CPU oracle on the same workload instead.
`--sweep` prints one line per point of the B x K roofline sweep.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft tokens/sec and logit GB/s (fraction of GB300 HBM peak), 1 GPU"
UNIT = "verified draft tokens/s"
B_DEF, K_DEF, V_DEF, T_DEF = 64, 8, 151_936, 1.0
GRAPH_STEPS = 100
PROFILE = os.path.join(ROOT, "profiles", "sv_verify_B64_K8_V151936_bf16_T1.md")


def _rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over the ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_step: float, steps: int, world: int, elapsed_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the max-over-ranks time
    (each rank is a replica that processes its own batch: weak scaling)."""
    return units_per_step * steps * world / (elapsed_ms / 1e3)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_sha():
    """Hash of the verify kernel's sources (its file and the shared header); ties a
    committed ncu summary to the kernel it measured."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_79_gb300", "csrc")
    for f in ("sv_common.cuh", "sv_verify.cu"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def _profiled_traffic():
    """DRAM bytes per launch of the verify kernel from the committed ncu summary, when it
    was taken on the current kernel sources; else None."""
    if not os.path.exists(PROFILE):
        return None
    txt = open(PROFILE).read()
    m = re.search(r"kernel sources sha:\s*([0-9a-f]+)", txt)
    t = re.search(r"dram bytes per launch \(full workload\):\s*([0-9]+)", txt)
    if not m or not t or m.group(1) != kernel_sha():
        return None
    return int(t.group(1))


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # let the sampler start before the timed region
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [[c.strip() for c in r] for r in csv.reader(io.StringIO(self.out)) if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [v for v in (num(r[1]) for r in rows) if v is not None]
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def _inputs(B, K, V, T, seed, device):
    import synth

    inp = synth.verify_inputs(B, K, V, dtype=torch.bfloat16, temperature=T, target_sigma=3.0,
                              draft_sigma=1.0, seed=seed, device=device)
    inp["conf"] = synth.confidences(B, K, seed=seed).to(device)
    return inp


def run_gpu(args):
    import speculative_decoding_verification_79_gb300 as sv
    import synth

    rank, world, local = _rank()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    B, K, V, T = args.B, args.K, args.V, args.T
    tau, budget = 0.0, B * K  # full-length blocks: nothing truncated, nothing trimmed
    sets = [_inputs(B, K, V, T, 1000 * rank + s, dev) for s in range(2)]  # 2 sets > L2
    ws = sv.Workspace(B, K, V, device=dev)
    st = torch.cuda.Stream(device=dev)
    out_len = torch.empty(B, dtype=torch.int32, device=dev)
    out_tok = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    out_acc = torch.empty(B, dtype=torch.int32, device=dev)

    def step(i, evs=None):
        g = sets[i & 1]
        if evs is not None:
            evs[0].record(st)
        sv.sv_schedule(g["conf"], tau, budget, ws, out_len=out_len, stream=st)
        if evs is not None:
            evs[1].record(st)
        sv.sv_verify(g["target"], g["draft"], g["draft_tok"], out_len, g["uniforms"], T, ws,
                     out_tok=out_tok, out_accepted=out_acc, stream=st)
        if evs is not None:
            evs[2].record(st)

    # Warm-up (eager), then capture GRAPH_STEPS steps with per-launch events.
    st.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(st):
        for i in range(max(3, args.warmup)):
            step(i)
    st.synchronize()
    n_graph = min(GRAPH_STEPS, args.steps)
    try:  # event-record nodes inside the graph time every launch of the last replay
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)]
               for _ in range(n_graph)]
    except TypeError:
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_graph)]
    # The timed graph holds the launches only; a second graph of the same steps with
    # event-record nodes between the launches gives the per-launch times.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        for i in range(n_graph):
            step(i)
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=st):
        for i in range(n_graph):
            step(i, evs[i])
    rem = args.steps % n_graph
    graph_rem = None
    if rem:
        graph_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_rem, stream=st):
            for i in range(rem):
                step(i)
    with torch.cuda.stream(st):  # replays go on the stream the events are recorded on
        for _ in range(2):  # graph warm-up
            graph.replay()
    st.synchronize()
    if ws.status(stream=st) != sv.SV_OK:
        raise RuntimeError("device status not OK after warm-up")

    reps = args.steps // n_graph
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with Clocks(dev.index if world == 1 else local) as clk, torch.cuda.stream(st):
        t0.record(st)
        for _ in range(reps):
            graph.replay()
        if graph_rem is not None:
            graph_rem.replay()
        t1.record(st)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    clocks = clk.summary()
    with torch.cuda.stream(st):  # per-launch times, after the timed region
        for _ in range(2):
            graph_ev.replay()
    st.synchronize()
    try:
        ver_ms = [e[1].elapsed_time(e[2]) for e in evs]
        sch_ms = [e[0].elapsed_time(e[1]) for e in evs]
        timing_src = ("event-record nodes around each launch in a replay of the same steps "
                      "after the timed region (the timed graph holds the launches only)")
    except RuntimeError:
        ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_graph)]
        with torch.cuda.stream(st):
            for i in range(n_graph):
                step(i, ev2[i])
        st.synchronize()
        ver_ms = [e[1].elapsed_time(e[2]) for e in ev2]
        sch_ms = [e[0].elapsed_time(e[1]) for e in ev2]
        timing_src = "eager launches with CUDA events right after the timed region"
    if ws.status(stream=st) != sv.SV_OK:
        raise RuntimeError("device status not OK after the timed region")

    L = out_len.cpu()
    tokens_per_step = int(L.sum().item())
    bytes_per_launch = synth.logit_bytes(L, V, 2, greedy=(T == 0.0))
    # For context: the rows a verifier would need if it stopped reading each request at
    # its first rejection j_b (positions 0..j_b, plus one row), from the last step's
    # outputs.
    jb = out_acc.cpu().clamp(min=0)
    early_exit = int(((2 * torch.minimum(jb + 1, L) + 1) * V * 2).sum().item())
    value = job_rate(tokens_per_step, args.steps, world, elapsed_ms)
    ver_avg = sum(ver_ms) / len(ver_ms)
    peak, peak_kind = _peaks()
    achieved = bytes_per_launch / (ver_avg / 1e3) / 1e9

    traffic = _profiled_traffic()
    traffic_src = (f"dram__bytes_read.sum + dram__bytes_write.sum of one ncu capture of this "
                   f"workload, from the committed summary {os.path.relpath(PROFILE, ROOT)}, "
                   f"taken on the same kernel sources (sha {kernel_sha()}); not measured in "
                   f"this run") if traffic is not None else (
                   "null: the committed ncu summary was taken on other kernel sources")
    e2e = run_e2e(args, sv, sets[0], ws, dev, tau, budget) if args.e2e_steps > 0 else None
    cpu = cpu_baseline(args) if (rank == 0 and not args.no_cpu) else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"schedule + verify, B={B} K={K} V={V} bf16 T={T}, draft noise "
                               "1.0, full-length blocks (tau=0, budget=B*K)",
                   "B": B, "K": K, "V": V, "temperature": T, "per_gpu_batch": B,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: two alternating input sets of "
                         f"{bytes_per_launch / 1e6:.0f} MB each (L2 129 MB)",
                   "timing": f"CUDA graph of {n_graph} steps replayed; CUDA events"},
        "logit_gbs": job_rate(bytes_per_launch, args.steps, world, elapsed_ms) / 1e9,
        "verify_us_avg": ver_avg * 1e3, "schedule_us_avg": sum(sch_ms) / len(sch_ms) * 1e3,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "traffic_source": traffic_src,
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
                     "kernel": "sv_verify_kernel<bf16, T>0>",
                     "algorithmic_bytes_per_launch": bytes_per_launch,
                     "per_launch_timing": timing_src,
                     "early_exit_min_bytes": early_exit,
                     "early_exit_min_frac_of_algorithmic": early_exit / bytes_per_launch},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def run_e2e(args, sv, g, ws, dev, tau, budget):
    """Public calls with host inputs: per step H2D of the step's inputs from pinned
    memory, schedule + verify, D2H of the emitted tokens and accepted counts. Two device
    input buffers alternate, so step i+1's copy (copy stream) runs under step i's
    schedule + verify (compute stream); each step's compute waits for its own copy, and
    a buffer is refilled only after the compute that read it has finished."""
    B, K = args.B, args.K
    host = {k: g[k].cpu().pin_memory() for k in ("target", "draft", "draft_tok", "uniforms",
                                                  "conf")}
    dbufs = [{k: torch.empty_like(g[k]) for k in host} for _ in range(2)]
    out_len = torch.empty(B, dtype=torch.int32, device=dev)
    out_tok = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    out_acc = torch.empty(B, dtype=torch.int32, device=dev)
    h_tok = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    h_acc = torch.empty(B, dtype=torch.int32).pin_memory()
    st = torch.cuda.Stream(device=dev)
    cp = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    for e in consumed:
        e.record(st)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = h_tok.numel() * 4 + h_acc.numel() * 4
    step = [0]

    def one():
        i = step[0] % 2
        step[0] += 1
        dbuf = dbufs[i]
        with torch.cuda.stream(cp):
            cp.wait_event(consumed[i])
            for k in host:
                dbuf[k].copy_(host[k], non_blocking=True)
            copied[i].record(cp)
        with torch.cuda.stream(st):
            st.wait_event(copied[i])
            sv.sv_schedule(dbuf["conf"], tau, budget, ws, out_len=out_len, stream=st)
            sv.sv_verify(dbuf["target"], dbuf["draft"], dbuf["draft_tok"], out_len,
                         dbuf["uniforms"], args.T, ws, out_tok=out_tok, out_accepted=out_acc,
                         stream=st)
            consumed[i].record(st)
            h_tok.copy_(out_tok, non_blocking=True)
            h_acc.copy_(out_acc, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        one()
    torch.cuda.synchronize(dev)
    dt = time.perf_counter() - t0
    tokens = int(out_len.sum().item()) * args.e2e_steps
    return {"value": tokens / dt, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
            "ms_per_step": dt / args.e2e_steps * 1e3}


def _oracle_args(inp, vlen=None):
    import synth

    return [synth.to_oracle(inp["target"]), synth.to_oracle(inp["draft"]),
            inp["draft_tok"].numpy(), inp["verify_len"].numpy() if vlen is None else vlen,
            inp["uniforms"].numpy()]


def _cpu_model():
    """The host CPU's model name (x86 /proc/cpuinfo, else lscpu, else platform)."""
    import platform
    import subprocess

    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def _oracle_rate(args, threads, seconds, seed):
    """Verified draft tokens/s of the float64 oracle (schedule + verify) on `threads`
    host threads, over as many passes of a sample batch as fit in about `seconds`."""
    import oracle

    inp = _inputs(1, args.K, args.V, args.T, seed, "cpu")
    t0 = time.perf_counter()
    oracle.verify(*_oracle_args(inp), args.T, nthreads=1, diag=False)
    one = time.perf_counter() - t0
    n_req = max(1, min(args.B, int(seconds * threads / max(one, 1e-6))))
    inp = _inputs(n_req, args.K, args.V, args.T, seed + 1, "cpu")
    conf = inp["conf"].numpy()
    oargs = _oracle_args(inp)
    threads = min(threads, n_req)
    reps, dt = 0, 0.0
    t0 = time.perf_counter()
    while reps == 0 or dt < seconds:
        oracle.schedule(conf, 0.0, n_req * args.K)
        oracle.verify(*oargs, args.T, nthreads=threads, diag=False)
        reps += 1
        dt = time.perf_counter() - t0
    return reps * n_req * args.K / dt, threads, reps, n_req, dt


def cpu_baseline(args):
    """The float64 oracle, as it stands, on a bounded sample of the same workload, scaled
    to verified draft tokens/s: on all host cores (the line's value) and on one core.
    The sample is the workload's batch of B requests (fewer if one batch alone would
    take longer than the time budget), run as many times as fit in about --cpu-seconds
    of wall time (half of it for the one-core figure)."""
    cores = os.cpu_count() or 1
    v, threads, reps, n_req, dt = _oracle_rate(args, cores, args.cpu_seconds, 7)
    v1, _, reps1, n1, dt1 = _oracle_rate(args, 1, args.cpu_seconds / 2, 17)
    return {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
            "value_1core": v1, "host_cpus": cores, "cpu_model": _cpu_model(),
            "sample": f"{reps} passes over {n_req} of the {args.B} requests (K={args.K}, "
                      f"V={args.V}, bf16 inputs, T={args.T}), schedule + verify, "
                      f"{dt:.1f} s wall on {threads} threads; one core: {reps1} passes over "
                      f"{n1} requests, {dt1:.1f} s"}


def run_reference(args):
    """--impl reference: the oracle on the host cores, each step a bounded sample of the
    workload sized so that warm-up plus the timed steps take about two minutes."""
    rank, world, _ = _rank()
    if rank != 0:
        return
    import oracle

    cores = os.cpu_count() or 1
    n_steps = args.steps + min(args.warmup, 3)
    per_step = 120.0 / max(1, n_steps)
    inp = _inputs(1, args.K, args.V, args.T, 2, "cpu")
    vl1 = torch.ones(1, dtype=torch.int32).numpy()
    t0 = time.perf_counter()
    oracle.verify(*_oracle_args(inp, vl1), args.T, nthreads=1, diag=False)
    t_l1 = time.perf_counter() - t0  # one request, one drafted position (3 rows)
    t_full = t_l1 * (2 * args.K + 1) / 3.0
    if per_step >= t_full:
        n_req = max(1, min(args.B, int(per_step * cores / t_full)))
        L = args.K
    else:
        n_req = 1
        L = max(1, min(args.K, int((per_step / t_l1 * 3.0 - 1.0) / 2.0)))
    inp = _inputs(n_req, args.K, args.V, args.T, 3, "cpu")
    conf = inp["conf"].numpy()
    a = _oracle_args(inp, torch.full((n_req,), L, dtype=torch.int32).numpy())
    threads = min(cores, n_req)

    def step():
        oracle.schedule(conf, 0.0, n_req * args.K)
        oracle.verify(*a, args.T, nthreads=threads, diag=False)

    for _ in range(min(args.warmup, 3)):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = n_req * L * args.steps / dt
    sample = (f"{n_req} of the {args.B} requests per step with verify length {L} (K={args.K}, "
              f"V={args.V}, bf16 inputs, T={args.T}), schedule + verify")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"schedule + verify, B={args.B} K={args.K} V={args.V} bf16 "
                               f"T={args.T}", "B": args.B, "K": args.K, "V": args.V},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_sweep(args):
    """One JSON line per roofline sweep point: the verify kernel alone, timed inside a CUDA
    graph (launch gaps excluded by event-record nodes around each launch), with enough
    alternating input sets that their total exceeds L2, so no launch reads the previous
    launch's data from L2."""
    import speculative_decoding_verification_79_gb300 as sv
    import synth

    dev = torch.device("cuda", 0)
    peak, _ = _peaks()
    temps = [float(t) for t in args.sweep_T.split(",")] if args.sweep_T else [args.T]
    st = torch.cuda.Stream(device=dev)
    for T in temps:
        for K in (args.sweep_K or synth.SWEEP_K):
            for B in (args.sweep_B or synth.SWEEP_B):
                nbytes1 = synth.logit_bytes([K] * B, synth.QWEN3_VOCAB, 2, greedy=(T == 0.0))
                nsets = max(2, -(-2 * (129 << 20) // max(1, nbytes1)))  # > 2x L2 in total
                sets = [synth.sweep_point(B, K, seed=s, device=dev) for s in range(nsets)]
                ws = sv.Workspace(B, K, synth.QWEN3_VOCAB, device=dev)
                outs = [(torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                         torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(2)]

                def launch(i):
                    g = sets[i % nsets]
                    o = outs[i & 1]
                    sv.sv_verify(g["target"], g["draft"] if T > 0 else None, g["draft_tok"],
                                 g["verify_len"], g["uniforms"] if T > 0 else None, T, ws,
                                 out_tok=o[0], out_accepted=o[1], stream=st)

                st.wait_stream(torch.cuda.current_stream(dev))
                with torch.cuda.stream(st):
                    for i in range(3):
                        launch(i)
                st.synchronize()
                n = max(args.sweep_reps, nsets)
                try:
                    evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
                           for _ in range(n)]
                except TypeError:
                    evs = None
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=st):
                    for i in range(n):
                        if evs:
                            evs[i][0].record(st)
                        launch(i)
                        if evs:
                            evs[i][1].record(st)
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(st):
                    graph.replay()
                    t0.record(st)
                    graph.replay()
                    t1.record(st)
                st.synchronize()
                if ws.status(stream=st) != sv.SV_OK:
                    raise RuntimeError("device status not OK in the sweep")
                try:
                    us = sorted(e[0].elapsed_time(e[1]) * 1e3 for e in evs)[n // 2]
                    src = "median of in-graph launch events"
                except (TypeError, RuntimeError):
                    us = t0.elapsed_time(t1) * 1e3 / n
                    src = "graph replay time / launches"
                tok = B * K
                print(json.dumps({"sweep": True, "T": T, "B": B, "K": K, "us": us,
                                  "tokens_per_s": tok / (us / 1e6),
                                  "gbs": nbytes1 / (us / 1e6) / 1e9,
                                  "frac": nbytes1 / (us / 1e6) / 1e9 / peak, "bytes": nbytes1,
                                  "input_sets": nsets, "timing": src}), flush=True)
                del sets, ws, graph


def _graph_median_us(fn, st, n=50):
    """Median per-call time of fn() captured n times in a CUDA graph, from event-record
    nodes around each call (launch gaps excluded)."""
    st.wait_stream(torch.cuda.current_stream(st.device))  # inputs are made on that stream
    with torch.cuda.stream(st):
        for _ in range(3):
            fn()
    st.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
           for _ in range(n)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        for i in range(n):
            evs[i][0].record(st)
            fn()
            evs[i][1].record(st)
    with torch.cuda.stream(st):
        graph.replay()
    st.synchronize()
    return sorted(e[0].elapsed_time(e[1]) * 1e3 for e in evs)[n // 2]


def run_calib(args):
    """One JSON line per configuration: per-call time of the plain schedule, the
    calibrated load-aware schedule, and the two calibration-loop kernels."""
    import speculative_decoding_verification_79_gb300 as sv
    import synth

    dev = torch.device("cuda", 0)
    st = torch.cuda.Stream(device=dev)
    for B, K in ((64, 8), (256, 16), (4096, 4)):
        conf = synth.confidences(B, K, seed=1).to(dev)
        temps = synth.temperatures(K, seed=1).to(dev)
        load = synth.load_state(seed=1).to(dev)
        c, vl, acc = (t.to(dev) for t in synth.calib_round(B, K, seed=1))
        ws = sv.Workspace(B, K, 16, device=dev)
        out_len = torch.empty(B, dtype=torch.int32, device=dev)
        cal = torch.empty(B, K, dtype=torch.float32, device=dev)
        tau = torch.empty(1, dtype=torch.float64, device=dev)
        stats = torch.zeros(sv.sv_calib_stats_len(K), dtype=torch.float64, device=dev)
        ece = torch.empty(1, dtype=torch.float64, device=dev)
        t_cur = temps.clone()
        budget = B * K // 2
        res = {"calib": True, "B": B, "K": K, "budget": budget}
        res["schedule_us"] = _graph_median_us(
            lambda: sv.sv_schedule(conf, 0.3, budget, ws, out_len=out_len, stream=st), st)
        res["schedule_cal_us"] = _graph_median_us(
            lambda: sv.sv_schedule_cal(conf, temps, load, 0.3, 0.2, 0.75, budget, ws,
                                       out_len=out_len, conf_cal=cal, tau_out=tau, stream=st), st)
        if B * K <= 8192:
            curve = synth.throughput_curve(8, seed=1).to(dev)
            res["schedule_curve_us"] = _graph_median_us(
                lambda: sv.sv_schedule_curve(conf, temps, load, 0.3, 0.2, 0.75, curve, budget, ws,
                                             out_len=out_len, stream=st), st)
        res["observe_us"] = _graph_median_us(
            lambda: sv.sv_calib_observe(c, vl, acc, stats, stream=st), st)
        res["update_us"] = _graph_median_us(
            lambda: sv.sv_calib_update(stats, t_cur, 0.01, 0.05, ece=ece, stream=st), st)
        if ws.status(stream=st) != sv.SV_OK:
            raise RuntimeError("device status not OK in the calibration timing")
        res["timing"] = "median of 50 in-graph call events"
        print(json.dumps(res), flush=True)


def run_markov(args):
    """One JSON line per rank r: the Markov logit-bias drafting loop (K positions) at the
    bench batch, timed per call inside a CUDA graph."""
    import speculative_decoding_verification_79_gb300 as sv
    import synth

    dev = torch.device("cuda", 0)
    st = torch.cuda.Stream(device=dev)
    peak, _ = _peaks()
    B, K, V = args.B, args.K, args.V
    for r in (128, 256):
        inp = {k: v.to(dev) for k, v in synth.markov_inputs(B, K, V, r, seed=3).items()}
        ws = sv.Workspace(B, K, 16, device=dev)
        corr = torch.empty_like(inp["logits"])
        tok = torch.empty((B, K), dtype=torch.int32, device=dev)
        keys = torch.empty(B * K, dtype=torch.int64, device=dev)
        us = _graph_median_us(lambda: sv.sv_markov_draft(inp["logits"], inp["U"], inp["Vm"],
                                                         inp["prev"], ws, corrected=corr,
                                                         draft_tok=tok, keys=keys, stream=st),
                              st, n=20)
        if ws.status(stream=st) != sv.SV_OK:
            raise RuntimeError("device status not OK in the Markov timing")
        nbytes = K * 2 * B * V * 2 + V * r * 2  # logits in and out per position, U once
        flops = K * 2.0 * V * r * B
        print(json.dumps({"markov": True, "B": B, "K": K, "V": V, "r": r, "us": us,
                          "us_per_position": us / K, "algorithmic_bytes": nbytes,
                          "gbs": nbytes / (us / 1e6) / 1e9,
                          "frac_hbm": nbytes / (us / 1e6) / 1e9 / peak,
                          "tflops": flops / (us / 1e6) / 1e12,
                          "timing": "median of 20 in-graph call events (a memset, one "
                                    "launch for the K positions at B <= 128, one token "
                                    "launch)"}),
              flush=True)


def run_tree(args):
    """One JSON line per batch size and temperature: tree verification of B trees of 16
    nodes (V=151,936 bf16; B from --tree-B, 64 by default), timed per call inside a CUDA
    graph with an L2 flush before each call. Algorithmic bytes are the rows the walk must read (the target row of every node
    on the accepted path and of the stop node, and the draft row of each of those with
    children), from the call's own outputs."""
    import speculative_decoding_verification_79_gb300 as sv
    import synth

    dev = torch.device("cuda", 0)
    st = torch.cuda.Stream(device=dev)
    peak, _ = _peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ws = sv.Workspace(1, 1, 1, device=dev)
    for B_t, T in [(b, t) for b in args.tree_B for t in (1.0, 0.0)]:
        inp = synth.tree_qwen3(T, seed=1, device=dev, B=B_t)
        B, N, V = inp["target"].shape
        outs = [torch.empty((B, N), dtype=torch.int32, device=dev),
                torch.empty(B, dtype=torch.int32, device=dev),
                torch.empty((B, N), dtype=torch.int32, device=dev)]
        st.wait_stream(torch.cuda.current_stream(dev))  # inputs are made on that stream

        def call():
            sv.sv_verify_tree(inp["target"], inp["draft"] if T > 0 else None, inp["parent"],
                              inp["draft_tok"], inp["n_nodes"],
                              inp["uniforms"] if T > 0 else None, T, ws, *outs, stream=st)

        with torch.cuda.stream(st):
            for _ in range(3):
                call()
        st.synchronize()
        n = 30
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
               for _ in range(n)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            for i in range(n):
                flush.zero_()
                evs[i][0].record(st)
                call()
                evs[i][1].record(st)
        with torch.cuda.stream(st):
            graph.replay()
        st.synchronize()
        us = sorted(e[0].elapsed_time(e[1]) * 1e3 for e in evs)[n // 2]
        if ws.status(stream=st) != sv.SV_OK:
            raise RuntimeError("device status not OK in the tree timing")
        acc = outs[1].cpu()
        nbytes = synth.tree_path_bytes(outs[2], acc, inp["parent"], V, 2, greedy=T == 0)
        all_rows = B * N * V * 2 * (1 if T == 0 else 2)
        emitted = int((acc + 1).sum())
        print(json.dumps({"tree": True, "B": B, "N": N, "V": V, "T": T, "dtype": "bf16",
                          "shape": "tree16", "us": us, "mean_accepted": float(acc.float().mean()),
                          "tokens_per_s": emitted / (us / 1e6),
                          "algorithmic_bytes": nbytes, "all_rows_bytes": all_rows,
                          "gbs": nbytes / (us / 1e6) / 1e9,
                          "frac_hbm": nbytes / (us / 1e6) / 1e9 / peak,
                          "timing": "median of 30 in-graph call events, L2 flushed before "
                                    "each call"}), flush=True)


def run_tree_once(args):
    """N untimed tree verification calls on the bench's tree workload (for ncu)."""
    import speculative_decoding_verification_79_gb300 as sv
    import synth

    dev = torch.device("cuda", 0)
    inp = synth.tree_qwen3(1.0, seed=1, device=dev)
    ws = sv.Workspace(1, 1, 1, device=dev)
    for _ in range(args.once):
        sv.sv_verify_tree(inp["target"], inp["draft"], inp["parent"], inp["draft_tok"],
                          inp["n_nodes"], inp["uniforms"], 1.0, ws)
    torch.cuda.synchronize()
    status = ws.status()
    print(json.dumps({"tree_once": args.once, "status": status}))
    if status != 0:
        sys.exit(1)


def run_curve_once(args):
    """N untimed calls of the throughput-curve schedule at B=64, K=8 (for ncu captures)."""
    import speculative_decoding_verification_79_gb300 as sv
    import synth

    dev = torch.device("cuda", 0)
    conf = synth.confidences(64, 8, seed=1).to(dev)
    curve = synth.throughput_curve(8, seed=1).to(dev)
    ws = sv.Workspace(64, 8, 16, device=dev)
    for _ in range(args.once):
        sv.sv_schedule_curve(conf, None, None, 0.3, 0.2, 0.75, curve, 256, ws)
    torch.cuda.synchronize()
    status = ws.status()
    print(json.dumps({"curve_once": args.once, "status": status}))
    if status != 0:
        sys.exit(1)


def run_markov_once(args):
    """N untimed calls of the Markov drafting loop at rank 256 (for ncu captures)."""
    import speculative_decoding_verification_79_gb300 as sv
    import synth

    dev = torch.device("cuda", 0)
    inp = {k: v.to(dev) for k, v in synth.markov_inputs(args.B, args.K, args.V, 256, seed=3).items()}
    ws = sv.Workspace(args.B, args.K, 16, device=dev)
    for _ in range(args.once):
        sv.sv_markov_draft(inp["logits"], inp["U"], inp["Vm"], inp["prev"], ws)
    torch.cuda.synchronize()
    status = ws.status()
    print(json.dumps({"markov_once": args.once, "status": status}))
    if status != 0:
        sys.exit(1)


def run_once(args):
    """N untimed steps on one input set of the configured workload (for ncu captures)."""
    import torch
    import speculative_decoding_verification_79_gb300 as sv

    dev = torch.device("cuda", 0)
    g = _inputs(args.B, args.K, args.V, args.T, 0, dev)
    ws = sv.Workspace(args.B, args.K, args.V)
    out_len = torch.empty(args.B, dtype=torch.int32, device=dev)
    for _ in range(args.once):
        sv.sv_schedule(g["conf"], 0.0, args.B * args.K, ws, out_len=out_len)
        sv.sv_verify(g["target"], g["draft"] if args.T > 0 else None, g["draft_tok"], out_len,
                     g["uniforms"] if args.T > 0 else None, args.T, ws)
    torch.cuda.synchronize()
    status = ws.status()
    print(json.dumps({"once": args.once, "status": status}))
    if status != 0:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--B", type=int, default=B_DEF)
    ap.add_argument("--K", type=int, default=K_DEF)
    ap.add_argument("--V", type=int, default=V_DEF)
    ap.add_argument("--T", type=float, default=T_DEF)
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--sweep-T", default=None)
    ap.add_argument("--sweep-reps", type=int, default=30)
    ap.add_argument("--calib", action="store_true",
                    help="time the calibrated schedule and the calibration-loop kernels")
    ap.add_argument("--markov", action="store_true",
                    help="time the Markov logit-bias drafting loop")
    ap.add_argument("--tree", action="store_true",
                    help="time tree (multi-candidate) verification")
    ap.add_argument("--tree-B", type=lambda x: [int(v) for v in x.split(",")], default=[64],
                    help="batch sizes of --tree, comma-separated")
    ap.add_argument("--sweep-B", type=lambda x: [int(v) for v in x.split(",")], default=None)
    ap.add_argument("--sweep-K", type=lambda x: [int(v) for v in x.split(",")], default=None)
    ap.add_argument("--once", type=int, default=0,
                    help="no timing: build one input set and run N schedule+verify steps "
                         "(a short, self-contained program for profilers)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.once > 0 and args.tree:
        run_tree_once(args)
    elif args.once > 0 and args.markov:
        run_markov_once(args)
    elif args.once > 0 and args.calib:
        run_curve_once(args)
    elif args.once > 0:
        run_once(args)
    elif args.sweep:
        run_sweep(args)
    elif args.calib:
        run_calib(args)
    elif args.markov:
        run_markov(args)
    elif args.tree:
        run_tree(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
