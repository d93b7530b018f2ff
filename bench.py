#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300: prints ONE JSON line (rank 0).

A step is one pass of the hot path over the single-prompt workload (B=1, H=32,
T=4096, K=V=128, bf16 q/k/v, fp32 gates/state, zero initial state, final state
returned): one ``kda_chunk_prefill_ws`` call (the 4-CTA cluster kernel that shares each
chunk's operands across the value tiles).  ``value`` is prefill tokens/s over all
ranks; the same run also times the paged-decode workload (256 sequences x 1 token,
H=32, K=V=128, 1024-slot fp32 pool, 64 steps carrying state in place) and reports
its state GB/s under "decode".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--only all|prefill|decode] [--decode-seqs S]

``--only`` and ``--decode-seqs`` exist for profiling captures of one kernel on a
smaller case; the default run measures everything.

Timing: CUDA events on the launching stream around each step, with L2 flushed
(a 256 MiB write) between timed steps; a short device sleep is queued ahead of each
start event so the event pair brackets the kernel, not the host-side launch.
N > 1 (torchrun): every rank runs its own replica of the workload (weak scaling),
step times are max-reduced over ranks.  ``--impl reference`` times the fp64 CPU
oracle on the host cores instead (a bounded sample of the same workload per step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

K_DIM = V_DIM = 128
CHUNK = 64
L2_FLUSH_BYTES = 256 << 20
DECODE_STEPS = 64


# ------------------------------------------------------------------ work accounting

def prefill_bytes_per_token_head(K=K_DIM, V=V_DIM, es=2):
    """Algorithmic HBM bytes per (token, head): q, k, v, o in bf16, g and beta fp32."""
    return (2 * K + 2 * V) * es + 4 * K + 4


def prefill_flops_per_token_head(K=K_DIM, V=V_DIM, C=CHUNK):
    """Lower-triangular chunk algebra: 6KV + C(3K + 2V) flops per (token, head)."""
    return 6 * K * V + C * (3 * K + 2 * V)


def decode_bytes_per_seq_head(K=K_DIM, V=V_DIM, es=2, state_es=4):
    """State read + write (fp32, or bf16 with state_es = 2) + q, k, v, o (bf16) + g (fp32) + beta."""
    return 2 * state_es * K * V + (2 * K + V) * es + 4 * K + 4 + V * es


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def load_traffic():
    """Per-launch DRAM bytes recorded from ncu captures in profiles/traffic.txt."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    out = {}
    try:
        with open(path) as f:
            for line in f:
                parts = line.split("#", 1)[0].split()
                if len(parts) == 2:
                    out[parts[0]] = None if parts[1] == "null" else int(parts[1])
    except OSError:
        pass
    return out


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons during a region."""
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, p in zip(names, parts[3:7]):
                if p.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[device_index] if vis else str(device_index)


# ------------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ our arm

def time_steps(fn, steps, warmup, stream, flush_buf, sleep_cycles=200_000):
    """Per-step device time (ms) with CUDA events on `stream`; L2 flushed between."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    with torch.cuda.stream(stream):
        for _ in range(steps):
            flush_buf.fill_(1.0)                      # evict L2 (256 MiB write)
            torch.cuda._sleep(sleep_cycles)           # keep the GPU busy while the host enqueues
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            e.synchronize()
            times.append(s.elapsed_time(e))
    return times


def measure_prefill(args, dev, stream, flush, world):
    """Device time of kda_chunk_prefill_ws on the single-prompt workload."""
    import torch
    from kimi_delta_attention_09_gb300 import _native, inputs
    case = inputs.single_prompt()
    T, H, K, V = case.T, case.H, case.K, case.V
    q, k, v = (x.to(dev) for x in (case.q, case.k, case.v))
    g, beta = case.g.to(dev), case.beta.to(dev)
    cu = case.cu_seqlens.to(dev)
    out = torch.empty_like(v)                       # bf16 output
    fin = torch.empty(case.N, H, K, V, dtype=torch.float32, device=dev)
    ws = torch.zeros(_native.kda_chunk_prefill_workspace_bytes(case.N, H, K, V, q.dtype),
                     dtype=torch.uint8, device=dev)

    def step():
        _native.kda_chunk_prefill_ws(q, k, v, g, beta, case.scale, None, cu, out, fin, ws, stream)

    barrier(world)
    with ClockSampler(gpu_id_for(dev.index)) as clk:
        times = time_steps(step, args.steps, args.warmup, stream, flush)
    torch.cuda.synchronize()
    barrier(world)
    return case, times, clk.summary(), (q, k, v, g, beta, cu, out, fin)


def measure_e2e(args, case, bufs, stream, flush, world):
    """The same prefill through the public host-to-host call (chunk_prefill_from_host):
    pinned host inputs in, pinned host output and final state out, every H2D and D2H
    copy inside the timed region (overlapped with the kernels piece by piece).  The
    working buffers of the first (untimed) call are passed back, as a serving loop
    would; the per-piece cu_seqlens they hold were copied once, outside the timing."""
    import torch
    import kimi_delta_attention_09_gb300 as kda
    hq, hk, hv, hg, hb = (x.pin_memory() for x in (case.q, case.k, case.v, case.g, case.beta))
    state = {"buffers": None}
    segments = 4

    def step():
        hout, hfin, state["buffers"] = kda.chunk_prefill_from_host(
            hq, hk, hv, hg, hb, case.scale, None, case.cu_seqlens, out_dtype=torch.bfloat16,
            segments=segments, buffers=state["buffers"])
        state["out"] = (hout, hfin)

    step()
    torch.cuda.synchronize()
    hout, hfin = state["out"]
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hg, hb))
    d2h = hout.numel() * hout.element_size() + hfin.numel() * hfin.element_size()
    n = max(3, args.steps // 2)
    times = time_steps(step, n, 3, stream, flush, sleep_cycles=0)
    return times, h2d, d2h, n * segments   # one prefill kernel per piece


def measure_decode(args, dev, stream, flush, world, bf16_state=False):
    """Device time per step of kda_recurrent_decode on the paged-decode workload
    (64 steps carrying the state in place through a 1024-slot fp32 pool); with
    bf16_state, of kda_recurrent_decode_bf16_state on the same pool stored in bf16."""
    import torch
    from kimi_delta_attention_09_gb300 import _native, inputs
    dcase = inputs.paged_decode(steps=DECODE_STEPS)
    N = min(args.decode_seqs, dcase.N)
    pool = dcase.pool.to(dev)
    if bf16_state:
        pool = pool.to(torch.bfloat16)
    fn = _native.kda_recurrent_decode_bf16_state if bf16_state else _native.kda_recurrent_decode
    idx = dcase.state_idx[:N].contiguous().to(dev)
    steps = [tuple(x[:N].contiguous().to(dev) for x in (s.q, s.k, s.v, s.g, s.beta))
             for s in dcase.steps]
    H, V = pool.shape[1], pool.shape[3]
    dout = torch.empty(N, H, V, dtype=torch.bfloat16, device=dev)
    counter = [0]

    def step():
        sq, sk, sv, sg, sb = steps[counter[0] % DECODE_STEPS]
        counter[0] += 1
        fn(sq, sk, sv, sg, sb, dcase.scale, pool, idx, dout, stream)

    barrier(world)
    times = time_steps(step, DECODE_STEPS if args.only != "decode" else max(args.steps, 1),
                       args.warmup, stream, flush)
    barrier(world)
    d_bytes = N * H * decode_bytes_per_seq_head(state_es=2 if bf16_state else 4)
    name = dcase.name if N == dcase.N else dcase.name.replace("N256", f"N{N}")
    if bf16_state:
        name += "_bf16_state"
    return name, N, times, d_bytes


def run_ours(args, rank, world, local):
    import torch

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks = load_peaks()
    peak_hbm = peaks["hbm_gbs"]
    traffic = load_traffic()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    line = {"metric": "KDA prefill tokens/s + TFLOP/s; decode state GB/s (fraction of roofline)",
            "value": None, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic"}
    launches = 0

    if args.only in ("all", "prefill"):
        case, ptimes, clocks, bufs = measure_prefill(args, dev, stream, flush, world)
        T, H, K, V = case.T, case.H, case.K, case.V
        p_ms = statistics.mean(ptimes)
        p_ms_max = max_over_ranks(p_ms, world)
        p_bytes = T * H * prefill_bytes_per_token_head() + case.N * H * K * V * 4
        p_flops = T * H * prefill_flops_per_token_head()
        p_gbs = p_bytes / (p_ms * 1e-3) / 1e9
        launches += args.steps
        line.update({
            "value": round(world * T / (p_ms_max * 1e-3), 1),
            "ms_per_step": round(p_ms_max, 5),
            "config": {"workload": case.name, "global_batch": world, "seq_len": T, "heads": H,
                       "head_dim_k": K, "head_dim_v": V, "chunk": CHUNK, "out_dtype": "bf16",
                       "parallelism": f"replicas{world}",
                       "l2": "flushed between timed steps (256 MiB write)"},
            "prefill": {"tokens_per_s": round(T / (p_ms * 1e-3), 1),
                        "tflops_algorithmic": round(p_flops / (p_ms * 1e-3) / 1e12, 3),
                        "gb_per_s_algorithmic": round(p_gbs, 1),
                        "ms_per_call": round(p_ms, 5), "ms_min": round(min(ptimes), 5),
                        "algorithmic_bytes": p_bytes, "algorithmic_flops": p_flops},
            "roofline": {"bound": "hbm", "kernel": "kda_prefill_rr_kernel",
                         "achieved": round(p_gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                         "frac": round(p_gbs / peak_hbm, 4), "peak_source": peaks["source"],
                         "traffic": traffic.get("prefill_rr_single_prompt")},
            "clocks": clocks,
        })
        if args.only == "all":
            etimes, h2d, d2h, n_e2e = measure_e2e(args, case, bufs, stream, flush, world)
            e_ms = max_over_ranks(statistics.mean(etimes), world)
            launches += n_e2e
            line["e2e"] = {"value": round(world * T / (e_ms * 1e-3), 1), "unit": "tokens/s",
                           "ms_per_step": round(e_ms, 4),
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_oracle_baseline(case, n_tokens=T)
        del bufs

    if args.only in ("all", "decode"):
        name, N, dtimes, d_bytes = measure_decode(args, dev, stream, flush, world)
        d_ms = statistics.mean(dtimes)
        d_ms_max = max_over_ranks(d_ms, world)
        d_gbs = d_bytes / (d_ms * 1e-3) / 1e9
        launches += len(dtimes)
        line["decode"] = {
            "workload": name, "metric": "state GB/s",
            "value": round(world * d_bytes / (d_ms_max * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(d_ms_max, 5), "steps": len(dtimes),
            "algorithmic_bytes_per_step": d_bytes,
            "roofline": {"bound": "hbm", "kernel": "kda_decode_kernel", "achieved": round(d_gbs, 1),
                         "peak": peak_hbm, "unit": "GB/s", "frac": round(d_gbs / peak_hbm, 4),
                         "traffic": traffic.get("decode_paged")}}
        name, N, dtimes, d_bytes = measure_decode(args, dev, stream, flush, world, bf16_state=True)
        d_ms = statistics.mean(dtimes)
        d_ms_max = max_over_ranks(d_ms, world)
        d_gbs = d_bytes / (d_ms * 1e-3) / 1e9
        launches += len(dtimes)
        line["decode_bf16_state"] = {
            "workload": name, "metric": "state GB/s",
            "value": round(world * d_bytes / (d_ms_max * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(d_ms_max, 5), "steps": len(dtimes),
            "algorithmic_bytes_per_step": d_bytes,
            "roofline": {"bound": "hbm", "kernel": "kda_decode_kernel (bf16 state)",
                         "achieved": round(d_gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                         "frac": round(d_gbs / peak_hbm, 4),
                         "traffic": traffic.get("decode_bf16_state_paged")}}
    line["gpu_launches"] = launches
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ oracle arm

def cpu_oracle_baseline(case, n_tokens):
    """The fp64 oracle (as it stands) on the first n_tokens of the workload."""
    import oracle
    sl = slice(0, n_tokens)
    threads = oracle.default_threads()
    used = min(threads, case.H)
    # repeat the sample until it has taken ~15 CPU-seconds on the threads in use
    reps, dt = 0, 0.0
    while reps == 0 or dt * used < 15.0:
        t0 = time.perf_counter()
        oracle.prefill(case.q[sl], case.k[sl], case.v[sl], case.g[sl], case.beta[sl], case.scale,
                       None, [0, n_tokens], nthreads=threads)
        dt += time.perf_counter() - t0
        reps += 1
    return {"value": round(reps * n_tokens / dt, 2), "unit": "tokens/s", "cores": used,
            "host_cores": threads, "kind": "oracle",
            "sample": f"first {n_tokens} tokens x {case.H} heads of {case.name}, {reps} repeats "
                      f"(fp64 token recurrence, {dt:.2f} s wall on {used} threads)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from kimi_delta_attention_09_gb300 import inputs
    import oracle
    case = inputs.single_prompt()
    n_tok = 1024
    sl = slice(0, n_tok)
    sample = [x[sl] for x in (case.q, case.k, case.v, case.g, case.beta)]
    threads = oracle.default_threads()

    def step():
        oracle.prefill(*sample, case.scale, None, [0, n_tok], nthreads=threads)

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    val = round(n_tok / (ms * 1e-3), 2)
    used = min(threads, case.H)
    line = {
        "impl": "reference",
        "metric": "KDA prefill tokens/s + TFLOP/s; decode state GB/s (fraction of roofline)",
        "value": val, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": case.name, "global_batch": 1, "seq_len": case.T, "heads": case.H,
                   "head_dim_k": case.K, "head_dim_v": case.V, "chunk": CHUNK,
                   "parallelism": "host threads over (sequence, head)"},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": used, "host_cores": threads,
                         "kind": "oracle",
                         "sample": f"first {n_tok} tokens x {case.H} heads of {case.name} per step"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "prefill", "decode"], default="all")
    ap.add_argument("--decode-seqs", type=int, default=256)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)          # at least 3 untimed warm-up steps
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; other ranks exit without work
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, rank, int(os.environ.get("WORLD_SIZE", "1")))
        return
    rank, world, local = dist_setup()
    run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
