#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300: prints ONE JSON line (rank 0).

A step is one pass of the hot path over the single-prompt workload (B=1, H=32,
T=4096, K=V=128, bf16 q/k/v, fp32 gates/state, zero initial state, final state
returned): one ``kda_chunk_prefill_ws`` call (the 4-CTA cluster kernel that shares each
chunk's operands across the value tiles).  ``value`` is prefill tokens/s.  The same run
also times the varlen packed workload (8 sequences, lengths U[256, 8192], nonzero
initial states) under "prefill_varlen", the long prompt (T=65536) under "prefill_long",
the paged-decode workload (256 sequences x 1 token, H=32, K=V=128, 1024-slot fp32
pool, 64 steps carrying state in place) under "decode" / "decode_bf16_state", and the
causal convolution in front of the op (width 4, SiLU, taps in paged slots) on the
varlen workload's 12,288 [q|k|v] channels ("conv_prefill") and on one token of 256
sequences ("conv_update").

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--only all|prefill|decode|conv] [--decode-seqs S] [--no-cpu-baseline]

``--only`` and ``--decode-seqs`` exist for profiling captures of one kernel on a
smaller case; the default run measures everything.  The end-to-end number ("e2e") is
the same single-prompt prefill through the C ABI's host-to-host call
(kda_chunk_prefill_host: pinned host buffers, every copy inside the timed region), with
the host link timed beside it.

Timing: CUDA events on the launching stream around each step, with L2 flushed
(a 256 MiB write) between timed steps; a short device sleep is queued ahead of each
start event so the event pair brackets the kernel, not the host-side launch.
The benchmark is single-GPU (every call of the library runs on one GPU): ``--gpus`` > 1
or a torchrun launch with WORLD_SIZE > 1 exits with an error line.  ``--impl reference``
times the fp64 CPU oracle on the host cores instead (a bounded sample of the same
workload per step; under torchrun rank 0 alone runs it).
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


def prefill_case_bytes(case):
    """Algorithmic HBM bytes of one prefill call: the per-(token, head) traffic plus the
    final states written and, when given, the initial states read (64 KiB each)."""
    T, H, K, V = case.T, case.H, case.K, case.V
    b = T * H * prefill_bytes_per_token_head() + case.N * H * K * V * 4
    if case.init_state is not None:
        b += case.N * H * K * V * 4
    return b


def time_prefill_case(args, case, dev, stream, flush, steps):
    """Device times of kda_chunk_prefill_ws (the cluster kernel) on one workload."""
    import torch
    from kimi_delta_attention_09_gb300 import _native
    H, K, V = case.H, case.K, case.V
    q, k, v = (x.to(dev) for x in (case.q, case.k, case.v))
    g, beta = case.g.to(dev), case.beta.to(dev)
    cu = case.cu_seqlens.to(dev)
    init = None if case.init_state is None else case.init_state.to(dev)
    out = torch.empty_like(v)                       # bf16 output
    fin = torch.empty(case.N, H, K, V, dtype=torch.float32, device=dev)
    ws = torch.zeros(_native.kda_chunk_prefill_workspace_bytes(case.N, H, K, V, q.dtype),
                     dtype=torch.uint8, device=dev)

    def step():
        _native.kda_chunk_prefill_ws(q, k, v, g, beta, case.scale, init, cu, out, fin, ws, stream)

    times = time_steps(step, steps, args.warmup, stream, flush)
    torch.cuda.synchronize()
    status = _native.kda_chunk_prefill_status(ws, stream)
    if status != _native.KDA_OK:
        raise RuntimeError(f"prefill on {case.name} reported device status {status}")
    return times, (q, k, v, g, beta, cu, out, fin)


def measure_prefill(args, dev, stream, flush):
    """Device time of kda_chunk_prefill_ws on the single-prompt workload."""
    from kimi_delta_attention_09_gb300 import inputs
    case = inputs.single_prompt()
    with ClockSampler(gpu_id_for(dev.index)) as clk:
        times, bufs = time_prefill_case(args, case, dev, stream, flush, args.steps)
    return case, times, clk.summary(), bufs


def prefill_block(case, times, peak_hbm, traffic_key, traffic, sample):
    """The JSON block of one timed prefill workload."""
    p_ms = statistics.mean(times)
    p_bytes = prefill_case_bytes(case)
    p_flops = case.T * case.H * prefill_flops_per_token_head()
    p_gbs = p_bytes / (p_ms * 1e-3) / 1e9
    return {"workload": case.name, "sequences": case.N, "tokens": case.T,
            "ms_per_step": round(p_ms, 5), "ms_min": round(min(times), 5), "steps": len(times),
            "tokens_per_s": round(case.T / (p_ms * 1e-3), 1),
            "tflops_algorithmic": round(p_flops / (p_ms * 1e-3) / 1e12, 3),
            "algorithmic_bytes": p_bytes, "algorithmic_flops": p_flops,
            "roofline": {"bound": "hbm", "kernel": "kda_prefill_rr_kernel",
                         "achieved": round(p_gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                         "frac": round(p_gbs / peak_hbm, 4), "traffic": traffic.get(traffic_key)},
            "cpu_baseline": sample}


def measure_e2e(args, case, bufs, stream, flush):
    """The same prefill through the public host-to-host call (chunk_prefill_from_host, the
    C ABI's kda_chunk_prefill_host): pinned host inputs in, pinned host output and final
    state out, every H2D and D2H copy inside the timed region (overlapped with the
    kernels piece by piece inside the library).  The device buffer and pinned outputs of
    the first (untimed) call are passed back, as a serving loop would.  Also times the
    link alone (one H2D copy of the step's inputs, one D2H copy of its outputs, from and to
    pinned memory, each alone and both at once), which bounds the end-to-end step from
    below."""
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
    # the link alone
    dev_in = torch.empty(h2d, dtype=torch.uint8, device=stream.device)
    dev_out = torch.empty(d2h, dtype=torch.uint8, device=stream.device)
    src = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    dst = torch.empty(d2h, dtype=torch.uint8).pin_memory()
    link = {}
    for name, fn, nb in (("h2d", lambda: dev_in.copy_(src, non_blocking=True), h2d),
                         ("d2h", lambda: dst.copy_(dev_out, non_blocking=True), d2h)):
        lt = time_steps(fn, 5, 2, stream, flush, sleep_cycles=0)
        link[name + "_gbs"] = round(nb / (statistics.median(lt) * 1e-3) / 1e9, 1)
    # both directions at once (the step's copies overlap in time): the link's real floor
    side = torch.cuda.Stream(stream.device)

    def both():
        ev = torch.cuda.Event()
        ev.record(stream)
        side.wait_event(ev)
        dev_in.copy_(src, non_blocking=True)
        with torch.cuda.stream(side):
            dst.copy_(dev_out, non_blocking=True)
        done = torch.cuda.Event()
        done.record(side)
        stream.wait_event(done)

    bt = time_steps(both, 5, 2, stream, flush, sleep_cycles=0)
    link["both_directions_ms"] = round(statistics.median(bt), 4)
    link["floor_ms"] = round(max(max(h2d / link["h2d_gbs"], d2h / link["d2h_gbs"]) / 1e6,
                                 link["both_directions_ms"]), 4)
    del dev_in, dev_out, src, dst
    return times, h2d, d2h, n * (segments + 1), link   # per piece one prefill; one cu kernel


def measure_decode(args, dev, stream, flush, bf16_state=False):
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

    times = time_steps(step, DECODE_STEPS if args.only != "decode" else max(args.steps, 1),
                       args.warmup, stream, flush)
    d_bytes = N * H * decode_bytes_per_seq_head(state_es=2 if bf16_state else 4)
    name = dcase.name if N == dcase.N else dcase.name.replace("N256", f"N{N}")
    if bf16_state:
        name += "_bf16_state"
    return name, N, times, d_bytes


def run_ours(args):
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks = load_peaks()
    peak_hbm = peaks["hbm_gbs"]
    traffic = load_traffic()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    line = {"metric": "KDA prefill tokens/s + TFLOP/s; decode state GB/s (fraction of roofline)",
            "value": None, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic"}
    launches = 0

    if args.only in ("all", "prefill"):
        case, ptimes, clocks, bufs = measure_prefill(args, dev, stream, flush)
        T, H, K, V = case.T, case.H, case.K, case.V
        p_ms = statistics.mean(ptimes)
        p_bytes = prefill_case_bytes(case)
        p_flops = T * H * prefill_flops_per_token_head()
        p_gbs = p_bytes / (p_ms * 1e-3) / 1e9
        launches += args.steps
        line.update({
            "value": round(T / (p_ms * 1e-3), 1),
            "ms_per_step": round(p_ms, 5),
            "config": {"workload": case.name, "global_batch": 1, "seq_len": T, "heads": H,
                       "head_dim_k": K, "head_dim_v": V, "chunk": CHUNK, "out_dtype": "bf16",
                       "parallelism": "one GPU",
                       "l2": "flushed between timed steps (256 MiB write)",
                       "also_timed": ["varlen_packed (prefill_varlen)", "long_prefill (prefill_long)",
                                      "paged_decode (decode, decode_bf16_state)"]},
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
            etimes, h2d, d2h, n_e2e, link = measure_e2e(args, case, bufs, stream, flush)
            e_ms = statistics.mean(etimes)
            launches += n_e2e
            line["e2e"] = {"value": round(T / (e_ms * 1e-3), 1), "unit": "tokens/s",
                           "ms_per_step": round(e_ms, 4), "call": "kda_chunk_prefill_host",
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                           "link": link, "of_link_floor": round(link["floor_ms"] / e_ms, 3)}
            if not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_oracle_baseline(case, n_tokens=T)
        del bufs
        if args.only in ("all", "prefill"):
            from kimi_delta_attention_09_gb300 import inputs
            for key, make, tkey in (("prefill_varlen", inputs.varlen_packed, "prefill_rr_varlen_packed"),
                                    ("prefill_long", inputs.long_prefill, "prefill_rr_long_prefill")):
                c = make()
                n = max(3, min(args.steps, 10))
                ctimes, cbufs = time_prefill_case(args, c, dev, stream, flush, n)
                del cbufs
                launches += n
                sample = None if args.no_cpu_baseline else cpu_oracle_baseline(c, n_tokens=1024, budget_s=5.0)
                line[key] = prefill_block(c, ctimes, peak_hbm, tkey, traffic, sample)
                del c

    if args.only in ("all", "decode"):
        name, N, dtimes, d_bytes = measure_decode(args, dev, stream, flush)
        d_ms = statistics.mean(dtimes)
        d_gbs = d_bytes / (d_ms * 1e-3) / 1e9
        launches += len(dtimes)
        line["decode"] = {
            "workload": name, "metric": "state GB/s",
            "value": round(d_gbs, 1), "unit": "GB/s",
            "ms_per_step": round(d_ms, 5), "steps": len(dtimes),
            "algorithmic_bytes_per_step": d_bytes,
            "roofline": {"bound": "hbm", "kernel": "kda_decode_kernel", "achieved": round(d_gbs, 1),
                         "peak": peak_hbm, "unit": "GB/s", "frac": round(d_gbs / peak_hbm, 4),
                         "traffic": traffic.get("decode_paged")}}
        name, N, dtimes, d_bytes = measure_decode(args, dev, stream, flush, bf16_state=True)
        d_ms = statistics.mean(dtimes)
        d_gbs = d_bytes / (d_ms * 1e-3) / 1e9
        launches += len(dtimes)
        line["decode_bf16_state"] = {
            "workload": name, "metric": "state GB/s",
            "value": round(d_gbs, 1), "unit": "GB/s",
            "ms_per_step": round(d_ms, 5), "steps": len(dtimes),
            "algorithmic_bytes_per_step": d_bytes,
            "roofline": {"bound": "hbm", "kernel": "kda_decode_kernel (bf16 state)",
                         "achieved": round(d_gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                         "frac": round(d_gbs / peak_hbm, 4),
                         "traffic": traffic.get("decode_bf16_state_paged")}}
    if args.only in ("all", "conv"):
        blocks, n_launch = measure_conv(args, dev, stream, flush, peak_hbm, traffic)
        line.update(blocks)
        launches += n_launch
    line["gpu_launches"] = launches
    print(json.dumps(line), flush=True)


def conv_bytes(case, prompt):
    """Algorithmic HBM bytes of one causal-convolution call: inputs read and outputs
    written once (bf16), the carried taps of every sequence read and written, the fp32
    weights and bias read."""
    T, D = case.x.shape
    W = case.weight.shape[1]
    es = case.x.element_size()
    N = case.state_idx.numel()
    return T * D * es * 2 + N * (W - 1) * D * es * 2 + D * (W + 1) * 4


def measure_conv(args, dev, stream, flush, peak_hbm, traffic):
    """The causal convolution in front of the op: the prompt pass on the varlen packed
    workload's [q|k|v] channels and the one-token update of the paged-decode workload
    (width 4, SiLU, taps carried in paged slots)."""
    import torch
    from kimi_delta_attention_09_gb300 import _native, inputs
    out_blocks, n_launch = {}, 0
    for key, make, prompt, tkey in (("conv_prefill", inputs.conv_varlen, True, "conv_fwd_varlen"),
                                    ("conv_update", inputs.conv_decode, False, "conv_update_decode")):
        c = make()
        x, w, b = c.x.to(dev), c.weight.to(dev), c.bias.to(dev)
        st, idx, cu = c.conv_state.to(dev), c.state_idx.to(dev), c.cu_seqlens.to(dev)
        out = torch.empty_like(x)

        if prompt:
            def step():
                _native.kda_causal_conv1d_fwd(x, w, b, st, idx, cu, out, _native.KDA_CONV_ACT_SILU, stream)
        else:
            def step():
                _native.kda_causal_conv1d_update(x, w, b, st, idx, out, _native.KDA_CONV_ACT_SILU, stream)

        n = max(3, min(args.steps, 20))
        times = time_steps(step, n, args.warmup, stream, flush)
        n_launch += n * (2 if prompt else 1)
        ms = statistics.mean(times)
        nbytes = conv_bytes(c, prompt)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out_blocks[key] = {
            "workload": c.name, "metric": "GB/s", "value": round(gbs, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "steps": n, "algorithmic_bytes": nbytes,
            "roofline": {"bound": "hbm", "kernel": "kda_conv_fwd_kernel" if prompt else "kda_conv_update_kernel",
                         "achieved": round(gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                         "frac": round(gbs / peak_hbm, 4), "traffic": traffic.get(tkey)}}
        del c, x, w, b, st, idx, cu, out
    return out_blocks, n_launch


# ------------------------------------------------------------------ oracle arm

def cpu_oracle_baseline(case, n_tokens, budget_s=15.0):
    """The fp64 oracle (as it stands) on the first n_tokens of the workload (of its first
    sequence), repeated until it has taken about `budget_s` CPU-seconds."""
    import oracle
    n_tokens = min(n_tokens, int(case.cu_seqlens[1]))
    sl = slice(0, n_tokens)
    threads = oracle.default_threads()
    used = min(threads, case.H)
    reps, dt = 0, 0.0
    while reps == 0 or dt * used < budget_s:
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
    ap.add_argument("--only", choices=["all", "prefill", "decode", "conv"], default="all")
    ap.add_argument("--decode-seqs", type=int, default=256)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)          # at least 3 untimed warm-up steps
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; other ranks exit without work
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, rank, int(os.environ.get("WORLD_SIZE", "1")))
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1 or args.gpus > 1:
        # every call of this library runs on one GPU (the prefill kernel's record hand-off
        # uses a cluster multicast load, kept to single-GPU runs), so there is no multi-GPU
        # step to time
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps({"error": "single-GPU benchmark: run with --gpus 1 and no torchrun",
                              "n_gpus": max(world, args.gpus)}), flush=True)
        sys.exit(2)
    run_ours(args)


if __name__ == "__main__":
    main()
