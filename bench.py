#!/usr/bin/env python3
"""Throughput of the DFlash hot path on GB300.

One step = block attention in each of the 5 draft layers, greedy verify of
sequences 0-31 and sampled verify of sequences 32-63, and the context-KV
materialisation of every sequence's committed rows -- the batched serving
workload at the Llama-3.1-8B shape (B = 64, block 16, ragged contexts of
512-8192 tokens in 16-token pages, vocabulary 128256), synthetic inputs.

Prints one JSON line. ``--impl reference`` times the CPU oracle instead (the
reference arm), on a bounded sample of the same workload.
Multi-GPU runs (torchrun) are independent replicas: each rank runs its own
batch; the barrier and the max over ranks bracket the timed region.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft+verify steps/s & verified tokens/s at 8B shape (B=64,k=16); % HBM roofline"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        sm_sorted = sorted(sm)
        med = sm_sorted[len(sm_sorted) // 2] if sm_sorted else None
        return {"sm_mhz": med, "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# replicas: every rank runs its own batch; the job's time is the slowest rank's
# ---------------------------------------------------------------------------
def max_over_ranks(x: float, world: int, device) -> float:
    """The maximum of ``x`` over all ranks (x itself when there is one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(steps: int, ms_max: float, world: int) -> float:
    """Steps per second of the whole job: all ranks' steps over the slowest
    rank's time (weak scaling: every rank has a full batch)."""
    return world * steps / (ms_max / 1e3)


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_step_estimate(wl, ctx_all, commit_rows, n_attn=2, n_verify=2, n_rows=4, seed=0):
    """Time the oracle on a bounded sample of one step and scale each part to
    the full step by its work units. Returns (seconds per full step, sample
    description)."""
    import numpy as np
    import torch

    import oracle as O
    from block_diffusion_speculative_fusion_gb300 import synth

    def f64(t):
        return t.float().numpy().astype(np.float64)

    # attention: n_attn sequences of one layer, scaled by keys and by L layers
    ctx = ctx_all[:n_attn].clone()
    w_a = dataclasses.replace(wl, B=n_attn)
    cache = synth.paged_cache(w_a, headroom=16, seed=seed, layers=1, ctx_len=ctx)
    blk = synth.block_qkv(w_a, 0, seed)
    args = [f64(blk["q"]), f64(blk["k_blk"]), f64(blk["v_blk"]), f64(cache.k_pools[0]), f64(cache.v_pools[0]),
            cache.page_table.numpy(), ctx.numpy(), wl.page_size]
    t0 = time.perf_counter()
    O.block_attn(*args)
    t_attn = time.perf_counter() - t0
    keys_sample = float((ctx + wl.k).sum())
    keys_all = float((ctx_all + wl.k).sum())
    attn_full = t_attn * keys_all / keys_sample * wl.L

    # verify: n_verify greedy and n_verify sampled sequences
    vb = synth.verify_batch(wl, seed, n_max=wl.n_draft, B=2 * n_verify, greedy_rows=n_verify)
    zt, zd = f64(vb["target_logits"]), f64(vb["draft_logits"])
    t0 = time.perf_counter()
    O.verify_greedy(zt[:n_verify], vb["cand"].numpy()[:n_verify], vb["n_draft"].numpy()[:n_verify])
    t_g = time.perf_counter() - t0
    t0 = time.perf_counter()
    O.verify_sample(zt[n_verify:], zd[n_verify:], vb["cand"].numpy()[n_verify:], vb["n_draft"].numpy()[n_verify:],
                    vb["u_acc"].numpy()[n_verify:], vb["u_final"].numpy()[n_verify:], wl.temperature)
    t_s = time.perf_counter() - t0
    verify_full = t_g * wl.n_greedy / n_verify + t_s * (wl.B - wl.n_greedy) / n_verify

    # materialise: n_rows committed rows of one sequence, scaled by committed rows
    w = synth.ctx_weights(wl, seed)
    hid = synth.captured_hidden(wl, n_rows, seed, B=1)
    pages = (n_rows + wl.page_size - 1) // wl.page_size + 1
    pt = np.arange(pages, dtype=np.int32)[None, :]
    pool = [np.zeros((pages, wl.page_size, wl.Hkv, wl.D)) for _ in range(wl.L)]
    t0 = time.perf_counter()
    O.materialize_ctx_kv(f64(hid), [n_rows], [0], f64(w["W_f"]), f64(w["b_f"]), f64(w["W_kv"]),
                         None if w["k_norm_w"] is None else f64(w["k_norm_w"]), wl.rms_eps, wl.rope_theta,
                         pool, [p.copy() for p in pool], pt, wl.page_size)
    t_m = time.perf_counter() - t0
    mat_full = t_m * commit_rows / n_rows
    total = attn_full + verify_full + mat_full
    sample = (f"attention: {n_attn} sequences x 1 layer (scaled by keys and x{wl.L} layers); verify: "
              f"{n_verify} greedy + {n_verify} sampled sequences (scaled to {wl.n_greedy}+{wl.B - wl.n_greedy}); "
              f"materialise: {n_rows} rows (scaled to {commit_rows} committed rows)")
    return total, sample, {"attn_s": attn_full, "verify_s": verify_full, "materialize_s": mat_full,
                           "sample_cpu_s": t_attn + t_g + t_s + t_m}


def abi_host_cost():
    """Host time of one enqueue through the C ABI per entry point (the C
    harness built beside the library; small problems, no synchronisation in
    the timed loop)."""
    from block_diffusion_speculative_fusion_gb300 import build as _b
    if not os.path.exists(_b.HOST_COST):
        return {"note": "harness not built"}
    try:
        r = subprocess.run([_b.HOST_COST], stdout=subprocess.PIPE, stderr=subprocess.STDOUT, timeout=120, text=True)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as exc:   # noqa: BLE001 - reported, not fatal
        return {"note": f"{type(exc).__name__}: {exc}"[:200]}


def workload_config(wl, world=1):
    """The ``config`` object of the JSON line: the workload, identical in both arms."""
    return {"workload": wl.name, "B": wl.B, "k": wl.k, "L": wl.L, "V": wl.V, "d": wl.d,
            "Hq/Hkv/D": f"{wl.Hq}/{wl.Hkv}/{wl.D}", "ctx": f"U[{wl.ctx_lo},{wl.ctx_hi}]",
            "page": wl.page_size, "verify": f"greedy {wl.n_greedy} + sampled {wl.B - wl.n_greedy}",
            "l2": "inputs larger than L2: ~5.7 GB of context K/V read per step (no flush needed)",
            "parallelism": f"replicas x{world}"}


def oracle_committed_rows(wl, seed=0):
    """Rows the step commits (sum of commit_len over the batch), from the
    oracle's accept rules on the step's verify inputs."""
    import numpy as np
    import oracle as O
    from block_diffusion_speculative_fusion_gb300 import synth
    vb = synth.verify_batch(wl, seed, n_max=wl.n_draft)
    f = lambda t: t.float().numpy().astype(np.float64)
    ng = wl.n_greedy
    g = O.verify_greedy(f(vb["target_logits"][:ng]), vb["cand"][:ng].numpy(), vb["n_draft"][:ng].numpy())
    s_ = O.verify_sample(f(vb["target_logits"][ng:]), f(vb["draft_logits"][ng:]), vb["cand"][ng:].numpy(),
                         vb["n_draft"][ng:].numpy(), vb["u_acc"][ng:].numpy(), vb["u_final"][ng:].numpy(),
                         wl.temperature)
    return int(g["commit_len"].sum() + s_["commit_len"].sum())


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


# ---------------------------------------------------------------------------
def run_reference(args, wl):
    """Reference arm: the CPU oracle as it stands, one bounded sample per step."""
    import torch
    from block_diffusion_speculative_fusion_gb300 import synth
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    ctx_all = synth.ctx_lengths(wl, 0)
    commit_rows = oracle_committed_rows(wl, 0)      # the step's committed rows (the GPU arm's count)
    for _ in range(args.warmup):
        oracle_step_estimate(wl, ctx_all, commit_rows, n_attn=1, n_verify=1, n_rows=2)
    est = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s, sample, parts = oracle_step_estimate(wl, ctx_all, commit_rows, n_attn=1, n_verify=1, n_rows=2)
        est.append(s)
    wall = time.perf_counter() - t0
    per_step = sum(est) / len(est)
    value = 1.0 / per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, args.gpus),
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": host_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": wall, "parts_s": parts,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def attn_bytes(ctx_mean_sum, wl):
    """Algorithmic HBM bytes of one block-attention launch (one draft layer):
    every context and block K/V row once, Q read once, O written once."""
    el = 2
    kv = (ctx_mean_sum + wl.B * wl.k) * wl.Hkv * wl.D * 2 * el
    qo = 2 * wl.B * wl.k * wl.Hq * wl.D * el
    return kv + qo


def traffic_from_profile(kernel_file):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of the kernel."""
    path = os.path.join(ROOT, "profiles", "attn_tc_kernel_llama8b_b64.md")
    src = os.path.join(ROOT, "block_diffusion_speculative_fusion_gb300", "csrc", kernel_file)
    if not os.path.exists(path) or not os.path.exists(src):
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha256_16") != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


def cuda_kernel_times(torch, fn, reps):
    """Device time of every kernel ``fn`` launches, from one CUPTI pass (torch
    profiler) over ``reps`` calls: {kernel name: [durations in us, in launch
    order]}. None when the profiler is unavailable."""
    try:
        from torch.profiler import ProfilerActivity, profile
    except Exception:   # noqa: BLE001
        return None
    try:
        torch.cuda.synchronize()
        if not getattr(cuda_kernel_times, "warm", False):
            # the first session in a process can miss kernels while CUPTI starts
            with profile(activities=[ProfilerActivity.CUDA]):
                fn()
                torch.cuda.synchronize()
            cuda_kernel_times.warm = True
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            for _ in range(reps):
                fn()
            torch.cuda.synchronize()
    except Exception as exc:   # noqa: BLE001 - reported, not fatal
        return {"_error": f"{type(exc).__name__}: {exc}"[:300]}
    evs = [e for e in prof.events() if str(getattr(e, "device_type", "")).endswith("CUDA")]
    if not evs:
        return {"_error": f"no device events among {len(prof.events())} profiler events"}
    return kernel_durations([(e.name, e.time_range.start, e.time_range.end) for e in evs])


def kernel_durations(events):
    """{kernel name: [durations]} from (name, start, end) device events. A
    programmatic dependent may start before the kernel it waits for has
    finished; its time is counted from that kernel's end."""
    out, last_end = {}, {}
    for raw, start, end in sorted(events, key=lambda x: x[1]):
        name = raw.split("(")[0].split("<")[0].strip().split(" ")[-1].split("::")[-1]
        for pred in PDL_PREDECESSORS.get(name, ()):
            if pred in last_end and last_end[pred] <= end:
                start = max(start, last_end[pred])
        out.setdefault(name, []).append(float(end - start))
        last_end[name] = end
    return out


# Kernels launched as programmatic dependents, with the kernels they wait for.
PDL_PREDECESSORS = {
    "attn_merge_kernel": ("attn_tc_kernel",),
    "gemm_tc_kernel": ("mat_gather_kernel", "mat_bias_kernel"),
    "gemm_simt_kernel": ("mat_gather_kernel", "mat_bias_kernel"),
    "mat_bias_kernel": ("gemm_tc_kernel", "gemm_simt_kernel"),
    "mat_epilogue_d128_kernel": ("gemm_tc_kernel", "gemm_simt_kernel"),
    "mat_epilogue_kernel": ("gemm_tc_kernel", "gemm_simt_kernel"),
    "sample_draw_kernel": ("sample_stats_kernel",),
}


def step_rooflines(torch, st, wl, hbm, tf, reps=4):
    """Per-kernel roofline of the step's kernels, each from its own device
    time (CUPTI, eager launches outside the timed region) and its algorithmic
    bytes: attention, the greedy and sampled verify kernels, the decode-sized
    materialisation GEMMs and the rest of the materialisation."""
    times = cuda_kernel_times(torch, st.step, reps)
    if not times or "_error" in times:
        return {"note": "torch profiler (CUPTI) unavailable", "detail": (times or {}).get("_error")}
    el = 2
    V, R, n = wl.V, wl.n_draft + 1, wl.n_draft
    ng, ns = wl.n_greedy, wl.B - wl.n_greedy
    acc = st.out["accept_len"][ng:].cpu()
    T = float(st.out["commit_len"].sum().item())
    rejected = int((acc < n).sum())
    md, N2 = wl.m * wl.d, wl.kv_out
    byts = {
        "greedy_kernel": ng * R * V * el,
        "sample_stats_kernel": ns * (R + n) * V * el,
        "sample_draw_kernel": (2 * rejected + (ns - rejected)) * V * el,
    }
    mean = lambda v: sum(v) / len(v)
    res = {}
    for name, nbytes in byts.items():
        if name in times:
            us = mean(times[name])
            res[name] = {"us": us, "bytes": nbytes, "GBps": nbytes / us / 1e3, "frac_hbm": nbytes / us / 1e3 / hbm,
                         "bound": "hbm"}
    if "gemm_tc_kernel" in times:
        g = times["gemm_tc_kernel"]
        g1, g2 = mean(g[0::2]), mean(g[1::2])
        b1 = wl.d * md * el + T * md * el + T * wl.d * el
        b2 = N2 * wl.d * el + T * wl.d * el + T * N2 * el
        res["gemm_tc_kernel (decode, fusion)"] = {"us": g1, "bytes": b1, "frac_hbm": b1 / g1 / 1e3 / hbm,
                                                  "bound": "hbm", "rows": T}
        res["gemm_tc_kernel (decode, K/V)"] = {"us": g2, "bytes": b2, "frac_hbm": b2 / g2 / 1e3 / hbm,
                                               "bound": "hbm", "rows": T}
    mat = [k_ for k_ in times if k_.startswith("mat_")]
    res["mat_other_us_per_step"] = {k_: sum(times[k_]) / reps for k_ in mat}
    if "attn_tc_kernel" in times:
        res["attn_tc_kernel_us"] = mean(times["attn_tc_kernel"])
    if "attn_merge_kernel" in times:
        res["attn_merge_kernel_us"] = mean(times["attn_merge_kernel"])
    return res


def prefill_roofline(torch, wl, tf, tf_sus):
    """The prefill-sized materialisation GEMMs (every context row of every
    sequence at once) against the dense bf16 tensor-core peak, from device
    kernel times (CUPTI)."""
    call, T, _ = prefill_materialize_call(wl, "cuda:0")
    for _ in range(2):
        call()
    times = cuda_kernel_times(torch, call, 3)
    if not times or "gemm_tc_kernel" not in times:
        return {"note": "torch profiler (CUPTI) unavailable", "detail": (times or {}).get("_error")}
    g = times["gemm_tc_kernel"]
    f1 = 2.0 * T * wl.m * wl.d * wl.d
    f2 = 2.0 * T * wl.d * wl.kv_out
    u1, u2 = sum(g[0::2]) / len(g[0::2]), sum(g[1::2]) / len(g[1::2])
    other = {k_: sum(v) / 3 for k_, v in times.items() if k_ != "gemm_tc_kernel"}
    return {"workload": wl.name, "rows": T, "bound": "tensor", "unit": "TFLOP/s",
            "gemm_fusion": {"us": u1, "tflops": f1 / u1 / 1e6, "frac": f1 / u1 / 1e6 / tf},
            "gemm_kv": {"us": u2, "tflops": f2 / u2 / 1e6, "frac": f2 / u2 / 1e6 / tf},
            "peak": tf, "peak_kind": "bf16_tflops (burst: the GEMMs are timed alone)",
            "other_kernels_us": other}


def capture_steps(torch, st, n):
    """One CUDA graph holding n steps, with a timing event (an external event
    node) around every call of the path. Returns (graph, events, None) or
    (None, None, reason)."""
    try:
        torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None, None, "torch.cuda.Event has no external flag"
    ev = {"attn": [], "verify": [], "mat": []}
    pending = {}

    def timer(tag):
        e = torch.cuda.Event(enable_timing=True, external=True)
        e.record()
        kind, edge = tag.rsplit("_", 1)
        if edge == "start":
            pending[kind] = e
        else:
            ev[kind].append((pending.pop(kind), e))

    try:
        g = st.capture(n, timer=timer)
    except Exception as exc:   # noqa: BLE001 - reported in the JSON line, the stream path runs instead
        torch.cuda.synchronize()
        return None, None, f"capture failed: {type(exc).__name__}: {exc}"[:200]
    return g, ev, None


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    import __graft_entry__
    __graft_entry__.build()
    from block_diffusion_speculative_fusion_gb300 import api
    from block_diffusion_speculative_fusion_gb300.step import DflashStep

    # stationary: every step decodes from the same initial context lengths, so
    # the timed steps all see the named workload (contexts do not drift)
    st = DflashStep(wl, seed=rank, device=dev, headroom_steps=2, pinned_inputs=True, stationary=True)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()

    ctx_start = st.ctx_len().clone()
    # ---------------- device-resident timed region ----------------
    ev = {"attn": [], "verify": [], "mat": []}
    pending = {}

    def timer(tag):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        kind, edge = tag.rsplit("_", 1)
        if edge == "start":
            pending[kind] = e
        else:
            ev[kind].append((pending.pop(kind), e))

    # The K timed steps are launched as one CUDA graph (the step is a fixed
    # sequence of launches on one stream), which removes the host launch gaps
    # between kernels. `value` is timed on a graph of the bare steps; the
    # per-call times come from a second graph of the same steps with a timing
    # event around every call, replayed apart (the event nodes add ~3 % to a
    # step, so they stay out of the timed region).
    graph, gev, launch_note = (None, None, "stream launches (--no-graph)")
    graph_plain = None
    if not args.no_graph:
        graph, gev, why = capture_steps(torch, st, args.steps)
        if graph is not None:
            try:
                graph_plain = st.capture(args.steps)
            except Exception as exc:   # noqa: BLE001 - the event graph is timed instead
                torch.cuda.synchronize()
                graph_plain = None
                why = f"plain capture failed: {type(exc).__name__}"
            for g_ in (graph, graph_plain):
                if g_ is not None:
                    g_.replay()          # upload and one untimed pass
            torch.cuda.synchronize()
            launch_note = (f"one CUDA graph of the {args.steps} timed steps" if graph_plain is not None else
                           f"one CUDA graph of the {args.steps} timed steps, with per-call events ({why})")
        else:
            launch_note = f"stream launches ({why})"

    def timed_region(mode):
        """mode: 'plain' (bare-step graph), 'events' (graph with per-call
        events) or 'stream' (stream launches with events)."""
        clocks = Clocks(local)
        barrier()
        torch.cuda.synchronize()
        clocks.start()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        if mode == "plain":
            graph_plain.replay()
        elif mode == "events":
            graph.replay()
        else:
            for _ in range(args.steps):
                st.step(timer=timer)
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
        clk_ = clocks.stop()
        src = gev if mode == "events" else ev
        pk = {k: (sum(a.elapsed_time(b) for a, b in v) / len(v)) * 1e3 for k, v in src.items() if v}
        return t_start.elapsed_time(t_end), pk, clk_

    if graph is not None:
        ms_ev, per_kernel, clk = timed_region("events")
        # the calls' event times must fit inside the step time
        calls_us = per_kernel.get("attn", 0.0) * wl.L + per_kernel.get("verify", 0.0) + per_kernel.get("mat", 0.0)
        step_us = ms_ev / args.steps * 1e3
        if not (0.5 * step_us < calls_us <= 1.02 * step_us):
            launch_note = f"stream launches (graph event times {calls_us:.0f} us vs step {step_us:.0f} us)"
            ms_total, per_kernel, clk = timed_region("stream")
        elif graph_plain is not None:
            ms_total, _, clk = timed_region("plain")
        else:
            ms_total = ms_ev
    else:
        ms_total, per_kernel, clk = timed_region("stream")
    ms_max = max_over_ranks(ms_total, world, dev)
    # a kernel that gave up a bounded wait (or met a bad page entry) leaves a
    # code in its workspace: such a run's numbers are not valid
    dev_errors = st.error_words()
    if any(dev_errors):
        raise RuntimeError(f"device error words after the timed region: {dev_errors}")
    commit_sum = float(st.out["commit_len"].sum().item())   # committed rows per step (every step alike)
    ms_per_step = ms_max / args.steps
    value = replica_throughput(args.steps, ms_max, world)
    tokens_per_s = value * commit_sum

    # ---------------- roofline of the dominant kernel (block attention) ----------------
    hbm, tf, tf_sus, peak_kind = _peaks()
    ctx_mean_sum = float(ctx_start.double().sum().item())
    ab = attn_bytes(ctx_mean_sum, wl)
    attn_us = per_kernel["attn"]
    achieved = ab / (attn_us * 1e-6) / 1e9
    roof = {"kernel": "attn_tc_kernel", "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind ==
            "measured" else "fallback 6.8 TB/s", "traffic": traffic_from_profile("attn.cu"),
            "algorithmic_bytes_per_launch": ab, "us_per_launch": attn_us}

    # ---------------- per-kernel rooflines (CUPTI device times, outside the timed region) ----------------
    roof_all = None
    if rank == 0:
        if args.no_cupti:
            roof_all = {"note": "skipped (--no-cupti)"}
        else:
            roof_all = step_rooflines(torch, st, wl, hbm, tf)
            if "attn_tc_kernel_us" in roof_all:
                # the attention kernel alone (the call's split merge is a second kernel)
                k_us = roof_all["attn_tc_kernel_us"]
                roof_all["attn_tc_kernel"] = {"us": k_us, "bytes": ab, "frac_hbm": ab / k_us / 1e3 / hbm,
                                              "bound": "hbm"}
            from block_diffusion_speculative_fusion_gb300 import workloads as W
            roof_all["prefill_gemms"] = prefill_roofline(torch, W.LLAMA8B_B1, tf, tf_sus)
        # step-level verify and materialisation, from the graph's own events
        el, V, R, n = 2, wl.V, wl.n_draft + 1, wl.n_draft
        ng, ns = wl.n_greedy, wl.B - wl.n_greedy
        vbytes = ng * R * V * el + ns * (R + n) * V * el + ns * 2 * V * el
        mbytes = (wl.d * wl.m * wl.d + wl.kv_out * wl.d) * el + commit_sum * (wl.m * wl.d + wl.kv_out) * el
        roof_all["verify_in_step"] = {"us": per_kernel.get("verify"), "bytes": vbytes,
                                      "frac_hbm": vbytes / per_kernel["verify"] / 1e3 / hbm}
        roof_all["materialize_in_step"] = {"us": per_kernel.get("mat"), "bytes": mbytes,
                                           "frac_hbm": mbytes / per_kernel["mat"] / 1e3 / hbm}
        st.reset()

    # ---------------- end to end through the public API with host buffers ----------------
    # Every step copies its inputs from pinned host memory and reads its
    # results back. The copies run on a second stream into the other of two
    # input sets while the previous step computes, and the host reads step i's
    # results while step i + 1 runs (overlap scheduling); each step's own H2D
    # copy and D2H read are inside the timed region.
    st.reset()
    h2d = st.input_bytes()
    sets = [st.inp, st.second_input_set()]
    outs = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in st.out.items()} for _ in range(2)]
    d2h = sum(v.numel() * v.element_size() for v in outs[0].values())
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]
    read = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_run(n, start=None):
        if start is not None:
            copy_stream.wait_event(start)   # no copy starts before the timed region
        with torch.cuda.stream(copy_stream):
            st.copy_inputs_from_host(sets[0])
            copied[0].record(copy_stream)
        for i in range(n):
            cur = i & 1
            if i + 1 < n:
                # the next step's inputs, once the step that last used that set is done
                copy_stream.wait_event(consumed[1 - cur])
                with torch.cuda.stream(copy_stream):
                    st.copy_inputs_from_host(sets[1 - cur])
                    copied[1 - cur].record(copy_stream)
            stream.wait_event(copied[cur])
            st.step(inp=sets[cur])
            consumed[cur].record(stream)
            for k, v in outs[cur].items():
                v.copy_(st.out[k], non_blocking=True)
            read[cur].record(stream)
            if i >= 1:
                read[1 - cur].synchronize()     # the host reads step i - 1's results
        read[(n - 1) & 1].synchronize()

    for s_ in (sets[0], sets[1]):
        for v in s_.values():
            v.record_stream(copy_stream)
    e2e_run(2)
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps, start=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = replica_throughput(args.steps, e2e_ms, world)

    # ---------------- per-call host cost of the C ABI, measured from C ----------------
    abi_host = None
    if rank == 0 and not args.no_cupti:
        abi_host = abi_host_cost()

    # ---------------- CPU baseline: the oracle on a bounded sample ----------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        est, sample, parts = oracle_step_estimate(wl, st.ctx0, int(round(commit_sum)), n_attn=4, n_verify=4,
                                                  n_rows=8)
        cpu = {"value": 1.0 / est, "unit": "steps/s", "cores": host_cores(), "kind": "oracle", "sample": sample,
               "parts_s": parts}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(wl, world),
            "launch": launch_note,
            "verified_tokens_per_s": tokens_per_s, "committed_rows_per_step": commit_sum,
            "kernels_us_per_step": {"attn_per_layer": per_kernel.get("attn"),
                                    "attn_total": per_kernel.get("attn", 0) * wl.L,
                                    "verify": per_kernel.get("verify"), "materialize": per_kernel.get("mat")},
            "roofline": roof,
            "roofline_all": roof_all,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": st.launches_per_step * args.steps,
            "device_error_words": dev_errors,
            "ms_per_step_with_call_events": ms_ev / args.steps if graph is not None else None,
            "abi_host_us_per_call": abi_host,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_kernel(args, wl):
    """One call of the step timed alone on the step's workload (attention: draft
    layer 0 only, so that one pool pair is resident)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from block_diffusion_speculative_fusion_gb300 import api, synth
    from block_diffusion_speculative_fusion_gb300.step import DflashStep
    if args.kernel == "prefill":
        # the prefill-sized materialisation GEMMs (Llama-3.1-8B shape, T = 2048 rows)
        from block_diffusion_speculative_fusion_gb300 import workloads as W
        call, T, flops = prefill_materialize_call(W.LLAMA8B_B1, "cuda:0")
        us = _time_calls(call, args.steps, args.warmup)
        print(json.dumps({"kernel": "prefill", "workload": W.LLAMA8B_B1.name, "rows": T, "us_per_call": us,
                          "tflops": flops / us / 1e6, "frac_bf16_peak": flops / us / 1e6 / _peaks()[1]}), flush=True)
        return
    if args.kernel == "materialize":
        # decode-sized: 64 sequences commit 1-8 rows each (seeded, ~4 on
        # average like the step's accept lengths) at their context ends; the
        # pools map only the pages those rows touch, so the call holds ~0.4 GB
        call, T, nbytes = decode_materialize_call(wl, "cuda:0")
        us = _time_calls(call, args.steps, args.warmup)
        print(json.dumps({"kernel": "materialize", "workload": wl.name, "rows": T, "us_per_call": us,
                          "bytes": nbytes, "frac_hbm": nbytes / us / 1e3 / _peaks()[0]}), flush=True)
        return
    if args.batch:
        wl = dataclasses.replace(wl, B=args.batch, n_greedy=min(wl.n_greedy, args.batch // 2))
    one = dataclasses.replace(wl, L=1) if args.kernel in ("attn", "verify") else wl
    st = DflashStep(one, seed=0, device="cuda:0", headroom_steps=4)
    inp = st.inp
    ng = wl.n_greedy

    def call():
        if args.kernel == "attn":
            api.block_attn(inp["q0"], inp["k_blk0"], inp["v_blk0"], st.k_pools[0], st.v_pools[0], st.page_table,
                           st.ctx[0], max_ctx=st.max_ctx, out=st.attn_out[0])
        elif args.kernel == "verify":
            api.verify_greedy(inp["target_logits"][:ng], inp["cand"][:ng], inp["n_draft"][:ng], out=st.out_g)
            api.verify_sample(inp["target_logits"][ng:], inp["draft_logits"], inp["cand"][ng:],
                              inp["u_acc"][ng:], inp["u_final"][ng:], wl.temperature, inp["n_draft"][ng:],
                              out=st.out_s)
        else:
            st.out["commit_len"].fill_(5)
            api.materialize_ctx_kv(inp["hidden"], st.out["commit_len"], st.ctx[0], st.W_f, st.b_f, st.W_kv,
                                   st.k_norm_w, wl.rms_eps, wl.rope_theta, st.k_pools, st.v_pools, st.page_table,
                                   new_len=st.ctx[1])
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    out = {"kernel": args.kernel, "workload": one.name, "B": one.B, "us_per_call": us}
    if args.kernel == "attn":
        ab = attn_bytes(float(st.ctx0.sum()), one)
        hbm = _peaks()[0]
        out.update({"bytes": ab, "GBps": ab / us / 1e3, "frac_hbm": ab / us / 1e3 / hbm})
    print(json.dumps(out), flush=True)


def _time_calls(fn, steps, warmup):
    """Mean device time of ``fn()`` in microseconds: ``steps`` calls captured in
    one CUDA graph and timed with CUDA events around its replay, so that the
    figure is the kernels' time and not the per-call host cost of the binding
    (stream launches only if the capture fails)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g):
            for _ in range(steps):
                fn()
        g.replay()
        torch.cuda.synchronize()
        _time_calls.mode = "cuda graph"
    except Exception:   # noqa: BLE001 - timed with stream launches instead
        torch.cuda.synchronize()
        g = None
        _time_calls.mode = "stream launches"
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    if g is not None:
        g.replay()
    else:
        for _ in range(steps):
            fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / steps


_time_calls.mode = "cuda graph"


def report_config(wl, args):
    """Per-kernel times and roofline fractions of one workload (one JSON line)."""
    import dataclasses as dc
    import torch
    from block_diffusion_speculative_fusion_gb300 import api, synth
    from block_diffusion_speculative_fusion_gb300.step import DflashStep
    hbm, tf, _, _ = _peaks()
    dev = "cuda:0"
    el = 2 if wl.dtype == "bf16" else 4
    out = {"config": wl.name, "B": wl.B, "k": wl.k, "V": wl.V}
    gbs = lambda nbytes, us: nbytes / us / 1e3
    if wl.stages == 1:
        # ---- one serving step through the step harness (stationary contexts) ----
        st = DflashStep(wl, seed=0, device=dev, headroom_steps=2, stationary=True)
        us_step = _time_calls(st.step, args.steps, args.warmup)
        rows = float(st.out["commit_len"].sum().item())
        out.update({"steps_per_s": 1e6 / us_step, "us_per_step": us_step, "verified_tokens_per_s": rows * 1e6 / us_step,
                    "committed_rows_per_step": rows})
        inp = st.inp
        us_attn = _time_calls(lambda: api.block_attn(inp["q0"], inp["k_blk0"], inp["v_blk0"], st.k_pools[0],
                                                     st.v_pools[0], st.page_table, st.ctx_start, max_ctx=st.max_ctx,
                                                     out=st.attn_out[0]), args.steps, args.warmup)
        ab = attn_bytes(float(st.ctx0.sum()), wl)
        out["attn_us_per_layer"] = us_attn
        # the in-block causal variant on the same inputs
        us_causal = _time_calls(lambda: api.block_attn(inp["q0"], inp["k_blk0"], inp["v_blk0"], st.k_pools[0],
                                                       st.v_pools[0], st.page_table, st.ctx_start,
                                                       max_ctx=st.max_ctx, out=st.attn_out[0], causal=True),
                                args.steps, args.warmup)
        out["attn_causal_us_per_layer"] = us_causal
        out["attn_causal_frac_hbm"] = gbs(ab, us_causal) / hbm
        # draft-side token choice over the MASK rows (argmax for greedy
        # workloads, inverse-CDF sampling otherwise), one pass over B x n_max rows
        sel = synth.draft_select_batch(wl, seed=0)
        sel = {k_: v_.to(dev) for k_, v_ in sel.items()}
        tsel = 0.0 if wl.n_greedy == wl.B else wl.temperature
        sel_out = api.draft_select(sel["draft_logits"], sel["anchor"], tsel, u_draft=sel["u_draft"])
        us_sel = _time_calls(lambda: api.draft_select(sel["draft_logits"], sel["anchor"], tsel,
                                                      u_draft=sel["u_draft"], out=sel_out), args.steps, args.warmup)
        if wl.name.startswith("qwen3_4b"):
            # DDTree on the same drafted positions: top-8 per position, a 512-node
            # best-first tree, then the greedy walk of the verified tree
            Kt, budget = 8, 512
            tk = api.ddtree_topk(sel["draft_logits"], Kt, 1.0)
            us_tk = _time_calls(lambda: api.ddtree_topk(sel["draft_logits"], Kt, 1.0, out=tk), args.steps, args.warmup)
            tr = api.ddtree_build(tk["tok"], tk["logp"], budget, V=wl.V)
            us_tb = _time_calls(lambda: api.ddtree_build(tk["tok"], tk["logp"], budget, V=wl.V, out=tr),
                                args.steps, args.warmup)
            torch.cuda.synchronize()
            zt = synth.ddtree_target_logits(wl, tr["node_token"], tr["node_parent"], tr["n_nodes"], seed=0,
                                            device=dev)
            tv = api.ddtree_verify_greedy(zt, tr["node_token"], tr["node_parent"], tr["n_nodes"], wl.n_max, Kt)
            us_tv = _time_calls(lambda: api.ddtree_verify_greedy(zt, tr["node_token"], tr["node_parent"], tr["n_nodes"],
                                                                 wl.n_max, Kt, out=tv), args.steps, args.warmup)
            out["ddtree"] = {"K": Kt, "budget": budget, "topk_us": us_tk,
                             "topk_frac_hbm": gbs(wl.B * wl.n_max * wl.V * el, us_tk) / hbm,
                             "build_us": us_tb, "verify_walk_us": us_tv,
                             "verify_walk_frac_hbm": gbs(wl.B * (budget + 1) * wl.V * el, us_tv) / hbm,
                             "mean_accept_len": float(tv["accept_len"].float().mean().item())}
            del zt
        out["draft_select_mode"] = "argmax" if tsel == 0.0 else f"sampled T={tsel}"
        out["draft_select_us"] = us_sel
        out["draft_select_frac_hbm"] = gbs(wl.B * wl.n_max * wl.V * el, us_sel) / hbm
        out["attn_frac_hbm"] = gbs(ab, us_attn) / hbm
        ng = wl.n_greedy
        R = wl.n_draft + 1
        if ng > 0:
            us_g = _time_calls(lambda: api.verify_greedy(inp["target_logits"][:ng], inp["cand"][:ng],
                                                         inp["n_draft"][:ng], out=st.out_g), args.steps, args.warmup)
            out["verify_greedy_us"] = us_g
            out["verify_greedy_frac_hbm"] = gbs(ng * R * wl.V * el, us_g) / hbm
        if ng < wl.B:
            ns = wl.B - ng
            us_s = _time_calls(lambda: api.verify_sample(
                inp["target_logits"][ng:], inp["draft_logits"], inp["cand"][ng:], inp["u_acc"][ng:],
                inp["u_final"][ng:], wl.temperature, inp["n_draft"][ng:], out=st.out_s), args.steps, args.warmup)
            out["verify_sample_us"] = us_s
            out["verify_sample_frac_hbm"] = gbs(ns * (2 * R - 1 + 2) * wl.V * el, us_s) / hbm
        del st
    else:
        # ---- DLoop looped step (DLoop page, mechanism 1 and the looped verify): stage s
        # drafts only where every earlier gate continued; the gates chain on the device
        # (stage s's active mask is stage s-1's cont) and count the drafted tokens; one
        # sampled verify then checks the S_b * k concatenated candidates, fed the gates'
        # row LSEs. Stage s's attention computes only the sequences still drafting
        # (dflash_block_attn_active with the previous gate's cont). ----
        n_q, k, S, n_max = wl.k, wl.n_draft, wl.stages, wl.n_max
        ctx = synth.ctx_lengths(wl, 0)
        cache = synth.paged_cache(wl, headroom=S + n_q, seed=0, layers=1, ctx_len=ctx, device=dev)
        pt, cl = cache.page_table.to(dev), cache.ctx_len.to(dev)
        blks = [{k_: v_.to(dev) for k_, v_ in synth.block_qkv(wl, 0, seed=0, n_kv_blk=n_q + s - 1).items()}
                for s in range(1, S + 1)]
        attn_out = [torch.empty_like(b_["q"]) for b_ in blks]
        vb = {k_: v_.to(dev) for k_, v_ in synth.verify_batch(wl, seed=0).items()}
        row_lse = torch.zeros(wl.B, n_max, dtype=torch.float32, device=dev)
        n_verify = torch.zeros(wl.B, dtype=torch.int32, device=dev)
        gouts = [{} for _ in range(S)]
        vout = {}

        def looped_step():
            n_verify.zero_()
            active = None
            for s in range(S):
                b_ = blks[s]
                for _ in range(wl.L):
                    api.block_attn(b_["q"], b_["k_blk"], b_["v_blk"], cache.k_pools[0], cache.v_pools[0], pt, cl,
                                   out=attn_out[s], active=active)
                api.gate_stage(vb["draft_logits"], vb["cand"], s, k, wl.temperature, wl.gate_g, active=active,
                               row_lse=row_lse, n_verify=n_verify, out=gouts[s])
                active = gouts[s]["cont"]
            api.verify_sample(vb["target_logits"], vb["draft_logits"], vb["cand"], vb["u_acc"], vb["u_final"],
                              wl.temperature, n_verify, draft_row_lse=row_lse, out=vout)

        us_loop = _time_calls(looped_step, args.steps, args.warmup)
        n_ver = n_verify.float()
        out["looped_step_us"] = us_loop
        out["looped_steps_per_s"] = 1e6 / us_loop
        out["looped_mean_stages"] = float(n_ver.mean().item()) / k
        out["looped_verified_tokens_per_s"] = float(vout["commit_len"].float().sum().item()) * 1e6 / us_loop
        masks = [None] + [g_["cont"].clone() for g_ in gouts[:-1]]
        for s in range(S):
            b_ = blks[s]
            us_a = _time_calls(lambda: api.block_attn(b_["q"], b_["k_blk"], b_["v_blk"], cache.k_pools[0],
                                                      cache.v_pools[0], pt, cl, out=attn_out[s]),
                               args.steps, args.warmup)
            if masks[s] is not None:
                # the stage as the looped step runs it: only the sequences still drafting
                out[f"stage{s + 1}_active_sequences"] = int(masks[s].sum().item())
                out[f"stage{s + 1}_attn_active_us_per_layer"] = _time_calls(
                    lambda: api.block_attn(b_["q"], b_["k_blk"], b_["v_blk"], cache.k_pools[0], cache.v_pools[0],
                                           pt, cl, out=attn_out[s], active=masks[s]), args.steps, args.warmup)
            us_g = _time_calls(lambda: api.gate_stage(vb["draft_logits"], vb["cand"], s, k, wl.temperature,
                                                      wl.gate_g, out=gouts[s]), args.steps, args.warmup)
            out[f"stage{s + 1}_attn_us_per_layer"] = us_a
            out[f"stage{s + 1}_gate_us"] = us_g
            if s == 0:
                out["attn_frac_hbm"] = gbs(attn_bytes(float(ctx.sum()), dc.replace(wl, k=n_q)), us_a) / hbm
                out["gate_frac_hbm"] = gbs(wl.B * k * wl.V * el, us_g) / hbm
        n = n_max
        us_v = _time_calls(lambda: api.verify_sample(vb["target_logits"], vb["draft_logits"], vb["cand"], vb["u_acc"],
                                                     vb["u_final"], wl.temperature, vb["n_draft"]),
                           args.steps, args.warmup)
        out["verify_sample_all_stages_us"] = us_v
        out["verify_sample_all_stages_frac_hbm"] = gbs(wl.B * (2 * n + 1 + 2) * wl.V * el, us_v) / hbm
        full_lse = api.gate(vb["draft_logits"], vb["cand"][:, 1:].contiguous(), wl.temperature, wl.gate_g,
                            want_row_lse=True)["row_lse"]
        us_vl = _time_calls(lambda: api.verify_sample(vb["target_logits"], vb["draft_logits"], vb["cand"],
                                                      vb["u_acc"], vb["u_final"], wl.temperature, vb["n_draft"],
                                                      draft_row_lse=full_lse), args.steps, args.warmup)
        out["verify_sample_gate_lse_all_stages_us"] = us_vl
        out["verify_sample_gate_lse_frac_hbm"] = gbs(wl.B * (n + 1 + 2) * wl.V * el, us_vl) / hbm
    if wl.dtype == "bf16" and wl.stages == 1 and wl.ctx_lo == wl.ctx_hi:
        # ---- prefill-sized materialisation: every context row of every sequence ----
        call_m, T, flops = prefill_materialize_call(wl, dev)
        us_m = _time_calls(call_m, max(3, args.steps // 4), 2)
        out["prefill_materialize_rows"] = T
        out["prefill_materialize_us"] = us_m
        out["prefill_materialize_tflops"] = flops / us_m / 1e6
        out["prefill_materialize_frac_bf16_peak"] = flops / us_m / 1e6 / tf
    out["timing"] = _time_calls.mode
    print(json.dumps(out), flush=True)


def prefill_materialize_call(wl, dev):
    """The context-KV materialisation of every context row of every sequence
    (prefill-sized T = B x context): returns (call, T, flops of both GEMMs)."""
    import torch
    from block_diffusion_speculative_fusion_gb300 import api, synth
    rows = wl.ctx_lo
    w = {k_: (v_.to(dev) if v_ is not None else None) for k_, v_ in synth.ctx_weights(wl, 0).items()}
    hid = synth.captured_hidden(wl, rows, 0, B=wl.B).to(dev)
    pc = synth.paged_cache(wl, headroom=0, seed=0, layers=wl.L, ctx_len=torch.full((wl.B,), rows, dtype=torch.int32),
                           device=dev)
    commit = torch.full((wl.B,), rows, dtype=torch.int32, device=dev)
    start = torch.zeros(wl.B, dtype=torch.int32, device=dev)
    pools_k = [t.to(dev) for t in pc.k_pools]
    pools_v = [t.to(dev) for t in pc.v_pools]
    ptab = pc.page_table.to(dev)

    def call():
        api.materialize_ctx_kv(hid, commit, start, w["W_f"], w["b_f"], w["W_kv"], w["k_norm_w"], wl.rms_eps,
                               wl.rope_theta, pools_k, pools_v, ptab)
    T = wl.B * rows
    return call, T, 2.0 * T * (wl.m * wl.d * wl.d + wl.d * wl.kv_out)


def decode_materialize_call(wl, dev):
    """One decode-sized materialisation at the throughput workload's shape:
    returns (call, committed rows T, algorithmic bytes: weights, the committed
    hidden rows and the K/V rows written)."""
    import torch
    from block_diffusion_speculative_fusion_gb300 import api, synth
    gen = torch.Generator().manual_seed(3)
    commit = torch.randint(1, 9, (wl.B,), generator=gen).to(torch.int32)
    start = synth.ctx_lengths(wl, 0)
    P = wl.page_size
    lo = (start // P).tolist()
    hi = ((start + commit - 1) // P).tolist()
    max_pages = max(hi) + 1
    pt = torch.full((wl.B, max_pages), -1, dtype=torch.int32)
    n = 0
    for b in range(wl.B):
        k = hi[b] - lo[b] + 1
        pt[b, lo[b]:hi[b] + 1] = torch.arange(n, n + k, dtype=torch.int32)
        n += k
    w = {k_: (v_.to(dev) if v_ is not None else None) for k_, v_ in synth.ctx_weights(wl, 0).items()}
    hid = synth.captured_hidden(wl, wl.k, 0).to(dev)
    dt = synth.io_dtype(wl)
    kp = [torch.zeros((n, P, wl.Hkv, wl.D), dtype=dt, device=dev) for _ in range(wl.L)]
    vp = [torch.zeros((n, P, wl.Hkv, wl.D), dtype=dt, device=dev) for _ in range(wl.L)]
    commit_d, start_d, pt_d = commit.to(dev), start.to(dev), pt.to(dev)

    def call():
        api.materialize_ctx_kv(hid, commit_d, start_d, w["W_f"], w["b_f"], w["W_kv"], w["k_norm_w"], wl.rms_eps,
                               wl.rope_theta, kp, vp, pt_d)
    T = int(commit.sum())
    el = 2
    nbytes = (wl.d * wl.m * wl.d + wl.kv_out * wl.d) * el + T * (wl.m * wl.d + wl.kv_out) * el
    return call, T, nbytes


def run_all_configs(args):
    import __graft_entry__
    __graft_entry__.build()
    from block_diffusion_speculative_fusion_gb300 import workloads as W
    for wl in W.ALL:
        report_config(wl, args)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    # for runs under a profiler: skip the CUPTI passes (a second CUPTI subscriber
    # beside ncu's) and the C host-cost child process
    ap.add_argument("--no-cupti", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the timed steps one by one (no CUDA graph)")
    ap.add_argument("--kernel", choices=["attn", "verify", "materialize", "prefill"], default=None,
                    help="time one call of the step in isolation (profiling aid)")
    ap.add_argument("--batch", type=int, default=None, help="override B (with --kernel)")
    ap.add_argument("--all-configs", action="store_true",
                    help="per-kernel times and roofline fractions of every workload, one JSON line each")
    args = ap.parse_args()
    from block_diffusion_speculative_fusion_gb300 import workloads as W
    wl = W.LLAMA8B_B64
    if args.impl == "reference":
        run_reference(args, wl)
    elif args.all_configs:
        run_all_configs(args)
    elif args.kernel:
        run_kernel(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
