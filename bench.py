"""Benchmark of the P-EAGLE parallel-draft step on GB300.

One step = the whole hot path over one synthetic batch: pe_prepare_inputs
(metadata, drafter input) -> pe_draft_step (fc, decoder layer with paged
attention, final norm) -> pe_argmax (LM head + greedy argmax).  The step is
captured as one CUDA graph (the way a serving engine runs the drafter) and
timed with CUDA events on its stream, max over ranks.  The roofline line's
kernel time comes from a loop of the LM head's own graph right after.  The
default line also carries, on one GPU, an "autoregressive" block (the same
batch drafted by the K-pass autoregressive baseline and by the parallel step,
at K = 7 and K = 3) and a "batched" block (the concurrency-64 post-norm
configuration, step and LM-head roofline); --no-extra leaves them out.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A verify_* workload times pe_verify_greedy (the greedy verification that yields
the next step's accepted counts and bonus tokens) instead of the draft step.  A
cod_* workload times pe_cod_sample_indices + pe_cod_mask (the training side's
COD index lists and asymmetric mask); its roofline line is the mask kernel, and
index_kernel_us is the whole call less the mask call timed alone.

Prints one JSON line.  --impl reference times the CPU oracle (the only
reference there is) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import ctypes
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_drafting_gb300 import workloads as W  # noqa: E402

METRIC = "parallel-draft step latency (us) and draft tokens/s at K=7; HBM GB/s %peak"
UNIT = "draft tokens/s"
DEFAULT_WORKLOAD = "gptoss_b1_k7"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the batched-step and autoregressive comparison blocks")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ----------------------------------------------------------------------------- ranks
# Several GPUs run independent replicas: each rank drafts (or verifies) its own
# seeded batch, no data crosses ranks, and the job's time is the slowest rank's.


def rank_workload(wl, rank):
    """The workload of one rank: the same recipe, its own seed."""
    return dataclasses.replace(wl, seed=wl.seed + rank)


def max_over_ranks(x, world, device):
    """The largest of every rank's x, on every rank (a no-op for one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms):
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / (ms / 1e3)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------------------------- algorithmic bytes


# workload -> (committed ncu summary, key of the dominant kernel's DRAM bytes per launch)
PROFILED = {"gptoss_b1_k7": ("lm_head_gemm_gptoss_b1_k7.md", "traffic_bytes_per_step"),
            "gptoss_b64_k7_postnorm": ("lm_head_gemm_gptoss_b64_k7.md", "traffic_bytes_per_step"),
            "verify_b64_k7": ("verify_greedy_b64_k7.md", "traffic_bytes_per_launch_f32"),
            "verify_b64_k7_bf16": ("verify_greedy_b64_k7.md", "traffic_bytes_per_launch_bf16"),
            "cod_s8192_a1024": ("cod_index_mask_s8192_a1024.md", "traffic_bytes_per_launch")}


def sources_digest(files):
    """sha256 over the sha256 digests of the listed files (paths from the repo root)."""
    digests = "".join(hashlib.sha256(open(os.path.join(ROOT, f), "rb").read()).hexdigest()
                      for f in files)
    return hashlib.sha256(digests.encode()).hexdigest()


def profiled_traffic(workload):
    """DRAM bytes (read + write) of the dominant kernel per launch from the committed
    ncu summary, while its sources are the ones it was captured with; else None."""
    if workload not in PROFILED:
        return None
    fname, key = PROFILED[workload]
    try:
        text = open(os.path.join(ROOT, "profiles", fname)).read()
        vals = dict(re.findall(r"^\s*(traffic_bytes_per_\w+|source_sha256|sources):\s*(\S.*)$",
                               text, re.M))
        if sources_digest(vals["sources"].split()) != vals["source_sha256"].strip():
            return None
        return int(vals[key])
    except (OSError, KeyError, ValueError):
        return None


def lm_head_bytes(dm, n_rows):
    """Bytes the LM head must move: W_lm once, the z rows, the fp32 argmax keys."""
    return dm.vocab * dm.d * 2 + n_rows * dm.d * 2 + n_rows * 8


def step_bytes(dm, batch):
    """Bytes the whole step must move: every weight once, the KV it reads and writes
    (in every layer), the captured hidden states and the embedding rows."""
    d, I, V = dm.d, dm.inter, dm.vocab
    n_l = max(1, getattr(dm, "n_layers", 1))
    w = (4 * d * d + n_l * (dm.qkv_rows * d + d * dm.n_heads * dm.head_dim + 3 * I * d) + V * d) * 2
    B, K = batch["B"], dm.K
    acc = batch["accepted"]
    pos0 = batch["prev_pos"][batch["qsl"][:-1] + acc]
    kv_read = n_l * int(np.sum(pos0 + K)) * dm.n_kv_heads * dm.head_dim * 2 * 2
    n_valid = int(np.sum(acc + K))
    kv_write = n_l * n_valid * dm.n_kv_heads * dm.head_dim * 2 * 2
    hid = batch["T_in"] * 3 * d * 2 + n_valid * d * 2
    return w + kv_read + kv_write + hid


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- CPU oracle leg


def oracle_sample(wl, batch, w, kc, vc, budget_s=20.0):
    """Time the oracle (as it stands) on whole requests of the workload until the
    budget is spent (at least one request).  Returns (draft tokens/s, sample text, threads)."""
    from oracle import pe_oracle as O

    t0 = time.perf_counter()
    done = 0
    for r in range(wl.batch):
        O.draft_step(wl.dims, w, batch, kc, vc, requests=[r])
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    try:
        from threadpoolctl import threadpool_info

        threads = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        threads = os.cpu_count() or 1
    sample = f"{done} of {wl.batch} requests of {wl.name} (full layer + LM head per request), {dt:.1f} s"
    return done * wl.dims.K / dt, sample, threads


# ----------------------------------------------------------------------------- reference arm


def warm_up(call, n, limit_s=60.0):
    """n untimed calls of call() before a reference arm's timed samples (the
    oracle's first calls pay numpy's and the BLAS library's set-up), at most
    limit_s in all.  Returns how many ran."""
    t0 = time.perf_counter()
    done = 0
    for _ in range(max(0, n)):
        call()
        done += 1
        if time.perf_counter() - t0 > limit_s:
            break
    return done


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = W.get(args.workload)
    batch = W.make_batch(wl)
    w = W.make_weights(wl)
    kc, vc = W.make_kv_cache(wl, batch["num_blocks"])
    # a zero budget: one request per warm-up step
    n_warm = warm_up(lambda: oracle_sample(wl, batch, w, kc, vc, budget_s=0.0), args.warmup)
    # each step: the oracle on whole requests of the workload, bounded in time;
    # the whole run stops after a few minutes
    per = []
    t_all = time.perf_counter()
    threads, sample = 1, ""
    for _ in range(max(1, args.steps)):
        v, sample, threads = oracle_sample(wl, batch, w, kc, vc, budget_s=10.0)
        per.append(v)
        if time.perf_counter() - t_all > 150:
            break
    value = statistics.median(per)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": len(per), "warmup": n_warm, "ms_per_step": 1000.0 * wl.batch * wl.dims.K / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "global_batch": wl.batch, "K": wl.dims.K,
                       "description": wl.description},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm


def warm_up_eager(r, stream, n=3):
    """n eager steps on `stream` (the step's first calls, before any capture)."""
    import torch

    with torch.cuda.stream(stream):
        for _ in range(n):
            r.run(stream=stream)
    stream.synchronize()


def capture_step_graph(r, stream):
    """The timed graph of one step: pe_prepare_inputs -> pe_draft_step ->
    pe_argmax exactly as the benchmark replays it (no logits store unless the
    runner asks for logits), captured on `stream`.  Every kernel boundary keeps
    its programmatic launch.  Returns (graph, kernel nodes in it)."""
    import torch

    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)  # kept to count its kernel nodes
    except TypeError:
        g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        r.prepare(stream=stream)
        r.step(stream=stream)
        r.argmax(stream=stream)
    n = graph_kernel_nodes(g)
    if hasattr(g, "instantiate"):
        try:
            g.instantiate()
        except RuntimeError:
            pass
    return g, n


def run_ours(args, rank, world, local):
    import torch

    from speculative_drafting_gb300 import build, runner

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    wl = W.get(args.workload)
    wl_rank = rank_workload(wl, rank)  # each rank drafts its own batch
    batch = W.make_batch(wl_rank)
    w = W.make_weights(wl)
    kc, vc = W.make_kv_cache(wl_rank, batch["num_blocks"])
    r = runner.StepRunner(wl, batch, w, kc, vc)
    # the step's inputs live in one device buffer (256-byte aligned parts), so that
    # the end-to-end loop moves them from one pinned host buffer with one copy
    dm = wl.dims
    stage_dev, stage_host = pack_step_inputs(r, batch)
    B, K = batch["B"], dm.K
    n_rows = B * K
    stream = torch.cuda.Stream()
    # eager warm-up, then capture
    warm_up_eager(r, stream)
    st, _ = r.status()
    if st:
        raise RuntimeError(f"device status {st:#x} on the benchmark batch")
    # the whole step is one graph; the LM head alone is a second graph, timed in
    # its own loop for the roofline line
    g_step, launches_per_step = capture_step_graph(r, stream)
    g_lm = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_lm, stream=stream):
        r.argmax(stream=stream)

    def one_step():
        g_step.replay()

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            one_step()
    stream.synchronize()

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for i in range(args.steps):
            g_step.replay()
        t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    step_ms = total_ms / args.steps
    # the LM head + argmax kernels alone, the same number of times, on the stream
    # they are launched on (its 1.16 GB weight stream is far larger than L2)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_lm.replay()
        for i in range(args.steps):
            ev[i][0].record(stream)
            g_lm.replay()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    lm_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    step_ms = max_over_ranks(step_ms, world, "cuda")

    # eager (no graph) step time, for reference
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e = max(10, args.steps // 4)
        e0.record(stream)
        for _ in range(n_e):
            r.run(stream=stream)
        e1.record(stream)
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / n_e

    # end to end through the C-ABI with host buffers: H2D of the step inputs from
    # pinned memory (one packed copy), the step, D2H of the draft tokens, every step
    # Each step ends with the host waiting for its drafts (what a scheduler pays
    # before it can use them), so the host clock times the loop.
    out_host = torch.empty(n_rows, dtype=torch.int32).pin_memory()
    h2d = stage_host.numel()
    d2h = out_host.numel() * 4
    n_e2e = max(10, args.steps // 2)
    with torch.cuda.stream(stream):
        for _ in range(3):
            stage_dev.copy_(stage_host, non_blocking=True)
            one_step()
            out_host.copy_(r.draft, non_blocking=True)
            stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            stage_dev.copy_(stage_host, non_blocking=True)
            one_step()
            out_host.copy_(r.draft, non_blocking=True)
            stream.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e2e_ms, world, "cuda")
    st, _ = r.status()
    if st:
        raise RuntimeError(f"device status {st:#x} after timing")

    peaks, src = measured_peaks()
    lm_avg_s = statistics.mean(lm_ms) / 1e3
    lm_bytes = lm_head_bytes(dm, n_rows)
    lm_flops = 2.0 * dm.vocab * dm.d * n_rows
    # the LM head's bound: DRAM for a few rows, the tensor cores for many (the
    # burst peak: the head is timed back to back on its own)
    if dm.dtype == "bf16" and lm_flops / (peaks["bf16_tflops"] * 1e12) > lm_bytes / (peaks["hbm_gbs"] * 1e9):
        achieved = lm_flops / lm_avg_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "algorithmic_flops": lm_flops}
    else:
        achieved = lm_bytes / lm_avg_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    total_tokens = n_rows * world
    value = job_throughput(n_rows, world, step_ms)
    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            v, sample, threads = oracle_sample(wl_rank, batch, w, kc, vc, budget_s=20.0)
            cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample}
        sb = step_bytes(dm, batch)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": step_ms, "step_latency_us": step_ms * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if
            dm.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": wl.name, "global_batch": B * world, "K": K,
                       "description": wl.description, "cuda_graph": True,
                       "l2": "inputs larger than L2: 1.41 GB of weights stream through every step"
                       if wl.name.startswith("gptoss") else "inputs larger than L2 (weights + KV)",
                       "parallelism": f"replica x{world} (independent requests per GPU)"},
            "eager_ms_per_step": eager_ms,
            "step_hbm": {"algorithmic_bytes": sb, "achieved_gbs": sb / (step_ms / 1e3) / 1e9,
                         "frac": sb / (step_ms / 1e3) / 1e9 / peaks["hbm_gbs"]},
            "clocks": clk,
            "e2e": {"value": total_tokens / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": (launches_per_step * args.steps if launches_per_step is not None
                             else None),
            "roofline": {"kernel": "gemm_tc_kernel (LM head + argmax epilogue)", **roof,
                         "traffic": profiled_traffic(wl.name),
                         "peak_source": src, "algorithmic_bytes": lm_bytes,
                         "avg_launch_us": lm_avg_s * 1e6},
            "cpu_baseline": cpu,
        }
        if world == 1 and not args.no_extra and wl.name == DEFAULT_WORKLOAD:
            line["autoregressive"] = autoregressive_block(wl, w, args.steps, stream)
            line["batched"] = batched_block("gptoss_b64_k7_postnorm", w, args.steps, stream, peaks,
                                            src)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def time_replays(g, stream, steps, warmup=3):
    """Device time (ms) per replay of graph g over `steps` back-to-back replays."""
    import torch

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(steps):
            g.replay()
        a1.record(stream)
    torch.cuda.synchronize()
    return a0.elapsed_time(a1) / steps


def autoregressive_block(wl, w, steps, stream):
    """The pages' comparison on this GPU ("P-EAGLE: parallel speculative decoding
    in vLLM", Solving the autoregressive drafting bottleneck, Performance
    benchmarks: K drafts cost K sequential passes; the autoregressive drafter
    peaks at K = 3, P-EAGLE at K = 7): the same batch drafted by the parallel
    step (one pass) and by pe_draft_autoregressive (K passes), each one CUDA
    graph, at K = 7 and K = 3 (K + 1 verify rows per request)."""
    import torch

    from speculative_drafting_gb300 import runner

    out = {}
    for K in (7, 3):
        wk = W.get(wl.name, K=K, n_prev=K + 1)
        batch = W.make_batch(wk)
        kc, vc = W.make_kv_cache(wk, batch["num_blocks"])
        r = runner.StepRunner(wk, batch, w, kc, vc)
        warm_up_eager(r, stream)
        g_par, n_par = capture_step_graph(r, stream)
        par_ms = time_replays(g_par, stream, steps)
        ws = r.drafter.autoregressive_workspace(r.B, r.T_in, r.inp["block_table"].shape[1])
        draft = torch.empty(r.B, K, dtype=torch.int32, device="cuda")
        with torch.cuda.stream(stream):
            for _ in range(3):
                r.autoregressive(draft, ws, stream=stream)
        stream.synchronize()
        st, _ = r.drafter.read_status(ws)
        if st:
            raise RuntimeError(f"device status {st:#x} in the autoregressive drafting")
        try:
            g_ar = torch.cuda.CUDAGraph(keep_graph=True)
        except TypeError:
            g_ar = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_ar, stream=stream):
            r.autoregressive(draft, ws, stream=stream)
        n_ar = graph_kernel_nodes(g_ar)
        if hasattr(g_ar, "instantiate"):
            try:
                g_ar.instantiate()
            except RuntimeError:
                pass
        ar_ms = time_replays(g_ar, stream, max(10, steps // 4))
        n_tok = r.B * K
        out[f"k{K}"] = {"workload": f"{wl.name} with K={K}", "parallel_step_us": par_ms * 1e3,
                        "parallel_kernels": n_par, "autoregressive_us": ar_ms * 1e3,
                        "autoregressive_kernels": n_ar,
                        "parallel_draft_tokens_per_s": n_tok / (par_ms / 1e3),
                        "autoregressive_draft_tokens_per_s": n_tok / (ar_ms / 1e3),
                        "speedup": ar_ms / par_ms}
        del r
    return out


def batched_block(name, w, steps, stream, peaks, src):
    """The concurrency-64 configuration ("P-EAGLE: parallel speculative decoding
    in vLLM", Performance benchmarks, c = 64), timed in the same process with the
    same method as the headline line: step graph, LM head graph, clocks."""
    import torch

    from speculative_drafting_gb300 import runner

    wl = W.get(name)
    batch = W.make_batch(wl)
    kc, vc = W.make_kv_cache(wl, batch["num_blocks"])
    r = runner.StepRunner(wl, batch, w, kc, vc)
    warm_up_eager(r, stream)
    st, _ = r.status()
    if st:
        raise RuntimeError(f"device status {st:#x} on the batched batch")
    g, n = capture_step_graph(r, stream)
    g_lm = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_lm, stream=stream):
        r.argmax(stream=stream)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    step_ms = time_replays(g, stream, steps)
    lm_ms = time_replays(g_lm, stream, steps)
    clk = clocks.stop()
    dm = wl.dims
    n_rows = batch["B"] * dm.K
    flops = 2.0 * dm.vocab * dm.d * n_rows
    ach = flops / (lm_ms / 1e3) / 1e12
    return {"workload": name, "description": wl.description, "global_batch": batch["B"],
            "step_us": step_ms * 1e3, "draft_tokens_per_s": n_rows / (step_ms / 1e3),
            "gpu_launches_per_step": n,
            "roofline": {"kernel": "gemm_tc_kernel (LM head + argmax epilogue)", "bound": "tensor",
                         "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": ach / peaks["bf16_tflops"], "algorithmic_flops": flops,
                         "avg_launch_us": lm_ms * 1e3, "peak_source": src,
                         "traffic": profiled_traffic(name)},
            "clocks": clk}


STEP_INPUTS = ("qsl", "prev_tok", "prev_pos", "accepted", "bonus", "block_table", "H_tgt")


def pack_step_inputs(r, batch):
    """Move the runner's input tensors into one device buffer, each part 256-byte
    aligned, and build the matching pinned host buffer from the batch's arrays.
    Returns (device buffer, pinned host buffer); r.inp now views the device one."""
    import torch

    host = {k: np.ascontiguousarray(batch[k]) for k in STEP_INPUTS}
    offs, total = {}, 0
    for k in STEP_INPUTS:
        offs[k] = total
        total = (total + host[k].nbytes + 255) // 256 * 256
    stage_dev = torch.zeros(total, dtype=torch.uint8, device=r.inp["qsl"].device)
    stage_host = torch.zeros(total, dtype=torch.uint8).pin_memory()
    hv = stage_host.numpy()
    for k in STEP_INPUTS:
        t = r.inp[k]
        nb = t.numel() * t.element_size()
        assert nb == host[k].nbytes, k
        view = stage_dev[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
        view.copy_(t)
        r.inp[k] = view
        hv[offs[k]:offs[k] + nb] = host[k].reshape(-1).view(np.uint8)
    return stage_dev, stage_host


def graph_kernel_nodes(graph):
    """Kernel launches in a captured step: the kernel nodes of its CUDA graph
    (driver query), or None where the driver or torch does not expose them."""
    try:
        cu = ctypes.CDLL("libcuda.so.1")
        h = ctypes.c_void_p(int(graph.raw_cuda_graph()))
        n = ctypes.c_size_t(0)
        if cu.cuGraphGetNodes(h, None, ctypes.byref(n)) != 0:
            return None
        nodes = (ctypes.c_void_p * n.value)()
        if cu.cuGraphGetNodes(h, nodes, ctypes.byref(n)) != 0:
            return None
        kinds = ctypes.c_int(0)
        k = 0
        for i in range(n.value):
            if cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(kinds)) == 0 and \
                    kinds.value == 0:  # CU_GRAPH_NODE_TYPE_KERNEL
                k += 1
        return k
    except (OSError, AttributeError, TypeError, ValueError, RuntimeError):
        return None


# ----------------------------------------------------------------------------- verification


VERIFY_METRIC = "greedy verification latency (us); HBM GB/s %peak"


def verify_oracle_sample(wl, b, budget_s):
    """Time the oracle's verification (as it stands) on whole batches until the
    budget is spent.  Returns (us per batch, sample text, threads)."""
    from oracle import pe_oracle as O

    t0 = time.perf_counter()
    done = 0
    while True:
        O.verify_greedy(b["qsl"], b["tok"], O.decode(b["logits"], wl.dtype))
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    sample = f"{done} whole batch(es) of {wl.name} ({b['T_in']} rows x {wl.vocab} logits), {dt:.1f} s"
    return dt / done * 1e6, sample, 1


def run_verify(args, rank, world, local):
    """pe_verify_greedy over one seeded verify batch per rank.  Inputs sit in HBM;
    L2 is flushed (a 256 MB write, then a read of it) before every timed call, and
    each call is timed alone with CUDA events on its stream."""
    import torch

    from speculative_drafting_gb300 import binding, build

    wl = W.get_verify(args.workload)
    if args.impl == "reference":
        if rank != 0:
            return
        b = W.make_verify_batch(wl)
        n_warm = warm_up(lambda: verify_oracle_sample(wl, b, budget_s=0.0), args.warmup)
        per, sample, threads = [], "", 1
        t_all = time.perf_counter()
        for _ in range(max(1, args.steps)):
            us, sample, threads = verify_oracle_sample(wl, b, budget_s=5.0)
            per.append(us)
            if time.perf_counter() - t_all > 150:
                break
        us = statistics.median(per)
        print(json.dumps({
            "impl": "reference", "metric": VERIFY_METRIC, "value": us, "unit": "us",
            "n_gpus": args.gpus, "steps": len(per), "warmup": n_warm, "ms_per_step": us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "global_batch": wl.batch,
                                            "description": wl.description},
            "cpu_baseline": {"value": us, "unit": "us", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    b = W.make_verify_batch(rank_workload(wl, rank))
    B, T_in, V = b["B"], b["T_in"], b["V"]
    esize = 2 if wl.dtype == "bf16" else 4
    code = binding.PE_DTYPE_BF16 if wl.dtype == "bf16" else binding.PE_DTYPE_F32
    lg_host = torch.from_numpy(b["logits"].view(np.int16) if wl.dtype == "bf16" else b["logits"])
    d = {"qsl": torch.from_numpy(b["qsl"]).cuda(), "tok": torch.from_numpy(b["tok"]).cuda(),
         "logits": lg_host.cuda()}
    target = torch.empty(T_in, dtype=torch.int32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    bon = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = binding.verify_workspace(T_in, V)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def call():
        binding.verify_greedy(B, T_in, d["qsl"], d["tok"], d["logits"], V, code, target, acc, bon,
                              ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    stream.synchronize()
    st, _ = binding.read_status_ws(ws, stream=stream)
    if st:
        raise RuntimeError(f"device status {st:#x} on the verify batch")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    def flush_l2():
        # write a buffer twice the size of L2, then read it back: the read evicts
        # the dirty lines, so no write-back lands inside the timed call
        flush.zero_()
        flush.max()

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            flush_l2()
            g.replay()
    stream.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_l2()
            ev[i][0].record(stream)
            g.replay()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    call_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    call_ms = max_over_ranks(call_ms, world, "cuda")
    # end to end: pinned host logits and tokens in, target tokens and counts out
    h_in = {"qsl": torch.from_numpy(b["qsl"]).pin_memory(),
            "tok": torch.from_numpy(b["tok"]).pin_memory(), "logits": lg_host.pin_memory()}
    h_out = [torch.empty(T_in, dtype=torch.int32).pin_memory(),
             torch.empty(B, dtype=torch.int32).pin_memory(),
             torch.empty(B, dtype=torch.int32).pin_memory()]
    n_e2e = max(5, args.steps // 4)
    with torch.cuda.stream(stream):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n_e2e):
            for k, t in h_in.items():
                d[k].copy_(t, non_blocking=True)
            g.replay()
            for hst, dev in zip(h_out, (target, acc, bon)):
                hst.copy_(dev, non_blocking=True)
        a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a0.elapsed_time(a1) / n_e2e
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    if rank == 0:
        peaks, src = measured_peaks()
        alg = T_in * V * esize + T_in * 4 * 2 + (B + 1) * 4 + 2 * B * 4
        achieved = alg / (call_ms / 1e3) / 1e9
        cpu = None
        if not args.no_cpu_baseline:
            us, sample, threads = verify_oracle_sample(wl, b, budget_s=10.0)
            cpu = {"value": us, "unit": "us", "cores": threads, "kind": "oracle", "sample": sample}
        print(json.dumps({
            "metric": VERIFY_METRIC, "value": call_ms * 1e3, "unit": "us", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": call_ms,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if wl.dtype == "f32" else "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "global_batch": B * world, "rows": T_in, "vocab": V,
                       "description": wl.description, "cuda_graph": True,
                       "l2": "flushed before every timed call (256 MB write, then a 256 MB "
                             "read, so no dirty line is written back inside the call)",
                       "parallelism": f"replica x{world} (independent batches per GPU)"},
            "clocks": clk,
            "e2e": {"value": e2e_ms * 1e3, "unit": "us", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": 2 * args.steps,
            "roofline": {"kernel": "verify_partial_kernel + verify_accept_kernel (whole call)",
                         "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": profiled_traffic(wl.name),
                         "peak_source": src, "algorithmic_bytes": alg,
                         "avg_launch_us": call_ms * 1e3},
            "cpu_baseline": cpu}), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------------------- COD training indices


COD_METRIC = "COD index lists + asymmetric mask per batch (us); HBM GB/s %peak of the mask write"


def cod_oracle_sample(wl, b, budget_s):
    """Time the oracle's index lists and dense mask (as they stand), one sequence
    at a time, until the budget is spent; scale to the whole batch.  Returns
    (us per batch, sample text, threads)."""
    from oracle import pe_cod as C

    t0 = time.perf_counter()
    done = 0
    while done < b["B"]:
        L = int(b["seq_len"][done])
        lv = C.cod_sample_indices(b["loss_mask"][done, :L], b["n_depth"], b["retain"],
                                  b["max_anchors"], b["u_anchor"][done, :L], b["u_keep"][done, :, :L])
        C.cod_mask(lv, L)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    sample = f"{done} of {b['B']} sequences of {wl.name}, {dt:.1f} s, scaled to the batch"
    return dt / done * b["B"] * 1e6, sample, 1


def run_cod(args, rank, world, local):
    """pe_cod_sample_indices + pe_cod_mask over one seeded batch of sequences per
    rank.  L2 is flushed before every timed call; the whole pair is one graph, and
    the mask call alone is a second graph, timed in its own loop for the
    roofline line."""
    import torch

    from speculative_drafting_gb300 import build, runner

    wl = W.get_cod(args.workload)
    if args.impl == "reference":
        if rank != 0:
            return
        b = W.make_cod_batch(wl)
        n_warm = warm_up(lambda: cod_oracle_sample(wl, b, budget_s=0.0), args.warmup)
        per, sample, threads = [], "", 1
        t_all = time.perf_counter()
        for _ in range(max(1, args.steps)):
            us, sample, threads = cod_oracle_sample(wl, b, budget_s=5.0)
            per.append(us)
            if time.perf_counter() - t_all > 150:
                break
        us = statistics.median(per)
        print(json.dumps({
            "impl": "reference", "metric": COD_METRIC, "value": us, "unit": "us",
            "n_gpus": args.gpus, "steps": len(per), "warmup": n_warm, "ms_per_step": us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic", "config": {"workload": wl.name, "global_batch": wl.batch,
                                            "description": wl.description},
            "cpu_baseline": {"value": us, "unit": "us", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    b = W.make_cod_batch(rank_workload(wl, rank))
    r = runner.CodRunner(b)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(3):
            r.run(stream=stream)
    stream.synchronize()
    st, _ = r.status()
    if st:
        raise RuntimeError(f"device status {st:#x} on the COD batch")
    g_all, g_mask = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all, stream=stream):
        r.run(stream=stream)
    with torch.cuda.graph(g_mask, stream=stream):
        r.build_mask(stream=stream)

    def flush_l2():
        flush.zero_()
        flush.max()

    def timed(graph, n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        with torch.cuda.stream(stream):
            for i in range(n):
                flush_l2()
                ev[i][0].record(stream)
                graph.replay()
                ev[i][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            flush_l2()
            g_all.replay()
    stream.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    call_ms = timed(g_all, args.steps)
    mask_ms = timed(g_mask, args.steps)
    clk = clocks.stop()
    call_ms = max_over_ranks(call_ms, world, "cuda")
    # end to end: pinned host inputs in, the lists, counts and masks out
    h_in = {k: torch.from_numpy(np.ascontiguousarray(b[k])).pin_memory()
            for k in ("seq_len", "loss_mask", "u_anchor", "u_keep")}
    counts = r.counts.cpu().numpy()
    lens = np.clip(b["seq_len"], 0, b["S_max"])
    Q = counts.sum(1)
    KV = lens + Q - counts[:, 0]
    width = (KV + 15) // 16 * 16
    h_mask = torch.empty(r.mask.numel(), dtype=torch.uint8).pin_memory()
    h_idx = torch.empty(r.idx.shape, dtype=torch.int32).pin_memory()
    h_cnt = torch.empty(r.counts.shape, dtype=torch.int32).pin_memory()
    n_e2e = max(3, args.steps // 8)
    with torch.cuda.stream(stream):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n_e2e):
            for k, t in h_in.items():
                r.inp[k].copy_(t, non_blocking=True)
            g_all.replay()
            h_idx.copy_(r.idx, non_blocking=True)
            h_cnt.copy_(r.counts, non_blocking=True)
            # each sequence's written rows (Q_b rows of its block)
            for s in range(r.B):
                nb = int(Q[s]) * r.ld
                if nb:
                    lo = s * r.mask_stride
                    h_mask[lo:lo + nb].copy_(r.mask[lo:lo + nb], non_blocking=True)
        a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a0.elapsed_time(a1) / n_e2e
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h_mask = int((Q * r.ld).sum())
    d2h = d2h_mask + h_idx.numel() * 4 + h_cnt.numel() * 4
    if rank == 0:
        peaks, src = measured_peaks()
        mask_bytes = int((Q * width).sum())
        # the mask kernel also reads each row's anchor and its chain places
        alg = mask_bytes + int(Q.sum()) * 4 + int((counts[:, 1:].sum(1)).sum()) * 4
        achieved = alg / (mask_ms / 1e3) / 1e9
        cpu = None
        if not args.no_cpu_baseline:
            us, sample, threads = cod_oracle_sample(wl, b, budget_s=10.0)
            cpu = {"value": us, "unit": "us", "cores": threads, "kind": "oracle", "sample": sample}
        print(json.dumps({
            "metric": COD_METRIC, "value": call_ms * 1e3, "unit": "us", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": call_ms,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic",
            "config": {"workload": wl.name, "global_batch": r.B * world, "seq_len": r.S,
                       "n_depth": r.D, "retain": r.retain, "max_anchors": r.max_anchors,
                       "mask_rows": int(Q.sum()), "mask_bytes": mask_bytes,
                       "description": wl.description, "cuda_graph": True,
                       "l2": "flushed before every timed call (256 MB write, then a 256 MB "
                             "read, so no dirty line is written back inside the call)",
                       "parallelism": f"replica x{world} (independent batches per GPU)"},
            "clocks": clk,
            "e2e": {"value": e2e_ms * 1e3, "unit": "us", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": 2 * args.steps,
            "roofline": {"kernel": "cod_mask_kernel", "bound": "hbm", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": profiled_traffic(wl.name),
                         "peak_source": src, "algorithmic_bytes": alg,
                         "avg_launch_us": mask_ms * 1e3},
            "index_kernel_us": (call_ms - mask_ms) * 1e3,
            "cpu_baseline": cpu}), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


PREP_METRIC = "metadata + hidden-state prep latency (us) per call; HBM GB/s %peak"


def prep_bytes(dm, batch):
    """Bytes pe_prepare_inputs must move: the verify batch's inputs and the block
    table entries it reads, the captured hidden states and embedding rows of the
    copied non-rejected rows (MASK rows share one h_shared and one emb(mask)),
    the drafter input rows it writes and the metadata tensors."""
    B, T_in, K, d = batch["B"], batch["T_in"], dm.K, dm.d
    acc = batch["accepted"].astype(np.int64)
    n_copied = int(np.sum(acc + 1))
    n_valid = int(np.sum(acc + K))
    T_out = T_in + B * (K - 1)
    inputs = (B + 1) * 4 + T_in * (4 + 8) + 2 * B * 4 + n_valid * 4
    hidden = n_copied * 3 * d * 2 + n_copied * d * 2 + 2 * d * 2
    out_a = n_valid * 4 * d * 2
    meta = T_out * (4 + 8 + 1 + 1 + 4 + 8 + 4) + 2 * (B + 1) * 4 + B * K * 4 + B * 4 + 4
    return inputs + hidden + out_a + meta


def prep_oracle_sample(wl, batch, w, budget_s=10.0):
    """The oracle's metadata + drafter input over the whole batch, repeated
    until the budget is spent.  Returns (us per call, sample text, threads)."""
    from oracle import pe_oracle as O

    t0 = time.perf_counter()
    done = 0
    while True:
        O.prepare_inputs(wl.dims, w, batch)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return dt / done * 1e6, f"{done} whole batches of {wl.name}, {dt:.1f} s", 1


def run_prep_reference(args, rank):
    if rank != 0:
        return
    wl = W.get(args.workload)
    batch = W.make_batch(wl)
    w = W.make_weights(wl)
    n_warm = warm_up(lambda: prep_oracle_sample(wl, batch, w, budget_s=0.0), args.warmup)
    per, sample, threads = [], "", 1
    t_all = time.perf_counter()
    for _ in range(max(1, args.steps)):
        us, sample, threads = prep_oracle_sample(wl, batch, w, budget_s=5.0)
        per.append(us)
        if time.perf_counter() - t_all > 150:
            break
    us = statistics.median(per)
    print(json.dumps({
        "impl": "reference", "metric": PREP_METRIC, "value": us, "unit": "us", "n_gpus": args.gpus,
        "steps": len(per), "warmup": n_warm, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "global_batch": wl.batch, "K": wl.dims.K,
                   "description": wl.description},
        "cpu_baseline": {"value": us, "unit": "us", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
        flush=True)


def run_prep(args, rank, world, local):
    """pe_prepare_inputs alone (metadata + drafter input), for the preparation
    workload that has no drafter layer.  L2 is flushed before every timed call
    (its ~30 MB fit in L2) and each call is timed alone with CUDA events."""
    import torch

    from speculative_drafting_gb300 import build, runner

    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    wl = W.get(args.workload)
    batch = W.make_batch(rank_workload(wl, rank))
    w = W.make_weights(wl)
    r = runner.StepRunner(wl, batch, w)
    stream = torch.cuda.Stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def flush_l2():
        flush.zero_()
        flush.max()

    with torch.cuda.stream(stream):
        for _ in range(3):
            r.prepare(stream=stream)
    stream.synchronize()
    st, _ = r.status()
    if st:
        raise RuntimeError(f"device status {st:#x} on the preparation batch")
    graphs = {}
    for name, with_a in (("call", True), ("meta", False)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            r.prepare(stream=stream, A=with_a)
        graphs[name] = g

    def timed(g, n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        with torch.cuda.stream(stream):
            for _ in range(max(args.warmup, 3)):
                flush_l2()
                g.replay()
            for i in range(n):
                flush_l2()
                ev[i][0].record(stream)
                g.replay()
                ev[i][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    call_ms = timed(graphs["call"], args.steps)
    meta_ms = timed(graphs["meta"], args.steps)
    clk = clocks.stop()
    call_ms = max_over_ranks(call_ms, world, "cuda")
    # end to end: the batch's inputs from one pinned host buffer, the metadata's
    # non-rejected row count read back, the host waiting for it every call
    stage_dev, stage_host = pack_step_inputs(r, batch)
    nv_host = torch.empty(1, dtype=torch.int32).pin_memory()
    n_e2e = max(10, args.steps // 2)
    with torch.cuda.stream(stream):
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            stage_dev.copy_(stage_host, non_blocking=True)
            graphs["call"].replay()
            nv_host.copy_(r.meta["n_valid"], non_blocking=True)
            stream.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
    if rank == 0:
        peaks, src = measured_peaks()
        alg = prep_bytes(wl.dims, batch)
        achieved = alg / (call_ms / 1e3) / 1e9
        cpu = None
        if not args.no_cpu_baseline:
            us, sample, threads = prep_oracle_sample(wl, batch, w, budget_s=10.0)
            cpu = {"value": us, "unit": "us", "cores": threads, "kind": "oracle", "sample": sample}
        print(json.dumps({
            "metric": PREP_METRIC, "value": call_ms * 1e3, "unit": "us", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": call_ms,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.dims.dtype, "data": "synthetic",
            "config": {"workload": wl.name, "global_batch": batch["B"] * world, "K": wl.dims.K,
                       "rows_in": batch["T_in"], "rows_out": r.T_out,
                       "description": wl.description, "cuda_graph": True,
                       "l2": "flushed before every timed call (256 MB write, then a 256 MB read)",
                       "parallelism": f"replica x{world} (independent requests per GPU)"},
            "meta_only_us": meta_ms * 1e3,
            "clocks": clk,
            "e2e": {"value": e2e_ms * 1e3, "unit": "us", "h2d_bytes_per_step": stage_host.numel(),
                    "d2h_bytes_per_step": 4, "ms_per_step": e2e_ms},
            "gpu_launches": 2 * args.steps,
            "roofline": {"kernel": "meta_kernel + input_kernel (the whole call)", "bound": "hbm",
                         "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": profiled_traffic(wl.name),
                         "peak_source": src, "algorithmic_bytes": alg,
                         "avg_launch_us": call_ms * 1e3},
            "cpu_baseline": cpu}), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.workload in W.VERIFY_WORKLOADS:
        run_verify(args, rank, world, local)
        return
    if args.workload in W.COD_WORKLOADS:
        run_cod(args, rank, world, local)
        return
    if not W.get(args.workload).has_drafter:
        if args.impl == "reference":
            run_prep_reference(args, rank)
            return
        run_prep(args, rank, world, local)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
