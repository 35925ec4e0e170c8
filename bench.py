"""Benchmark of the paged KV cache decode step on GB300.

A step is one pass of the whole hot path over one batch: the decode-step slot
mapping, kv_store of the appended tokens, and paged_decode -- per layer for
multi-layer workloads.  Default workload: the Qwen3-0.6B-shaped layer (batch
64, 16 q / 8 kv heads, head_dim 128, block_size 256, context_lens U[512,4096]).

Prints ONE JSON line (rank 0).  `value` is the achieved HBM bandwidth of the
step in GB/s (algorithmic bytes / step time, whole job); the line also carries
seq-steps/s, the roofline of the dominant kernel (paged_decode) and the CPU
oracle baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference] [--workload NAME]

Under torchrun (N > 1) every rank runs its own batch (seed + rank) on its own
GPU with no collective on the data path (weak scaling); the time is the max
over ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: achieved HBM GB/s (% of peak) and seq-steps/sec"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 126 * 1024 * 1024
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "paged_decode_qwen3_0p6b.txt")


# ----------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(workload: str, rank: int) -> int:
    """Seed of this rank's batch: every rank runs its own, different batch (weak scaling)."""
    from paged_kv_cache_62_gb300 import workloads
    return workloads.SEED_BASE + workloads.ORDER.index(workload) + 1000 * rank


def reduce_over_ranks(x: float, op: str, device) -> float:
    """max / min of a per-rank scalar over all ranks (identity for one process)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.MIN)
    return float(t.item())


def job_bandwidth(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank moves bytes_per_rank_step per step; the step time is the slowest rank's."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def step_bytes(wl) -> dict:
    """Algorithmic bytes of one step: every K and V row of every sequence's context read once, q read and
    the output written (bf16), the context length and block-table entries read, and the new token's
    k, v rows read and stored."""
    s = wl.spec
    lens = wl.lens_host().astype(np.int64)
    B, Hq, Hkv, D = s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim
    row = Hkv * D * 2
    decode = int(lens.sum()) * row * 2 + B * Hq * D * 2 * 2          # K+V rows read, q read, out written
    decode_index = B * 4 + int(sum(-(-int(L) // s.block_size) for L in lens)) * 4
    # the step stores each sequence's new token in the decode launch itself (pkv_paged_decode_store):
    # its k, v rows read and its cache rows written (the length and table entry are in decode_index)
    store = B * row * 2 * 2
    L = s.layers
    return {"decode": decode + decode_index, "store": store, "fused": decode + decode_index + store,
            "step": L * (decode + decode_index + store), "decode_kv_only": int(lens.sum()) * row * 2}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.proc = None
        self.gpu = gpu_index
        self.out = b""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", self.gpu], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = list(csv.reader(io.StringIO(self.out.decode(errors="replace"))))
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_sha() -> str:
    """SHA-256 over the sources the decode kernel is compiled from (the kernel header, its entry-point
    file and the device helpers), in that order."""
    csrc = os.path.join(ROOT, "paged_kv_cache_62_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("pkv_decode_kernel.cuh", "pkv_decode.cu", "pkv_device.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_from_profile():
    """DRAM bytes per paged_decode launch from the committed ncu summary, if it matches the current source."""
    try:
        kv = {}
        with open(PROFILE_TRAFFIC) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, _, v = line.partition(":")
                    kv[k.strip()] = v.strip()
        sha = kernel_source_sha()
        if kv.get("src_sha256") != sha:
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


def warm_up(step, min_steps: int, min_seconds: float) -> int:
    """Untimed steps right before a timed region: at least min_steps, and at least min_seconds of them (a GB300
    idles at a low clock and takes a moment to ramp up; the per-SM split settles over the first calls on a
    workspace).  Returns the number of steps run."""
    n, t0 = 0, time.perf_counter()
    while n < min_steps or time.perf_counter() - t0 < min_seconds:
        for _ in range(max(1, min_steps)):
            step()
        n += max(1, min_steps)
        torch.cuda.synchronize()
    return n


def launch_distribution(us):
    """Summary of per-launch times (us, in launch order): mean, median, extremes, and the first and last five
    (a settling or clock-ramp effect shows up as first5 above last5)."""
    a = np.asarray(us, dtype=np.float64)
    return {"launches": int(a.size), "mean_us": round(float(a.mean()), 2), "median_us": round(float(np.median(a)), 2),
            "min_us": round(float(a.min()), 2), "max_us": round(float(a.max()), 2),
            "first5_mean_us": round(float(a[:5].mean()), 2), "last5_mean_us": round(float(a[-5:].mean()), 2)}


def time_calls(call, reps: int, stream) -> tuple[float, float]:
    """Mean us per call of `call`, issued `reps` times back to back with CUDA events around the whole run
    (as a loop issues it), then mean us with an event pair around every call (the pairs cut the overlap of
    a launch's set-up with the previous launch's tail).  Five untimed calls come first."""
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(reps):
        call()
    t1.record(stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for c0, c1 in evs:
        c0.record(stream)
        call()
        c1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) * 1e3 / reps, float(np.mean([c0.elapsed_time(c1) for c0, c1 in evs])) * 1e3


def source_sha() -> str:
    """SHA-256 over every library source and the public header (the product as built), in sorted order."""
    csrc = os.path.join(ROOT, "paged_kv_cache_62_gb300", "csrc")
    h = hashlib.sha256()
    for p in sorted(os.path.join(csrc, n) for n in os.listdir(csrc)) + [os.path.join(ROOT, "include", "pkv.h")]:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def run_metadata(dev) -> dict:
    """GPU name, git commit (when the checkout has its .git), source hash and host CPU model."""
    git = None
    try:
        r = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"], capture_output=True, text=True, timeout=10)
        if r.returncode == 0:
            git = r.stdout.strip()
    except Exception:
        pass
    cpu = None
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.startswith("Model name:"):
                cpu = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if cpu is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        cpu = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    import platform
    return {"gpu_name": torch.cuda.get_device_name(dev), "git_commit": git, "source_sha256": source_sha(),
            "host_cpu_model": cpu or platform.machine(), "host_cores": os.cpu_count(),
            "torch": torch.__version__, "cuda": torch.version.cuda}


def config_block(name, dev, rank, peak, warmup):
    """One workload's decode step (pkv_paged_decode_store per layer, issued through pkv.DecodeStoreStep, the
    binding a serving loop keeps across steps), after `warmup` steps: back to back (CUDA events around all the
    steps), per launch with CUDA events around each (the event pairs themselves add a few microseconds to a
    short launch), and as one captured CUDA graph replayed back to back."""
    from paged_kv_cache_62_gb300 import pkv, workloads
    wl = workloads.make(name, dev, seed=rank_seed(name, rank))
    s = wl.spec
    B, Hq, Hkv, D = s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim
    max_ctx = int(wl.lens_host().max())
    outs = [torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev) for _ in wl.layers]
    ws = pkv.alloc_workspace(B, Hq, Hkv, D, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    k_step = [lay.k_new[:B].contiguous() for lay in wl.layers]
    v_step = [lay.v_new[:B].contiguous() for lay in wl.layers]
    bound = [pkv.DecodeStoreStep(lay.q, k_step[li], v_step[li], lay.k_cache, lay.v_cache, wl.block_tables,
                                 wl.context_lens, wl.scale, outs[li], ws, max_context_len=max_ctx, err_word=err)
             for li, lay in enumerate(wl.layers)]

    def step(evs=None, st=None):
        h = (stream if st is None else st).cuda_stream
        for li in range(len(bound)):
            if evs is not None:
                evs[li][0].record(st if st is not None else stream)
            bound[li].run(h)
            if evs is not None:
                evs[li][1].record(st if st is not None else stream)

    nl = len(wl.layers)
    n_steps = 300 if nl == 1 else 12
    warm_up(step, max(warmup, 3), 0.1)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(n_steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    step_ms = t0.elapsed_time(t1) / n_steps
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nl)]
           for _ in range(n_steps)]
    for i in range(n_steps):
        step(evs[i])
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) * 1e3 for row in evs for (a, b) in row]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(st=torch.cuda.current_stream(dev))  # the capture stream
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g_steps = 300 if nl == 1 else 20
    t0.record(stream)
    for _ in range(g_steps):
        graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    g_ms = t0.elapsed_time(t1) / g_steps
    assert err.item() == 0, f"{name}: device error word {err.item():#x}"
    nb = step_bytes(wl)
    dist = launch_distribution(per)
    res = {"workload": s.description, "layers": nl, "batch": B, "launches_per_step": nl,
           "algorithmic_bytes_per_launch": nb["fused"], "algorithmic_bytes_per_step": nb["step"],
           "launch_us": dist, "back_to_back_launch_us": round(step_ms * 1e3 / nl, 2),
           "launch_gbs_median": round(nb["fused"] / (dist["median_us"] * 1e-6) / 1e9, 1),
           "launch_frac_median": round(nb["fused"] / (dist["median_us"] * 1e-6) / 1e9 / peak, 4),
           "step_ms": round(step_ms, 5), "step_gbs": round(nb["step"] / (step_ms * 1e-3) / 1e9, 1),
           "step_frac": round(nb["step"] / (step_ms * 1e-3) / 1e9 / peak, 4),
           "seq_steps_per_sec": round(B / (step_ms * 1e-3), 1),
           "graph_step_ms": round(g_ms, 5), "graph_gbs": round(nb["step"] / (g_ms * 1e-3) / 1e9, 1),
           "graph_seq_steps_per_sec": round(B / (g_ms * 1e-3), 1)}
    if name == "long_mixed":
        uniq, logical = wl.kv_bytes_unique(), wl.kv_bytes_logical()
        ub = nb["fused"] - logical + uniq
        res["logical_kv_bytes_per_launch"] = logical
        res["unique_kv_bytes_per_launch"] = uniq
        res["unique_bytes_per_launch"] = ub
        res["unique_gbs_median"] = round(ub / (dist["median_us"] * 1e-6) / 1e9, 1)
        res["unique_frac_median"] = round(ub / (dist["median_us"] * 1e-6) / 1e9 / peak, 4)
        res["note"] = ("groups of 8 sequences share up to 64 leading blocks, which later readers find in L2: the "
                       "logical figure can pass the copy peak, the unique one counts each cached row once")
    del wl, outs, ws, graph
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- GPU arm
def run_pkv(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_62_gb300 import pkv, workloads

    wl = workloads.make(args.workload, dev, seed=rank_seed(args.workload, rank))
    s = wl.spec
    B, Hq, Hkv, D = s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim
    max_ctx = int(wl.lens_host().max())
    outs = [torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev) for _ in wl.layers]
    wsbuf = pkv.alloc_workspace(B, Hq, Hkv, D, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    launches_per_step = len(wl.layers)
    # one new token per sequence: rows [0, B) of the step's k / v (the workload's extra padding rows are
    # for the unfused kv_store's slot -1 path and are not stored by a decode step)
    k_step = [lay.k_new[:B].contiguous() for lay in wl.layers]
    v_step = [lay.v_new[:B].contiguous() for lay in wl.layers]
    # one launch per layer (the new token's K/V stored into the cache and attended), through the binding a
    # serving loop keeps across steps (buffers checked once)
    bound = [pkv.DecodeStoreStep(lay.q, k_step[li], v_step[li], lay.k_cache, lay.v_cache, wl.block_tables,
                                 wl.context_lens, wl.scale, outs[li], wsbuf, max_context_len=max_ctx, err_word=err)
             for li, lay in enumerate(wl.layers)]

    def step(dec_events=None, st=None):
        st = stream if st is None else st
        h = st.cuda_stream
        for li in range(len(bound)):
            if dec_events is not None:
                dec_events[li][0].record(st)
            bound[li].run(h)
            if dec_events is not None:
                dec_events[li][1].record(st)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    if args.steps is None:
        # size the run to about 2 s of GPU work (untimed calls, before the warm-up below)
        step()
        torch.cuda.synchronize()
        tw = time.perf_counter()
        for _ in range(10):
            step()
        torch.cuda.synchronize()
        per = (time.perf_counter() - tw) / 10
        args.steps = int(min(50000, max(50, 2.0 / per)))
        args.steps = int(reduce_over_ranks(args.steps, "min", dev))

    nlay = len(wl.layers)
    dec_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nlay)]
              for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local] \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else str(local)
    with ClockSampler(gpu_index) as clocks:
        time.sleep(0.3)  # nvidia-smi's first sample
        # The warm-up runs here, right before the timed steps: an idle GB300 drops to its idle clock within
        # a fraction of a second, and the first call after an idle gap then runs ~1.5x slower.
        n_warm = warm_up(step, max(args.warmup, 3), 0.2)
        assert err.item() == 0, f"device error word {err.item():#x}"
        barrier()
        torch.cuda.synchronize()
        # the timed region: the steps back to back, as a decode loop issues them (events around the whole)
        t0.record(stream)
        for i in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        barrier()
        # then the same steps with an event pair around every launch, for the per-launch distribution (the
        # pairs cut the overlap of a launch's set-up with the previous launch's tail, so these read longer)
        for i in range(args.steps):
            step(dec_ev[i])
        torch.cuda.synchronize()
        time.sleep(0.3)
    ms = t0.elapsed_time(t1) / args.steps
    dec_mean_ms = ms / launches_per_step  # the timed region's average per launch
    dec_ms = [a.elapsed_time(b) for row in dec_ev for (a, b) in row]
    launch_stats = launch_distribution([x * 1e3 for x in dec_ms])
    ms = reduce_over_ranks(ms, "max", dev)

    # ---- the same step captured once as a CUDA graph and replayed (how a serving engine runs its
    # decode step): no host work between launches, and each kernel's set-up overlaps the previous
    # kernel's tail through programmatic dependent launch.  Same inputs, same workspace.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(st=torch.cuda.current_stream(dev))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g_steps = max(10, min(args.steps, 20000))
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    g0.record(stream)
    for _ in range(g_steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    g_ms = reduce_over_ranks(g0.elapsed_time(g1) / g_steps, "max", dev)
    assert err.item() == 0, f"device error word {err.item():#x}"

    # ---- several new tokens per sequence (pkv_paged_attention) on layer 0, causal over each sequence's
    # cache: the last nq tokens of every sequence as queries
    mixed = None
    if not args.no_fp8:
        lay0 = wl.layers[0]
        lens_h = wl.lens_host().astype(np.int64)
        row = Hkv * D * 2 * 2

        def time_attention(nq, offsets, reps):
            """Mean us of a pkv_paged_attention call with nq new tokens per sequence (given by offsets, or
            as new_per_seq = nq), back to back (and with an event pair around each call)."""
            cu = torch.arange(0, (B + 1) * nq, nq, dtype=torch.int32, device=dev) if offsets else None
            qa = torch.randn(B * nq, Hq, D, device=dev).bfloat16()
            oa = torch.empty_like(qa)
            wsa = pkv.alloc_attention_workspace(B * nq, Hq, Hkv, D, dev)

            def call():
                pkv.paged_attention(qa, lay0.k_cache, lay0.v_cache, wl.block_tables, cu, wl.context_lens, wl.scale,
                                    oa, wsa, max_context_len=max_ctx, err_word=err, stream=stream,
                                    new_per_seq=0 if offsets else nq)
            us, us_ev = time_calls(call, reps, stream)
            assert err.item() == 0, f"device error word {err.item():#x}"
            return us, us_ev

        nq = 4
        if lens_h.min() >= nq:
            # a speculative-decoding verify step: the 4 queries of a sequence as 4 x G virtual heads
            us_m, us_m_ev = time_attention(nq, False, 50)
            unique = int(lens_h.sum()) * row
            streamed = int(sum(L - nq + 1 + i for L in lens_h for i in range(nq))) * row
            mixed = {"kernel": "pkv_paged_attention (paged_decode_kernel, the 4 queries of a sequence as 4 x G "
                               "virtual heads over one pass of its keys)",
                     "query_rows": B * nq, "new_tokens_per_sequence": nq, "mean_call_us": round(us_m, 2),
                     "event_pair_mean_call_us": round(us_m_ev, 2),
                     "unique_kv_bytes": unique, "streamed_kv_bytes": streamed,
                     "unique_gbs": round(unique / (us_m * 1e-6) / 1e9, 1),
                     "streamed_gbs": round(streamed / (us_m * 1e-6) / 1e9, 1),
                     "note": "K/V read once per sequence; streamed_* counts one pass per query row, for comparison "
                             "with running the rows separately"}
        nv = 8
        if lens_h.min() >= nv:
            # a verify step with the offsets given: chunks of max(1, 16 // G) queries on regular CTAs
            us_v, us_v_ev = time_attention(nv, True, 50)
            unique = int(lens_h.sum()) * row
            mixed = dict(mixed or {})
            mixed["verify_offsets"] = {
                "kernel": "pkv_paged_attention (expand_rows_kernel + paged_decode_kernel, chunks of up to "
                          "16 / G queries)", "query_rows": B * nv, "new_tokens_per_sequence": nv,
                "mean_call_us": round(us_v, 2), "event_pair_mean_call_us": round(us_v_ev, 2), "unique_kv_bytes": unique,
                "unique_gbs": round(unique / (us_v * 1e-6) / 1e9, 1)}
        npf = 64
        if lens_h.min() >= npf and B * npf <= 16384:
            # the last npf tokens of every sequence as one prefill chunk over its cached prefix (offsets
            # given): query-split CTAs, 8 x max(1, 16 // G) queries per K/V pass
            us_p, us_p_ev = time_attention(npf, True, 30)
            qe = max(1, 16 // (Hq // Hkv)) * 8
            chunk_rows = int(sum(L - npf + min(c + qe, npf) for L in lens_h for c in range(0, npf, qe))) * row
            per_query = int(sum(L - npf + 1 + i for L in lens_h for i in range(npf))) * row
            mixed = dict(mixed or {})
            mixed["prefill_chunk"] = {
                "kernel": "pkv_paged_attention (expand_rows_kernel + paged_decode_kernel on tensor-memory "
                          "query-split CTAs (tcgen05.mma, 128 rows per tile), %d queries share each K/V pass)" % qe,
                "query_rows": B * npf, "new_tokens_per_sequence": npf, "mean_call_us": round(us_p, 2),
                "event_pair_mean_call_us": round(us_p_ev, 2),
                "chunk_streamed_kv_bytes": chunk_rows, "per_query_kv_bytes": per_query,
                "chunk_streamed_gbs": round(chunk_rows / (us_p * 1e-6) / 1e9, 1),
                "note": "the last %d tokens of every sequence as a prefill chunk over its cached prefix; "
                        "chunk_streamed counts one K/V pass per group of queries sharing it (what the kernel "
                        "reads), per_query one pass per query row" % npf}

    # ---- copy-on-write block copies (pkv_copy_blocks) on this workload's pool: owned blocks copied
    # into blocks no sequence holds, as many pairs as there are such blocks (up to 256)
    cow = None
    bt_h = wl.block_tables.cpu().numpy()
    owned = np.unique(bt_h[bt_h >= 0])
    free_ids = np.setdiff1d(np.arange(wl.num_blocks), owned)
    n_cow = int(min(256, len(free_ids), len(owned)))
    if n_cow >= 8:
        lay0 = wl.layers[0]
        cow_pairs = torch.from_numpy(np.stack([owned[:n_cow], free_ids[:n_cow]], 1).astype(np.int32)).to(dev)
        cow_us, cow_us_ev = time_calls(lambda: pkv.copy_blocks(lay0.k_cache, lay0.v_cache, cow_pairs, err, stream),
                                       50, stream)
        assert err.item() == 0, f"device error word {err.item():#x}"
        block_bytes = s.block_size * Hkv * D * 2
        cow_bytes = n_cow * 2 * block_bytes * 2  # K and V blocks, each read once and written once
        cow = {"kernel": "pkv_copy_blocks (copy_blocks_kernel)", "pairs": n_cow, "block_bytes": block_bytes,
               "bytes_per_launch": cow_bytes, "mean_launch_us": round(cow_us, 2),
               "event_pair_mean_launch_us": round(cow_us_ev, 2),
               "achieved": round(cow_bytes / (cow_us * 1e-6) / 1e9, 1), "unit": "GB/s",
               "note": "bytes read + written; peak is the measured copy bandwidth (read + write)"}

    # ---- the same decode over E4M3 (fp8) caches: layer 0's caches quantised per kv head
    # (scale = max |x| / 448), the same queries, tables and lengths
    fp8 = None
    if not args.no_fp8:
        lay0 = wl.layers[0]
        fin = lambda x: torch.nan_to_num(x.float(), nan=0.0)
        ks8 = (fin(lay0.k_cache).abs().amax(dim=(0, 1, 3)) / 448).clamp_min(1e-6).contiguous()
        vs8 = (fin(lay0.v_cache).abs().amax(dim=(0, 1, 3)) / 448).clamp_min(1e-6).contiguous()
        q8 = lambda x, sc: (x.float() / sc.view(1, 1, -1, 1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn) \
            .view(torch.uint8).contiguous()  # NaN canaries stay NaN (clamp keeps NaN)
        kc8, vc8 = q8(lay0.k_cache, ks8), q8(lay0.v_cache, vs8)
        out8 = torch.empty_like(outs[0])

        def dec8():
            pkv.paged_decode_fp8(lay0.q, kc8, vc8, ks8, vs8, wl.block_tables, wl.context_lens, wl.scale, out8,
                                 wsbuf, max_context_len=max_ctx, err_word=err, stream=stream)
        n8 = max(20, min(args.steps, 500))
        us8, us8_ev = time_calls(dec8, n8, stream)
        assert err.item() == 0, f"device error word {err.item():#x}"
        nb0 = step_bytes(wl)
        bytes8 = nb0["decode"] - nb0["decode_kv_only"] // 2  # K/V at one byte an element
        fp8 = {"kernel": "pkv_paged_decode_fp8 (paged_decode_kernel, E4M3 caches)", "bytes_per_launch": bytes8,
               "mean_launch_us": round(us8, 2), "event_pair_mean_launch_us": round(us8_ev, 2),
               "achieved": round(bytes8 / (us8 * 1e-6) / 1e9, 1), "unit": "GB/s",
               "seq_steps_per_sec_decode_only": round(B / (us8 * 1e-6), 1),
               "speedup_vs_bf16_decode": round(dec_mean_ms * 1e3 / us8, 3),
               "note": "layer 0 of the workload, caches quantised per kv head (scale = max|x| / 448)"}

    # ---- end to end: host buffers in, host result out, through the same public calls.  A step's inputs
    # (every layer's q and new k / v rows, the block tables, the lengths) sit packed in one pinned host
    # buffer and go over in one copy; the outputs come back in one copy (as a serving loop stages them).
    parts = [lay.q for lay in wl.layers] + k_step + v_step + [wl.block_tables, wl.context_lens]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += -(-(t.numel() * t.element_size()) // 256) * 256  # 256-byte aligned segments
    h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(parts, offs):
        n = t.numel() * t.element_size()
        h_in[o:o + n].copy_(t.contiguous().view(torch.uint8).view(-1).cpu())
        views.append(d_in[o:o + n].view(t.dtype).view(t.shape))
    nl = len(wl.layers)
    d_q, d_k, d_v = views[:nl], views[nl:2 * nl], views[2 * nl:3 * nl]
    d_bt, d_lens = views[3 * nl], views[3 * nl + 1]
    d_out = torch.empty(nl, B, Hq, D, dtype=torch.bfloat16, device=dev)
    h_out = [torch.empty(nl, B, Hq, D, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = total
    d2h = d_out.numel() * d_out.element_size()
    done = [torch.cuda.Event(), torch.cuda.Event()]
    e2e_bound = [pkv.DecodeStoreStep(d_q[li], d_k[li], d_v[li], lay.k_cache, lay.v_cache, d_bt, d_lens, wl.scale,
                                     d_out[li], wsbuf, max_context_len=max_ctx, err_word=err)
                 for li, lay in enumerate(wl.layers)]
    h_stream = stream.cuda_stream

    def e2e_step(i):
        # a serving loop: the host issues step i, then waits for step i - 1's results (read back into the
        # other host buffer) before it goes on, so the host's issue time overlaps the GPU's work.  (Copies on
        # a stream of their own, overlapping the kernels, measured slower: the host-side cost of the extra
        # events and stream switches outweighs the ~8 us of copies per Qwen3-0.6B-shaped step.)
        d_in.copy_(h_in, non_blocking=True)
        for li in range(nl):
            e2e_bound[li].run(h_stream)
        h_out[i % 2].copy_(d_out, non_blocking=True)
        done[i % 2].record(stream)
        if i > 0:
            done[(i - 1) % 2].synchronize()

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_steps = max(10, min(args.steps, 200))
    barrier()
    te = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - te) * 1e3 / e2e_steps
    e2e_ms = reduce_over_ranks(e2e_ms, "max", dev)
    torch.cuda.synchronize()
    assert err.item() == 0, f"device error word {err.item():#x}"

    nb = step_bytes(wl)
    peak, peak_kind = hbm_peak()
    gbs = job_bandwidth(nb["step"], ws, ms)
    dec_gbs = nb["fused"] / (dec_mean_ms * 1e-3) / 1e9
    traffic = traffic_from_profile() if args.workload == "qwen3_0p6b" else None
    line = {
        "metric": METRIC,
        "value": round(gbs, 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": n_warm,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",  # the arithmetic (fp32 products and sums); K/V, q and out are stored as bf16
        "data": "synthetic (seeded N(0,1) bf16 K/V/q, shuffled block pool, NaN canaries in unowned rows)",
        "config": {"workload": f"{args.workload}: {s.description}", "storage": "bf16", "layers": s.layers,
                   "batch_per_gpu": B,
                   "q_heads": Hq, "kv_heads": Hkv, "head_dim": D, "block_size": s.block_size,
                   "mean_context_len": float(wl.lens_host().mean()), "parallelism": f"replicas x{ws}",
                   "l2": f"inputs larger than L2 (KV pool {2 * wl.layers[0].k_cache.numel() * 2 / 2**20:.0f} MiB"
                         f" per layer > {L2_BYTES / 2**20:.0f} MiB)"},
        "seq_steps_per_sec": round(B * ws / (ms * 1e-3), 1),
        "pct_of_peak": {"measured_copy": round(100 * gbs / ws / peak, 2) if peak_kind == "measured" else None,
                        "nominal_8TBps": round(100 * gbs / ws / NOMINAL_HBM_GBS, 2)},
        "algorithmic_bytes_per_step": nb["step"],
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"kernel": "pkv_paged_decode_store (paged_decode_kernel: store of the new token, attention, "
                               "split-K merge)", "bound": "hbm",
                     "achieved": round(dec_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(dec_gbs / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": nb["fused"], "mean_launch_us": round(dec_mean_ms * 1e3, 2),
                     "mean_launch_us_note": "the timed region's steps back to back, per launch",
                     "event_pair_median_launch_us": launch_stats["median_us"],
                     "frac_event_pair_median": round(nb["fused"] / (launch_stats["median_us"] * 1e-6) / 1e9 / peak,
                                                     4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s"},
        "e2e": {"value": round(job_bandwidth(nb["step"], ws, e2e_ms), 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "note": "every step: one copy of the packed pinned host q/k/v/block_tables/context_lens in, "
                        "one copy of the bf16 outputs back; "
                        "the host waits for step i - 1's results before issuing step i + 1 (two steps in flight, "
                        "as a serving loop runs); wall clock over all steps"},
        "graph": {"value": round(job_bandwidth(nb["step"], ws, g_ms), 1), "unit": "GB/s",
                  "ms_per_step": round(g_ms, 5), "steps": g_steps,
                  "note": "the step captured once as a CUDA graph and replayed back to back (CUDA events around "
                          "all replays); the headline value above is plain stream launches"},
        "clocks": clocks.summary(),
        "launches": dict(launch_stats, note="the same steps after the timed region, an event pair around every "
                                             "launch"),
        "meta": run_metadata(dev),
    }
    if mixed is not None:
        line["mixed"] = mixed
    if fp8 is not None:
        fp8["peak"] = peak
        fp8["frac"] = round(fp8["achieved"] / peak, 4)
        line["fp8"] = fp8
    if cow is not None:
        cow["peak"] = peak
        cow["frac"] = round(cow["achieved"] / peak, 4)
        line["cow_copy"] = cow
    if args.workload == "long_mixed":
        line["config"]["unique_kv_bytes_per_launch"] = wl.kv_bytes_unique()
        line["config"]["logical_kv_bytes_per_launch"] = wl.kv_bytes_logical()
    if ws == 1 and not args.no_configs:
        # every workload of the suite, one after the other (the headline one included, measured afresh)
        line["configs"] = {name: config_block(name, dev, rank, peak, args.warmup) for name in workloads.ORDER}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------------------- CPU oracle legs
def host_copy(wl):
    from paged_kv_cache_62_gb300 import workloads
    lays = [{k: workloads.bits(getattr(layer, k)) for k in ("q", "k_new", "v_new", "k_cache", "v_cache")}
            for layer in wl.layers]
    return lays, wl.block_tables.cpu().numpy(), wl.context_lens.cpu().numpy()


def oracle_step(wl, lays, bt, lens, seqs, nthreads):
    """Slot mapping + kv_store + paged decode of `seqs` (a prefix of the batch) in the fp64 oracle."""
    import oracle
    s = wl.spec
    sub_bt, sub_lens = bt[:seqs], lens[:seqs]
    slot = oracle.decode_slot_mapping(sub_bt, sub_lens, s.block_size, seqs)
    for t in wl.skip_tokens:
        if t < seqs:
            slot[t] = -1
    out = None
    for L in lays:
        oracle.kv_store(L["k_new"][:seqs], L["v_new"][:seqs], slot, L["k_cache"], L["v_cache"])
        out = oracle.paged_decode(L["q"][:seqs], L["k_cache"], L["v_cache"], sub_bt, sub_lens, wl.scale,
                                  nthreads=nthreads)
    return out


def cpu_baseline(wl, budget_s=12.0):
    """The oracle as it stands, on the host cores, over a bounded sample of the same workload.

    The sample is a prefix of the batch on the first layer; for multi-layer
    workloads the per-step figures are scaled by the layer count.
    """
    from paged_kv_cache_62_gb300 import workloads
    first = wl.layers[0]
    lays = [{k: workloads.bits(getattr(first, k)) for k in ("q", "k_new", "v_new", "k_cache", "v_cache")}]
    bt, lens = wl.block_tables.cpu().numpy(), wl.context_lens.cpu().numpy()
    cores = os.cpu_count() or 1
    s = wl.spec
    seqs = min(s.num_seqs, 4)
    t = time.perf_counter()
    oracle_step(wl, lays, bt, lens, seqs, cores)
    dt = max(time.perf_counter() - t, 1e-6)
    seqs = int(max(1, min(s.num_seqs, seqs * (budget_s / 3) / dt)))
    reps, elapsed = 0, 0.0
    t = time.perf_counter()
    while elapsed < budget_s * 0.6 or reps == 0:
        oracle_step(wl, lays, bt, lens, seqs, cores)
        reps += 1
        elapsed = time.perf_counter() - t
    per_layer = elapsed / reps
    lens_s = lens[:seqs].astype(np.int64)
    row = s.num_kv_heads * s.head_dim * 2
    nbytes = int(lens_s.sum()) * row * 2 + seqs * s.num_q_heads * s.head_dim * 4 + seqs * row * 4
    per_step = per_layer * s.layers
    # the same oracle on one thread, over a smaller prefix (about a quarter of the budget)
    seqs1 = int(max(1, min(seqs, seqs * (budget_s / 4) / (per_layer * cores))))
    t = time.perf_counter()
    oracle_step(wl, lays, bt, lens, seqs1, 1)
    dt1 = max(time.perf_counter() - t, 1e-6)
    lens_1 = lens[:seqs1].astype(np.int64)
    nbytes1 = int(lens_1.sum()) * row * 2 + seqs1 * s.num_q_heads * s.head_dim * 4 + seqs1 * row * 4
    single = {"value": round(nbytes1 / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
              "seq_steps_per_sec": round(seqs1 / (dt1 * s.layers), 3),
              "sample": f"first {seqs1} sequences, one repetition in {dt1:.1f} s"}
    return {"value": round(nbytes / per_layer / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "single_thread": single,
            "seq_steps_per_sec": round(seqs / per_step, 3), "seconds_per_step": round(per_step, 4),
            "sample": f"first {seqs} of {s.num_seqs} sequences of the {s.name} batch"
                      + (f", layer 0 of {s.layers} (time x{s.layers} per step)" if s.layers > 1 else "")
                      + f"; slot mapping + kv_store + fp64 paged decode; {reps} repetition(s) in {elapsed:.1f} s"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    from paged_kv_cache_62_gb300 import workloads
    wl = workloads.make(args.workload, "cpu", layers=1 if args.workload == "full_depth" else None)
    s = wl.spec
    lays, bt, lens = host_copy(wl)
    cores = os.cpu_count() or 1
    # size one step to ~1 s so that --steps K --warmup W stays within minutes
    t = time.perf_counter()
    oracle_step(wl, lays, bt, lens, min(4, s.num_seqs), cores)
    dt = max(time.perf_counter() - t, 1e-6)
    seqs = int(max(1, min(s.num_seqs, min(4, s.num_seqs) * 1.0 / dt)))
    if args.steps is None:
        args.steps = 10
    for _ in range(args.warmup):
        oracle_step(wl, lays, bt, lens, seqs, cores)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(wl, lays, bt, lens, seqs, cores)
    per_step = (time.perf_counter() - t) / args.steps
    lens_s = lens[:seqs].astype(np.int64)
    row = s.num_kv_heads * s.head_dim * 2
    nbytes = int(lens_s.sum()) * row * 2 + seqs * s.num_q_heads * s.head_dim * 4 + seqs * row * 4
    value = nbytes / per_step / 1e9
    sample = (f"first {seqs} of {s.num_seqs} sequences of the {s.name} batch"
              + (", one of 28 layers" if s.name == "full_depth" else "")
              + ", slot mapping + kv_store + fp64 paged decode per step")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16 inputs, CPU generator)",
            "config": {"workload": f"{args.workload}: {s.description}", "parallelism": "host cores"},
            "seq_steps_per_sec": round(seqs / per_step, 3),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: about 2 s of GPU work)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--workload", default="qwen3_0p6b")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the E4M3-cache decode measurement")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload block of all five workloads")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_pkv(args)


if __name__ == "__main__":
    main()
