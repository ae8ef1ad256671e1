"""Benchmark: one step = the whole hot path (dispatch layout, RDMA token
count, dispatch, identity expert, weighted combine) on the high-throughput
prefill workload: 8 logical EP ranks x 4096 tokens/rank, hidden 7168 bf16,
256 experts, top-8 routing from N(0,1) logits, rank-major receive buffers.

Prints ONE JSON line on rank 0.  ``value`` is tokens/s of the whole step
with inputs resident in HBM; ``e2e`` is the same step through the C ABI from
pinned host buffers (host->device copies of x / topk_idx / topk_weights and
the device->host copy of the combined output inside the timed region).
``--impl reference`` times the CPU oracle instead, on a bounded sample of
the same workload.  Multi-GPU (torchrun): every rank runs an independent
replica (the emulated EP ranks already live inside one GPU); value is the
sum of all ranks' tokens over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from combine_ep_layout_05_gb300 import inputs  # noqa: E402

WORKLOAD = "prefill_r8_t4096"
METRIC = "dispatch+combine tokens/s and effective HBM GB/s (% of GB300 peak) vs tokens/rank"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# algorithmic bytes (decimal GB convention of the pages: bytes / 1e9 / s)
# ---------------------------------------------------------------------------

def wire_row_bytes(H, combine_fmt):
    """Bytes of one row in a combine wire format (payload + scales)."""
    if combine_fmt == "mxfp8":
        return H + H // 32
    if combine_fmt == "nvfp4":
        return H // 2 + (H // 16) * 2
    return H * 2


def algorithmic_bytes(T, H, k, R, E, N, D, dtype="bf16", combine_fmt="bf16", A=None):
    """Bytes each step must move at least once, per kernel.

    layout:   read topk_idx (T*k*8) once; write is_token_in_rank (T*R),
              rank_slot and token-major offset (2*T*R*4), expert_slot
              (T*k*4); the RDMA token counts come out of the same pass
    dispatch: read x (T*H*2) and rank_slot (T*R*4); write D rows
              (D*H*2, or D*(H + H/128*4) for FP8)
    combine:  read D rows (D*H*2), topk_idx + weights (T*k*12), rank_slot
              (T*R*4); write out (T*H*2)
    """
    row_out = H * 2 if dtype == "bf16" else H + (H // 128) * 4
    byt = {
        "layout": T * k * 8 + T * R + 2 * T * R * 4 + T * k * 4,
        "dispatch": T * H * 2 + T * R * 4 + D * row_out,
        "combine": D * H * 2 + T * k * 12 + T * R * 4 + T * H * 2,
    }
    if dtype != "bf16":
        # identity expert for an FP8 payload: read the payload and scales of
        # each live row, write its bf16 expert output
        byt["expert"] = D * (row_out + H * 2)
    if A is not None:
        # two-level: dispatch stages A = algo rows (one per (token, node)) and
        # forwards them; combine writes A node partials and sums them
        byt["dispatch"] = T * H * 2 + T * R * 4 + A * H * 2 + (A * H * 2 + D * H * 2)
        byt["combine"] = D * H * 2 + T * k * 12 + T * R * 4 + A * H * 2 + (A * H * 2 + T * H * 2)
    if combine_fmt != "bf16":
        # expert-side cast to the wire format, then combine reads wire rows
        wb = wire_row_bytes(H, combine_fmt)
        byt["wire"] = D * (H * 2 + wb)
        byt["combine"] = D * wb + T * k * 12 + T * R * 4 + T * H * 2
    return byt


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(kernel_key, src_files, workload=WORKLOAD):
    """Per-launch DRAM bytes from the committed ncu summary of this kernel on
    this workload, or None if absent or taken on a different source."""
    path = os.path.join(ROOT, "profiles", f"{kernel_key}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    h = re.search(r"source_sha256:\s*([0-9a-f]+)", txt)
    if not m or not h or h.group(1) != source_hash(src_files):
        return None
    return float(m.group(1))


def same_mix_peak(workload=WORKLOAD):
    """The HBM bound measured for the dispatch's own read:write mix (each
    token row read once, written to its ~5.3 destination rows) by the
    `--mix-bound` probe on this machine's GPUs, from its committed summary; None
    if absent."""
    path = os.path.join(ROOT, "profiles", f"hbm_mix_{workload}.md")
    if not os.path.exists(path):
        return None
    m = re.search(r"same_mix_bound_gbs:\s*([0-9.eE+]+)", open(path).read())
    return (float(m.group(1)), os.path.relpath(path, ROOT)) if m else None


def source_hash(files):
    hs = hashlib.sha256()
    for f in files:
        hs.update(open(os.path.join(ROOT, f), "rb").read())
    return hs.hexdigest()[:16]


_CS = "combine_ep_layout_05_gb300/csrc/"
KERNEL_SOURCES = {
    "dispatch": [_CS + "dispatch.cu", _CS + "dispatch_device.cuh", _CS + "ep_internal.cuh"],
    "combine": [_CS + "combine.cu", _CS + "combine_device.cuh", _CS + "ep_internal.cuh", _CS + "vec8.cuh"],
    "combine_mxfp8": [_CS + "combine_wire.cu", _CS + "combine_device.cuh", _CS + "ep_internal.cuh"],
    "combine_nvfp4": [_CS + "combine_wire.cu", _CS + "combine_device.cuh", _CS + "ep_internal.cuh"],
    "layout": [_CS + "layout.cu", _CS + "layout_device.cuh", _CS + "ep_internal.cuh"],
    "layout_dispatch": [_CS + "fused.cu", _CS + "dispatch_device.cuh", _CS + "layout_device.cuh",
                        _CS + "ep_internal.cuh"],
    # two-level: hop 1 runs the dispatch kernels, hop 2 the forwarding kernel;
    # combine = node partials + cross-node sum (traffic of the pair)
    "dispatch_two_level": [_CS + "dispatch.cu", _CS + "dispatch_device.cuh", _CS + "two_level.cu",
                           _CS + "ep_internal.cuh", _CS + "vec8.cuh"],
    "combine_two_level": [_CS + "two_level.cu", _CS + "dispatch_device.cuh", _CS + "ep_internal.cuh",
                          _CS + "vec8.cuh"],
    # the identity expert of an FP8 payload and the expert-side wire cast
    "expert": [_CS + "dequant.cu", _CS + "dispatch_device.cuh", _CS + "ep_internal.cuh", _CS + "vec8.cuh"],
    "wire_mxfp8": [_CS + "wire.cu", _CS + "dispatch_device.cuh", _CS + "ep_internal.cuh", _CS + "vec8.cuh"],
    "wire_nvfp4": [_CS + "wire.cu", _CS + "dispatch_device.cuh", _CS + "ep_internal.cuh", _CS + "vec8.cuh"],
}


def traffic_key(dom, args):
    """Profile key of the dominant kernel (or kernel pair) of this run."""
    if getattr(args, "two_level", False) and dom in ("dispatch", "combine"):
        return f"{dom}_two_level"
    if dom in ("combine", "wire") and getattr(args, "combine_fmt", "bf16") != "bf16":
        return f"{dom}_{args.combine_fmt}"
    return dom


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0, t1):
        samples = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                samples.append((ts + frac, float(parts[1]), float(parts[2]), parts[4:8]))
            except Exception:
                continue
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [s for s in samples if t0 - 0.05 <= s[0] <= t1 + 0.05]
        note = "during timed region"
        if not inside:   # region shorter than the sampling period: nearest samples
            inside = sorted(samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))[:3]
            note = "nearest samples (timed region shorter than the sampling period)"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i, v in enumerate(s[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([s[1] for s in inside])), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside), "window": note}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample_step(x, idx, w, wl, t0, t1, lay=None):
    """One oracle step on tokens [t0, t1): layout of the whole problem (slots
    depend on every earlier token), RDMA counts, dispatch and combine of the
    sampled tokens."""
    import oracle
    R, G, E = wl.ranks, wl.gpus_per_node, wl.experts
    lay, _ = oracle.layout(idx, E, R, G)
    oracle.rdma_token_count(idx, E, R, G)
    rows = oracle.recv_rows(x.shape[0], E, R, wl.layout)
    recv = np.zeros((rows, x.shape[1]), np.uint16)
    oracle.dispatch(x, idx, lay, E, R, G, layout_name=wl.layout, recv=recv, t0=t0, t1=t1)
    oracle.combine(recv, idx, w, lay, E, R, G, layout_name=wl.layout, t0=t0, t1=t1)


def cpu_baseline(x, idx, w, wl, budget_s=12.0):
    """Oracle throughput: source-rank segments one after another until the
    budget is spent or the whole workload is done (single thread)."""
    Tr = wl.tokens_per_rank
    done, t_start = 0, time.perf_counter()
    for s in range(wl.ranks):
        oracle_sample_step(x, idx, w, wl, s * Tr, (s + 1) * Tr)
        done += Tr
        if time.perf_counter() - t_start > budget_s:
            break
    el = time.perf_counter() - t_start
    return {"value": done / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done // Tr} of {wl.ranks} source-rank segments ({done} of {wl.tokens} tokens), one "
                      f"oracle step each (layout + RDMA count over all tokens, dispatch + combine of the "
                      f"segment), single thread, {el:.1f} s"}


def _cpu_worker(wl, segs, budget_s, barrier, queue):
    """One process of the all-cores oracle baseline: regenerates the seeded
    inputs, waits for the others, then runs oracle steps on its source-rank
    segments until the budget is spent."""
    x, idx, w = inputs.make_workload_inputs(wl)
    Tr = wl.tokens_per_rank
    barrier.wait()
    t0 = time.monotonic()
    done, i = 0, 0
    while True:
        s = segs[i % len(segs)]
        oracle_sample_step(x, idx, w, wl, s * Tr, (s + 1) * Tr)
        done += Tr
        i += 1
        if time.monotonic() - t0 > budget_s:
            break
    queue.put((done, t0, time.monotonic()))


def cpu_baseline_all_cores(wl, budget_s=8.0):
    """The oracle on every host core: one spawned process per core, each
    repeating oracle steps on source-rank segments (independent work, the
    oracle unchanged) for the budget; value = all tokens / wall time."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    P = max(1, min(os.cpu_count() or 1, 64))
    barrier, queue = ctx.Barrier(P), ctx.Queue()
    procs = [ctx.Process(target=_cpu_worker, args=(wl, [p % wl.ranks], budget_s, barrier, queue))
             for p in range(P)]
    for pr in procs:
        pr.start()
    try:
        res = [queue.get(timeout=budget_s + 300) for _ in range(P)]
    except Exception as e:   # a worker died: no all-cores figure
        for pr in procs:
            pr.kill()
        return {"value": None, "unit": "tokens/s", "cores": P, "kind": "oracle", "error": repr(e)}
    for pr in procs:
        pr.join()
    done = sum(r[0] for r in res)
    wall = max(r[2] for r in res) - min(r[1] for r in res)
    return {"value": done / wall, "unit": "tokens/s", "cores": P, "kind": "oracle",
            "sample": f"{P} processes, each repeating oracle steps (layout + RDMA count over all {wl.tokens} tokens, "
                      f"dispatch + combine of one source-rank segment of {wl.tokens_per_rank} tokens) for "
                      f"{budget_s:.0f} s; {done} tokens in {wall:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = inputs.WORKLOADS[WORKLOAD]
    x, idx, w = inputs.make_workload_inputs(wl)
    Tr = wl.tokens_per_rank
    sample = min(Tr, 512)      # tokens per step: one bounded slice of source rank 0
    for _ in range(args.warmup):
        oracle_sample_step(x, idx, w, wl, 0, sample)
    t0 = time.perf_counter()
    for i in range(args.steps):
        s = (i % wl.ranks) * Tr
        oracle_sample_step(x, idx, w, wl, s, s + sample)
    el = time.perf_counter() - t0
    val = sample * args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(wl),
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: oracle layout + RDMA count over all {wl.tokens} tokens, "
                                       f"dispatch + combine of {sample} tokens of one source rank, single thread"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def bench_workload(args):
    """The prefill workload (or, with --workload, another one), optionally
    with fewer tokens per rank for profiling a smaller case of the same
    kernels."""
    import dataclasses
    wl = inputs.WORKLOADS[args.workload]
    if args.tokens_per_rank and args.tokens_per_rank != wl.tokens_per_rank:
        wl = dataclasses.replace(wl, name=f"{wl.name.rsplit('_t', 1)[0]}_t{args.tokens_per_rank}",
                                 tokens_per_rank=args.tokens_per_rank)
    return wl


def _routing_label(wl):
    if wl.routing == "group_limited":
        return (f"group-limited: |N(0,1)|+1 scores, top {min(wl.nodes, 4)} of {wl.nodes} node groups by group max, "
                f"then top-{wl.topk}; softmax weights")
    if wl.zipf_s:
        return (f"top-{wl.topk} of N(0,1) logits + log p_e, p_e ~ 1/(e+1)^{wl.zipf_s:g} (Zipf expert popularity), "
                "softmax weights")
    return f"top-{wl.topk} of N(0,1) logits, softmax weights (uniform expert popularity)"


def _config(wl, args=None):
    extra = {}
    if args is not None and getattr(args, "combine_fmt", "bf16") != "bf16":
        extra["combine_wire_format"] = args.combine_fmt
    if args is not None and getattr(args, "fused", False):
        extra["layout_dispatch"] = "fused (one launch)"
    if args is not None and getattr(args, "two_level", False):
        extra["dispatch_combine"] = "two-level (node forwarding)"
    return {**extra, "workload": wl.name, "ranks": wl.ranks, "tokens_per_rank": wl.tokens_per_rank, "tokens": wl.tokens,
            "hidden": wl.hidden, "experts": wl.experts, "topk": wl.topk, "gpus_per_node": wl.gpus_per_node,
            "layout": wl.layout, "dispatch_dtype": wl.dtype,
            "routing": _routing_label(wl),
            "l2": f"inputs larger than L2 (x {wl.tokens * wl.hidden * 2 / 1e6:.0f} MB, receive buffer "
                  f"{wl.ranks * wl.tokens * wl.hidden * 2 / 1e9:.2f} GB)", "parallelism": "replicas",
            **({"zipf_s": wl.zipf_s} if wl.zipf_s else {})}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def hold_gpu(us: float):
    """Enqueues a spin of about `us` microseconds on the current stream, so
    that the host has enqueued the launches that follow before the GPU
    reaches them: the events around small kernels then time the device, not
    the host's launch rate.  Runs before a timed region starts, never inside
    one."""
    import torch
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None and us > 0:
        sleep(int(us * 2100))   # cycles at up to 2.1 GHz

def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from combine_ep_layout_05_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    barrier(world)
    from combine_ep_layout_05_gb300.pipeline import EpPipeline

    wl = bench_workload(args)
    T, H, k, E, R, G = wl.tokens, wl.hidden, wl.topk, wl.experts, wl.ranks, wl.gpus_per_node
    x_h, idx_h, w_h = inputs.make_workload_inputs(wl)
    dev = torch.device("cuda", local)
    x = torch.from_numpy(x_h.view(np.int16)).to(dev).view(torch.bfloat16)
    idx = torch.from_numpy(idx_h).to(dev)
    w = torch.from_numpy(w_h).to(dev)
    pipe = EpPipeline(T, H, k, E, R, G, wl.layout, wl.dtype, dev, fused=args.fused, combine_fmt=args.combine_fmt,
                      two_level=args.two_level)
    args.fused = pipe.fused
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(3, args.warmup)):
        pipe.step(x, idx, w, stream)
    torch.cuda.synchronize()
    # live receive rows: one per (token, rank) in the rank-major layout, one
    # per (token, expert) in the expert-major layout
    D = int((pipe.buf.recv_tokens_per_rank if wl.layout == "rank_major" else pipe.buf.tokens_per_expert)
            .sum().item())
    A = int(pipe.buf.algo_per_rank.sum().item())
    P = int(pipe.buf.physical_exact_per_rank.sum().item())
    st = int(pipe.status.item())
    if st:
        raise RuntimeError(f"device status {st} on the benchmark workload")

    # ---- timed region: inputs resident in HBM -------------------------------
    names = ["layout_dispatch", "combine"] if args.fused else ["layout", "dispatch", "combine"]
    # the identity expert of an FP8 payload and the expert-side wire cast are
    # steps of their own
    names += (["expert"] if wl.dtype != "bf16" else []) + (["wire"] if args.combine_fmt != "bf16" else [])
    evs = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] for n in names}
    # the K timed steps run as `repeats` back-to-back groups, each bracketed
    # by a barrier and a synchronize; value uses their total time, the
    # groups' spread says how repeatable it is
    reps = max(1, min(args.repeats, args.steps))
    groups = [args.steps // reps + (1 if g < args.steps % reps else 0) for g in range(reps)]
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.2 if sampler else 0)
    group_ms = []
    i = 0
    wall0 = time.time()
    for n_g in groups:
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        hold_gpu(40.0 * n_g * pipe.kernels_per_step())
        start.record(stream)
        for _ in range(n_g):
            if args.fused:
                e = evs["layout_dispatch"][i]; e[0].record(stream); pipe.layout_dispatch_step(x, idx, stream)
                e[1].record(stream)
            else:
                e = evs["layout"][i]; e[0].record(stream); pipe.layout_step(idx, stream); e[1].record(stream)
                e = evs["dispatch"][i]; e[0].record(stream); pipe.dispatch_step(x, idx, stream); e[1].record(stream)
            if "expert" in evs:
                e = evs["expert"][i]; e[0].record(stream); pipe.expert_step(idx, stream); e[1].record(stream)
            if "wire" in evs:
                e = evs["wire"][i]; e[0].record(stream); pipe.wire_step(idx, stream); e[1].record(stream)
            e = evs["combine"][i]; e[0].record(stream); pipe.combine_step(idx, w, stream); e[1].record(stream)
            i += 1
        stop.record(stream)
        torch.cuda.synchronize()
        group_ms.append(start.elapsed_time(stop))
    wall1 = time.time()
    barrier(world)
    el_ms = float(sum(group_ms))
    el_ms_max = reduce_max(el_ms, world, dev)
    per_step_groups = [gm / n_g for gm, n_g in zip(group_ms, groups)]
    per_kernel = {n: float(np.mean([a.elapsed_time(b) for a, b in evs[n]])) for n in names}

    # ---- the same step replayed from a CUDA graph ---------------------------
    graph_ms = []
    if args.graph_steps > 0:
        gsteps = args.graph_steps
        graph = pipe.capture(x, idx, w, steps=gsteps)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        for _ in range(reps):
            a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            hold_gpu(50.0)
            a_ev.record()
            graph.replay()
            b_ev.record()
            torch.cuda.synchronize()
            graph_ms.append(a_ev.elapsed_time(b_ev) / gsteps)
        del graph
        st = int(pipe.status.item())
        if st:
            raise RuntimeError(f"device status {st} in the graph replay")

    # ---- end to end: pinned host buffers through the C ABI ------------------
    # HostBatchRunner overlaps each step's host->device input copies and the
    # previous step's device->host output copy with the kernels
    from combine_ep_layout_05_gb300.pipeline import HostBatchRunner
    runner = HostBatchRunner(pipe, 2, dev)
    x_pin = torch.from_numpy(x_h.view(np.int16)).pin_memory()
    idx_pin = torch.from_numpy(idx_h).pin_memory()
    w_pin = torch.from_numpy(w_h).pin_memory()
    outs_pin = [torch.empty((T, H), dtype=torch.int16).pin_memory() for _ in range(2)]
    batches = lambda n: ((x_pin, idx_pin, w_pin, outs_pin[i % 2]) for i in range(n))
    runner.run(batches(max(3, args.warmup)))
    torch.cuda.synchronize()
    barrier(world)
    s2, t2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(runner.s_in)
    runner.run(batches(args.steps))
    runner.s_out.wait_stream(runner.s_in)
    runner.s_out.wait_stream(runner.s_comp)
    t2.record(runner.s_out)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(s2.elapsed_time(t2), world, dev)
    assert torch.equal(outs_pin[(args.steps - 1) % 2], pipe.out.view(torch.int16).cpu()), \
        "end-to-end output differs from the device-resident step"

    if sampler:
        sampler.stop()
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    ms_step = el_ms_max / args.steps
    value = world * T / (ms_step / 1e3)
    byt = algorithmic_bytes(T, H, k, R, E, R // G, D, wl.dtype, args.combine_fmt, A if args.two_level else None)
    step_bytes = sum(byt.values())
    peak, peak_src = measured_peak()
    if args.fused:
        byt["layout_dispatch"] = byt.pop("layout") + byt.pop("dispatch")
    dom = max(per_kernel, key=lambda n: per_kernel[n])
    tkey = traffic_key(dom, args)
    dc_bytes = sum(v for n, v in byt.items() if n in ("dispatch", "layout_dispatch", "combine"))
    ach = byt[dom] / (per_kernel[dom] / 1e3) / 1e9
    dc_ms = sum(v for n, v in per_kernel.items() if n in ("dispatch", "layout_dispatch", "combine"))
    clocks = sampler.summary(wall0, wall1) if sampler else {}
    # the dispatch against the bound for its own 16:84 read:write mix (the
    # copy peak above is a 50:50 stream)
    same_mix = None
    smp = same_mix_peak(wl.name) if (dom in ("dispatch", "layout_dispatch") and wl.dtype == "bf16"
                                     and not args.two_level) else None
    if smp:
        same_mix = {"kernel": dom, "achieved": ach, "peak": smp[0], "unit": "GB/s", "frac": ach / smp[0],
                    "peak_source": smp[1]}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded numpy: x ~ N(0,1) bf16, routing top-8)",
        "config": _config(wl, args),
        "effective_hbm_gbs": step_bytes / (ms_step / 1e3) / 1e9,
        "effective_hbm_frac": step_bytes / (ms_step / 1e3) / 1e9 / peak,
        "dispatch_combine_tokens_per_s": T / (dc_ms / 1e3),
        "dispatch_combine_hbm_gbs": dc_bytes / (dc_ms / 1e3) / 1e9,
        "kernel_ms": per_kernel,
        "dispatched_rows": D,
        # the pages' fabric accounting: inter-node rows (algo incl. the local
        # node, physical without it, and the page's formula) and bytes/s
        "rdma": {"algo_tokens": A, "physical_exact_tokens": P,
                 "physical_formula_tokens": A * (R // G - 1) / (R // G),
                 "algo_bytes_per_s": A * H * 2 / (dc_ms / 1e3), "nvl_recv_bytes_per_s": D * H * 2 / (dc_ms / 1e3)},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": peak, "unit": "GB/s",
                     "frac": ach / peak, "peak_source": f"{peak_src} hbm_gbs",
                     "algorithmic_bytes_per_launch": byt[dom],
                     "traffic": (profile_traffic(tkey, KERNEL_SOURCES[tkey], wl.name)
                                 if tkey in KERNEL_SOURCES else None),
                     "traffic_profile": f"profiles/{tkey}_{wl.name}.md"},
        "repeats": {"n": reps, "steps_each": groups,
                    "ms_per_step_median": float(np.median(per_step_groups)),
                    "ms_per_step_min": float(min(per_step_groups)), "ms_per_step_max": float(max(per_step_groups)),
                    "spread_pct": 100.0 * (max(per_step_groups) - min(per_step_groups)) / float(np.median(per_step_groups))},
        "clocks": clocks,
        "gpu_launches": args.steps * pipe.kernels_per_step(),
        "e2e": {"value": world * T / (e2e_ms / args.steps / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": x_h.nbytes + idx_h.nbytes + w_h.nbytes, "d2h_bytes_per_step": T * H * 2,
                "ms_per_step": e2e_ms / args.steps},
    }
    if same_mix:
        line["roofline"]["same_mix"] = same_mix
    if graph_ms:
        gmed = float(np.median(graph_ms))
        line["graph"] = {"steps_per_graph": args.graph_steps, "replays": len(graph_ms), "ms_per_step_median": gmed,
                         "ms_per_step_min": float(min(graph_ms)), "ms_per_step_max": float(max(graph_ms)),
                         "tokens_per_s": world * T / (gmed / 1e3)}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x_h, idx_h, w_h, wl)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(wl)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_sweep(args):
    """Tokens-per-rank sweep (8 ranks, rank-major): one JSON line per point on
    stdout, each a full step (layout, RDMA count, dispatch, identity expert,
    combine) timed with CUDA events; L2 flushed between steps when the
    point's working set fits in L2."""
    import torch
    from combine_ep_layout_05_gb300 import build
    build.build()
    from combine_ep_layout_05_gb300.pipeline import EpPipeline
    dev = torch.device("cuda", 0)
    peak, peak_src = measured_peak()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)   # 512 MB > L2
    points = inputs.sweep_workloads(args.sweep_hidden, args.sweep_experts, args.sweep_dtype)
    if args.sweep_tokens:
        keep = {int(v) for v in args.sweep_tokens.split(",")}
        points = [wl for wl in points if wl.tokens_per_rank in keep]
    for wl in points:
        T, H, k, E, R, G = wl.tokens, wl.hidden, wl.topk, wl.experts, wl.ranks, wl.gpus_per_node
        x_h, idx_h, w_h = inputs.make_workload_inputs(wl)
        x = torch.from_numpy(x_h.view(np.int16)).to(dev).view(torch.bfloat16)
        idx = torch.from_numpy(idx_h).to(dev)
        w = torch.from_numpy(w_h).to(dev)
        pipe = EpPipeline(T, H, k, E, R, G, wl.layout, wl.dtype, dev, fused=args.fused,
                          combine_fmt=args.combine_fmt)
        for _ in range(3):
            pipe.step(x, idx, w)
        torch.cuda.synchronize()
        D = int(pipe.buf.recv_tokens_per_rank.sum().item())
        small = (x_h.nbytes * 2 + D * H * 2) < 256e6
        times, dc, parts = [], [], {n: [] for n in ("layout", "dispatch", "expert", "combine")}
        for _ in range(args.steps):
            if small:
                flush.fill_(1)
            hold_gpu(40.0 * pipe.kernels_per_step())
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            ev[0].record()
            if pipe.fused:
                ev[1].record()
                pipe.layout_dispatch_step(x, idx)
            else:
                pipe.layout_step(idx)
                ev[1].record()
                pipe.dispatch_step(x, idx)
            ev[2].record()
            pipe.expert_step(idx)
            pipe.wire_step(idx)
            ev[3].record()
            pipe.combine_step(idx, w)
            ev[4].record()
            torch.cuda.synchronize()
            times.append(ev[0].elapsed_time(ev[4]))
            dc.append(ev[1].elapsed_time(ev[4]) - ev[2].elapsed_time(ev[3]))
            for i, n in enumerate(("layout", "dispatch", "expert", "combine")):
                parts[n].append(ev[i].elapsed_time(ev[i + 1]))
        ms = float(np.median(times))
        # the same step replayed from a CUDA graph (one launch per step)
        graph = pipe.capture(x, idx, w)
        gt = []
        for _ in range(args.steps):
            if small:
                flush.fill_(1)
            hold_gpu(30.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            torch.cuda.synchronize()
            gt.append(a.elapsed_time(b))
        gms = float(np.median(gt))
        del graph
        byt = algorithmic_bytes(T, H, k, R, E, R // G, D, wl.dtype, args.combine_fmt)
        tot = sum(byt.values())
        print(json.dumps({"workload": wl.name, "tokens_per_rank": wl.tokens_per_rank, "tokens": T, "hidden": H,
                          "experts": E, "dtype": wl.dtype, "combine_fmt": args.combine_fmt,
                          "fused": pipe.fused, "dispatched_rows": D, "ms_per_step": ms,
                          "tokens_per_s": T / (ms / 1e3),
                          "dispatch_combine_tokens_per_s": T / (float(np.median(dc)) / 1e3),
                          "effective_hbm_gbs": tot / (ms / 1e3) / 1e9,
                          "hbm_frac": tot / (ms / 1e3) / 1e9 / peak, "peak_source": peak_src,
                          "kernel_us": {n: 1e3 * float(np.median(v)) for n, v in parts.items()},
                          "ms_p10": float(np.percentile(times, 10)), "ms_p90": float(np.percentile(times, 90)),
                          "graph_ms_per_step": gms, "graph_tokens_per_s": T / (gms / 1e3),
                          "graph_ms_p10": float(np.percentile(gt, 10)), "graph_ms_p90": float(np.percentile(gt, 90)),
                          "bytes": byt, "l2_flushed": small}), flush=True)
        del pipe, x, idx, w
        torch.cuda.empty_cache()
    return 0


PROBE_SRC = os.path.join(ROOT, "combine_ep_layout_05_gb300", "probe", "hbm_mix.cu")
PROBE_BIN = os.path.join(ROOT, "combine_ep_layout_05_gb300", "probe", "hbm_mix")


def run_mix_bound():
    """Builds (if needed) and runs the HBM same-mix probe: the bandwidth
    plain streaming kernels reach for the dispatch's read:write mix (each
    token row read once, written to its ~5.3 destinations) on this GPU;
    prints its JSON line."""
    if not os.path.exists(PROBE_BIN) or os.path.getmtime(PROBE_BIN) < os.path.getmtime(PROBE_SRC):
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                               PROBE_SRC, "-o", PROBE_BIN])
    out = subprocess.run([PROBE_BIN], check=True, capture_output=True, text=True).stdout
    print(out.strip().splitlines()[-1], flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--repeats", type=int, default=5,
                    help="the timed steps run as this many groups; their spread is reported")
    ap.add_argument("--graph-steps", type=int, default=10,
                    help="steps captured in one CUDA graph for the replayed-step figure (0: skip)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fused", dest="fused", action="store_const", const=True, default=None,
                    help="layout + dispatch as one launch (ep_layout_dispatch); default: where it is the faster")
    ap.add_argument("--unfused", dest="fused", action="store_const", const=False,
                    help="layout and dispatch as two calls (ep_layout, ep_dispatch)")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(inputs.WORKLOADS),
                    help="workload (the default is the headline one)")
    ap.add_argument("--two-level", action="store_true",
                    help="node-forwarding dispatch and combine (ep_dispatch_two_level / ep_combine_two_level)")
    ap.add_argument("--combine-fmt", default="bf16", choices=["bf16", "mxfp8", "nvfp4"],
                    help="combine wire format (expert-side cast + decode-on-the-fly combine)")
    ap.add_argument("--tokens-per-rank", type=int, default=0,
                    help="profiling only: the prefill shape with this many tokens per rank")
    ap.add_argument("--sweep", action="store_true", help="tokens/rank sweep, one JSON line per point")
    ap.add_argument("--mix-bound", action="store_true",
                    help="measure the HBM bound for the dispatch's 16:84 read:write mix (probe program)")
    ap.add_argument("--sweep-hidden", type=int, default=7168)
    ap.add_argument("--sweep-experts", type=int, default=256)
    ap.add_argument("--sweep-dtype", default="bf16", choices=["bf16", "fp8_e4m3"])
    ap.add_argument("--sweep-tokens", default="", help="comma-separated tokens/rank points (default: all)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.mix_bound:
        return run_mix_bound()
    if args.sweep:
        return run_sweep(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
