"""Benchmark of one decode step (partition pass + reduce) of paged-KV GQA decode attention.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  The headline workload is the largest configuration, the long
context (4 sequences of 32 768 tokens, 8 KV heads, QG 8, 32-token blocks, 32 partitions of 1280
tokens); the line's "other_workloads" list times every other configuration the same way in the
same run (the fp8 one among them).  A step is one pass of the whole hot path over one batch:
pda_decode (the partition kernel) then pda_reduce, both through the C ABI, inputs resident in
HBM.  Between timed steps, outside the timed events, L2 is flushed: a 512 MiB write, then a
256 MiB read of another buffer, so that the step starts with an L2 holding none of its inputs
and no dirty lines (otherwise the timed kernels would also pay for writing the flush back).
  value        (sequence, KV head) units per second, all ranks
  e2e          the same metric through the public API with host buffers: H2D of the step's
               query, block table and context lengths from pinned memory, the two launches,
               D2H of the bf16 output; the KV cache is device-resident state
  roofline     the partition kernel: algorithmic bytes per launch / its CUDA-event time,
               against the measured copy bandwidth of the GB300 (MEASURED_PEAKS.json)
  cpu_baseline the fp64 CPU oracle on the host cores, on a bounded sample of the same step
Multi-GPU: replicas only (each rank runs the whole workload; no collective in the step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_gqa_block_gb300 import workloads as wl   # noqa: E402

# the headline: the largest configuration (the long-context one, 537 MB of KV per step)
DEFAULT_WORKLOAD = "b4_hk8_qg8_bs32_ctx32768_g5p32"
METRIC = "decode seq-head-steps/s and KV-read HBM GB/s (fraction of ~8 TB/s), 1 GB300"
UNIT = "seq-head-steps/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
L2_CLEAN_READ_BYTES = 256 << 20
L2_BYTES = 129e6        # GB300 L2: a step whose KV reads exceed it gets no reuse from one step to the next
# the files that make up the partition kernel (its ncu counters go stale when one changes)
PARTITION_KERNEL_SOURCES = ("pda_decode.cuh", "pda_group.cuh", "pda_rows.cuh", "pda_merge.cuh", "pda_ptx.cuh", "pda_launch.cuh",
                            "pda_internal.h", "pda_decode_bf16.cu", "pda_decode_fp8.cu", "pda_decode_tq4.cu",
                            "pda_api.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=wl.WORKLOAD_ORDER)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="two", choices=["fused", "two"],
                    help="fused: pda_decode_fused (one launch); two: pda_decode then pda_reduce")
    ap.add_argument("--graph", action="store_true", help="replay each step from a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--variant", type=int, default=0, choices=[0, 1, 2, 3],
                    help="partition-kernel layout for --workload: 0 automatic, 1 head warps, 2 head groups (fp8), "
                         "3 row halves (bf16, QG 16)")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="time only --workload (by default the other configurations are timed too)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(dist, values, device="cpu"):
    """Replicas: every rank times its own copy of the step and the slowest rank sets the time.
    Returns the element-wise maximum of `values` over all ranks (the values themselves when
    there is no process group)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def replica_throughput(world: int, units_per_rank: int, seconds_per_step: float) -> float:
    """Units processed per second by all ranks together (each rank runs the whole step)."""
    return world * units_per_rank / seconds_per_step


KV_NAMES = {wl.KV_BF16: "bf16", wl.KV_FP8_E4M3: "fp8_e4m3", wl.KV_TQ4: "tq4"}


def kv_bytes_per_token_head(w: wl.Workload) -> int:
    """K and V bytes of one token of one KV head, metadata fields included (fp8: two fp32
    scales; TQ4: three fp16 fields)."""
    return w.token_head_bytes + w.meta_region_bytes // (w.num_kv_heads * w.kv_block_size)


def algorithmic_bytes(w: wl.Workload, ctx: np.ndarray, W: int) -> dict:
    """Bytes the step must move at minimum (per step)."""
    Hk, QG, D = w.num_kv_heads, w.query_group_size, w.head_dim
    tok = int(ctx.sum())
    kv = tok * Hk * kv_bytes_per_token_head(w)
    nvalid = int(np.sum(-(-ctx.astype(np.int64) // W)))
    q = w.num_seqs * Hk * QG * D * 2
    bt = int(np.sum(-(-ctx.astype(np.int64) // w.kv_block_size))) * 4
    partials = nvalid * Hk * QG * (D * 4 + 8)
    out = w.num_seqs * Hk * QG * D * 2
    return {"kv": kv, "decode": kv + q + bt + 4 * w.num_seqs + partials, "reduce": partials + out,
            "tokens": tok, "units": w.num_seqs * Hk}


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_gqa_block_gb300", "csrc")
    for f in PARTITION_KERNEL_SOURCES:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM traffic per launch of the partition kernel from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        d = json.load(open(path))
    except Exception:
        return None
    e = d.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.samples = []
        if self.proc is None:
            return
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                try:
                    self.samples.append({"sm": float(parts[0]), "max": float(parts[1]), "power": float(parts[2]),
                                         "hw_slowdown": parts[4], "hw_thermal": parts[5], "sw_thermal": parts[6],
                                         "sw_power_cap": parts[7]})
                except ValueError:
                    pass

    def summary(self):
        s = getattr(self, "samples", [])
        if not s:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm_max = max(x["max"] for x in s)
        load = [x for x in s if x["power"] > 0.25 * max(y["power"] for y in s)] or s
        reasons = set()
        for x in s:
            for k in ("hw_slowdown", "hw_thermal", "sw_thermal", "sw_power_cap"):
                if x[k].lower() == "active":
                    reasons.add(k)
        return {"sm_mhz": statistics.median(x["sm"] for x in load), "sm_max_mhz": sm_max,
                "reasons": sorted(reasons), "samples": len(s)}


# ------------------------------------------------------------------------------------ oracle leg
def oracle_units_per_s(inp: wl.Inputs, budget_s: float, rng_seed: int = 0, threads_cap: int | None = None):
    """The fp64 oracle as it stands, on the host cores, on a random sample of (sequence, KV head)
    units of the step sized to about budget_s seconds (whole passes over the step's units when the
    step is smaller than that).  Returns (units/s, threads, description)."""
    import oracle
    from tests import oracle_helpers as oh
    oracle.build()
    w = inp.workload
    rng = np.random.default_rng(rng_seed)
    order = rng.permutation(w.num_seqs * w.num_kv_heads)
    cores = threads_cap or os.cpu_count() or 1
    n = min(len(order), cores)
    t0 = time.perf_counter()
    r = oh.run_oracle(inp, units=order[:n], threads=cores)
    dt = time.perf_counter() - t0
    done, threads, passes = n, r["threads"], 0
    while dt < budget_s:
        if done < len(order):            # first pass: the rest of the units, sized to the budget
            more = int(min(len(order) - done, max(1, done * (budget_s - dt) / max(dt, 1e-3))))
            chunk = order[done:done + more]
        else:                            # the whole step again
            chunk = order
            passes += 1
        t1 = time.perf_counter()
        r = oh.run_oracle(inp, units=chunk, threads=cores)
        dt += time.perf_counter() - t1
        done += len(chunk)
        threads = max(threads, r["threads"])
    what = (f"{done} units: the step's {len(order)} (sequence, KV head) units {passes + 1} times" if passes
            else f"{done} of {len(order)} (sequence, KV head) units drawn at random")
    return done / dt, threads, f"{what}, {dt:.1f} s"


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = wl.WORKLOADS[args.workload]
    inp = wl.generate(w)
    import oracle
    from tests import oracle_helpers as oh
    oracle.build()
    cores = os.cpu_count() or 1
    order = np.random.default_rng(0).permutation(w.num_seqs * w.num_kv_heads)
    # size each step so that warmup + steps stay within ~2 minutes
    t0 = time.perf_counter()
    oh.run_oracle(inp, units=order[:cores], threads=cores)
    per_batch = time.perf_counter() - t0
    per_step_budget = max(0.002, 120.0 / max(1, args.steps + args.warmup))
    n = max(1, min(len(order), int(cores * per_step_budget / max(per_batch, 1e-6))))
    times, threads = [], 0
    for i in range(args.warmup + args.steps):
        units = np.roll(order, -i * n)[:n]
        t = time.perf_counter()
        r = oh.run_oracle(inp, units=units, threads=cores)
        dt = time.perf_counter() - t
        threads = max(threads, r["threads"])
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = n * len(times) / total
    sample = f"{n} of {len(order)} (sequence, KV head) units per step, fp64, {threads} threads"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "global_batch": w.num_seqs, "num_kv_heads": w.num_kv_heads,
                   "query_group_size": w.query_group_size, "kv_dtype": KV_NAMES[w.kv_dtype]},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ------------------------------------------------------------------------------------ our leg
class _Step:
    """One workload resident on the device: inputs, plan, workspace, and the calls of one step."""

    def __init__(self, pda, w, inp, dev, stream, path, variant=0):
        import torch
        self.w, self.inp, self.path, self.stream, self.pda = w, inp, path, stream, pda
        self.p = pda.plan(w.num_seqs, w.num_kv_heads, w.query_group_size, w.kv_block_size, w.max_blocks_per_seq,
                          w.tile_groups_per_partition, w.max_partitions, w.kv_dtype, w.softmax_scale,
                          kernel_variant=variant)
        # the step's per-call inputs (query, block table, context lengths) live in one device buffer,
        # so that the end-to-end loop moves them from host memory with a single copy
        parts = [inp.query.view(np.uint8).reshape(-1), inp.block_table.view(np.uint8).reshape(-1),
                 inp.context_lens.view(np.uint8).reshape(-1)]
        offs, total = [], 0
        for x in parts:
            offs.append(total)
            total += (x.size + 255) // 256 * 256
        self.step_in_host = torch.zeros(total, dtype=torch.uint8).pin_memory()
        for x, o in zip(parts, offs):
            self.step_in_host[o:o + x.size] = torch.from_numpy(x)
        self.step_in = self.step_in_host.to(dev)

        def views(buf):
            return (buf[offs[0]:offs[0] + parts[0].size].view(torch.bfloat16).view(inp.query.shape),
                    buf[offs[1]:offs[1] + parts[1].size].view(torch.int32).view(inp.block_table.shape),
                    buf[offs[2]:offs[2] + parts[2].size].view(torch.int32))
        self.q, self.bt, self.ctx = views(self.step_in)
        self.qh, self.bth, self.ctxh = views(self.step_in_host)
        self.cache = torch.from_numpy(inp.cache).to(dev)
        self.tq4 = w.kv_dtype == wl.KV_TQ4
        self.cent = torch.from_numpy(inp.extra["centroids"]).to(dev) if self.tq4 else None
        if self.tq4 and path == "fused":
            raise SystemExit("the fused step does not read TQ4 caches; use --path two")
        self.ws = pda.workspace(self.p, dev)
        self.out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
        self.outh = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.cnt = pda.counters(self.p, dev)
        self.launches_per_step = 1 if path == "fused" else 2
        self.units = w.num_seqs * w.num_kv_heads

    def decode_on(self, qx, btx, ctxx):
        w, ws, pda = self.w, self.ws, self.pda
        if self.tq4:
            pda.decode_tq4(self.p, qx, self.cache, w.num_cache_blocks, self.cent, btx, ctxx, ws["partial_out"],
                           ws["exp_sums"], ws["max_logits"], err_word=self.err, stream=self.stream)
        else:
            pda.decode(self.p, qx, self.cache, w.num_cache_blocks, btx, ctxx, ws["partial_out"], ws["exp_sums"],
                       ws["max_logits"], err_word=self.err, stream=self.stream)

    def step_on(self, qx, btx, ctxx, outx):
        w, ws, pda = self.w, self.ws, self.pda
        if self.path == "fused":
            pda.decode_fused(self.p, qx, self.cache, w.num_cache_blocks, btx, ctxx, ws["partial_out"],
                             ws["exp_sums"], ws["max_logits"], self.cnt, outx, err_word=self.err, stream=self.stream)
        else:
            self.decode_on(qx, btx, ctxx)
            pda.reduce(self.p, ctxx, ws["partial_out"], ws["exp_sums"], ws["max_logits"], outx, err_word=self.err,
                       stream=self.stream)

    def step(self):
        self.step_on(self.q, self.bt, self.ctx, self.out)

    def decode(self):
        self.decode_on(self.q, self.bt, self.ctx)

    def check_err(self):
        if int(self.err.item()) != 0:
            raise RuntimeError(f"{self.w.name}: device error word {int(self.err.item())}")


def event_times(fn, n, flush, stream, before=None):
    """Device time of `fn` on `stream` for n calls (CUDA events on that stream, L2 flushed before
    each call outside the events); seconds."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush()
        a, b = ev[i]
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e-3 for a, b in ev]


def back_to_back_times(fn, n, stream, batches=10):
    """Device time of n calls of `fn` issued back to back on `stream` (CUDA events around each of
    `batches` equal batches, nothing between the calls); seconds per call, one figure per batch."""
    import torch
    if n % batches:   # exactly n calls: one batch unless n divides evenly
        batches = 1
    per = n // batches
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(batches)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        for _ in range(per):
            fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e-3 / per for a, b in ev]


def timing_mode(w, inp, W) -> str:
    """How the steps are timed: back to back when the step's KV reads exceed L2 (no step then finds
    the previous step's KV in L2), else each step alone after an L2 flush."""
    return "back_to_back" if algorithmic_bytes(w, inp.context_lens, W)["kv"] > L2_BYTES else "flushed"


def l2_note(mode, w, inp, W) -> str:
    if mode == "back_to_back":
        kv = algorithmic_bytes(w, inp.context_lens, W)["kv"]
        return (f"inputs larger than L2: {kv / 1e6:.0f} MB of KV per step > {L2_BYTES / 1e6:.0f} MB L2; "
                "steps timed back to back, no flush")
    return "flushed between timed steps (512 MiB write, then 256 MiB read)"


def rates(w, inp, p, mean_step, mean_dec, world, peak, peaks, kernel="pda_partition_kernel"):
    ab = algorithmic_bytes(w, inp.context_lens, p.partition_tokens)
    achieved = ab["decode"] / mean_dec / 1e9
    kv_gbs = ab["kv"] / mean_step / 1e9
    return ab, {
        "kv_read_gbs": kv_gbs * world,
        "kv_read_frac_of_8tbs": kv_gbs / NOMINAL_HBM_GBS,
        "kv_read_frac_of_measured": kv_gbs / peak,
        "decode_ms": mean_dec * 1e3,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": committed_traffic(w.name), "kernel": kernel,
                     "algorithmic_bytes_per_launch": ab["decode"],
                     "peak_source": "measured" if peaks else "fallback"},
    }


def run_ours(args, rank, world, local_rank):
    import torch
    import paged_kv_gqa_block_gb300 as pda
    from paged_kv_gqa_block_gb300 import _build
    _build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = wl.WORKLOADS[args.workload]
    inp = wl.generate(w)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean_buf = torch.zeros(L2_CLEAN_READ_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.zero_()       # evicts everything from L2 ...
        clean_buf.sum()         # ... and leaves it holding clean lines of another buffer
    if args.graph:      # graphs are captured on a non-default stream: run everything on one
        torch.cuda.set_stream(torch.cuda.Stream(dev))
    stream = torch.cuda.current_stream(dev)
    S = _Step(pda, w, inp, dev, stream, args.path, args.variant)
    step = S.step
    mode = timing_mode(w, inp, S.p.partition_tokens)

    for _ in range(args.warmup):
        if mode == "flushed":
            flush()
        step()
    torch.cuda.synchronize()
    if args.graph:      # capture one step; the timed loops replay it
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            S.step()
        torch.cuda.synchronize()

        def step():
            graph.replay()
        for _ in range(3):
            flush()
            step()
        torch.cuda.synchronize()
    S.check_err()

    # ---- device-resident timing on the launching stream (nothing between the two launches of a
    # step, so the reduce can be scheduled while the partition pass drains): the K steps back to
    # back when the step's KV exceeds L2, else events around each step after an L2 flush
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        wall0 = time.perf_counter()
        if mode == "back_to_back":
            t_step = back_to_back_times(step, args.steps, stream)
        else:
            t_step = event_times(step, args.steps, flush, stream)
        wall = time.perf_counter() - wall0
    if dist:
        dist.barrier()
    # the partition kernel alone (roofline of the dominant kernel): each launch after an L2 flush,
    # so its duration includes the cold start of every launch
    dec_steps = max(20, min(args.steps, 500))
    t_dec = event_times(S.decode, dec_steps, flush, stream)
    mean_step, mean_dec = sum(t_step) / len(t_step), sum(t_dec) / len(t_dec)
    med_step, min_step = float(np.median(t_step)), min(t_step)
    flushed = None
    if mode == "back_to_back":   # the same step alone after an L2 flush, for comparison
        t_fl = event_times(step, max(20, min(args.steps, 500)), flush, stream)
        flushed = {"ms_per_step": sum(t_fl) / len(t_fl) * 1e3, "step_ms_median": float(np.median(t_fl)) * 1e3,
                   "how": "each step alone between CUDA events, L2 flushed before it"}
    if dist:
        mean_step, mean_dec = max_over_ranks(dist, [mean_step, mean_dec], dev)

    # ---- end to end through the public API with host buffers.  Reported: the C ABI called with the
    # step's inputs (query, block table, context lengths) and its bf16 output in pinned host
    # memory, which the kernels read and write across the host link.  Beside it: the same step
    # with one explicit copy of the packed inputs in and one of the output out.  The KV cache is
    # device-resident state in both.
    e2e_steps = max(10, min(args.steps, 500))

    def step_with_copies():
        S.step_in.copy_(S.step_in_host, non_blocking=True)
        step()
        S.outh.copy_(S.out, non_blocking=True)

    def step_on_host():
        S.step_on(S.qh, S.bth, S.ctxh, S.outh)
    e2e, e2e_zc = [], []
    if mode == "back_to_back":
        for fn, acc in ((step_with_copies, e2e), (step_on_host, e2e_zc)):
            for _ in range(3):
                fn()
            acc.extend(back_to_back_times(fn, e2e_steps, stream))
    else:
        for fn, acc in ((step_with_copies, e2e), (step_on_host, e2e_zc)):
            for i in range(e2e_steps + 3):
                flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                b.synchronize()
                if i >= 3:
                    acc.append(a.elapsed_time(b) * 1e-3)
    mean_e2e = sum(e2e) / len(e2e)
    mean_e2e_zc = sum(e2e_zc) / len(e2e_zc)
    if dist:
        mean_e2e, mean_e2e_zc = max_over_ranks(dist, [mean_e2e, mean_e2e_zc], dev)
    torch.cuda.synchronize()
    S.check_err()

    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks and peaks.get("hbm_gbs") else FALLBACK_HBM_GBS
    p = S.p
    units = S.units

    # ---- the other configurations, timed the same way in the same run (device-resident inputs;
    # back to back when their KV exceeds L2, else L2 flushed between steps); each is generated,
    # timed and freed in turn
    others = []
    if not args.no_other_workloads:
        del S
        n_other = max(50, min(args.steps, 500))
        for name in wl.WORKLOAD_ORDER:
            if name == w.name:
                continue
            wo = wl.WORKLOADS[name]
            io = wl.generate(wo)
            So = _Step(pda, wo, io, dev, stream, "two")
            mo = timing_mode(wo, io, So.p.partition_tokens)
            for _ in range(max(3, args.warmup)):
                if mo == "flushed":
                    flush()
                So.step()
            torch.cuda.synchronize()
            So.check_err()
            if mo == "back_to_back":
                ts = back_to_back_times(So.step, n_other, stream)
            else:
                ts = event_times(So.step, n_other, flush, stream)
            td = event_times(So.decode, n_other, flush, stream)
            So.check_err()
            ms, md = sum(ts) / len(ts), sum(td) / len(td)
            if dist:
                ms, md = max_over_ranks(dist, [ms, md], dev)
            _, r = rates(wo, io, So.p, ms, md, world, peak, peaks, kernel_name(pda, So.p))
            others.append({"workload": name, "kv_dtype": KV_NAMES[wo.kv_dtype], "steps": n_other,
                           "value": replica_throughput(world, So.units, ms), "unit": UNIT,
                           "ms_per_step": ms * 1e3, "step_ms_median": float(np.median(ts)) * 1e3,
                           "l2": l2_note(mo, wo, io, So.p.partition_tokens), **r})
            del So, io
            torch.cuda.empty_cache()

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    ab, r = rates(w, inp, p, mean_step, mean_dec, world, peak, peaks, kernel_name(pda, p))
    res = {
        "metric": METRIC, "value": replica_throughput(world, units, mean_step), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_step * 1e3,
        "higher_is_better": True, "step_ms_median": med_step * 1e3, "step_ms_min": min_step * 1e3,
        "scaling": "weak", "vs_baseline": None,
        "dtype": KV_NAMES[w.kv_dtype],
        "data": "synthetic",
        "config": {"workload": w.name, "global_batch": world * w.num_seqs, "num_kv_heads": w.num_kv_heads,
                   "query_group_size": w.query_group_size, "kv_block_size": w.kv_block_size,
                   "tile_groups_per_partition": p.resolved_tile_groups, "num_partitions": p.num_partitions,
                   "context_tokens": ab["tokens"], "seq_len_max": int(inp.context_lens.max()),
                   "parallelism": f"replicas{world}", "l2": l2_note(mode, w, inp, p.partition_tokens)},
        "query_head_steps_per_s": replica_throughput(world, units * w.query_group_size, mean_step),
        **r,
        "e2e": {"value": replica_throughput(world, units, mean_e2e_zc), "unit": UNIT,
                "h2d_bytes_per_step": int(inp.query.nbytes + inp.block_table.nbytes + inp.context_lens.nbytes),
                "d2h_bytes_per_step": int(w.num_seqs * w.num_q_heads * w.head_dim * 2),
                "how": "inputs and output in pinned host memory, read and written by the kernels"},
        "e2e_with_copies": {"value": replica_throughput(world, units, mean_e2e), "unit": UNIT,
                            "h2d_bytes_per_step": int(e2e_in_bytes(inp)),
                            "d2h_bytes_per_step": int(w.num_seqs * w.num_q_heads * w.head_dim * 2),
                            "how": "one copy of the packed inputs in, one copy of the output out"},
        "gpu_launches": (1 if args.path == "fused" else 2) * args.steps,
        "kernel_variant": args.variant,
        "step_path": ("pda_decode_fused (one launch)" if args.path == "fused" else "pda_decode + pda_reduce") +
                     (", replayed from a CUDA graph" if args.graph else ""),
        "decode_launches_timed_separately": dec_steps,
        "decode_timing": "each partition-kernel launch alone between CUDA events, L2 flushed before it",
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
    }
    if flushed:
        res["flushed"] = flushed
    if others:
        res["other_workloads"] = others
    if not args.no_cpu_baseline and world >= 1:
        v, threads, sample = oracle_units_per_s(inp, args.cpu_budget_s)
        res["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample}
        v1, _, sample1 = oracle_units_per_s(inp, args.cpu_budget_s / 3, threads_cap=1)
        res["cpu_baseline_1thread"] = {"value": v1, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample1}
    print(json.dumps(res))
    if dist:
        dist.destroy_process_group()


def kernel_name(pda, p) -> str:
    """The partition kernel pda_decode launches for plan p (its roofline is the line's)."""
    v = pda.kernel_variant(p)
    return {pda.VARIANT_HEAD_GROUPS: "pda_group_kernel", pda.VARIANT_ROW_HALVES: "pda_rows_kernel"}.get(
        v, "pda_partition_kernel")


def e2e_in_bytes(inp) -> int:
    """Bytes of the packed per-step inputs copied in by the end-to-end loop (each part padded to 256)."""
    return sum((x.nbytes + 255) // 256 * 256 for x in (inp.query, inp.block_table, inp.context_lens))


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
