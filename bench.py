"""Benchmark of the paged-attention hot path on GB300.

One step is one full ``attn_decode_paged`` call (paged decode kernel plus split
merge) over the Llama-2-7B-shaped batch: bf16, batch 16, 32 query heads = 32
KV heads, head_dim 128, KV lengths U[512, 4096], page 16, 8192-page pool. The
metric is HBM GB/s of algorithmic bytes: each sequence's K and V read once.
The same JSON line carries the causal prefill figure (bf16, batch 8, T 1024,
32 heads, d 128) in TFLOP/s of causal FLOPs.

``python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]``.
With N > 1 it runs one replica per GPU under torchrun (the path shards by sequence
with no exchange); started without torchrun, it starts N ranks itself through
``torch.distributed.run``. Rank 0 prints one JSON line.

The CPU baseline is the fp64 oracle as it stands, timed after the GPU measurements on
every host core (worker processes, one BLAS thread each) and on one core.
"""
from __future__ import annotations

import os

# The CPU baseline (the fp64 oracle) runs one BLAS thread per process, the processes spread
# over the host's cores: pin BLAS threads before numpy loads (spawned workers inherit it).
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import math
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attn HBM GB/s (% of peak); causal prefill attn TFLOP/s (% peak)"
WORKLOAD = ("llama7b_batched_decode: bf16, batch 16, 32 query heads = 32 KV heads, head_dim 128, "
            "kv_len U[512,4096] seeded, page_size 16, 8192-page pool, one query token per sequence")
PREFILL_WORKLOAD = "causal_prefill_llama7b: bf16, batch 8, T 1024, 32/32 heads, head_dim 128, [B,T,H,D]"
# decode workloads: (builder name, description, explicit split count or 0 for automatic)
DECODE_WORKLOADS = {
    "llama7b_batched_decode": ("llama7b_batched_decode", WORKLOAD, 0),
    "long_context_gqa_decode": ("long_context_gqa_decode",
                                "long_context_gqa_decode: bf16, batch 4, 32 query heads over 8 KV heads, "
                                "head_dim 128, kv_len 32768, page_size 16, 8192-page shuffled pool, 32 KV splits",
                                32),
}
FALLBACK_HBM = 6800.0
FALLBACK_BF16 = 1900.0
L2_FLUSH_BYTES = 256 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return FALLBACK_HBM, FALLBACK_BF16, 1700.0, "fallback"


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_attention_28_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key, src_hash, units_now):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this exact source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel_key)
    if not d or d.get("source_hash") != src_hash:
        return None
    return d["dram_bytes_per_launch"] * units_now / d["units"]


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons around the timed region.

    ``mark_start``/``mark_end`` bracket the timed region. The summary uses the
    samples taken inside it, or the nearest sample on each side when the region
    is shorter than the sampling period. ``settle`` keeps the GPU busy until a
    sample exists on the needed side, so that the samples reflect clocks under load.
    """

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def _rows(self):
        import datetime
        rows = []
        if self.path is None:
            return rows
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(p[1]), float(p[2]), p[5:9]))
                except ValueError:
                    continue
        return rows

    def settle(self, busy, after=None, timeout=5.0):
        """Run ``busy()`` until a sample exists (after time ``after`` when given)."""
        if self.proc is None:
            return
        t_end = time.time() + timeout
        while time.time() < t_end:
            rows = self._rows()
            if rows and (after is None or rows[-1][0] > after):
                return
            for _ in range(20):
                busy()
            torch.cuda.synchronize()

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = self._rows()
        inside = [r for r in rows if self.t0 <= r[0] <= self.t1]
        used = inside
        if not used:
            before = [r for r in rows if r[0] < self.t0][-1:]
            after = [r for r in rows if r[0] > self.t1][:1]
            used = before + after
        reasons = set()
        for r in used:
            for n, v in zip(self.NAMES, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        sm = [r[1] for r in used]
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": used[-1][2] if used else None, "reasons": sorted(reasons),
               "samples_in_region": len(inside), "samples_used": len(used)}
        if not inside and used:
            out["note"] = ("the timed region is shorter than the 100 ms sampling period: the nearest "
                           "sample on each side, both taken while the same step ran back to back")
        return out


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def weak_scaling_rate(units_per_step, steps, world, seconds):
    """Whole-job throughput of `world` replicas that each process `units_per_step` per step
    for `steps` steps: every rank's units over the slowest rank's time (max over ranks)."""
    return units_per_step * steps * world / seconds


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle arm

def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def oracle_decode_rate(case, budget_s, workers):
    """Times the fp64 oracle, as it stands, on whole passes over the decode batch (every
    (sequence, KV head) unit) until ``budget_s`` has elapsed, on ``workers`` processes.
    Returns (GB/s of algorithmic bytes, passes, seconds)."""
    from oracle import timing
    r = timing.decode_runner(case.q.double().numpy(), case.k_pages.float().numpy(),
                             case.v_pages.float().numpy(), case.block_table.numpy(),
                             case.kv_lens.numpy(), case.scale, workers)
    try:
        passes, el = timing.time_passes(r, budget_s)
    finally:
        r.close()
    return case.kv_bytes() * passes / el / 1e9, passes, el


def oracle_prefill_rate(case, workers):
    """One timed pass of the fp64 causal-prefill oracle over the whole workload (it builds
    every 1024 x 1024 score matrix), after an untimed one. Returns (TFLOP/s of causal FLOPs,
    seconds)."""
    from oracle import timing
    r = timing.prefill_runner(case.q.float().numpy(), case.k.float().numpy(), case.v.float().numpy(),
                              case.scale, workers)
    try:
        _, el = timing.time_passes(r, 0.0)
    finally:
        r.close()
    return case.causal_flops() / el / 1e12, el


def cpu_baselines(case, budget_s=8.0):
    """The decode oracle on every host core and on one core."""
    cores = host_cores()
    all_rate = oracle_decode_rate(case, budget_s, cores)
    one_rate = oracle_decode_rate(case, budget_s, 1)
    return {"value": all_rate[0], "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{all_rate[1]} whole pass(es) of the fp64 oracle over the full decode batch in "
                      f"{all_rate[2]:.1f} s on {cores} worker processes (one BLAS thread each), after one "
                      "untimed pass",
            "value_1core": one_rate[0],
            "sample_1core": f"{one_rate[1]} pass(es) in {one_rate[2]:.1f} s in one process"}


def other_cpu_baselines(workloads, budget_s=3.0):
    """The fp64 oracle, as it stands, on every host core and on one core, for the three other
    configurations: the single-sequence fp32 decode, the long-context GQA decode and the
    shared-prefix decode. Each leg runs whole passes over the whole workload until
    ``budget_s`` has elapsed, after one untimed pass. GB/s of the same algorithmic bytes as
    the GPU line."""
    from oracle import timing
    cores = host_cores()
    cases = {
        "single_seq_decode_f32": workloads.single_seq_decode_f32(),
        "long_context_gqa_decode": workloads.long_context_gqa_decode(poison=False),
        "cascade_shared_prefix_decode": workloads.cascade_shared_prefix_decode(poison=False),
    }
    res = {}
    for name, c in cases.items():
        def runner(workers):
            if name == "cascade_shared_prefix_decode":
                return timing.cascade_runner(c.q.double().numpy(), c.k_pages.float().numpy(),
                                             c.v_pages.float().numpy(), c.prefix_table.numpy(), c.prefix_len,
                                             c.suffix_table.numpy(), c.suffix_lens.numpy(), c.scale, workers)
            return timing.decode_runner(c.q.double().numpy(), c.k_pages.float().numpy(),
                                        c.v_pages.float().numpy(), c.block_table.numpy(), c.kv_lens.numpy(),
                                        c.scale, workers)
        legs = {}
        for label, workers in (("all", cores), ("one", 1)):
            r = runner(workers)
            try:
                passes, el = timing.time_passes(r, budget_s)
            finally:
                r.close()
            legs[label] = (c.kv_bytes() * passes / el / 1e9, passes, el)
        res[name] = {"value": legs["all"][0], "unit": "GB/s", "cores": cores, "kind": "oracle",
                     "sample": f"{legs['all'][1]} whole pass(es) of the fp64 oracle over the full workload in "
                               f"{legs['all'][2]:.1f} s on {cores} worker processes, after one untimed pass",
                     "value_1core": legs["one"][0],
                     "sample_1core": f"{legs['one'][1]} pass(es) in {legs['one'][2]:.1f} s in one process"}
    return res


def prefill_cpu_baseline(case):
    cores = host_cores()
    tf_all, s_all = oracle_prefill_rate(case, cores)
    tf_one, s_one = oracle_prefill_rate(case, 1)
    return {"value": tf_all, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"one whole pass of the fp64 causal-prefill oracle (full 1024 x 1024 scores per "
                      f"(batch, head), causal FLOPs counted) in {s_all:.2f} s on {cores} worker processes",
            "seconds": s_all, "value_1core": tf_one, "seconds_1core": s_one}


def run_reference(args, rank, world):
    """The oracle timed on the host cores: the reference arm of this benchmark."""
    if rank != 0:
        return
    from paged_kv_attention_28_gb300 import workloads
    case = workloads.llama7b_batched_decode(poison=False)
    cores = host_cores()
    from oracle import timing
    r = timing.decode_runner(case.q.double().numpy(), case.k_pages.float().numpy(),
                             case.v_pages.float().numpy(), case.block_table.numpy(),
                             case.kv_lens.numpy(), case.scale, cores)
    try:
        for _ in range(args.warmup):
            r.one_pass()
        per_step = max(0.5, 20.0 / max(1, args.steps))
        rates, secs = [], []
        for _ in range(args.steps):
            passes, el = 0, 0.0
            t0 = time.perf_counter()
            while passes == 0 or el < per_step:
                r.one_pass()
                passes += 1
                el = time.perf_counter() - t0
            rates.append(case.kv_bytes() * passes / el / 1e9)
            secs.append(el / passes)
    finally:
        r.close()
    value = statistics.mean(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas{world}"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "whole passes of the fp64 oracle over the full decode batch on "
                                   f"{cores} worker processes (~{per_step:.1f} s per step)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def run_ours(args, rank, world, local):
    from paged_kv_attention_28_gb300 import build as _b
    if rank == 0:
        _b.build(quiet=True)
    barrier(world)
    from paged_kv_attention_28_gb300 import binding as B
    from paged_kv_attention_28_gb300 import workloads

    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, bf16_peak, bf16_sust, peak_src = peaks()

    stream = torch.cuda.current_stream(dev)
    if args.only in OTHER_PARTS:
        res = other_workloads(B, workloads, dev, stream, args.steps, hbm_peak, parts=(args.only,))
        if rank == 0:
            print(json.dumps({"metric": METRIC, "only": args.only, "also": res}), flush=True)
        return
    if args.only == "prefill":
        pre = prefill_bench(B, workloads, dev, stream, args, world, bf16_peak, bf16_sust, peak_src)
        if rank == 0:
            print(json.dumps({"metric": METRIC, "only": "prefill", "prefill": pre}), flush=True)
        return
    builder, workload_desc, req_splits = DECODE_WORKLOADS[args.workload]
    case = getattr(workloads, builder)(poison=False)

    # The per-step inputs (q, block table, lengths) and outputs (out, lse) each live in one
    # device buffer, so that the end-to-end loop moves them with one copy each way.
    B_, Hq, D = case.q.shape
    in_specs = [(t.shape, t.dtype) for t in (case.q, case.block_table, case.kv_lens)]
    out_specs = [(case.q.shape, case.q.dtype), ((B_, Hq), torch.float32)]
    d_in, (q, bt, lens) = packed(in_specs, dev)
    h_in, h_in_views = packed(in_specs, "cpu", pin=True)
    for view, src in zip(h_in_views, (case.q, case.block_table, case.kv_lens)):
        view.copy_(src)
    d_in.copy_(h_in)
    d_out, (out, lse) = packed(out_specs, dev)
    h_out, _ = packed(out_specs, "cpu", pin=True)
    kp = case.k_pages.to(dev)
    vp = case.v_pages.to(dev)
    S = B.decode_num_splits(B_, case.max_blocks, Hq, case.n_kv_heads, D, case.page_size, req_splits,
                            B.PKV_BF16)
    ws = B.alloc_workspace(B.decode_workspace_size(B_, case.max_blocks, Hq, case.n_kv_heads, D,
                                                   case.page_size, req_splits, B.PKV_BF16), dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    launches_per_step = 1 + (1 if S > 1 else 0)
    algo_bytes = case.kv_bytes()

    def step():
        B.decode_paged(q, kp, vp, bt, lens, case.scale, num_splits=req_splits, out=out, lse=lse,
                       workspace=ws, err_flag=err)

    # Warm-up steps as the timed ones run them (L2 flush, then the call), so that nothing
    # happens for the first time inside the timed region; then at least half a second of
    # calls, so that the GPU is at its clocks.
    for i in range(max(3, args.warmup)):
        flush_l2(flush, i)
        step()
    torch.cuda.synchronize()
    busy_for(step, 0.5)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        clk.settle(step)                          # a sample under load exists before the region
        barrier(world)
        torch.cuda.synchronize()
        clk.mark_start()
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush_l2(flush, i)                    # evict L2 between steps (not timed)
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        wall = time.perf_counter() - t0
        clk.mark_end()
        clk.settle(step, after=clk.t1)            # and one after it
        clocks = clk.summary()
    assert int(err.item()) == 0, f"device error flag {int(err.item())}"
    times_ms = [a.elapsed_time(b) for a, b in ev]
    total_s = sum(times_ms) / 1e3
    total_s = max_over_ranks(total_s, world)
    value = weak_scaling_rate(algo_bytes, args.steps, world, total_s) / 1e9
    ms_per_step = 1000 * total_s / args.steps
    kernel_gbs = algo_bytes / (statistics.mean(times_ms) / 1e3) / 1e9

    # ---- end to end through the public call: pinned host inputs in, results out, every step
    # (one packed copy in, q + block table + lengths; one packed copy out, out + lse)
    e2e_steps = args.steps
    for _ in range(2):
        d_in.copy_(h_in, non_blocking=True)
        step()
        h_out.copy_(d_out, non_blocking=True)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(e2e_steps):
        d_in.copy_(h_in, non_blocking=True)
        step()
        h_out.copy_(d_out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    e2e_value = weak_scaling_rate(algo_bytes, e2e_steps, world, e2e_s) / 1e9
    h2d = h_in.numel()
    d2h = h_out.numel()

    # ---- the same end-to-end steps pipelined as a serving loop would run them: step i+1's
    # inputs go in on one copy stream while step i computes, and step i's results come back
    # on another. Two sets of packed input/output buffers; every step still moves its own.
    d_in2, (q2, bt2, lens2) = packed(in_specs, dev)
    d_out2, (out2, lse2) = packed(out_specs, dev)
    sets = [(d_in, q, bt, lens, d_out, out, lse), (d_in2, q2, bt2, lens2, d_out2, out2, lse2)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]
    ev_read = [torch.cuda.Event(), torch.cuda.Event()]  # a set's results are back on the host

    def pipelined(n):
        with torch.cuda.stream(s_h2d):
            sets[0][0].copy_(h_in, non_blocking=True)
            ev_in[0].record(s_h2d)
        for i in range(n):
            k = i % 2
            if i + 1 < n:
                with torch.cuda.stream(s_h2d):
                    if i >= 1:
                        s_h2d.wait_event(ev_done[1 - k])  # step i-1 is done with that set
                    sets[1 - k][0].copy_(h_in, non_blocking=True)
                    ev_in[1 - k].record(s_h2d)
            stream.wait_event(ev_in[k])
            if i >= 2:
                stream.wait_event(ev_read[k])  # step i-2's results have left this set
            _, qk, btk, lk, _, ok_, lsek = sets[k]
            B.decode_paged(qk, kp, vp, btk, lk, case.scale, num_splits=req_splits, out=ok_, lse=lsek,
                           workspace=ws, err_flag=err)
            ev_done[k].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[k])
                h_out.copy_(sets[k][4], non_blocking=True)
                ev_read[k].record(s_d2h)

    pipelined(4)
    torch.cuda.synchronize()
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    p0.record(s_h2d)
    pipelined(e2e_steps)
    s_d2h.wait_stream(stream)
    s_d2h.wait_stream(s_h2d)
    p1.record(s_d2h)
    torch.cuda.synchronize()
    pipe_s = max_over_ranks(p0.elapsed_time(p1) / 1e3, world)
    pipe_value = weak_scaling_rate(algo_bytes, e2e_steps, world, pipe_s) / 1e9

    units = int(case.kv_lens.sum())
    traffic = profiled_traffic(args.workload, source_hash("decode_kernel.cuh", "decode.cu", "ptx.cuh"), units)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc, "parallelism": f"replicas{world}", "num_splits": S,
                   "algorithmic_bytes_per_step": algo_bytes,
                   "l2": f"inputs ({algo_bytes / 1e6:.0f} MB of K/V) exceed the 129 MB L2, and a 256 MiB buffer is written and then read between timed steps (the L2 holds no dirty lines when a step starts)",
                   "timing": "CUDA events around each call on the launch stream; sum over steps; max over ranks"},
        "roofline": {"bound": "hbm", "achieved": kernel_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": kernel_gbs / hbm_peak, "peak_source": f"{peak_src} hbm_gbs",
                     "traffic": traffic, "kernel": "decode_paged_kernel (+ merge_splits_kernel inside the same events)"},
        "e2e_pipelined": {"value": pipe_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                          "d2h_bytes_per_step": d2h,
                          "note": "the e2e steps with step i+1's inputs copied in on one stream and step i's results copied out on another while step i computes; two sets of packed buffers; like the serial e2e, no L2 flush between steps (the 682 MB of K/V exceed the L2), and back-to-back steps hide each other's launch gaps"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "q, block_table and kv_lens copied in from one pinned host buffer and out, lse copied back into another, one copy each way every step; the KV page pool is resident device state"},
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "wall_s": wall,
    }
    # ---- causal prefill on the same line (its own roofline against dense bf16)
    pre = None
    if args.only == "all":
        pre = prefill_bench(B, workloads, dev, stream, args, world, bf16_peak, bf16_sust, peak_src)
    if pre is not None:
        line["prefill"] = pre
        line["gpu_launches"] += pre.pop("launches")
    if args.only == "all" and args.workload == "llama7b_batched_decode":
        line["also"] = other_workloads(B, workloads, dev, stream, min(args.steps, 200), hbm_peak)

    # ---- the CPU baseline: the fp64 oracle on the host's cores (rank 0, one GPU only), after
    # every GPU measurement so that no timed GPU region follows an idle GPU
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baselines(case)
        if pre is not None:
            pre["cpu_baseline"] = prefill_cpu_baseline(workloads.causal_prefill_llama7b())
        if "also" in line:
            for name, cb in other_cpu_baselines(workloads).items():
                if name in line["also"]:
                    line["also"][name]["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)


def busy_for(fn, seconds):
    """Calls ``fn`` until ``seconds`` of wall time have passed (untimed warm-up)."""
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        for _ in range(10):
            fn()
        torch.cuda.synchronize()


def packed(specs, device, pin=False):
    """One byte buffer holding a tensor per (shape, dtype), each starting on a 256-byte
    boundary; returns the buffer and the tensors as views into it."""
    offs, n = [], 0
    for shape, dtype in specs:
        offs.append(n)
        nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        n = (n + nbytes + 255) // 256 * 256
    buf = torch.empty(n, dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = []
    for (shape, dtype), off in zip(specs, offs):
        nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        views.append(buf[off:off + nbytes].view(dtype).view(shape))
    return buf, views


def flush_l2(buf, i):
    """Evicts L2 between timed steps (not timed): write a buffer larger than L2, then read
    it back, so that the write-back of the dirty lines happens here and not inside the
    next timed step."""
    buf.fill_(float(i))
    buf.sum()


def time_calls(fn, steps, stream, dev):
    """Mean device time (ms) of ``fn`` over ``steps`` calls, L2 flushed before each call."""
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for i in range(3):
        flush_l2(flush, i)
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush_l2(flush, i)
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / steps


OTHER_PARTS = ("fp8", "gqa", "cascade", "chunk", "flat_gemm", "single")


def other_workloads(B, workloads, dev, stream, steps, hbm_peak, parts=OTHER_PARTS):
    """The remaining workloads, each timed on its own: GB/s of algorithmic K/V bytes (TFLOP/s for
    the chunked prefill). ``parts`` picks which (all by default; one for a profiler capture)."""
    res = {}

    def entry(name, nbytes, ms, extra=None):
        gbs = nbytes / (ms / 1e3) / 1e9
        d = {"value": gbs, "unit": "GB/s", "ms_per_call": ms, "algorithmic_bytes": nbytes,
             "frac_of_measured_hbm": gbs / hbm_peak}
        if extra:
            d.update(extra)
        res[name] = d

    if "fp8" in parts:
        # The Llama-7B batch (same lengths, same page order) over FP8 E4M3 page pools with
        # per-(page, KV head) scales: half the K/V bytes of the bf16 headline.
        c = workloads.llama7b_batched_decode_fp8(poison=False)
        q, kc, vc, ks, vs, bt, ln = (t.to(dev) for t in (c.q, c.k_codes, c.v_codes, c.k_scale,
                                                         c.v_scale, c.block_table, c.kv_lens))
        out = torch.empty_like(q)
        lse = torch.empty(c.batch, c.n_qo_heads, dtype=torch.float32, device=dev)
        S = B.decode_num_splits(c.batch, c.max_blocks, c.n_qo_heads, c.n_kv_heads, c.head_dim,
                                c.page_size, 0, B.PKV_FP8_E4M3)
        ws = B.alloc_workspace(B.decode_workspace_size(c.batch, c.max_blocks, c.n_qo_heads, c.n_kv_heads,
                                                       c.head_dim, c.page_size, 0, B.PKV_FP8_E4M3), dev)
        ms = time_calls(lambda: B.decode_paged_fp8(q, kc, vc, ks, vs, bt, ln, c.scale, out=out, lse=lse,
                                                   workspace=ws), steps, stream, dev)
        toks = int(c.kv_lens.sum())
        entry("llama7b_batched_decode_fp8", c.kv_bytes(), ms,
              {"num_splits": S, "tokens_per_s": toks / (ms / 1e3),
               "bytes_note": "E4M3 codes of every token's K and V plus the scales of the pages read"})
        del q, kc, vc, ks, vs, bt, ln, ws

    if "gqa" in parts:
        c = workloads.long_context_gqa_decode(poison=False)
        q, kp, vp, bt, ln = (t.to(dev) for t in (c.q, c.k_pages, c.v_pages, c.block_table, c.kv_lens))
        out = torch.empty_like(q)
        lse = torch.empty(c.batch, c.n_qo_heads, dtype=torch.float32, device=dev)
        S = workloads.LONG_CONTEXT_SPLITS
        ws = B.alloc_workspace(B.decode_workspace_size(c.batch, c.max_blocks, c.n_qo_heads,
                                                       c.n_kv_heads, c.head_dim, 16, S, B.PKV_BF16), dev)
        ms = time_calls(lambda: B.decode_paged(q, kp, vp, bt, ln, c.scale, num_splits=S, out=out,
                                               lse=lse, workspace=ws), steps, stream, dev)
        entry("long_context_gqa_decode", c.kv_bytes(), ms, {"num_splits": S})
        fb = torch.zeros(1, dtype=torch.int32, device=dev)
        ms = time_calls(lambda: B.decode_paged(q, kp, vp, bt, ln, c.scale, num_splits=S, out=out,
                                               lse=lse, workspace=ws, unified_phi=0.0,
                                               fallback_count=fb), steps, stream, dev)
        entry("long_context_gqa_decode_unified_max", c.kv_bytes(), ms,
              {"num_splits": S, "phi": 0.0, "fallbacks_total": int(fb.item())})
        del q, kp, vp, bt, ln, ws
        # the same lengths and pool with 8 query heads per KV head (64 query heads)
        c = workloads.long_context_gqa8_decode(poison=False)
        q, kp, vp, bt, ln = (t.to(dev) for t in (c.q, c.k_pages, c.v_pages, c.block_table, c.kv_lens))
        out = torch.empty_like(q)
        lse = torch.empty(c.batch, c.n_qo_heads, dtype=torch.float32, device=dev)
        ws = B.alloc_workspace(B.decode_workspace_size(c.batch, c.max_blocks, c.n_qo_heads,
                                                       c.n_kv_heads, c.head_dim, 16, S, B.PKV_BF16), dev)
        ms = time_calls(lambda: B.decode_paged(q, kp, vp, bt, ln, c.scale, num_splits=S, out=out,
                                               lse=lse, workspace=ws), steps, stream, dev)
        entry("long_context_gqa8_decode", c.kv_bytes(), ms, {"num_splits": S, "group": 8})
        del q, kp, vp, bt, ln, ws
        # the GQA-8 batch over FP8 E4M3 pools (the tensor-core path with in-kernel conversion)
        c = workloads.long_context_gqa8_decode_fp8(poison=False)
        q, kc, vc, ks, vs, bt, ln = (t.to(dev) for t in (c.q, c.k_codes, c.v_codes, c.k_scale, c.v_scale,
                                                         c.block_table, c.kv_lens))
        out = torch.empty_like(q)
        lse = torch.empty(c.batch, c.n_qo_heads, dtype=torch.float32, device=dev)
        ws = B.alloc_workspace(B.decode_workspace_size(c.batch, c.max_blocks, c.n_qo_heads, c.n_kv_heads,
                                                       c.head_dim, 16, S, B.PKV_FP8_E4M3), dev)
        ms = time_calls(lambda: B.decode_paged_fp8(q, kc, vc, ks, vs, bt, ln, c.scale, num_splits=S, out=out,
                                                   lse=lse, workspace=ws), steps, stream, dev)
        toks = int(c.kv_lens.sum())
        entry("long_context_gqa8_decode_fp8", c.kv_bytes(), ms,
              {"num_splits": S, "group": 8, "tokens_per_s": toks / (ms / 1e3),
               "bytes_note": "E4M3 codes of every token's K and V plus the scales of the pages read"})
        del q, kc, vc, ks, vs, bt, ln, ws

    if "cascade" in parts:
        c = workloads.cascade_shared_prefix_decode(poison=False)
        q, kp, vp, pt, st, sl = (t.to(dev) for t in (c.q, c.k_pages, c.v_pages, c.prefix_table,
                                                     c.suffix_table, c.suffix_lens))
        out = torch.empty_like(q)
        lse = torch.empty(c.n_requests, c.n_qo_heads, dtype=torch.float32, device=dev)
        ws = B.alloc_workspace(B.cascade_workspace_size(c.n_requests, c.prefix_len, st.shape[1],
                                                        c.n_qo_heads, c.n_kv_heads, c.head_dim,
                                                        c.page_size), dev)
        ms = time_calls(lambda: B.decode_cascade(q, kp, vp, pt, c.prefix_len, st, sl, c.scale, out=out,
                                                 lse=lse, workspace=ws), steps, stream, dev)
        entry("cascade_shared_prefix_decode", c.kv_bytes(), ms,
              {"bytes_note": "shared prefix K/V counted once plus every suffix"})
        del q, kp, vp, pt, st, sl, ws

    if "chunk" in parts:
        # Chunked prefill over the paged cache: 8 sequences of Llama-7B heads, each appending
        # 1024 tokens to a 3072-token prefix (the new tokens' K/V already in the pages).
        n_seq, C, L0 = 8, 1024, 3072
        c = workloads.make_paged_decode(1006, n_seq, 32, 32, 128, 16, [L0 + C] * n_seq, dtype="bf16",
                                        poison=False)
        gen = torch.Generator().manual_seed(1007)
        qc = torch.randn((n_seq, C, 32, 128), generator=gen, dtype=torch.float32).to(torch.bfloat16).to(dev)
        kp, vp, bt = c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev)
        pl = torch.full((n_seq,), L0, dtype=torch.int32, device=dev)
        out = torch.empty_like(qc)
        lse = torch.empty((n_seq, 32, C), dtype=torch.float32, device=dev)
        ms = time_calls(lambda: B.prefill_paged_chunk(qc, kp, vp, bt, pl, c.scale, out=out, lse=lse),
                        steps, stream, dev)
        flops = 4 * 128 * 32 * n_seq * (C * L0 + C * (C + 1) // 2)
        tf = flops / (ms / 1e3) / 1e12
        res["chunked_prefill_paged"] = {
            "value": tf, "unit": "TFLOP/s", "ms_per_call": ms, "flops": flops,
            "frac_of_measured_bf16": tf / peaks()[1],
            "workload": f"{n_seq} sequences x {C} new tokens after a {L0}-token prefix, 32/32 heads, d 128, "
                        "page 16, bf16 (attended pairs only)"}
        del qc, kp, vp, bt, pl, out, lse

    if "flat_gemm" in parts:
        # The flat GEMMs either side of attention in a Llama-2-7B-shaped decode step: the QKV
        # projection (n 12288) and the O projection (n 4096), k 4096, for 1, 8 and 16 tokens.
        # Bytes moved: the bf16 weights, tokens and result once each (the weights dominate;
        # the QKV weights, 100 MB, would fit in the L2, which is flushed before every call).
        fg = {}
        for proj, builder in (("qkv", workloads.llama7b_qkv_projection), ("o", workloads.llama7b_o_projection)):
            for m in (1, 8, 16):
                c = builder(m)
                x, w = c.x.to(dev), c.w.to(dev)
                y = torch.empty((m, c.n), dtype=torch.bfloat16, device=dev)
                ms = time_calls(lambda: B.flat_gemm(x, w, out=y), steps, stream, dev)
                gbs = c.bytes_moved() / (ms / 1e3) / 1e9
                fg[f"{proj}_m{m}"] = {"value": gbs, "unit": "GB/s", "ms_per_call": ms, "bytes": c.bytes_moved(),
                                      "frac_of_measured_hbm": gbs / hbm_peak, "m": m, "n": c.n, "k": c.k,
                                      "cluster": B.flat_gemm_num_splits(m, c.n, c.k),
                                      "tflops": 2 * m * c.n * c.k / (ms / 1e3) / 1e12}
                del x, w, y
        res["flat_gemm"] = {"workload": "Llama-2-7B-shaped decode projections, bf16 x[m, 4096] w[n, 4096]^T, "
                                        "synthetic weights", "cases": fg}

    if "single" in parts:
        c = workloads.single_seq_decode_f32()
        q, kp, vp, bt, ln = (t.to(dev) for t in (c.q, c.k_pages, c.v_pages, c.block_table, c.kv_lens))
        ms = time_calls(lambda: B.decode_paged(q, kp, vp, bt, ln, c.scale), steps, stream, dev)
        entry("single_seq_decode_f32", c.kv_bytes(), ms,
              {"note": "1 MiB of K/V: launch-latency bound; L2 flushed before each call"})
        # The same call captured once into a CUDA graph and replayed: the library never
        # allocates, copies to the host or synchronises, so the decode and its split merge
        # replay as one graph launch on the current buffers.
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        ws = B.alloc_workspace(B.decode_workspace_size(c.batch, c.max_blocks, c.n_qo_heads, c.n_kv_heads,
                                                       c.head_dim, c.page_size, 0, B.PKV_F32), dev)

        def call():
            B.decode_paged(q, kp, vp, bt, ln, c.scale, out=out, lse=lse, workspace=ws)

        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            call()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        ms = time_calls(graph.replay, steps, stream, dev)
        entry("single_seq_decode_f32_graph", c.kv_bytes(), ms,
              {"note": "the same call replayed from a CUDA graph captured once; L2 flushed before each replay"})

        # What a graph is for: a model step makes one such call per layer. 32 layers, each
        # with its own query, outputs and K/V pool, called back to back from Python, against
        # the same 32 calls captured once and replayed as one graph launch. Timed as a
        # group (CUDA events around all 32, L2 flushed before the group): the direct calls
        # also pay the host's per-call launch cost whenever it exceeds the kernel's time.
        n_layers = 32
        layers = []
        for _ in range(n_layers):
            layers.append((torch.randn_like(q), kp.clone(), vp.clone(), torch.empty_like(q),
                           torch.empty(q.shape[:2], dtype=torch.float32, device=dev)))

        def all_layers():
            for ql, kl, vl, ol, ll in layers:
                B.decode_paged(ql, kl, vl, bt, ln, c.scale, out=ol, lse=ll, workspace=ws)

        side.wait_stream(stream)
        with torch.cuda.stream(side):
            all_layers()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph_l = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_l):
            all_layers()
        ms_direct = time_calls(all_layers, max(3, steps // 10), stream, dev)
        ms_graph = time_calls(graph_l.replay, max(3, steps // 10), stream, dev)
        entry("single_seq_decode_f32_32_layers_direct", n_layers * c.kv_bytes(), ms_direct,
              {"us_per_layer": 1000 * ms_direct / n_layers,
               "note": "32 calls (one per layer, own q, out and K/V pool) from Python back to back"})
        entry("single_seq_decode_f32_32_layers_graph", n_layers * c.kv_bytes(), ms_graph,
              {"us_per_layer": 1000 * ms_graph / n_layers,
               "note": "the same 32 calls captured once into a CUDA graph, replayed as one launch"})

    return res

def prefill_bench(B, workloads, dev, stream, args, world, bf16_peak, bf16_sust, peak_src):
    case = workloads.causal_prefill_llama7b()
    q, k, v = case.q.to(dev), case.k.to(dev), case.v.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty(case.batch, case.n_qo_heads, case.seq_len, dtype=torch.float32, device=dev)
    try:
        B.prefill_causal(q, k, v, case.scale, out=out, lse=lse)
    except B.AttnError as e:
        if e.status == B.PKV_ERR_UNSUPPORTED:
            return None
        raise
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for i in range(max(3, args.warmup)):
        flush_l2(flush, i)
        B.prefill_causal(q, k, v, case.scale, out=out, lse=lse)
    busy_for(lambda: B.prefill_causal(q, k, v, case.scale, out=out, lse=lse), 0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2(flush, i)
        ev[i][0].record(stream)
        B.prefill_causal(q, k, v, case.scale, out=out, lse=lse)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / 1e3, world)
    flops = case.causal_flops()
    tflops = flops * args.steps * world / t / 1e12
    per = flops * args.steps / t / 1e12
    return {"workload": PREFILL_WORKLOAD, "value": tflops, "unit": "TFLOP/s",
            "ms_per_step": 1000 * t / args.steps, "causal_flops_per_step": flops,
            "roofline": {"bound": "tensor", "achieved": per, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": per / bf16_peak, "peak_source": f"{peak_src} bf16_tflops (burst)",
                         "traffic": profiled_traffic("causal_prefill_llama7b",
                                                     source_hash("prefill.cu", "tcgen05.cuh", "ptx.cuh"), 1),
                         "kernel": "attn_tile_kernel<causal>"},
            "launches": args.steps}


def torchrun_command(n, port, script, argv):
    """The command that runs ``script argv`` as ``n`` ranks on this node (127.0.0.1 rendezvous)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr=127.0.0.1", f"--master-port={port}", script] + list(argv)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--master-port", type=int, default=29531,
                    help="rendezvous port when bench.py starts its own ranks (--gpus N > 1)")
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "decode", "prefill"] + list(OTHER_PARTS), default="all",
                    help="run one part only (for profiler captures)")
    ap.add_argument("--workload", choices=sorted(DECODE_WORKLOADS), default="llama7b_batched_decode",
                    help="decode workload of the timed step (the headline is llama7b_batched_decode)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # Not started by torchrun: start N ranks (one replica per GPU) through it.
        sys.exit(subprocess.call(torchrun_command(args.gpus, args.master_port, os.path.abspath(__file__),
                                                  sys.argv[1:])))
    rank, world, local = dist_init()
    if world != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE is {world}")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
