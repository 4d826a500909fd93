#!/usr/bin/env python
"""Benchmark of the paged-KV decode step on one GB300 (per rank).

A step is one pass of the decode hot path over the batch-32 mixed-length
workload: append one new token per row into its pool slot
(paged_kv_append), then batched paged decode attention of every row's query
over its block table, with the 1024-token shared prefix read once for all 32
rows (paged_decode_attention).  Workload: bf16, 32 q / 8 kv heads, head_dim
128, block size 16, suffixes uniform on 0..7168 (seed 1002), block ids
shuffled.  The K/V read per step (about 0.47 GB) is larger than L2, so no
flush is needed between steps.

value    = unique K/V bytes the step attends (the prefix once, every row's own
           tokens) / device time per step, in GB/s (whole job: all ranks).
e2e      = the same metric with the step's inputs (q, new K/V, slots, lengths)
           copied from pinned host memory and the output copied back inside
           the timed region.
roofline = the dominant kernel (the decode kernel: shared-prefix and split-KV
           CTAs in one launch) timed with CUDA events on its own stream during
           the timed region; its algorithmic bytes are the unique K/V tiles it
           reads (512 B per token and kv head; the prefix once).

``--impl reference`` times the CPU oracle (single thread) on a bounded sample
of the same workload instead.
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

import pkv_inputs as gen  # noqa: E402

METRIC = "paged decode KV GB/s (% of 8 TB/s) and decode tok/s at batch 32, 1×GB300"
NOMINAL_HBM_GBS = 8000.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1900.0


def workload_bytes(w: gen.Workload):
    """Unique K/V bytes a decode step attends and the split kernel's share."""
    D, hkv, eb = w.head_dim, w.num_kv_heads, w.elem_bytes
    per_token = 2 * hkv * D * eb  # K and V, every kv head
    P = w.shared_prefix_tokens
    unique_tokens = P + int(np.sum(w.seq_lens.astype(np.int64) - P))
    suffix_tokens = int(np.sum(w.seq_lens.astype(np.int64) - P))
    return unique_tokens * per_token, suffix_tokens * per_token


# ---------------------------------------------------------------------------
# clocks sampled with nvidia-smi during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu=timestamp,{self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return None
        # samples from the loaded part of the run: SM clock above idle
        load = [r for r in rows if r[0] > 0.5 * r[1]] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(load)}


# ---------------------------------------------------------------------------
# the library arm
# ---------------------------------------------------------------------------
def kernel_source_sha():
    h = hashlib.sha256()
    for f in ("decode_kernel.cuh", "decode_coop.cuh", "decode_bf16.cu", "decode_common.cuh", "pkv_device.cuh",
              "pkv_internal.h"):
        with open(os.path.join(ROOT, "block_paged_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(sha):
    path = os.path.join(ROOT, "profiles", "decode_split_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("source_sha") != sha:
        return None
    return d.get("dram_bytes_per_launch_full_workload")


PROF_EVERY = 4     # roofline loop: one decode launch in this many carries events
ROOF_SAMPLES = 64  # roofline loop: timed decode launches (the median is reported)


def barrier(world):
    """All ranks meet (no-op for one rank)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, dev):
    """The largest of the ranks' values of x (a time): the job is as slow as
    its slowest rank."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank_step, world, ms, steps):
    """Whole-job throughput: every rank processes units_per_rank_step per step
    (replicas over disjoint row batches, no exchange), and the job takes the
    max-over-ranks time ms for `steps` steps.  Units per second."""
    return world * units_per_rank_step / (ms / steps / 1e3)


def run_pkv(args, rank, world, local):
    import torch
    import block_paged_kv_gb300 as pkv

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = gen.shared_prefix_b32()
    bytes_step, bytes_split = workload_bytes(w)

    def up(a):
        if w.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    k_pool, v_pool = up(w.k_pool), up(w.v_pool)
    q, k_new, v_new = up(w.q), up(w.k_new), up(w.v_new)
    tables = torch.from_numpy(w.block_tables).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    slots_h = pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows, w.new_pos,
                                    w.block_size)
    slots = torch.from_numpy(slots_h).to(dev)
    desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, w.block_size, dev)
    max_len = int(w.seq_lens.max())
    ws = pkv.alloc_workspace(pkv.decode_workspace_size(w.batch, w.num_q_heads, w.num_kv_heads,
                                                       w.head_dim, w.block_size, max_len, 0, desc), dev)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(qx=q, kx=k_new, vx=v_new, sx=slots, lx=lens, ox=out):
        pkv.paged_kv_append(k_pool, v_pool, sx, kx, vx, status=status)
        pkv.paged_decode_attention(qx, k_pool, v_pool, tables, lx, 0, w.scale, out=ox,
                                   workspace=ws, max_seq_len=max_len, prefix=desc, status=status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = pkv.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = pkv.launch_count() - n0
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)

    # the decode kernel's own duration, for the roofline: a loop of its own
    # right after the timed steps, of ROOF_SAMPLES timed launches (whatever
    # --steps is), each the decode launch of one step among unsampled ones.
    # The events around a launch cost it its overlap with its neighbours
    # (programmatic dependent launch), so only one step in PROF_EVERY carries
    # them; the median launch is reported
    pkv.profile_enable([])  # clear the records
    for i in range(ROOF_SAMPLES * PROF_EVERY):
        sample = i % PROF_EVERY == 0
        if sample:
            pkv.profile_mask([pkv.KERNEL_DECODE_SPLIT])
        step()
        if sample:
            pkv.profile_mask([])
    torch.cuda.synchronize()
    split_times = pkv.profile_times(pkv.KERNEL_DECODE_SPLIT)
    nsplit = len(split_times)
    split_med_ms = statistics.median(split_times)
    clk = clocks.stop() if rank == 0 else None
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    # end to end: every step's inputs come from pinned host memory and its
    # output goes back to pinned host memory, through the same public calls.
    # The copies run on a second stream under the kernels (two buffer sets):
    # step i+1's uploads and step i's download overlap step i's kernels, as a
    # serving loop would run them; each step's copies are inside the timed
    # region, which ends when the last download has landed
    # A step's five inputs are staged together in one pinned host buffer and
    # go up in one copy (one call per step instead of five, as a serving loop
    # would batch them); on the device each buffer set holds the five tensors
    # as views of one byte buffer, each at a 256-byte aligned offset.
    srcs = (q, k_new, v_new, slots, lens)
    nbytes = [t.numel() * t.element_size() for t in srcs]
    offs, total = [], 0
    for n in nbytes:
        offs.append(total)
        total += (n + 255) // 256 * 256
    in_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o, n in zip(srcs, offs, nbytes):
        in_h[o:o + n].copy_(t.cpu().contiguous().reshape(-1).view(torch.uint8))

    def input_views(raw):
        return tuple(raw[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(srcs, offs, nbytes))

    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    raws = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    bufs = [(*input_views(raw), torch.empty_like(out)) for raw in raws]
    h2d = total
    d2h = out_h[0].numel() * out_h[0].element_size()
    # at least 200 end-to-end steps (about 20 ms), so that the pipeline's
    # fill and drain do not weigh on a short --steps run
    e2e_steps = max(200, min(args.steps, 1000))
    cs = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def upload(bset):  # on the copy stream, once the set's last step is done
        with torch.cuda.stream(cs):
            cs.wait_event(ev_done[bset])
            raws[bset].copy_(in_h, non_blocking=True)
            ev_in[bset].record(cs)

    def e2e_run(nsteps, start_event=None):
        if start_event is not None:
            cs.wait_event(start_event)
        upload(0)
        for i in range(nsteps):
            bset = i % 2
            stream.wait_event(ev_in[bset])
            stream.wait_event(ev_out[bset])  # this set's previous download has landed
            qx, kx, vx, sx, lx, ox = bufs[bset]
            step(qx, kx, vx, sx, lx, ox)
            ev_done[bset].record(stream)
            if i + 1 < nsteps:
                upload(1 - bset)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_done[bset])
                out_h[bset].copy_(ox, non_blocking=True)
                ev_out[bset].record(cs)
        stream.wait_event(ev_out[(nsteps - 1) % 2])

    e2e_run(3)
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    e2e_run(e2e_steps, start_event=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    secondary = secondary_measurements(args, pkv, torch, dev) if (rank == 0 and args.secondary) else None

    if rank != 0:
        return
    peak, peak_kind = peaks()
    t_step = ms / args.steps / 1e3
    value = job_rate(bytes_step, world, ms, args.steps) / 1e9
    split_avg_s = split_med_ms / 1e3
    achieved = bytes_step / split_avg_s / 1e9
    sha = kernel_source_sha()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) cast to bf16; shuffled block ids)",
        "config": contract_config(w, world),
        "pct_of_8TBps": round(100 * value / world / NOMINAL_HBM_GBS, 1),
        "tok_per_s": round(job_rate(w.batch, world, ms, args.steps), 1),
        "clocks": clk,
        "e2e": {"value": round(job_rate(bytes_step, world, e2e_ms, e2e_steps) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms / e2e_steps, 5),
                "copies": "one pinned host staging buffer up and the output down per step, on a "
                          "second stream, overlapped with the previous step's kernels"},
        "gpu_launches": int(launches),
        "roofline": {"kernel": "decode_split_kernel<128, bf16> (shared-prefix + split-KV decode, one launch)",
                     "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 3), "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": committed_traffic(sha), "algorithmic_bytes_per_launch": bytes_step,
                     "avg_launch_us": round(split_avg_s * 1e6, 2),
                     "launch_us_stat": "median of the timed launches", "launches_timed": nsplit,
                     "launch_us_mean": round(1e3 * statistics.mean(split_times), 2),
                     "launch_us_min": round(1e3 * min(split_times), 2),
                     "launch_us_max": round(1e3 * max(split_times), 2),
                     "source_sha": sha},
    }
    if secondary is not None:
        line["secondary"] = secondary
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)


def time_loop(torch, fn, steps, warmup, flush=None):
    """Mean device time of fn() (seconds).  Every iteration is enqueued
    without a host sync, with its own pair of events: the host stays ahead
    of the GPU, so its launch work does not count; the L2 flush (if any) runs
    before each iteration's start event."""
    for _ in range(warmup):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for e0, e1 in ev:
        if flush is not None:
            flush()
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps / 1e3


def fp8_b32_setup(pkv, torch, dev):
    """The batch-32 shared-prefix workload on FP8 (E4M3) pools: its context is
    appended (quantized) once; returns (workload, step = append one token per
    row + shared-prefix decode, decode alone, K/V bytes a decode reads, status)."""
    w = gen.shared_prefix_b32()
    ks, vs = float(gen.FP8_K_SCALE), float(gen.FP8_V_SCALE)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    kp, vp = pkv.fp8_pools(w.num_blocks, w.num_kv_heads, w.head_dim, dev)
    cs, ckr, cvr = gen.live_slots(w)
    pkv.paged_kv_append(kp, vp, torch.from_numpy(cs).to(dev), up(ckr), up(cvr),
                        k_scale=ks, v_scale=vs)
    del ckr, cvr
    q, kn, vn = up(w.q), up(w.k_new), up(w.v_new)
    t = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    slots = torch.from_numpy(pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows,
                                                   w.new_pos, 16)).to(dev)
    desc = pkv.make_prefix_desc(w.block_tables, w.seq_lens, 16, dev)
    ml = int(w.seq_lens.max())
    ws = pkv.alloc_workspace(pkv.decode_workspace_size(w.batch, w.num_q_heads, w.num_kv_heads,
                                                       w.head_dim, 16, ml, 0, desc), dev)
    out = torch.empty_like(q)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def decode():
        pkv.paged_decode_attention(q, kp, vp, t, sl, 0, w.scale, out=out, workspace=ws,
                                   max_seq_len=ml, prefix=desc, status=st, k_scale=ks, v_scale=vs)

    def step():
        pkv.paged_kv_append(kp, vp, slots, kn, vn, status=st, k_scale=ks, v_scale=vs)
        decode()

    return w, step, decode, workload_bytes(w)[0] // 2, st


def fp8_prefill_measure(pkv, torch, dev, steps, warmup, flush=None):
    """The chunked-prefill workload (4 x 512 queries vs a 16384-token prefix)
    with its K/V in FP8 pools."""
    w = gen.chunked_prefill()
    ks, vs = float(gen.FP8_K_SCALE), float(gen.FP8_V_SCALE)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    kp, vp = pkv.fp8_pools(w.num_blocks, w.num_kv_heads, w.head_dim, dev)
    cs, ckr, cvr = gen.live_slots(w)
    pkv.paged_kv_append(kp, vp, torch.from_numpy(cs).to(dev), up(ckr), up(cvr), k_scale=ks, v_scale=vs)
    slots = pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows, w.new_pos, 16)
    pkv.paged_kv_append(kp, vp, torch.from_numpy(slots).to(dev), up(w.k_new), up(w.v_new),
                        k_scale=ks, v_scale=vs)
    q = up(w.q)
    t = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    cu = torch.from_numpy(w.cu_q_lens).to(dev)
    out = torch.empty_like(q)
    C = int(w.cu_q_lens[1] - w.cu_q_lens[0])
    ml = int(w.seq_lens.max())
    s = time_loop(torch, lambda: pkv.paged_prefill_chunk_attention(q, cu, kp, vp, t, sl, C, 0, w.scale,
                                                                   out=out, max_seq_len=ml,
                                                                   k_scale=ks, v_scale=vs),
                  steps, warmup, flush)
    keys = sum(int(L) - C + i + 1 for L in w.seq_lens for i in range(C))
    flops = 4 * w.head_dim * keys * w.num_q_heads
    return {"us": round(s * 1e6, 2), "TFLOP/s": round(flops / s / 1e12, 1), "flop": flops,
            "frac_of_bf16_peak": round(flops / s / 1e12 / bf16_peak(), 3),
            "peak": "measured bf16_tflops (burst): the products are f16, whose dense rate is bf16's",
            "l2": "flushed before each call" if flush else "not flushed"}


def run_fp8_prefill_case(args, local):
    """The chunked prefill on FP8 pools timed alone (for profiling)."""
    import torch
    import block_paged_kv_gb300 as pkv
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    r = fp8_prefill_measure(pkv, torch, dev, args.steps, args.warmup)
    print(json.dumps(dict(case="fp8_prefill", **r)), flush=True)


def run_fp8_case(args, local):
    """The FP8 decode of the batch-32 shared-prefix workload timed alone (for profiling)."""
    import torch
    import block_paged_kv_gb300 as pkv
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w, _, decode, b, st = fp8_b32_setup(pkv, torch, dev)
    for _ in range(args.warmup):
        decode()
    torch.cuda.synchronize()
    pkv.profile_enable([pkv.KERNEL_DECODE_SPLIT])
    for _ in range(args.steps):
        decode()
    torch.cuda.synchronize()
    n, t = pkv.profile_read(pkv.KERNEL_DECODE_SPLIT)
    pkv.profile_enable([])
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    s = t / max(n, 1) / 1e3
    print(json.dumps({"case": "fp8_decode", "workload": w.name.replace("bf16", "fp8"),
                      "split_kernel_us": round(s * 1e6, 2), "GB/s": round(b / s / 1e9, 1),
                      "frac_of_hbm_peak": round(b / s / 1e9 / peaks()[0], 3)}), flush=True)


def run_long_case(args, local, sliding=False):
    """One group of the long-context workload (4 rows x 32768 tokens, 8 q / 1
    kv head, head_dim 256) decoded alone: the full-attention group, or the
    sliding-window group (window 512, expired blocks as -1 sentinels); its
    split and merge kernels timed by their own events (for profiling)."""
    import torch
    import block_paged_kv_gb300 as pkv
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = gen.long_two_groups()[1 if sliding else 0]

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    kp, vp, q = up(w.k_pool), up(w.v_pool), up(w.q)
    t = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    out = torch.empty_like(q)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ml = int(w.seq_lens.max())
    ws = pkv.alloc_workspace(pkv.decode_workspace_size(w.batch, w.num_q_heads, w.num_kv_heads,
                                                       w.head_dim, 16, ml, w.window), dev)

    def decode():
        pkv.paged_decode_attention(q, kp, vp, t, sl, w.window, w.scale, out=out, workspace=ws,
                                   max_seq_len=ml, status=st)

    for _ in range(args.warmup):
        decode()
    torch.cuda.synchronize()
    pkv.profile_enable([pkv.KERNEL_DECODE_SPLIT, pkv.KERNEL_DECODE_COMBINE])
    for _ in range(args.steps):
        decode()
    torch.cuda.synchronize()
    n, ts = pkv.profile_read(pkv.KERNEL_DECODE_SPLIT)
    n2, tc = pkv.profile_read(pkv.KERNEL_DECODE_COMBINE)
    pkv.profile_enable([])
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    if w.window:
        b = w.batch * min(w.window, ml) * 2 * w.num_kv_heads * w.head_dim * 2
    else:
        b = workload_bytes(w)[0]
    s = ts / max(n, 1) / 1e3
    print(json.dumps({"case": "sliding_decode" if sliding else "long_decode", "workload": w.name,
                      "split_kernel_us": round(s * 1e6, 2),
                      "merge_kernel_us": round(tc / max(n2, 1) * 1e3, 2),
                      "split_GB/s": round(b / s / 1e9, 1),
                      "split_frac_of_hbm_peak": round(b / s / 1e9 / peaks()[0], 3)}), flush=True)


def run_append_case(args, local, fp8=False):
    """The bulk append of every private-suffix token of the batch-32 workload
    (124,682 tokens) into bf16 pools, or quantized into FP8 pools, timed alone
    (for profiling)."""
    import torch
    import block_paged_kv_gb300 as pkv
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = gen.shared_prefix_b32()
    n = int(np.sum(w.seq_lens - 1024))
    rows = np.repeat(np.arange(w.batch), w.seq_lens - 1024).astype(np.int32)
    pos = np.concatenate([np.arange(1024, L) for L in w.seq_lens]).astype(np.int32)
    slots = torch.from_numpy(pkv.slot_mapping_host(w.block_tables, w.num_blocks, rows, pos, 16)).to(dev)
    kn = torch.randn((n, 8, 128), dtype=torch.bfloat16, device=dev)
    vn = torch.randn_like(kn)
    if fp8:
        kp, vp = pkv.fp8_pools(w.num_blocks, 8, 128, dev)
        ks, vs = float(gen.FP8_K_SCALE), float(gen.FP8_V_SCALE)
        fn = lambda: pkv.paged_kv_append(kp, vp, slots, kn, vn, k_scale=ks, v_scale=vs)  # noqa: E731
        b = 2 * n * 8 * 128 * (2 + 1) + 4 * n   # bf16 rows in, E4M3 codes out
    else:
        kp = torch.empty((w.num_blocks, 8, 16, 128), dtype=torch.bfloat16, device=dev)
        vp = torch.empty_like(kp)
        fn = lambda: pkv.paged_kv_append(kp, vp, slots, kn, vn)  # noqa: E731
        b = 2 * 2 * n * 8 * 128 * 2 + 4 * n     # rows read and written, K and V
    s = time_loop(torch, fn, args.steps, args.warmup)
    print(json.dumps({"case": "fp8_append" if fp8 else "append", "tokens": n, "us": round(s * 1e6, 2),
                      "GB/s": round(b / s / 1e9, 1), "frac_of_hbm_peak": round(b / s / 1e9 / peaks()[0], 3)}),
          flush=True)


def secondary_measurements(args, pkv, torch, dev):
    """The other workloads, shorter runs: dense decode (L2 flushed), long
    context full + sliding, bulk append of a whole context."""
    res = {}
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.add_(1)

    def up(w, a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    # dense decode (33.5 MB of K/V: L2-sized, so L2 is flushed before each step)
    w = gen.dense_bf16()
    kp, vp, q = up(w, w.k_pool), up(w, w.v_pool), up(w, w.q)
    t = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    out = torch.empty_like(q)
    ws = pkv.alloc_workspace(pkv.decode_workspace_size(w.batch, w.num_q_heads, w.num_kv_heads,
                                                       w.head_dim, 16, 2048, 0), dev)
    s = time_loop(torch, lambda: pkv.paged_decode_attention(q, kp, vp, t, sl, 0, w.scale, out=out,
                                                            workspace=ws, max_seq_len=2048),
                  200, 10, flush)
    b = workload_bytes(w)[0]
    res["dense_bf16_decode"] = {"us": round(s * 1e6, 2), "GB/s": round(b / s / 1e9, 1),
                                "kv_bytes": b, "l2": "flushed before each step"}
    del kp, vp
    # long context: full group and sliding group, one call each
    full, sliding = gen.long_two_groups()
    for name, w in (("long_full_bf16_decode", full), ("long_sliding_bf16_decode", sliding)):
        kp, vp, q = up(w, w.k_pool), up(w, w.v_pool), up(w, w.q)
        t = torch.from_numpy(w.block_tables).to(dev)
        sl = torch.from_numpy(w.seq_lens).to(dev)
        out = torch.empty_like(q)
        ml = int(w.seq_lens.max())
        ws = pkv.alloc_workspace(pkv.decode_workspace_size(w.batch, w.num_q_heads, w.num_kv_heads,
                                                           w.head_dim, 16, ml, w.window), dev)
        s = time_loop(torch, lambda: pkv.paged_decode_attention(q, kp, vp, t, sl, w.window, w.scale,
                                                                out=out, workspace=ws, max_seq_len=ml),
                      100, 5, flush)
        if w.window:
            b = w.batch * min(w.window, ml) * 2 * w.num_kv_heads * w.head_dim * 2
        else:
            b = workload_bytes(w)[0]
        res[name] = {"us": round(s * 1e6, 2), "GB/s": round(b / s / 1e9, 1), "kv_bytes": b}
        del kp, vp
    # the same two groups in one fused launch (split + merge), against the two
    # calls one after the other
    gdev = []
    for w in (full, sliding):
        kp, vp, q = up(w, w.k_pool), up(w, w.v_pool), up(w, w.q)
        gdev.append((w, kp, vp, q, torch.from_numpy(w.block_tables).to(dev),
                     torch.from_numpy(w.seq_lens).to(dev), torch.empty_like(q)))
    groups = [pkv.DecodeGroup(q, kp, vp, t, sl, w.window, w.scale, out=o,
                              max_seq_len=int(w.seq_lens.max()))
              for w, kp, vp, q, t, sl, o in gdev]
    gws = pkv.alloc_workspace(pkv.decode_groups_workspace_size(groups), dev)
    sws = [pkv.alloc_workspace(pkv.decode_workspace_size(w.batch, w.num_q_heads, w.num_kv_heads,
                                                         w.head_dim, 16, int(w.seq_lens.max()),
                                                         w.window), dev) for w, *_ in gdev]

    def two_calls():
        for (w, kp, vp, q, t, sl, o), wsx in zip(gdev, sws):
            pkv.paged_decode_attention(q, kp, vp, t, sl, w.window, w.scale, out=o, workspace=wsx,
                                       max_seq_len=int(w.seq_lens.max()))

    s_two = time_loop(torch, two_calls, 100, 5, flush)
    s_fused = time_loop(torch, lambda: pkv.paged_decode_attention_groups(groups, workspace=gws),
                        100, 5, flush)
    b = workload_bytes(full)[0] + full.batch * sliding.window * 2 * sliding.num_kv_heads * sliding.head_dim * 2
    res["long_two_groups_fused"] = {"us": round(s_fused * 1e6, 2), "GB/s": round(b / s_fused / 1e9, 1),
                                    "two_calls_us": round(s_two * 1e6, 2), "kv_bytes": b,
                                    "note": "full + sliding group of the long-context workload, one split "
                                            "launch and one merge launch; each timed back to back on the device"}
    del gdev, groups
    # chunked prefill: 4 rows x 512 queries against a 16384-token paged prefix
    w = gen.chunked_prefill()
    kp, vp, q = up(w, w.k_pool), up(w, w.v_pool), up(w, w.q)
    kn, vn = up(w, w.k_new), up(w, w.v_new)
    t = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    cu = torch.from_numpy(w.cu_q_lens).to(dev)
    slots = torch.from_numpy(pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows,
                                                   w.new_pos, 16)).to(dev)
    pkv.paged_kv_append(kp, vp, slots, kn, vn)
    out = torch.empty_like(q)
    C = int(w.cu_q_lens[1] - w.cu_q_lens[0])
    ml = int(w.seq_lens.max())
    s = time_loop(torch, lambda: pkv.paged_prefill_chunk_attention(q, cu, kp, vp, t, sl, C, 0, w.scale,
                                                                   out=out, max_seq_len=ml),
                  30, 5, flush)
    keys = sum(int(L) - C + i + 1 for L in w.seq_lens for i in range(C))
    flops = 4 * w.head_dim * keys * w.num_q_heads
    res["chunked_prefill"] = {"us": round(s * 1e6, 2), "TFLOP/s": round(flops / s / 1e12, 1),
                              "flop": flops, "frac_of_bf16_peak": round(flops / s / 1e12 / bf16_peak(), 3),
                              "peak": "measured bf16_tflops (burst)", "l2": "flushed before each call"}
    del kp, vp
    # the same chunked prefill on FP8 pools (context appended quantized)
    res["chunked_prefill_fp8"] = fp8_prefill_measure(pkv, torch, dev, 30, 5, flush)
    # speculative verify: 32 rows x 4 queries over 1024..8192-token contexts
    w = gen.verify_steps()
    kp, vp, q = up(w, w.k_pool), up(w, w.v_pool), up(w, w.q)
    kn, vn = up(w, w.k_new), up(w, w.v_new)
    t = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    cu = torch.from_numpy(w.cu_q_lens).to(dev)
    slots = torch.from_numpy(pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows,
                                                   w.new_pos, 16)).to(dev)
    pkv.paged_kv_append(kp, vp, slots, kn, vn)
    out = torch.empty_like(q)
    C = int(w.cu_q_lens[1] - w.cu_q_lens[0])
    ml = int(w.seq_lens.max())
    s = time_loop(torch, lambda: pkv.paged_prefill_chunk_attention(q, cu, kp, vp, t, sl, C, 0, w.scale,
                                                                   out=out, max_seq_len=ml),
                  50, 5, flush)
    b = int(np.sum(w.seq_lens)) * 2 * w.num_kv_heads * w.head_dim * 2
    res["verify_4q"] = {"workload": w.name, "us": round(s * 1e6, 2), "GB/s": round(b / s / 1e9, 1),
                        "kv_bytes": b, "queries_per_s": round(w.batch * C / s, 1),
                        "l2": "flushed before each call"}
    del kp, vp
    # host block allocator: the batch-32 workload's requests (a 1024-token
    # shared prompt + private suffixes) through find / reserve / publish /
    # release, timed on the host
    alloc = pkv.BlockAllocator(16, 1024, 1 << 20)
    wl = gen.shared_prefix_b32()
    prompts = [np.concatenate([np.arange(1024, dtype=np.int32),
                               np.arange(int(L) - 1024, dtype=np.int32) + 10**6 * (i + 1)])
               for i, L in enumerate(wl.seq_lens)]
    t0 = time.perf_counter()
    rounds = 20
    for _ in range(rounds):
        ids = []
        for ptoks in prompts:
            r = alloc.begin()
            alloc.find_cached_prefix(r, ptoks)
            alloc.reserve(r, len(ptoks) + 1)
            alloc.publish(r, ptoks)
            ids.append(r)
        for r in ids:
            alloc.release(r)
    dt = time.perf_counter() - t0
    res["block_allocator"] = {"requests_per_s": round(rounds * len(prompts) / dt, 1),
                              "us_per_batch32": round(dt / rounds * 1e6, 1),
                              "tokens_per_batch": int(sum(len(x) for x in prompts)),
                              "pool_blocks": alloc.stats()[0],
                              "note": "host, single thread, via the Python binding"}
    # FP8 (E4M3) pools: the batch-32 shared-prefix step with the K/V cache in
    # FP8 (per-layer scales), timed like the contract line: steps back to
    # back, the split kernel's own duration from events on sampled steps
    w, fp8_step, fp8_decode, b, st = fp8_b32_setup(pkv, torch, dev)
    steps = 400
    for _ in range(10):
        fp8_step()
    torch.cuda.synchronize()
    pkv.profile_enable([])
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        if i % PROF_EVERY == 0:
            pkv.profile_mask([pkv.KERNEL_DECODE_SPLIT])
        fp8_step()
        if i % PROF_EVERY == 0:
            pkv.profile_mask([])
    e1.record()
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    s_step = e0.elapsed_time(e1) / steps / 1e3
    s_split = statistics.median(pkv.profile_times(pkv.KERNEL_DECODE_SPLIT)) / 1e3
    peak = peaks()[0]
    res["fp8_decode_b32"] = {"workload": w.name.replace("bf16", "fp8"), "step_us": round(s_step * 1e6, 2),
                             "tok_per_s": round(w.batch / s_step, 1),
                             "step_GB/s": round(b / s_step / 1e9, 1),
                             "split_kernel_us": round(s_split * 1e6, 2),
                             "split_kernel_us_stat": f"median of {steps // PROF_EVERY} timed launches",
                             "split_kernel_GB/s": round(b / s_split / 1e9, 1),
                             "split_kernel_frac_of_hbm_peak": round(b / s_split / 1e9 / peak, 3),
                             "kv_bytes": b, "scales": [float(gen.FP8_K_SCALE), float(gen.FP8_V_SCALE)],
                             "step": "append 1 token/row (quantized) + shared-prefix paged decode",
                             "l2": "no flush: 0.26 GB of K/V per step exceeds the 129 MB L2"}
    del fp8_step, fp8_decode
    # bulk append: every token of the batch-32 workload's private suffixes
    w = gen.shared_prefix_b32()
    n = int(np.sum(w.seq_lens - 1024))
    kp = torch.empty((w.num_blocks, 8, 16, 128), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    rows = np.repeat(np.arange(w.batch), w.seq_lens - 1024).astype(np.int32)
    pos = np.concatenate([np.arange(1024, L) for L in w.seq_lens]).astype(np.int32)
    slots = torch.from_numpy(pkv.slot_mapping_host(w.block_tables, w.num_blocks, rows, pos, 16)).to(dev)
    kn = torch.randn((n, 8, 128), dtype=torch.bfloat16, device=dev)
    vn = torch.randn_like(kn)
    s = time_loop(torch, lambda: pkv.paged_kv_append(kp, vp, slots, kn, vn), 50, 5)
    b = 2 * 2 * n * 8 * 128 * 2 + 4 * n
    res["bulk_append"] = {"tokens": n, "us": round(s * 1e6, 2), "GB/s": round(b / s / 1e9, 1),
                          "bytes": b}
    del kp, vp
    kp, vp = pkv.fp8_pools(w.num_blocks, 8, 128, dev)
    ks, vs = float(gen.FP8_K_SCALE), float(gen.FP8_V_SCALE)
    s = time_loop(torch, lambda: pkv.paged_kv_append(kp, vp, slots, kn, vn, k_scale=ks, v_scale=vs),
                  50, 5)
    b = 2 * n * 8 * 128 * (2 + 1) + 4 * n   # bf16 rows in, E4M3 codes out
    res["bulk_append_fp8"] = {"tokens": n, "us": round(s * 1e6, 2), "GB/s": round(b / s / 1e9, 1),
                              "bytes": b}
    return res


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline field)
# ---------------------------------------------------------------------------
def _oracle_setup(w):
    import oracle
    orc = oracle.load()
    slots, bad = orc.slot_mapping(w.block_tables, w.num_blocks, w.new_rows, w.new_pos, w.block_size)
    kp, vp = w.k_pool.copy(), w.v_pool.copy()
    orc.append(kp, vp, w.dtype, slots, w.k_new, w.v_new)
    return orc, kp, vp


def host_cpu():
    """(logical cores, CPU model string) of this host."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return os.cpu_count() or 1, model or "unknown"


def _oracle_rate(w, orc, kp, vp, budget_s, rows_order, threads=1):
    """Oracle rate for whole rows (all q heads each) taken in the given order,
    again from the start when every row is done, until about budget_s of wall
    time; the full step's time is extrapolated by attended keys.  With
    threads > 1 that many host threads each decode whole rows at once (the
    oracle's C calls release the interpreter lock), one row per call."""
    import threading
    bytes_step, _ = workload_bytes(w)
    full_keys = float(np.sum(w.seq_lens.astype(np.int64))) * w.num_q_heads
    lock = threading.Lock()
    state = {"next": 0, "keys": 0.0, "rows": []}
    t_start = time.perf_counter()

    def worker():
        while True:
            with lock:
                if time.perf_counter() - t_start >= budget_s:
                    return
                r = int(rows_order[state["next"] % len(rows_order)])
                state["next"] += 1
            pairs = np.array([[r, h] for h in range(w.num_q_heads)], dtype=np.int32)
            orc.decode(w.q, kp, vp, w.dtype, w.block_tables, w.seq_lens, w.window, w.scale,
                       pairs=pairs)
            with lock:
                state["keys"] += float(w.seq_lens[r]) * w.num_q_heads
                state["rows"].append(r)

    if threads == 1:
        worker()
    else:
        pool = [threading.Thread(target=worker) for _ in range(threads)]
        for t in pool:
            t.start()
        for t in pool:
            t.join()
    spent = time.perf_counter() - t_start
    t_full = spent * full_keys / state["keys"]
    return bytes_step / t_full / 1e9, state["rows"], spent


def cpu_baseline(w, budget_s=10.0):
    """The oracle timed on this host: one thread, then every logical core."""
    orc, kp, vp = _oracle_setup(w)
    order = gen.permutation(77, "cpu_rows", w.batch)
    nproc, model = host_cpu()
    value, rows, spent = _oracle_rate(w, orc, kp, vp, budget_s, order)
    value_all, rows_all, spent_all = _oracle_rate(w, orc, kp, vp, budget_s, order, threads=nproc)
    passes = len(rows) / w.batch
    return {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"decode of {len(rows)} whole rows ({passes:.2f} passes over the "
                      f"{w.batch} rows in the order {[int(r) for r in order]}; all "
                      f"{w.num_q_heads} q heads each; {spent:.1f} s single-threaded); "
                      "full-step time extrapolated by attended keys",
            "value_all_cores": round(value_all, 4), "cores_all": nproc,
            "sample_all_cores": f"{len(rows_all)} whole rows in the same order on {nproc} threads "
                                f"(one row per oracle call), {spent_all:.1f} s of wall time",
            "nproc": nproc, "cpu_model": model}


def contract_config(w, world):
    """The workload description both arms print (the same keys and values)."""
    return {"workload": w.name, "batch": w.batch, "q_heads": w.num_q_heads,
            "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
            "shared_prefix_tokens": w.shared_prefix_tokens, "suffix_tokens": "uniform 0..7168",
            "step": "append 1 token/row + shared-prefix paged decode",
            "kv_bytes_per_step": workload_bytes(w)[0], "parallelism": f"replicas x{world} (rows shard)",
            "l2": "no flush: 0.47 GB of K/V per step exceeds the 129 MB L2"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: every host core decodes whole rows of
    the batch-32 workload for a bounded time per step."""
    if rank != 0:
        return
    w = gen.shared_prefix_b32()
    orc, kp, vp = _oracle_setup(w)
    order = gen.permutation(77, "cpu_rows", w.batch)
    nproc, model = host_cpu()
    total_steps = args.steps + args.warmup
    per_step = max(0.05, min(5.0, 120.0 / max(total_steps, 1)))
    vals = []
    for i in range(total_steps):
        rot = np.roll(order, -i)
        v, rows, spent = _oracle_rate(w, orc, kp, vp, per_step, rot, threads=nproc)
        if i >= args.warmup:
            vals.append((v, spent, rows))
    value = statistics.median(v for v, _, _ in vals)
    ms_step = 1e3 * workload_bytes(w)[0] / (value * 1e9)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": contract_config(w, world),
            "arm": "the CPU oracle (IEEE double), bounded sample of whole rows per step",
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nproc, "kind": "oracle",
                             "cpu_model": model,
                             "sample": f"each step: whole rows (all q heads) on {nproc} threads for about "
                                       f"{per_step:.2f} s; full-step time extrapolated by attended keys"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_prefill_case(args, local):
    """Chunked prefill (4 x 512 queries vs a 16384-token prefix) timed alone."""
    import torch
    import block_paged_kv_gb300 as pkv
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = gen.chunked_prefill()

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    kp, vp, q, kn, vn = up(w.k_pool), up(w.v_pool), up(w.q), up(w.k_new), up(w.v_new)
    t = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    cu = torch.from_numpy(w.cu_q_lens).to(dev)
    slots = torch.from_numpy(pkv.slot_mapping_host(w.block_tables, w.num_blocks, w.new_rows,
                                                   w.new_pos, 16)).to(dev)
    pkv.paged_kv_append(kp, vp, slots, kn, vn)
    out = torch.empty_like(q)
    C = int(w.cu_q_lens[1] - w.cu_q_lens[0])
    s = time_loop(torch, lambda: pkv.paged_prefill_chunk_attention(q, cu, kp, vp, t, sl, C, 0, w.scale,
                                                                   out=out),
                  args.steps, args.warmup)
    keys = sum(int(L) - C + i + 1 for L in w.seq_lens for i in range(C))
    flops = 4 * w.head_dim * keys * w.num_q_heads
    print(json.dumps({"case": "chunked_prefill", "workload": w.name, "us": round(s * 1e6, 2),
                      "TFLOP/s": round(flops / s / 1e12, 1),
                      "frac_of_bf16_peak": round(flops / s / 1e12 / bf16_peak(), 3)}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--no-secondary", dest="secondary", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--case", choices=["step", "prefill", "fp8_decode", "append", "fp8_append",
                                       "fp8_prefill", "long_decode", "sliding_decode"],
                    default="step",
                    help="step: the decode step (the contract line); prefill / fp8_decode / append / "
                         "fp8_append / fp8_prefill / long_decode: time the chunked prefill, the FP8 "
                         "decode, the bulk append into bf16 or FP8 pools, the FP8 chunked prefill "
                         "or the long-context full-attention or sliding-window decode alone (for "
                         "profiling)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.case == "prefill":
        run_prefill_case(args, local)
    elif args.case == "fp8_decode":
        run_fp8_case(args, local)
    elif args.case == "fp8_append":
        run_append_case(args, local, fp8=True)
    elif args.case == "append":
        run_append_case(args, local)
    elif args.case == "fp8_prefill":
        run_fp8_prefill_case(args, local)
    elif args.case == "long_decode":
        run_long_case(args, local)
    elif args.case == "sliding_decode":
        run_long_case(args, local, sliding=True)
    else:
        run_pkv(args, rank, world, local)


if __name__ == "__main__":
    main()
