#!/usr/bin/env python
"""Benchmark of the paged KV-cache hot path on GB300.

One step = one decode step of one attention layer over a batch of sequences
whose K/V already sit in the paged pool: the new token of every sequence is
written through its slot mapping (kv_append), then paged decode attention
reads every sequence's blocks through its block table (split-KV partitions
plus the log-sum-exp merge when the plan has more than one split).

Default workload: Llama-3-8B-shaped paged decode (64 sequences, context
lengths uniform in [512, 4096], 32 query / 8 kv heads, head_dim 128, bf16,
16-token blocks shuffled across a pool 1.2x the blocks needed).

Metric: KV bytes read by decode attention per second (valid tokens only:
sum_b L_b * 2 * Hkv * D * 2 bytes) -- "value" -- plus decode tokens/s.

On one GPU the default run also measures, in the same process and with
short runs, the Yi-6B-shaped long-context decode (paged on the balanced
schedule and on the grid plan, and the contiguous path, with the
paged-vs-contiguous slowdown), the shared-prefix step and the Yi-34B-shaped
prefill with its chunk append; they go under "other_workloads"
(--no-extras skips them).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       [--splits S] [--plan auto|grid|balanced] [--prefix-splits P] [--impl reference]
Under torchrun each rank runs an independent replica (weak scaling).
Prints exactly one JSON line on stdout (rank 0).
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attn KV-read GB/s (fraction of HBM peak); decode tokens/s"
L2_BYTES = 129 * 1000 ** 2
FALLBACK_HBM_GBS = 6800.0

DESCR = {
    "llama3_8b_decode": "Llama-3-8B-shaped paged decode: 64 seqs, ctx U[512,4096], 32q/8kv heads, "
                        "head_dim 128, bf16, 16-token blocks shuffled in a 1.2x pool",
    "yi6b_long_decode": "Yi-6B-shaped long-context paged decode: 8 seqs, ctx log-U[32768,196608], "
                        "32q/4kv heads, head_dim 128, bf16, split-KV + LSE merge",
    "yi6b_long_decode_contig": "Yi-6B-shaped long-context decode on the contiguous "
                               "(cuMemMap-backed) KV path, same inputs as yi6b_long_decode",
    "yi34b_prefill": "Yi-34B-shaped chunked causal paged prefill: 4 seqs x (8192 cached + 2048 "
                     "new) tokens in shuffled 16-token blocks, 56q/8kv heads, head_dim 128, bf16",
    "vmm_pages": "vAttention page mapping: 8 requests reserved for 196608 tokens (4 kv heads, d128, "
                 "bf16) mapped to their lengths page by page, with and without the background page "
                 "pool",
    "swap_blocks": "swap 2048 shuffled 64 KiB blocks (Llama-3-8B-shaped pool, 8 kv heads, d128, "
                   "bf16) out to pinned host memory and back in",
    "shared_prefix_step": "append + decode step with shared prefix: 256 seqs, ctx U[128,2048], groups "
                          "of 16 share a 1024-token prefix (refcounted blocks, copy-on-write), "
                          "32q/8kv heads, head_dim 128, bf16",
}
PREFILL_METRIC = "chunked causal paged prefill tensor TFLOP/s (fraction of dense bf16 peak)"


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(*rel):
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, src_hash: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel \
                and parts[1] == workload and parts[2] == src_hash:
            return float(parts[3])
    return None


def max_over_ranks(ms: float, device=None) -> float:
    """The slowest rank's time (ms).  All ranks call it; with one process it
    returns ms unchanged."""
    import torch
    import torch.distributed as tdist

    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, steps: int, world: int, slowest_ms: float) -> float:
    """Whole-job rate: every rank processed units_per_rank per step (weak
    scaling), the job took the slowest rank's time."""
    return world * units_per_rank * steps / (slowest_ms * 1e-3)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# Workload set-up (shared by both arms: host arrays only)
# --------------------------------------------------------------------------
def kv_type(args):
    """The storage type of the K/V cache (and of q, the new rows and the
    output): the library's code and the workloads' name for it."""
    import paged_kv_cache_196_gb300 as pk
    f16 = getattr(args, "kv_dtype", "bf16") == "f16"
    return (pk.KV_F16 if f16 else pk.KV_BF16), ("f16" if f16 else "bf16")


def decode_workload(name, dtype=None):
    base = name.replace("_contig", "")
    cfg = W.CONFIGS[base]
    lens = W.decode_lengths(base)
    need = int(sum((int(L) + 15) // 16 for L in lens))  # blocks the contexts occupy
    nb = int(math.ceil(cfg["pool_factor"] * need))
    t0 = time.time()
    inp = W.decode_inputs(base, nb, dtype=dtype)
    log(f"[bench] generated {name} inputs in {time.time() - t0:.1f}s "
        f"({nb} blocks, {int(lens.sum())} tokens)")
    max_blocks = (cfg["len_hi"] + 15) // 16
    return cfg, inp, nb, max_blocks


# --------------------------------------------------------------------------
# Our arm
# --------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch

    import paged_kv_cache_196_gb300 as pk

    torch.cuda.set_device(local_rank)
    dist = world > 1
    if dist:
        import torch.distributed as tdist

    contig = args.workload.endswith("_contig")
    KVT, kvt = kv_type(args)
    cfg, inp, nb, max_blocks = decode_workload(args.workload, kvt)
    lens = inp["lens"]
    B, hq, hkv, d = len(lens), cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    e = 2
    kv_bytes = int(lens.sum()) * 2 * hkv * d * e
    scale = 1.0 / math.sqrt(d)

    # ---- host block manager: the allocation of every context's blocks
    alloc = pk.kv_allocator_create(nb)
    pk.kv_allocator_set_order(alloc, inp["perm"])
    tables = np.full((B, max_blocks), -1, np.int32)
    for b, L in enumerate(lens):
        pk.kv_prepare_append(alloc, tables[b], 0, 0, int(L), np.zeros(int(L), np.int64),
                             np.zeros(0, np.int32), np.zeros(0, np.int32))
    pk.kv_allocator_destroy(alloc)
    last = lens.astype(np.int64) - 1  # the new token of sequence b is its last position

    # ---- device state: the cache (paged pool or per-request virtual ranges)
    if not contig:
        pool = pk.kv_pool_create(nb, 16, hkv, d, KVT)
        if args.launch_overlap:
            pk.kv_pool_set_launch_overlap(pool, True)
        kp, vp = pk.kv_pool_ptrs(pool)
        _fill(kp, torch.from_numpy(inp["pool_k"].view(np.int16)))
        _fill(vp, torch.from_numpy(inp["pool_v"].view(np.int16)))
        d_tables = torch.from_numpy(tables).cuda()
        slots = tables[np.arange(B), last // 16].astype(np.int64) * 16 + last % 16
    else:
        ctx = pk.kv_contig_create(B, cfg["len_hi"], hkv, d, KVT)
        if args.launch_overlap:
            pk.kv_contig_set_launch_overlap(ctx, True)
        t0 = time.time()
        for b, L in enumerate(lens):
            pk.kv_contig_reserve(ctx, b)
            pk.kv_contig_ensure(ctx, b, int(L))
        map_s = time.time() - t0
        head_stride, page, _ = pk.kv_contig_layout(ctx)
        # sequence b's logical K/V (its blocks of the shuffled pool, in table
        # order) written through the library's contiguous append
        for b, L in enumerate(lens):
            j = np.arange(int(L))
            blk = tables[b, j // 16]
            rk = torch.from_numpy(np.ascontiguousarray(inp["pool_k"][blk, :, j % 16]).view(np.int16)).cuda()
            rv = torch.from_numpy(np.ascontiguousarray(inp["pool_v"][blk, :, j % 16]).view(np.int16)).cuda()
            pk.kv_contig_append(ctx, rk, rv,
                                torch.full((int(L),), b, dtype=torch.int32, device="cuda"),
                                torch.arange(int(L), dtype=torch.int32, device="cuda"), int(L))
            torch.cuda.synchronize()
            del rk, rv
        req_ids = torch.arange(B, dtype=torch.int32, device="cuda")
    d_lens = torch.from_numpy(lens).cuda()
    q = torch.from_numpy(inp["q"].view(np.int16)).cuda()
    g = W.rng(cfg["seed"] + 1000 + rank)
    k_new = torch.from_numpy(W.normal(g, (B, hkv, d), kvt).view(np.int16)).cuda()
    v_new = torch.from_numpy(W.normal(g, (B, hkv, d), kvt).view(np.int16)).cuda()
    out = torch.empty((B, hq, d), dtype=torch.int16, device="cuda")
    # the split plan: from the host-known lengths unless forced on the command line
    splits = args.splits if args.splits > 0 else pk.kv_decode_plan(lens, hkv, max_blocks)
    ws_bytes = pk.kv_decode_workspace_size(B, hq, hkv, d, max_blocks, splits)
    ws = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device="cuda")
    part_blocks, max_splits = pk.kv_decode_split_plan(B, hkv, max_blocks, splits)
    balanced = False
    if not contig:
        d_slots = torch.from_numpy(slots).cuda()
        # the grid takes the sequences longest first (one wave loads the SMs evenly)
        h_order = np.zeros(B, np.int32)
        pk.kv_decode_order(lens.astype(np.int32), h_order)
        d_order = torch.from_numpy(h_order).cuda()
        # or: one wave of CTAs with equal runs of blocks (host-made schedule);
        # "auto" takes it when its runs are long enough for the deep ring
        h_sched = pk.kv_decode_schedule(lens.astype(np.int32), hkv, max_blocks,
                                        num_ctas=args.sched_ctas, ring_stages=args.sched_ring,
                                        flags=pk.KV_SCHED_WHOLE_PIECES if args.sched_whole else 0)
        balanced = args.plan == "balanced" or (args.plan == "auto" and int(h_sched[4]) == 1)
        if balanced:
            d_sched = torch.from_numpy(h_sched).cuda()
            ws_bytes = pk.kv_decode_schedule_workspace_size(h_sched, hq, d)
            ws = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device="cuda")
            max_splits = int(h_sched[2])

    # One step: the new tokens' K/V go into their slots (contiguous path:
    # position seq_lens - 1 of each request), then decode over all tokens, in
    # one call (the append fused into the decode kernel).
    def step():
        if contig:
            pk.contig_append_and_decode(ctx, q, k_new, v_new, req_ids, d_lens, B, hq, scale, out,
                                        KVT, None, splits, ws, ws_bytes)
        elif balanced:
            pk.paged_decode_attention_scheduled(pool, q, d_tables, max_blocks, d_lens, B, hq, scale,
                                                h_sched, d_sched, out, KVT, None, ws,
                                                ws_bytes, k_new=k_new, v_new=v_new,
                                                slot_mapping=d_slots)
        else:
            pk.paged_append_and_decode(pool, q, k_new, v_new, d_slots, d_tables, max_blocks, d_lens,
                                       B, hq, scale, out, KVT, None, splits, ws, ws_bytes,
                                       seq_order=d_order)

    # merge_kernel runs only for plans of more than 32 splits
    launches_per_step = 1 + (1 if max_splits > 32 else 0)

    # ---- warm-up
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    err = pk.kv_contig_get_device_error(ctx) if contig else pk.kv_get_device_error(pool)
    if err:
        raise RuntimeError(f"device error word {err:#x} after warm-up")

    # ---- timed region (device time, inputs resident in HBM): K steps back to
    # back between two events
    K = args.steps
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if dist:
        tdist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for i in range(K):
        step()
    t_end.record()
    torch.cuda.synchronize()
    if dist:
        tdist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    # ---- the decode launch on its own, for the roofline: a shorter run of the
    # same steps with an event pair around each decode launch (the pairs cost
    # the steps a few microseconds, so they stay out of the timed region)
    Ka = min(K, 500)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(Ka)]
    for i in range(Ka):
        ev[i][0].record()
        step()
        ev[i][1].record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    attend_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    total_ms = max_over_ranks(total_ms, device="cuda")
    ms_per_step = total_ms / K
    value = job_throughput(kv_bytes, K, world, total_ms) / 1e9
    tokens_per_s = job_throughput(B, K, world, total_ms)

    # ---- end to end through the public API with host buffers, two ways.
    # First with staging copies: each step plans its grid order (or balanced
    # schedule) on the host from the host copy of the lengths, copies its
    # inputs (q, the new k/v, the slots or positions, the lengths, the order
    # or schedule) from a pinned host buffer in a single transfer, runs the
    # step on views of the device copy, and reads its output back.  Two pinned
    # input buffers, two device input buffers and two output buffers: step i's
    # inputs travel on a copy stream while step i - 1 computes, its output
    # travels back on another while step i + 1 computes (the steps themselves
    # stay in order on the compute stream).  Then without them (below).
    # Every step is the same decode step (same lengths, same slots), so the
    # slot mapping is planned once, before the loops.
    Ke = min(K, 2000)
    h_parts = [torch.from_numpy(inp["q"].view(np.int16)), k_new.cpu(), v_new.cpu()]
    if not contig:
        h_parts.append(torch.from_numpy(slots))
    h_parts.append(torch.from_numpy(lens))
    if not contig:
        h_parts.append(torch.from_numpy(h_sched if balanced else h_order))
    offs, total = [], 0
    for t in h_parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_ins = [torch.empty(total, dtype=torch.uint8).pin_memory() for _ in range(2)]
    for h_in in h_ins:
        for t, o in zip(h_parts, offs):
            n = t.numel() * t.element_size()
            h_in[o:o + n].view(t.dtype).copy_(t.reshape(-1))
    # numpy views of each pinned buffer's order / schedule slot, planned into per step
    plan_views = []
    if not contig:
        pt, po = h_parts[5], offs[5]
        for h_in in h_ins:
            plan_views.append(h_in[po:po + pt.numel() * 4].view(torch.int32).numpy())

    sched_scratch = (np.zeros(pk.kv_decode_schedule_capacity(B, hkv, max_blocks), np.int32)
                     if balanced else None)

    def plan(dst):
        if balanced:  # planned at the capacity bound, the used part copied in
            used = pk.kv_decode_schedule(lens.astype(np.int32), hkv, max_blocks,
                                         num_ctas=args.sched_ctas, ring_stages=args.sched_ring,
                                         flags=pk.KV_SCHED_WHOLE_PIECES if args.sched_whole else 0,
                                         out=sched_scratch)
            dst[:len(used)] = used
        else:
            pk.kv_decode_order(lens.astype(np.int32), dst)
    d_ins = [torch.empty(total, dtype=torch.uint8, device="cuda") for _ in range(2)]
    bufs = []
    for d_in in d_ins:
        views = []
        for t, o in zip(h_parts, offs):
            n = t.numel() * t.element_size()
            views.append(d_in[o:o + n].view(t.dtype).view(t.shape))
        bufs.append(views)
    outs = [out, torch.empty_like(out)]
    h_outs = [torch.empty((B, hq, d), dtype=torch.int16).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_parts)
    d2h = h_outs[0].numel() * 2
    s_comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def use(views, o):
        nonlocal q, k_new, v_new, d_slots, d_lens, d_sched, d_order, out
        q, k_new, v_new = views[0], views[1], views[2]
        if contig:  # q, k_new, v_new, lengths
            d_lens = views[3]
        else:  # q, k_new, v_new, slots, lengths, schedule or order
            d_slots = views[3]
            d_lens = views[4]
            if balanced:
                d_sched = views[5]
            else:
                d_order = views[5]
        out = o

    if dist:
        tdist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_comp)
    for i in range(Ke):
        bi = i % 2
        if plan_views:
            ev_in[bi].synchronize()  # step i - 2's copy out of this pinned buffer is done
            plan(plan_views[bi])
        s_in.wait_event(ev_comp[bi])  # step i - 2 has read this input buffer
        with torch.cuda.stream(s_in):
            d_ins[bi].copy_(h_ins[bi], non_blocking=True)
        ev_in[bi].record(s_in)
        s_comp.wait_event(ev_in[bi])
        s_comp.wait_event(ev_out[bi])  # step i - 2's output has been read back
        use(bufs[bi], outs[bi])
        step()
        ev_comp[bi].record(s_comp)
        s_out.wait_event(ev_comp[bi])
        with torch.cuda.stream(s_out):
            h_outs[bi].copy_(outs[bi], non_blocking=True)
        ev_out[bi].record(s_out)
    for bi in range(2):
        s_comp.wait_event(ev_out[bi])
    e1.record(s_comp)
    torch.cuda.synchronize()
    copy_ms = e0.elapsed_time(e1)
    copy_ms = max_over_ranks(copy_ms, device="cuda")
    copy_value = job_throughput(kv_bytes, Ke, world, copy_ms) / 1e9
    assert torch.equal(h_outs[(Ke - 1) % 2], outs[(Ke - 1) % 2].cpu())
    last_out = outs[(Ke - 1) % 2].clone()

    # ---- the same loop without staging copies: on a GB300 the GPU reads and
    # writes pinned host memory directly over NVLink-C2C, so each step's call
    # gets its inputs in a pinned host buffer (planned into on the host, as
    # above) and writes its output to a pinned host buffer, which the host
    # reads once the step is done.  A ring of NZ buffer pairs: before step i
    # reuses pair i % NZ, the host waits for step i - NZ (an event recorded
    # after each step) and reads that step's output.
    NZ = 4
    z_ins = [torch.empty(total, dtype=torch.uint8).pin_memory() for _ in range(NZ)]
    z_views, z_plans = [], []
    for z_in in z_ins:
        z_in.copy_(h_ins[0])
        views = []
        for t, o in zip(h_parts, offs):
            n = t.numel() * t.element_size()
            views.append(z_in[o:o + n].view(t.dtype).view(t.shape))
        z_views.append(views)
        if not contig:
            z_plans.append(z_in[po:po + pt.numel() * 4].view(torch.int32).numpy())
    z_outs = [torch.empty((B, hq, d), dtype=torch.int16).pin_memory() for _ in range(NZ)]
    z_done = [torch.cuda.Event() for _ in range(NZ)]
    z_read = 0
    torch.cuda.synchronize()
    e0.record(s_comp)
    for i in range(Ke):
        zi = i % NZ
        if i >= NZ:
            z_done[zi].synchronize()
            z_read ^= int(z_outs[zi][0, 0, 0])  # the host reads step i - NZ's output
        if z_plans:
            plan(z_plans[zi])
        use(z_views[zi], z_outs[zi])
        step()
        z_done[zi].record(s_comp)
    e1.record(s_comp)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, device="cuda")
    e2e_value = job_throughput(kv_bytes, Ke, world, e2e_ms) / 1e9
    # the same step's output, bit for bit, through both loops
    assert torch.equal(z_outs[(Ke - 1) % NZ], last_out.cpu())

    err = pk.kv_contig_get_device_error(ctx) if contig else pk.kv_get_device_error(pool)
    if err:
        raise RuntimeError(f"device error word {err:#x} after the timed region")

    peak, peak_kind = read_peaks()
    # With one launch per step the timed region is K back-to-back launches of
    # the kernel: its length over K bounds the mean launch duration from above
    # (it adds the gaps between launches).  Otherwise the event-pair run.
    pair_ms = attend_ms
    if launches_per_step == 1:
        attend_ms = min(attend_ms, total_ms / K)
    achieved = kv_bytes / (attend_ms * 1e-3) / 1e9
    src = source_hash("paged_kv_cache_196_gb300/csrc/decode.cu",
                      "paged_kv_cache_196_gb300/csrc/common.cuh")
    # bf16 / head_dim 128 with >= 3 query heads per kv head runs the tensor-core kernel
    kname = "decode_tc_kernel" if (hq // hkv >= 3 and d == 128) else "decode_kernel"
    if balanced:
        kname = "decode_tc_sched_kernel"
    traffic = recorded_traffic(kname, args.workload + ("_f16" if kvt == "f16" else ""), src)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": kvt,
        "data": "synthetic",
        "config": {
            "workload": DESCR[args.workload],
            "name": args.workload,
            "kv_dtype": kvt,
            "batch": B,
            "tokens": int(lens.sum()),
            "kv_bytes_per_step": kv_bytes,
            "num_splits": splits,
            "part_blocks": part_blocks,
            "max_splits": max_splits,
            "launch_overlap": bool(args.launch_overlap),
            "plan": ("balanced schedule%s: %d CTAs of up to %d blocks, %d-stage ring"
                     % (" (whole pieces, longest first)" if args.sched_whole else "",
                        int(h_sched[0]), int(h_sched[3]), 8 if int(h_sched[4]) else 4)
                     if balanced else "grid-indexed" + ("" if contig else ", longest first")),
            "l2": f"inputs larger than L2 ({kv_bytes / 1e6:.0f} MB of KV read per step vs "
                  f"{L2_BYTES / 1e6:.0f} MB L2); no flush",
            "parallelism": f"replicas x{world}",
        },
        "decode_tokens_per_s": round(tokens_per_s, 1),
        "roofline": {
            "bound": "hbm",
            "kernel": ("contig_append_and_decode" if contig else
                       "paged_decode_attention_scheduled" if balanced else "paged_append_and_decode")
                      + f" ({kname}" + ("" if kname == "decode_kernel" else ", the append fused")
                      + (" + split merge kernel)" if max_splits > 32 else ")"),
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} HBM copy bandwidth",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": kv_bytes,
            "avg_launch_ms": round(attend_ms, 5),
            "launch_ms_source": ("timed region / K (one launch per step)"
                                 if launches_per_step == 1 and attend_ms < pair_ms else
                                 "event pairs around %d launches" % Ka),
            "event_pair_ms": round(pair_ms, 5),
        },
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms / Ke, 5),
                "steps": Ke,
                "transfers": "the step's call reads its inputs from a pinned host buffer and writes "
                             "its output to a pinned host buffer over NVLink-C2C (no staging "
                             "copies); the host plans each step's order or schedule into the "
                             "buffer and reads each step's output; a ring of %d buffer pairs" % NZ},
        "e2e_copy_engine": {"value": round(copy_value, 1), "unit": "GB/s",
                            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                            "ms_per_step": round(copy_ms / Ke, 5), "steps": Ke,
                            "copies": "the same steps with staging copies: step i's inputs go "
                                      "host to device on a copy stream while step i - 1 computes, "
                                      "its output comes back on another while step i + 1 computes"},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
    }
    if contig:
        line["config"]["vmm"] = {"page_bytes": page, "map_seconds": round(map_s, 4),
                                 "head_stride_tokens": head_stride}
    if contig:
        pk.kv_contig_destroy(ctx)
    else:
        pk.kv_pool_destroy(pool)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp, nb, max_blocks)
    if dist:
        tdist.barrier()
    return line


def _fill(ptr, src):
    """Copies a host tensor into library-owned device memory (set-up only)."""
    import torch

    class _Raw:
        pass

    raw = _Raw()
    raw.__cuda_array_interface__ = {"shape": tuple(src.shape), "typestr": "<i2",
                                    "data": (ptr, False), "version": 3}
    torch.as_tensor(raw, device="cuda").copy_(src.cuda())


# --------------------------------------------------------------------------
# CPU oracle timings (baseline leg and reference arm)
# --------------------------------------------------------------------------
def _oracle_tables(inp, max_blocks):
    import oracle

    return oracle.build_block_tables(inp["lens"], 16, inp["perm"], max_blocks)


def cpu_baseline(cfg, inp, nb, max_blocks, budget_s=12.0):
    """The oracle, as it stands, on a bounded sample: sequences taken in
    order (all query heads), in growing batches, wrapping around the batch,
    until about budget_s seconds of CPU work."""
    import oracle

    tables = _oracle_tables(inp, max_blocks)
    hkv, d, hq = cfg["num_kv_heads"], cfg["head_dim"], cfg["num_q_heads"]
    lens = inp["lens"]
    B = len(lens)
    done, spent, nbytes, S = 0, 0.0, 0, 1
    while spent < budget_s:
        seqs = [(done + i) % B for i in range(S)]
        items = [(b, h) for b in seqs for h in range(hq)]
        t0 = time.time()
        oracle.paged_decode(inp["pool_k"], inp["pool_v"], tables, lens, inp["q"],
                            1 / math.sqrt(d), items=items)
        spent += time.time() - t0
        nbytes += int(lens[seqs].sum()) * 2 * hkv * d * 2
        done += S
        S = min(2 * S, 4 * B)
    return {"value": round(nbytes / spent / 1e9, 4), "unit": "GB/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{done} sequence decodes ({done / B:.1f} passes over the {B}-sequence "
                      f"batch), all {hq} query heads each, fp64 reassemble-then-softmax, "
                      f"{spent:.1f}s"}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is one (sequence, query
    head) of the workload, cycling through the batch."""
    import oracle

    cfg, inp, nb, max_blocks = decode_workload(args.workload)
    tables = _oracle_tables(inp, max_blocks)
    lens = inp["lens"]
    B, hq, hkv, d = len(lens), cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]

    def step(i):
        b, h = (i // hq) % B, i % hq
        oracle.paged_decode(inp["pool_k"], inp["pool_v"], tables, lens, inp["q"],
                            1 / math.sqrt(d), items=[(b, h)])
        return int(lens[b]) * 2 * d * 2  # this head's K and V bytes

    for i in range(args.warmup):
        step(i)
    t0 = time.time()
    nbytes = sum(step(args.warmup + i) for i in range(args.steps))
    dt = time.time() - t0
    value = nbytes / dt / 1e9
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": DESCR[args.workload], "name": args.workload, "batch": B},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "one (sequence, query head) per step, cycling the batch; "
                                   "a single item runs on one core"},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def read_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def run_prefill(args, rank, world, local_rank):
    """One prefill step: append the chunk's K/V through the slot mapping, then
    chunked causal paged prefill attention of the chunk's queries."""
    import torch

    import paged_kv_cache_196_gb300 as pk

    torch.cuda.set_device(local_rank)
    KVT, kvt = kv_type(args)
    cfg = W.CONFIGS["yi34b_prefill"]
    B, hq, hkv, d = cfg["batch"], cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    c_len, t_len = cfg["cached_len"], cfg["chunk_len"]
    L = c_len + t_len
    max_blocks = (L + 15) // 16
    nb = int(math.ceil(cfg["pool_factor"] * B * max_blocks))
    t0 = time.time()
    inp = W.prefill_inputs("yi34b_prefill", nb, dtype=kvt)
    log(f"[bench] generated yi34b_prefill inputs in {time.time() - t0:.1f}s")
    lens = np.full(B, L, np.int32)
    alloc = pk.kv_allocator_create(nb)
    pk.kv_allocator_set_order(alloc, inp["perm"])
    tables = np.full((B, max_blocks), -1, np.int32)
    slots = []
    for b in range(B):
        s = np.zeros(L, np.int64)
        pk.kv_prepare_append(alloc, tables[b], 0, 0, L, s, np.zeros(0, np.int32),
                             np.zeros(0, np.int32))
        slots.append(s[c_len:])
    pk.kv_allocator_destroy(alloc)
    slots = np.concatenate(slots)
    pool = pk.kv_pool_create(nb, 16, hkv, d, KVT)
    kp, vp = pk.kv_pool_ptrs(pool)
    _fill(kp, torch.from_numpy(inp["pool_k"].view(np.int16)))
    _fill(vp, torch.from_numpy(inp["pool_v"].view(np.int16)))
    T = B * t_len
    q = torch.from_numpy(inp["q"].view(np.int16)).cuda()
    k_new = torch.from_numpy(inp["k_new"].view(np.int16)).cuda()
    v_new = torch.from_numpy(inp["v_new"].view(np.int16)).cuda()
    d_slots = torch.from_numpy(slots).cuda()
    d_tables = torch.from_numpy(tables).cuda()
    d_lens = torch.from_numpy(lens).cuda()
    cu = torch.from_numpy(np.arange(0, T + 1, t_len, dtype=np.int32)).cuda()
    out = torch.empty((T, hq, d), dtype=torch.int16, device="cuda")
    scale = 1.0 / math.sqrt(d)
    pairs = B * hq * (t_len * c_len + t_len * (t_len + 1) // 2)
    flops = 4 * d * pairs

    def append():
        pk.kv_append(pool, k_new, v_new, d_slots, T)

    def attend():
        pk.paged_prefill_attention(pool, q, cu, T, t_len, d_tables, max_blocks, d_lens, B, hq,
                                   scale, out, KVT, None)

    for _ in range(args.warmup):
        append()
        attend()
    torch.cuda.synchronize()
    if pk.kv_get_device_error(pool):
        raise RuntimeError("device error word set after warm-up")
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(K):
        ea[i].record()
        append()
        ev[i][0].record()
        attend()
        ev[i][1].record()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = e0.elapsed_time(e1)
    attend_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    append_ms = float(np.mean([a.elapsed_time(b[0]) for a, b in zip(ea, ev)]))
    append_bytes = 2 * 2 * T * hkv * d * 2 + 8 * T  # read k/v_new, write the pool, slots
    if pk.kv_get_device_error(pool):
        raise RuntimeError("device error word set after the timed region")
    pk.kv_pool_destroy(pool)
    # The append alone, launches back to back between two events (an event
    # pair around a ~10 us kernel adds microseconds of its own).  Four chunks
    # of new K/V with disjoint destination blocks are taken in turn, 268 MB
    # of sources and destinations together, more than L2: each launch reads
    # its inputs from HBM and its destination lines are written back.
    R = 4
    apool = pk.kv_pool_create(R * T // 16, 16, hkv, d, KVT)
    g_app = W.rng(cfg["seed"] + 2000)
    sets = []
    for r in range(R):
        ks = torch.from_numpy(W.normal(g_app, (T, hkv, d), kvt).view(np.int16)).cuda()
        vs = torch.from_numpy(W.normal(g_app, (T, hkv, d), kvt).view(np.int16)).cuda()
        # chunk r's tokens fill the blocks of region r of the pool, shuffled
        perm = W.permutation(g_app, T // 16).astype(np.int64)
        j = np.arange(T, dtype=np.int64)
        sl = torch.from_numpy((r * (T // 16) + perm[j // 16]) * 16 + j % 16).cuda()
        sets.append((ks, vs, sl))
    for r in range(R):
        pk.kv_append(apool, sets[r][0], sets[r][1], sets[r][2], T)
    Kb = min(K, 200) // R * R or R
    eb0 = torch.cuda.Event(enable_timing=True)
    eb1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    eb0.record()
    for i in range(Kb):
        ks, vs, sl = sets[i % R]
        pk.kv_append(apool, ks, vs, sl, T)
    eb1.record()
    torch.cuda.synchronize()
    append_b2b_ms = eb0.elapsed_time(eb1) / Kb
    if pk.kv_get_device_error(apool):
        raise RuntimeError("device error word set after the append timing")
    pk.kv_pool_destroy(apool)
    # context: one plain device copy of the same bytes (a buffer the size of
    # the new K and V together into another), cycled over four such pairs
    srcs = [torch.cat([k_.reshape(-1), v_.reshape(-1)]) for k_, v_, _ in sets]
    dsts = [torch.empty_like(x) for x in srcs]
    torch.cuda.synchronize()
    eb0.record()
    for i in range(Kb):
        dsts[i % R].copy_(srcs[i % R])
    eb1.record()
    torch.cuda.synchronize()
    copy_ms = eb0.elapsed_time(eb1) / Kb
    del sets, srcs, dsts
    peak, kind = read_tensor_peak()
    achieved = flops / (attend_ms * 1e-3) / 1e12
    sfx = "_f16" if kvt == "f16" else ""
    line = {
        "metric": PREFILL_METRIC, "value": round(flops * K / (total_ms * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": kvt, "data": "synthetic",
        "config": {"workload": DESCR["yi34b_prefill"], "name": "yi34b_prefill", "kv_dtype": kvt,
                   "flop_per_step": flops, "append_tokens_per_step": T,
                   "l2": "KV 168 MB + Q 117 MB per step, larger than L2; no flush"},
        "prefill_tokens_per_s": round(T * K / (total_ms * 1e-3), 1),
        "append": {"tokens": T, "bytes": append_bytes,
                   "avg_ms": round(append_b2b_ms, 5),
                   "gbs": round(append_bytes / (append_b2b_ms * 1e-3) / 1e9, 1),
                   "frac_of_hbm_peak": round(append_bytes / (append_b2b_ms * 1e-3) / 1e9 /
                                             read_peaks()[0], 4),
                   "timing": f"{Kb} appends back to back between two events, cycling {R} "
                             f"chunks with disjoint destinations ({R * append_bytes / 1e6:.0f} MB "
                             "of sources and destinations, more than L2)",
                   "in_step_event_pair_ms": round(append_ms, 5),
                   "same_bytes_device_copy_ms": round(copy_ms, 5),
                   "frac_of_same_bytes_copy": round(copy_ms / append_b2b_ms, 4),
                   "kernel": "kv_append (append_kernel)",
                   "traffic": recorded_traffic("append_kernel", "yi34b_prefill_chunk" + sfx, source_hash(
                       "paged_kv_cache_196_gb300/csrc/pool.cu"))},
        "roofline": {"bound": "tensor", "kernel": "paged_prefill_attention (prefill_kernel)",
                     "achieved": round(achieved, 2), "peak": peak,
                     "peak_kind": f"{kind} dense bf16 (cuBLAS burst)" + (
                         "; fp16 has the same nominal dense rate (ratio 1)" if sfx else ""),
                     "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic("prefill_kernel", "yi34b_prefill" + sfx, source_hash(
                         "paged_kv_cache_196_gb300/csrc/prefill.cu",
                         "paged_kv_cache_196_gb300/csrc/tc.cuh",
                         "paged_kv_cache_196_gb300/csrc/common.cuh")),
                     "algorithmic_flop_per_launch": flops, "avg_launch_ms": round(attend_ms, 4)},
        "gpu_launches": 2 * K, "clocks": clk,
    }
    return line


def run_shared_prefix(args, rank, world, local_rank):
    """One decode step over sequences that share prefix blocks: the planned
    copy-on-write block copies, the append of every sequence's new token and
    decode attention over the L+1 tokens -- the cascade decode (each group's
    shared blocks read once), with the plain paged decode of the same step
    timed beside it."""
    import torch

    import paged_kv_cache_196_gb300 as pk

    torch.cuda.set_device(local_rank)
    inp = W.shared_prefix_inputs()
    lens = inp["lens"]
    B, G, P = len(lens), inp["group_size"], inp["prefix_len"]
    hkv, d = inp["new_k"].shape[1], inp["new_k"].shape[2]
    hq = inp["q"].shape[1]
    max_blocks = (int(lens.max()) + 1 + 15) // 16
    need = sum(-(-(int(L) + 1) // 16) for L in lens)
    nb = int(math.ceil(1.2 * need)) + (B // G + 1) * (P // 16)
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16)
    alloc = pk.kv_pool_allocator(pool)
    pk.kv_allocator_set_order(alloc, W.permutation(W.rng(W.CONFIGS["shared_prefix_step"]["seed"] + 7), nb))
    none = np.zeros(0, np.int32)
    tables = np.full((B, max_blocks), -1, np.int32)
    nblocks = np.zeros(B, np.int32)
    templates = {}

    def put(k, v, slots):
        if len(slots):
            pk.kv_append(pool, torch.from_numpy(np.ascontiguousarray(k).view(np.int16)).cuda(),
                         torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).cuda(),
                         torch.from_numpy(np.asarray(slots, np.int64)).cuda(), len(slots))

    for b in range(B):  # the cache as it stands before the step (shared prefixes)
        g, L = b // G, int(lens[b])
        if g not in templates:
            row = np.full(P // 16, -1, np.int32)
            s = np.zeros(P, np.int64)
            pk.kv_prepare_append(alloc, row, 0, 0, P, s, none, none)
            put(inp["prefix_k"][g], inp["prefix_v"][g], s)
            templates[g] = row
        nbp = -(-min(L, P) // 16)
        tables[b, :nbp] = templates[g][:nbp]
        pk.kv_allocator_share(alloc, tables[b, :nbp])
        nblocks[b] = nbp
        if L > P:
            s = np.zeros(L - P, np.int64)
            nblocks[b], _ = pk.kv_prepare_append(alloc, tables[b], int(nblocks[b]), P, L - P, s,
                                                 none, none)
            put(inp["suffix_k"][b], inp["suffix_v"][b], s)
    for row in templates.values():
        pk.kv_allocator_free(alloc, row)
    # ---- host step: plan the whole batch's appends (new blocks, copy-on-write)
    slots = np.zeros(B, np.int64)
    cow_src, cow_dst = np.zeros(B, np.int32), np.zeros(B, np.int32)
    t0 = time.perf_counter()
    n_cow = pk.kv_prepare_append_batch(alloc, tables, nblocks, lens.astype(np.int64),
                                       np.ones(B, np.int32), slots, cow_src, cow_dst)
    plan_ms = (time.perf_counter() - t0) * 1e3
    new_lens = (lens + 1).astype(np.int32)
    logical_bytes = int(new_lens.sum()) * 2 * hkv * d * 2
    held = {}  # tokens each distinct physical block holds for its longest user
    for b in range(B):
        for i in range(int(nblocks[b])):
            blk = int(tables[b, i])
            held[blk] = max(held.get(blk, 0), min(16, int(new_lens[b]) - 16 * i))
    unique_tokens = sum(held.values())
    unique_bytes = unique_tokens * 2 * hkv * d * 2
    d_src = torch.from_numpy(cow_src[:max(n_cow, 1)]).cuda()
    d_dst = torch.from_numpy(cow_dst[:max(n_cow, 1)]).cuda()
    d_slots = torch.from_numpy(slots).cuda()
    d_tables = torch.from_numpy(tables).cuda()
    d_lens = torch.from_numpy(new_lens).cuda()
    k_new = torch.from_numpy(inp["new_k"].view(np.int16)).cuda()
    v_new = torch.from_numpy(inp["new_v"].view(np.int16)).cuda()
    q = torch.from_numpy(inp["q"].view(np.int16)).cuda()
    out = torch.empty((B, hq, d), dtype=torch.int16, device="cuda")
    splits = args.splits if args.splits > 0 else pk.kv_decode_plan(new_lens, hkv, max_blocks)
    ws_bytes = pk.kv_decode_workspace_size(B, hq, hkv, d, max_blocks, splits)
    ws = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    # cascade: a sequence's shared tokens are its leading table entries that
    # are still its group's prefix blocks after this step's copy-on-write plan
    groups = -(-B // G)
    group_seqs = np.full((groups, G), -1, np.int32)
    shared = np.zeros(B, np.int32)
    for b in range(B):
        group_seqs[b // G, b % G] = b
        tpl = templates[b // G]
        k = 0
        while k < len(tpl) and tables[b, k] == tpl[k]:
            k += 1
        shared[b] = k * 16
    prefix_blocks = P // 16
    psplits = pk.kv_cascade_plan(groups, hkv, prefix_blocks, args.prefix_splits)
    suffix_lens = np.maximum(new_lens - (shared // 16) * 16, 1).astype(np.int32)
    csplits = args.splits if args.splits > 0 else pk.kv_decode_plan(suffix_lens, hkv, max_blocks)
    wsc_bytes = pk.kv_cascade_workspace_size(B, hq, hkv, d, max_blocks, csplits, psplits)
    wsc = torch.empty(max(wsc_bytes // 4, 1), dtype=torch.float32, device="cuda")
    d_groups = torch.from_numpy(group_seqs).cuda()
    d_shared = torch.from_numpy(shared).cuda()
    # the suffix grid's order: longest own part first, the one-block suffixes
    # after the first 40% (kv_cascade_order)
    s_order = np.zeros(B, np.int32)
    pk.kv_cascade_order(suffix_lens, s_order)
    d_sorder = torch.from_numpy(s_order).cuda()

    def decode_plain():
        pk.paged_decode_attention(pool, q, d_tables, max_blocks, d_lens, B, hq, scale, out,
                                  pk.KV_BF16, None, splits, ws, ws_bytes)

    def decode_cascade():
        pk.paged_decode_attention_cascade(pool, q, d_tables, max_blocks, d_lens, B, hq, scale,
                                          d_groups, groups, G, d_shared, prefix_blocks, psplits,
                                          out, pk.KV_BF16, None, csplits, wsc, wsc_bytes,
                                          seq_order=d_sorder)

    def step(ev=None, decode=decode_cascade):
        if n_cow:
            pk.kv_copy_blocks(pool, d_src, d_dst, n_cow)
        pk.kv_append(pool, k_new, v_new, d_slots, B)
        if ev is not None:
            ev[0].record()
        decode()
        if ev is not None:
            ev[1].record()

    for _ in range(args.warmup):
        step()
        step(decode=decode_plain)
    torch.cuda.synchronize()
    if pk.kv_get_device_error(pool):
        raise RuntimeError("device error word set after warm-up")
    # the plain paged decode of the same step, for comparison (not the timed value)
    pl = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for i in range(args.steps):
        step(pl[i], decode=decode_plain)
    torch.cuda.synchronize()
    plain_ms = float(np.mean([a.elapsed_time(b) for a, b in pl]))
    K = args.steps
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(K):
        step()
    e1.record()
    torch.cuda.synchronize()
    total_ms = e0.elapsed_time(e1)
    # the cascade decode on its own (event pairs around it), outside the timed steps
    Ka = min(K, 500)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ka)]
    for i in range(Ka):
        step(evs[i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    dec_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    if pk.kv_get_device_error(pool):
        raise RuntimeError("device error word set after the timed region")
    peak, peak_kind = read_peaks()
    achieved = unique_bytes / (dec_ms * 1e-3) / 1e9
    pk.kv_pool_destroy(pool)
    return {
        "metric": METRIC, "value": round(logical_bytes * K / (total_ms * 1e-3) / 1e9, 1),
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": DESCR["shared_prefix_step"], "name": "shared_prefix_step",
                   "batch": B, "logical_kv_bytes_per_step": logical_bytes,
                   "unique_kv_bytes_per_step": unique_bytes, "cow_copies_per_step": n_cow,
                   "cow_bytes_per_step": n_cow * 2 * hkv * 16 * d * 2 * 2,
                   "host_plan_ms": round(plan_ms, 3), "num_splits": csplits,
                   "prefix_splits": psplits, "groups": groups,
                   "l2": f"unique KV read per step ({unique_bytes / 1e6:.0f} MB) larger than L2; "
                         "no flush"},
        "decode_tokens_per_s": round(B * K / (total_ms * 1e-3), 1),
        "decode_ms": {"cascade": round(dec_ms, 5), "plain_paged": round(plain_ms, 5),
                      "plain_paged_logical_gbs": round(logical_bytes / (plain_ms * 1e-3) / 1e9, 1)},
        "roofline": {"bound": "hbm",
                     "kernel": "paged_decode_attention_cascade (cascade_prefix_kernel + decode_tc_kernel)",
                     "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth; algorithmic bytes = unique KV "
                                  "(shared blocks once per group, each sequence's own blocks)",
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "algorithmic_bytes_per_launch": unique_bytes, "avg_launch_ms": round(dec_ms, 5)},
        "gpu_launches": (4 if n_cow else 3) * K, "clocks": clk,
    }


def run_swap(args, rank, world, local_rank):
    """Swap-out then swap-in of 2048 blocks between the pool and pinned host
    memory (kernels that store to / load from the host buffer directly),
    against one copy-engine transfer of the same bytes each way."""
    import torch

    import paged_kv_cache_196_gb300 as pk

    torch.cuda.set_device(local_rank)
    cfg = W.CONFIGS["llama3_8b_decode"]
    hkv, d, nb, n = cfg["num_kv_heads"], cfg["head_dim"], 8192, 2048
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16)
    ids = torch.from_numpy(W.permutation(W.rng(cfg["seed"]), nb)[:n]).cuda()
    nbytes = pk.kv_swap_bytes(pool, n)
    buf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def time_it(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    t_out = time_it(lambda: pk.kv_swap_out(pool, ids, n, buf))
    t_in = time_it(lambda: pk.kv_swap_in(pool, ids, n, buf))
    t_d2h = time_it(lambda: buf.copy_(dbuf, non_blocking=True))
    t_h2d = time_it(lambda: dbuf.copy_(buf, non_blocking=True))
    if pk.kv_get_device_error(pool):
        raise RuntimeError("device error word set")
    gbs = lambda ms: round(nbytes / (ms * 1e-3) / 1e9, 1)
    total_ms = t_out + t_in
    return {
        "metric": "swap block-copy GB/s (pool <-> pinned host)", "value": round(2 * nbytes / (total_ms * 1e-3) / 1e9, 1),
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": DESCR["swap_blocks"], "name": "swap_blocks", "blocks": n,
                   "bytes_each_way": nbytes},
        "swap_out_gbs": gbs(t_out), "swap_in_gbs": gbs(t_in),
        "roofline": {"bound": "host link", "kernel": "swap_blocks_kernel",
                     "achieved": round(nbytes / (min(t_out, t_in) * 1e-3) / 1e9, 1),
                     "peak": max(gbs(t_d2h), gbs(t_h2d)),
                     "peak_kind": "copy-engine transfer of the same bytes measured in this run",
                     "unit": "GB/s", "frac": round(min(t_d2h, t_h2d) / min(t_out, t_in), 4),
                     "traffic": None, "copy_engine_d2h_gbs": gbs(t_d2h), "copy_engine_h2d_gbs": gbs(t_h2d)},
        "gpu_launches": 2 * args.steps, "clocks": None,
    }


def run_vmm(args, rank, world, local_rank):
    """Host latency of the contiguous path's page mapping: kv_contig_ensure
    (cuMemCreate + cuMemMap + cuMemSetAccess per 2 MiB page) against the same
    with pages pre-created by the background pool, and kv_contig_release
    (unmap + release) against unmap + recycle."""
    import torch

    import paged_kv_cache_196_gb300 as pk

    torch.cuda.set_device(local_rank)
    cfg = W.CONFIGS["yi6b_long_decode"]
    lens = W.decode_lengths("yi6b_long_decode")
    res = {}
    for mode in ("cold", "pool"):
        ctx = pk.kv_contig_create(len(lens), cfg["len_hi"], cfg["num_kv_heads"], cfg["head_dim"],
                                  pk.KV_BF16)
        if mode == "pool":
            pk.kv_contig_page_pool(ctx, 512, 1024)
            t0 = time.time()
            while pk.kv_contig_page_stats(ctx)["spare"] < 512 and time.time() - t0 < 30:
                time.sleep(0.01)
        t0 = time.perf_counter()
        for b, L in enumerate(lens):
            pk.kv_contig_reserve(ctx, b)
            pk.kv_contig_ensure(ctx, b, int(L))
        t_map = time.perf_counter() - t0
        t0 = time.perf_counter()
        for b in range(len(lens)):
            pk.kv_contig_release(ctx, b)
        t_rel = time.perf_counter() - t0
        st = pk.kv_contig_page_stats(ctx)
        res[mode] = {"map_us_per_page": round(st["map_us"], 2), "unmap_us_per_page": round(st["unmap_us"], 2),
                     "ensure_total_ms": round(t_map * 1e3, 2), "release_total_ms": round(t_rel * 1e3, 2),
                     "pages_created": st["created"], "pages_reused": st["reused"]}
        pk.kv_contig_destroy(ctx)
    pages = res["cold"]["pages_created"]
    return {
        "metric": "contiguous-path page mapping latency (host, per 2 MiB page)",
        "value": res["pool"]["map_us_per_page"], "unit": "us/page", "n_gpus": world, "steps": 1,
        "warmup": 0, "ms_per_step": res["pool"]["ensure_total_ms"], "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": DESCR["vmm_pages"], "name": "vmm_pages", "pages": pages},
        "cold": res["cold"], "pool": res["pool"], "gpu_launches": 0, "clocks": None,
    }


# --------------------------------------------------------------------------
# The other workloads, measured in the same process as the headline
# --------------------------------------------------------------------------
def _summary(line):
    r = line.get("roofline", {})
    out = {"value": line["value"], "unit": line["unit"], "ms_per_step": line["ms_per_step"],
           "steps": line["steps"],
           "roofline": {k: r.get(k) for k in ("bound", "kernel", "achieved", "peak", "unit", "frac",
                                              "avg_launch_ms")},
           "clocks": line.get("clocks")}
    if "e2e" in line:
        out["e2e"] = {"value": line["e2e"]["value"], "unit": line["e2e"]["unit"]}
    if "e2e_copy_engine" in line:
        out["e2e_copy_engine"] = {"value": line["e2e_copy_engine"]["value"],
                                  "unit": line["e2e_copy_engine"]["unit"]}
    plan = line["config"].get("plan")
    if plan:
        out["plan"] = plan
    return out


def run_extras(args, local_rank):
    """Short runs of the Yi-6B decode (paged, balanced schedule and grid plan;
    contiguous), the shared-prefix step, the Yi-34B prefill (with its chunk
    append), and the Llama-3-8B decode and Yi-34B prefill on fp16 storage,
    one after another in this process, for the headline line."""
    sub = argparse.Namespace(**vars(args))
    sub.steps = max(20, min(args.steps, 300))
    sub.warmup = max(3, min(args.warmup, 10))
    sub.no_cpu_baseline = True
    sub.splits = 0
    res = {}
    runs = [("yi6b_long_decode", "auto"), ("yi6b_long_decode_grid", "grid"),
            ("yi6b_long_decode_contig", "auto"), ("shared_prefix_step", "auto"),
            ("yi34b_prefill", "auto"), ("llama3_8b_decode_f16", "auto"), ("yi34b_prefill_f16", "auto")]
    for key, plan in runs:
        sub.workload = key.replace("_grid", "").replace("_f16", "")
        sub.kv_dtype = "f16" if key.endswith("_f16") else "bf16"
        sub.plan = plan
        t0 = time.time()
        if sub.workload == "yi34b_prefill":
            line = run_prefill(sub, 0, 1, local_rank)
        elif sub.workload == "shared_prefix_step":
            line = run_shared_prefix(sub, 0, 1, local_rank)
        else:
            line = run_ours(sub, 0, 1, local_rank)
        res[key] = _summary(line)
        if key == "yi34b_prefill":
            res["prefill_chunk_append"] = line["append"]
        if key == "shared_prefix_step":
            res[key]["decode_ms"] = line["decode_ms"]
        log(f"[bench] extra workload {key}: {line['value']} {line['unit']} "
            f"({time.time() - t0:.1f}s)")
    paged = res["yi6b_long_decode"]["value"]
    grid = res["yi6b_long_decode_grid"]["value"]
    contig = res["yi6b_long_decode_contig"]["value"]
    # slowdown = t_paged / t_contig - 1 over the same KV bytes; positive: paged slower
    res["yi6b_paged_vs_contiguous"] = {
        "paged_gbs": paged, "paged_grid_gbs": grid, "contiguous_gbs": contig,
        "slowdown_paged_balanced": round(contig / paged - 1, 4),
        "slowdown_paged_same_grid_plan": round(contig / grid - 1, 4),
        "target": "paged no more than 5% slower (slowdown <= 0.05)"}
    return res



def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="llama3_8b_decode", choices=sorted(DESCR))
    ap.add_argument("--splits", type=int, default=0,
                    help="0 = plan from the host-known lengths (kv_decode_plan)")
    ap.add_argument("--plan", default="auto", choices=["auto", "grid", "balanced"],
                    help="paged decode: grid-indexed split plan, balanced schedule, or auto "
                         "(balanced when its runs take the deep ring: long contexts)")
    ap.add_argument("--sched-ctas", type=int, default=0,
                    help="balanced plan: CTAs (0 = kv_decode_schedule's rule)")
    ap.add_argument("--sched-whole", action="store_true",
                    help="balanced plan: one piece per CTA (KV_SCHED_WHOLE_PIECES)")
    ap.add_argument("--sched-ring", type=int, default=0, choices=[0, 4, 8],
                    help="balanced plan: ring stages (0 = kv_decode_schedule's rule)")
    ap.add_argument("--launch-overlap", action=argparse.BooleanOptionalAction, default=True,
                    help="decode: back-to-back launches may overlap (kv_pool_set_launch_overlap, "
                         "kv_contig_set_launch_overlap; on by default)")
    ap.add_argument("--prefix-splits", type=int, default=0,
                    help="shared-prefix step: key-range partitions of each group's prefix "
                         "(0 = kv_cascade_plan)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "f16"],
                    help="storage type of the K/V cache, q and the output (decode and prefill "
                         "workloads); the workloads' inputs are the same draws rounded to it")
    ap.add_argument("--no-extras", action="store_true",
                    help="default workload: skip the short runs of the other workloads that "
                         "the headline line reports under other_workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return  # the reference arm runs on rank 0 only
        if args.workload in ("yi34b_prefill", "shared_prefix_step", "swap_blocks", "vmm_pages"):
            print(json.dumps({"impl": "reference", "unavailable":
                              "the reference arm times the decode workloads only"}), flush=True)
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as tdist

        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.workload == "yi34b_prefill":
        line = run_prefill(args, rank, world, local_rank)
    elif args.workload == "shared_prefix_step":
        line = run_shared_prefix(args, rank, world, local_rank)
    elif args.workload == "swap_blocks":
        line = run_swap(args, rank, world, local_rank)
    elif args.workload == "vmm_pages":
        line = run_vmm(args, rank, world, local_rank)
    else:
        line = run_ours(args, rank, world, local_rank)
    if world == 1 and args.workload == "llama3_8b_decode" and not args.no_extras:
        line["other_workloads"] = run_extras(args, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as tdist

        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
