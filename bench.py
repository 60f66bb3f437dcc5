#!/usr/bin/env python3
"""Benchmark of the paged KV-cache hot path on GB300.

Workload (per GPU): the batched-decode batch -- 64 sequences with context lengths uniform in
[512, 4096], 32 query / 8 KV heads, head_dim 128, 16-position pages shuffled over a pool
with 10% free pages, bf16 K/V ~ N(0,1) (seeded, synthetic).

One step = the whole decode hot path over that batch:
    slot mapping of the 64 new tokens -> store of their K/V -> split-K paged decode -> merge.
`value` is algorithmic bytes per step (K/V of every cached position read once, Q read, O
written, new K/V read and written) over device time, inputs resident in HBM, L2 flushed
between steps.  The line also carries the append-prefill leg (KV-rewind workload: 1,000
documents x 50 new tokens over 300 cached, page sizes 16 and 64) with its TFLOP/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvc|reference]

`--impl reference` times the CPU oracle (fp64) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "paged decode attention HBM GB/s (% of GB300 peak); append-prefill TFLOP/s"
WORKLOAD = ("batched-decode: 64 seqs, ctx U[512,4096], 32 q / 8 kv heads, head_dim 128, "
            "page 16, bf16, 10% free pages, pages shuffled")


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["kvc", "reference"], default="kvc")
    p.add_argument("--flush-mb", type=int, default=512,
                   help="L2 flush: MB written, then half as many read")
    p.add_argument("--append-steps", type=int, default=60)
    p.add_argument("--append-docs", type=int, default=1000,
                   help="documents in the rewind-append leg (smaller for profiler captures)")
    p.add_argument("--no-append", action="store_true")
    p.add_argument("--no-legs", action="store_true",
                   help="skip the shared-prefix and long-context decode legs")
    p.add_argument("--leg-steps", type=int, default=30)
    p.add_argument("--legs", type=lambda v: v.split(","),
                   default=["tiny_decode", "shared_prefix", "long_decode", "int8_decode",
                            "hnd_decode", "page_copy"],
                   help="comma-separated decode legs to run (default: all)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-headline", action="store_true",
                   help="skip the batched-decode step and print only the legs (profiler captures)")
    p.add_argument("--append-page-sizes", type=lambda v: [int(x) for x in v.split(",")],
                   default=[16, 64], help="page sizes of the rewind-append leg")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=5.0,
                   help="seconds of oracle passes over the headline batch (the other legs' "
                        "oracle runs take one pass of their workload)")
    return p.parse_args()


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------------------

def decode_bytes(case) -> int:
    """K and V of every cached position read once, Q read, O written (bf16)."""
    per_pos = 2 * case.kv_heads * case.head_dim * 2
    qo = 2 * case.num_seqs * case.q_heads * case.head_dim * 2
    return int(case.context_lens.astype(np.int64).sum()) * per_pos + qo


def store_bytes(case) -> int:
    """New K/V read and written, slots written and read."""
    row = case.kv_heads * case.head_dim * 2
    return case.num_tokens * (2 * row * 2 + 8)


def fused_work(case) -> int:
    """Bytes of one kvc_append_store: the chunk's K/V read once and written to the pools, the
    cached positions' K/V read, Q read, O written."""
    row = 2 * case.kv_heads * case.head_dim * 2          # K and V of one position
    cached = int((case.context_lens - case.q_lens).clip(min=0).sum())
    qo = 2 * case.num_tokens * case.q_heads * case.head_dim * 2
    return 2 * case.num_tokens * row + cached * row + qo


def append_work(case, int8: bool = False):
    """(bytes, flops) of one append: K/V of each sequence's visible positions read once, Q
    read, O written; 4*D flops per (query head, visible key) pair (QK and PV).  INT8 pages:
    D one-byte codes and a 4-byte scale per cached vector."""
    vec = case.head_dim + 4 if int8 else case.head_dim * 2
    per_pos = 2 * case.kv_heads * vec
    q_lens = case.q_lens.astype(np.int64)
    ctx = case.context_lens.astype(np.int64)
    kv = int(ctx.sum()) * per_pos
    qo = 2 * case.num_tokens * case.q_heads * case.head_dim * 2
    # token i sees ctx - q_len + i + 1 keys
    pairs = int((q_lens * (ctx - q_lens) + q_lens * (q_lens + 1) // 2).sum())
    flops = 4 * case.head_dim * case.q_heads * pairs
    return kv + qo, flops


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.2)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.remove(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; timing only -- the path has no collective)
# ---------------------------------------------------------------------------------------

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "kvc" else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def rank_seed(config: int, rank: int):
    """Workload seed of a rank: rank 0 runs the named configuration's own inputs, every other
    rank a different seeded batch of the same shape (replicas process distinct work)."""
    from workloads.configs import SEED_BASE
    return None if rank == 0 else SEED_BASE + config + 1000 * rank


def whole_job_value(world: int, bytes_per_step: int, steps: int, max_total_ms: float) -> float:
    """GB/s over all ranks: every rank moved bytes_per_step per step; time is the slowest
    rank's total over the timed steps."""
    return world * bytes_per_step * steps / (max_total_ms / 1e3) / 1e9


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# Sources (under the package's csrc/) that make up each profiled kernel, hashed in this order.
PROFILE_SOURCES = {
    "decode_batched": ("kvc_decode.cu", "kvc_decode_cta.cuh", "kvc_device.cuh"),
    "grouped_shared_prefix": ("kvc_grouped.cu", "kvc_decode_cta.cuh", "kvc_device.cuh"),
    "decode_int8_batched": ("kvc_decode_int8.cu", "kvc_device.cuh"),
    "append_rewind_p16": ("kvc_append_tc.cu", "kvc_append_items.cuh", "kvc_device.cuh"),
    "append_int8_rewind_p16": ("kvc_append_int8.cu", "kvc_append_items.cuh", "kvc_device.cuh"),
    "append_rewind_p64": ("kvc_append_tc.cu", "kvc_append_items.cuh", "kvc_device.cuh"),
    "long_decode": ("kvc_decode.cu", "kvc_decode_cta.cuh", "kvc_device.cuh"),
    "merge_long_decode": ("kvc_decode.cu", "kvc_device.cuh"),
    "store_rewind": ("kvc_store.cu", "kvc_device.cuh"),
}


def profile_digest(kernel_tag: str) -> str:
    h = hashlib.sha256()
    for f in PROFILE_SOURCES[kernel_tag]:
        h.update(open(os.path.join(ROOT, "pagedattention_kvc_store_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def traffic_from_profile(kernel_tag: str):
    """DRAM bytes per launch recorded by ncu for this kernel, if none of its sources has
    changed since (the summary records their sha256 prefix)."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s+source_sha256:\s*([0-9a-f]+)",
                  text)
    if not m:
        return None
    return float(m.group(1)) if profile_digest(kernel_tag).startswith(m.group(2)) else None


# ---------------------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------------------

class L2Flush:
    """The L2 flush run before every timed GPU step, outside its events: a write of a buffer
    larger than L2 (evicting every input), then a read of another one (256 MB) so that the
    write's own dirty lines go back to HBM here rather than during the timed step, whose
    reads would otherwise evict them and pay for their write-back (up to an L2's worth of
    DRAM writes that are not the step's work)."""

    def __init__(self, torch, mb, dev):
        self.write_buf = torch.empty(mb << 20, dtype=torch.uint8, device=dev)
        self.read_buf = torch.ones(max(mb // 2, 1) << 18, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)
        self.torch = torch

    def __call__(self):
        self.write_buf.zero_()
        self.torch.sum(self.read_buf, dim=0, out=self.sink)


def time_graph(torch, fn, stream, flush, steps):
    """Capture fn in a CUDA graph; median device time (ms) over `steps` replays, L2 flushed
    between replays outside the timed events."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    del g
    return statistics.median(ts)


def host_rows(out):
    """A GPU output as fp64 rows on the host (for the oracle comparison)."""
    return out.float().cpu().numpy().astype(np.float64)


def run_tiny(torch, kvc, args, dev, stream, flush, rank):
    """The tiny decode (4 sequences of 1, 17, 33 and 100 positions, 4 / 2 heads, head_dim 64,
    16-position pages in a 32-page pool): too small for a rate, so its step time is reported
    (one kvc_decode_store call as a graph, and the separate slot mapping + store + decode),
    with its output checked against the oracle."""
    from workloads import config_case
    from workloads.device import to_device

    case = config_case(1, seed=rank_seed(1, rank))
    d = to_device(case, dev)
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.bfloat16,
                      device=dev)
    slots = torch.empty(case.num_tokens, dtype=torch.int32, device=dev)
    pool = kvc.pool_desc(d.k_pool)
    splits, chunk, ws = kvc.kvc_decode_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, 0)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)

    def separate():
        kvc.kvc_slot_mapping(slots, d.block_table, d.context_lens, None, case.page_size)
        kvc.kvc_store(d.k_pool, d.v_pool, d.k_new, d.v_new, slots)
        kvc.kvc_decode(out, d.q, d.k_pool, d.v_pool, d.block_table, d.context_lens,
                       case.max_ctx, num_splits=0, workspace=work)
    with torch.cuda.stream(stream):
        t_sep = time_graph(torch, separate, stream, flush, args.leg_steps)
        t = time_graph(torch, lambda: kvc.kvc_decode_store(
            out, d.q, d.k_new, d.v_new, d.k_pool, d.v_pool, d.block_table, d.context_lens,
            case.max_ctx, num_splits=0, workspace=work), stream, flush, args.leg_steps)
    got = host_rows(out)
    r = {"workload": "4 seqs, ctx {1,17,33,100}, 4/2 heads, D 64, P 16, 32-page pool; decode "
                     "step with the store of the 4 new tokens",
         "us": round(t * 1e3, 2), "separate_us": round(t_sep * 1e3, 2),
         "bytes": decode_bytes(case) + store_bytes(case), "splits": splits,
         "gpu_launches_per_step": 2 if splits > 1 else 1}
    del d, out, work, slots
    if args.cpu_on:
        r["cpu_baseline"] = oracle_leg(case, got, "GB/s")
    return r


def run_decode_legs(torch, kvc, args, dev, stream, flush, peaks, rank):
    """Shared-prefix decode (grouped vs plain) and long-context split-K decode."""
    from workloads import config_case
    from workloads.device import i32_tensor, to_device

    legs = {}
    per_pos = lambda c: 2 * c.kv_heads * c.head_dim * 2
    qo = lambda c: 2 * c.num_seqs * c.q_heads * c.head_dim * 2
    if "shared_prefix" in args.legs:
        # shared prefix: 32 groups x 8 sequences over 2,048 shared positions
        case = config_case(3, seed=rank_seed(3, rank))
        d = to_device(case, dev)
        slots = torch.empty(case.num_tokens, dtype=torch.int32, device=dev)
        kvc.kvc_slot_mapping(slots, d.block_table, d.context_lens, None, case.page_size)
        kvc.kvc_store(d.k_pool, d.v_pool, d.k_new, d.v_new, slots)
        out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.bfloat16,
                          device=dev)
        indptr = np.arange(0, case.num_seqs + 1, 8, dtype=np.int32)
        prefix = np.full(len(case.groups), case.shared_positions, np.int32)
        gi, gs, gp = (i32_tensor(indptr, dev), i32_tensor(np.concatenate(case.groups), dev),
                      i32_tensor(prefix, dev))
        pool = kvc.pool_desc(d.k_pool)
        ws_g = kvc.kvc_decode_shared_prefix_plan(case.num_seqs, case.q_heads, pool, case.max_ctx,
                                                 len(case.groups), int(prefix.max()))
        work_g = torch.empty(ws_g, dtype=torch.uint8, device=dev)
        _, _, ws_p = kvc.kvc_decode_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, 0)
        work_p = torch.empty(max(ws_p, 16), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            t_g = time_graph(torch, lambda: kvc.kvc_decode_shared_prefix(
                out, d.q, d.k_pool, d.v_pool, d.block_table, d.context_lens, case.max_ctx, gi, gs,
                gp, 8, int(prefix.max()), work_g), stream, flush, args.leg_steps)
            got_grouped = host_rows(out)
            t_p = time_graph(torch, lambda: kvc.kvc_decode(
                out, d.q, d.k_pool, d.v_pool, d.block_table, d.context_lens, case.max_ctx,
                num_splits=0, workspace=work_p), stream, flush, args.leg_steps)
            got_plain = host_rows(out)
        # the same step with the groups found on the device from the block tables: the prepass
        # alone, and prepass + decode over its fixed-capacity group list (S / 2 slots, unused
        # ones empty; at most 8 members; prefix bound max_ctx), with no host read of the count
        cap = case.num_seqs // 2
        di = torch.empty(cap + 1, dtype=torch.int32, device=dev)
        ds = torch.empty(case.num_seqs, dtype=torch.int32, device=dev)
        dp = torch.empty(cap, dtype=torch.int32, device=dev)
        dn = torch.empty(1, dtype=torch.int32, device=dev)
        ws_d = kvc.kvc_decode_shared_prefix_plan(case.num_seqs, case.q_heads, pool, case.max_ctx,
                                                 cap, case.max_ctx)
        work_d = torch.empty(ws_d, dtype=torch.uint8, device=dev)

        def detect():
            kvc.kvc_shared_prefix_groups(di, ds, dp, dn, d.block_table, d.context_lens,
                                         case.page_size, 8)

        def detect_and_decode():
            detect()
            kvc.kvc_decode_shared_prefix(out, d.q, d.k_pool, d.v_pool, d.block_table,
                                         d.context_lens, case.max_ctx, di, ds, dp, 8,
                                         case.max_ctx, work_d)
        with torch.cuda.stream(stream):
            t_det = time_graph(torch, detect, stream, flush, args.leg_steps)
            t_gd = time_graph(torch, detect_and_decode, stream, flush, args.leg_steps)
        torch.cuda.synchronize()
        got_device = host_rows(out)
        found = int(dn.item())
        unique_pos = int(case.context_lens.sum()) - 7 * len(case.groups) * int(prefix[0])
        unique_b = unique_pos * per_pos(case) + qo(case)
        logical_b = int(case.context_lens.sum()) * per_pos(case) + qo(case)
        legs["shared_prefix"] = {
            "workload": "32 groups x 8 seqs, 2,048 shared positions + U[64,512] own, 32/8 heads, "
                        "D 128, P 16",
            "grouped_us": round(t_g * 1e3, 1), "plain_us": round(t_p * 1e3, 1),
            "unique_bytes": unique_b, "logical_bytes": logical_b,
            "grouped_unique_gbs": round(unique_b / (t_g / 1e3) / 1e9, 1),
            "grouped_frac_of_hbm": round(unique_b / (t_g / 1e3) / 1e9 / peaks["hbm"], 4),
            "plain_unique_gbs": round(unique_b / (t_p / 1e3) / 1e9, 1),
            "plain_effective_gbs": round(logical_b / (t_p / 1e3) / 1e9, 1),
            "gpu_launches_per_step": {"grouped": 3, "plain": 2, "device_groups": 5},
            "traffic_grouped_decode_kernel": traffic_from_profile("grouped_shared_prefix"),
            "device_groups": {"groups_found": found, "detect_us": round(t_det * 1e3, 2),
                              "detect_and_grouped_us": round(t_gd * 1e3, 1),
                              "unique_gbs": round(unique_b / (t_gd / 1e3) / 1e9, 1)},
        }
        del d, out, work_g, work_p, slots, work_d
        torch.cuda.empty_cache()
        if args.cpu_on:
            o = oracle_leg(case, got_grouped, "GB/s",
                           also={"plain_decode": got_plain, "device_groups": got_device})
            o["unit_note"] = "logical bytes (every sequence's positions, shared ones per member)"
            legs["shared_prefix"]["cpu_baseline"] = o
        del case
    if "long_decode" in args.legs:
        # long context: 8 sequences of 32k..128k positions
        case = config_case(5, seed=rank_seed(5, rank))
        d = to_device(case, dev)
        slots = torch.empty(case.num_tokens, dtype=torch.int32, device=dev)
        kvc.kvc_slot_mapping(slots, d.block_table, d.context_lens, None, case.page_size)
        kvc.kvc_store(d.k_pool, d.v_pool, d.k_new, d.v_new, slots)
        out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.bfloat16,
                          device=dev)
        pool = kvc.pool_desc(d.k_pool)
        splits, chunk, ws = kvc.kvc_decode_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, 0)
        work = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            t = time_graph(torch, lambda: kvc.kvc_decode(
                out, d.q, d.k_pool, d.v_pool, d.block_table, d.context_lens, case.max_ctx,
                num_splits=0, workspace=work), stream, flush, args.leg_steps)
        got = host_rows(out)
        b = int(case.context_lens.sum()) * per_pos(case) + qo(case)
        legs["long_decode"] = {
            "workload": "8 seqs, ctx U[32768,131072], 64/8 heads, D 128, P 64, split-K + merge",
            "us": round(t * 1e3, 1), "bytes": b, "gbs": round(b / (t / 1e3) / 1e9, 1),
            "frac_of_hbm": round(b / (t / 1e3) / 1e9 / peaks["hbm"], 4), "splits": splits,
            "chunk": chunk, "gpu_launches_per_step": 2,
            "traffic_decode_kernel": traffic_from_profile("long_decode"),
            "traffic_merge_kernel": traffic_from_profile("merge_long_decode"),
        }
        del d, out, work, slots
        torch.cuda.empty_cache()
        if args.cpu_on:
            legs["long_decode"]["cpu_baseline"] = oracle_leg(case, got, "GB/s")
        del case
    if "int8_decode" in args.legs:
        # INT8 pages: the batched-decode batch quantised by kvc_store_int8 (every slot of the bf16
        # pools, as if each were a new token), decoded by kvc_decode_int8 beside kvc_decode
        case = config_case(2, seed=rank_seed(2, rank))
        d = to_device(case, dev)
        slots = torch.empty(case.num_tokens, dtype=torch.int32, device=dev)
        kvc.kvc_slot_mapping(slots, d.block_table, d.context_lens, None, case.page_size)
        kvc.kvc_store(d.k_pool, d.v_pool, d.k_new, d.v_new, slots)
        pages, P, H, D = (int(x) for x in d.k_pool.shape)
        kc = torch.empty(pages, P, H, D, dtype=torch.int8, device=dev)
        vc = torch.empty_like(kc)
        ks = torch.empty(pages, H, P, dtype=torch.float32, device=dev)
        vs = torch.empty_like(ks)
        all_slots = torch.arange(pages * P, dtype=torch.int32, device=dev)
        kvc.kvc_store_int8(kc, vc, ks, vs, d.k_pool.view(pages * P, H, D),
                           d.v_pool.view(pages * P, H, D), all_slots)
        out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.bfloat16,
                          device=dev)
        pool = kvc.pool_desc(d.k_pool)
        splits, chunk, ws = kvc.kvc_decode_int8_plan(case.num_seqs, case.q_heads, pool,
                                                     case.max_ctx, 0)
        _, _, ws16 = kvc.kvc_decode_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, 0)
        work = torch.empty(max(ws, ws16, 16), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            t8 = time_graph(torch, lambda: kvc.kvc_decode_int8(
                out, d.q, kc, vc, ks, vs, d.block_table, d.context_lens, case.max_ctx,
                num_splits=0, workspace=work), stream, flush, args.leg_steps)
            t16 = time_graph(torch, lambda: kvc.kvc_decode(
                out, d.q, d.k_pool, d.v_pool, d.block_table, d.context_lens, case.max_ctx,
                num_splits=0, workspace=work), stream, flush, args.leg_steps)
            # the whole INT8 step: quantise and store each sequence's new token, then decode
            # (the pools already hold those tokens, so every replay writes the same bytes)
            t8_fused = time_graph(torch, lambda: kvc.kvc_decode_int8_store(
                out, d.q, d.k_new, d.v_new, kc, vc, ks, vs, d.block_table, d.context_lens,
                case.max_ctx, num_splits=0, workspace=work), stream, flush, args.leg_steps)

            def int8_separate():
                kvc.kvc_slot_mapping(slots, d.block_table, d.context_lens, None, case.page_size)
                kvc.kvc_store_int8(kc, vc, ks, vs, d.k_new, d.v_new, slots)
                kvc.kvc_decode_int8(out, d.q, kc, vc, ks, vs, d.block_table, d.context_lens,
                                    case.max_ctx, num_splits=0, workspace=work)
            t8_sep = time_graph(torch, int8_separate, stream, flush, args.leg_steps)
        b8 = int(case.context_lens.sum()) * 2 * H * (D + 4) + qo(case)
        b16 = decode_bytes(case)
        legs["int8_decode"] = {
            "workload": "batched decode on INT8 pages: 64 seqs, ctx U[512,4096], 32/8 heads, D 128, "
                        "P 16 (132 B per vector)",
            "us": round(t8 * 1e3, 1), "bytes": b8, "gbs": round(b8 / (t8 / 1e3) / 1e9, 1),
            "frac_of_hbm": round(b8 / (t8 / 1e3) / 1e9 / peaks["hbm"], 4),
            "bf16_us": round(t16 * 1e3, 1), "bf16_bytes": b16,
            "speedup_vs_bf16": round(t16 / t8, 3), "ctas": splits,
            "gpu_launches_per_step": 2 if splits > 1 else 1,
            "traffic_decode_int8_kernel": traffic_from_profile("decode_int8_batched"),
            "step_store_decode_us": {"fused": round(t8_fused * 1e3, 1),
                                     "separate": round(t8_sep * 1e3, 1),
                                     "launches": {"fused": 2 if splits > 1 else 1,
                                                  "separate": 4 if splits > 1 else 3}},
        }
        del d, out, work, slots, kc, vc, ks, vs, all_slots
        torch.cuda.empty_cache()
    if "hnd_decode" in args.legs:
        # HND pools (one contiguous block per page and kv head): the batched-decode batch
        case = config_case(2, seed=rank_seed(2, rank))
        d = to_device(case, dev)
        kh = d.k_pool.permute(0, 2, 1, 3).contiguous()
        vh = d.v_pool.permute(0, 2, 1, 3).contiguous()
        del d.k_pool, d.v_pool
        slots = torch.empty(case.num_tokens, dtype=torch.int32, device=dev)
        kvc.kvc_slot_mapping(slots, d.block_table, d.context_lens, None, case.page_size)
        kvc.kvc_store(kh, vh, d.k_new, d.v_new, slots, layout="hnd")
        out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.bfloat16,
                          device=dev)
        pool = kvc.pool_desc(kh, "hnd")
        splits, chunk, ws = kvc.kvc_decode_plan(case.num_seqs, case.q_heads, pool, case.max_ctx, 0)
        work = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            t = time_graph(torch, lambda: kvc.kvc_decode(
                out, d.q, kh, vh, d.block_table, d.context_lens, case.max_ctx, num_splits=0,
                workspace=work, layout="hnd"), stream, flush, args.leg_steps)
        b = decode_bytes(case)
        legs["hnd_decode"] = {
            "workload": "batched decode on HND pools: 64 seqs, ctx U[512,4096], 32/8 heads, D 128, "
                        "P 16",
            "us": round(t * 1e3, 1), "bytes": b, "gbs": round(b / (t / 1e3) / 1e9, 1),
            "frac_of_hbm": round(b / (t / 1e3) / 1e9 / peaks["hbm"], 4), "splits": splits,
            "gpu_launches_per_step": 2 if splits > 1 else 1,
        }
        del d, out, work, slots, kh, vh
        torch.cuda.empty_cache()
    if "page_copy" in args.legs:
        # copy-on-write page copies: 4,096 pages of P 16 x 8 kv heads x D 128 (32 KB per pool)
        # from one half of a 16,384-page pool to shuffled pages of the other half
        n_pages, n_copy = 16384, 4096
        rng = np.random.default_rng(rank_seed(6, rank) or 6)
        kp = torch.empty(n_pages, 16, 8, 128, dtype=torch.bfloat16, device=dev).normal_()
        vp = torch.empty_like(kp).normal_()
        perm = rng.permutation(n_pages).astype(np.int32)
        src, dst = i32_tensor(perm[:n_copy], dev), i32_tensor(perm[n_copy:2 * n_copy], dev)
        with torch.cuda.stream(stream):
            t = time_graph(torch, lambda: kvc.kvc_copy_pages(kp, vp, src, dst), stream, flush,
                           args.leg_steps)
        b = 2 * 2 * n_copy * 16 * 8 * 128 * 2          # K and V, read and written
        legs["page_copy"] = {
            "workload": "copy-on-write of 4,096 pages (P 16, 8 kv heads, D 128) in a 16,384-page pool",
            "us": round(t * 1e3, 1), "bytes": b, "gbs": round(b / (t / 1e3) / 1e9, 1),
            "frac_of_hbm": round(b / (t / 1e3) / 1e9 / peaks["hbm"], 4), "gpu_launches_per_step": 1,
        }
        del kp, vp
        torch.cuda.empty_cache()
    return legs


def headline_config(case, args, world):
    """The headline workload's description, printed alike by both arms."""
    return {"workload": WORKLOAD, "num_seqs": case.num_seqs, "q_heads": case.q_heads,
            "kv_heads": case.kv_heads, "head_dim": case.head_dim, "page_size": case.page_size,
            "sum_ctx": int(case.context_lens.sum()),
            "l2": (f"flushed between GPU steps ({args.flush_mb} MB write, then a "
                   f"{max(args.flush_mb // 2, 1)} MB read that drains its dirty lines)"),
            "parallelism": f"replicas x{world} (sequences sharded, no collective)"}


def summary_of(line):
    """Each leg's headline figure, its roofline fraction, its oracle time and its parity, in
    a few hundred bytes."""
    def pick(d, *path):
        for k in path:
            if not isinstance(d, dict) or k not in d:
                return None
            d = d[k]
        return d

    def par(d):
        p = pick(d, "cpu_baseline", "parity_vs_gpu")
        return None if p is None else [p["max_abs"], p["mean_abs"]]

    def osec(d):
        return pick(d, "cpu_baseline", "seconds_per_pass")

    legs = line.get("decode_legs") or {}
    app = line.get("append") or {}
    out = {"decode_step_gbs": line["value"], "decode_frac": line["roofline"]["frac"],
           "decode_parity": par(line), "decode_oracle_s": osec(line)}
    if "tiny_decode" in line:
        t = line["tiny_decode"]
        out["tiny_us"] = t["us"]
        out["tiny_parity"] = par(t)
    for P in ("p16", "p64"):
        if P in app:
            out[f"append_{P}_frac"] = app[P]["roofline_frac"]
            out[f"append_{P}_tflops"] = app[P]["tflops"]
            out[f"append_{P}_parity"] = par(app[P])
            out[f"append_{P}_oracle_s"] = osec(app[P])
            out[f"int8_append_{P}_frac"] = pick(app, P, "int8", "roofline_frac")
    if "shared_prefix" in legs:
        out["shared_prefix_frac"] = legs["shared_prefix"]["grouped_frac_of_hbm"]
        out["shared_prefix_parity"] = par(legs["shared_prefix"])
        out["shared_prefix_oracle_s"] = osec(legs["shared_prefix"])
    if "long_decode" in legs:
        out["long_decode_frac"] = legs["long_decode"]["frac_of_hbm"]
        out["long_decode_parity"] = par(legs["long_decode"])
        out["long_decode_oracle_s"] = osec(legs["long_decode"])
    if "int8_decode" in legs:
        out["int8_decode_frac"] = legs["int8_decode"]["frac_of_hbm"]
    if "e2e" in line:
        out["e2e_gbs"] = line["e2e"]["value"]
    return out


def run_kvc(args):
    import torch

    import pagedattention_kvc_store_gb300 as kvc
    from workloads import config_case
    from workloads.device import to_device

    rank, world, local = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    # the oracle (timed on the host cores, and compared with each leg's output) runs on rank 0
    # of a 1-GPU run only
    args.cpu_on = rank == 0 and world == 1 and not args.no_cpu_baseline
    if args.no_headline:
        # the legs alone (for profiler captures of one leg's kernels); not a bench line
        flush = L2Flush(torch, args.flush_mb, dev)
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            legs = {}
            if not args.no_append:
                legs["append"] = run_append(torch, kvc, args, dev, stream, flush, peaks, rank)
            if not args.no_legs:
                legs["decode_legs"] = run_decode_legs(torch, kvc, args, dev, stream, flush,
                                                      peaks, rank)
        if rank == 0:
            print(json.dumps({"legs_only": True, **legs}), flush=True)
        return

    # each rank decodes its own batch of 64 sequences (weak scaling, no collective)
    case = config_case(2, seed=rank_seed(2, rank))
    d = to_device(case, dev)
    S, Hq, D = case.num_seqs, case.q_heads, case.head_dim
    slots = torch.empty(case.num_tokens, dtype=torch.int32, device=dev)
    out = torch.empty(S, Hq, D, dtype=torch.bfloat16, device=dev)
    pool = kvc.pool_desc(d.k_pool)
    splits, chunk, ws = kvc.kvc_decode_plan(S, Hq, pool, case.max_ctx, 0)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
    flush = L2Flush(torch, args.flush_mb, dev)

    def store_part():
        kvc.kvc_slot_mapping(slots, d.block_table, d.context_lens, None, case.page_size)
        kvc.kvc_store(d.k_pool, d.v_pool, d.k_new, d.v_new, slots)

    def decode_part():
        kvc.kvc_decode(out, d.q, d.k_pool, d.v_pool, d.block_table, d.context_lens,
                       case.max_ctx, num_splits=0, workspace=work)

    def fused_step():
        # slot mapping + store + decode + merge through kvc_decode_store: the decode CTA that
        # holds each sequence's newest position stores its new K / V first
        kvc.kvc_decode_store(out, d.q, d.k_new, d.v_new, d.k_pool, d.v_pool, d.block_table,
                             d.context_lens, case.max_ctx, num_splits=0, workspace=work)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        store_part()
        decode_part()
        torch.cuda.synchronize()
        K, W = args.steps, args.warmup
        # The step (slot mapping, store, decode, merge: one kvc_decode_store call) runs as one
        # graph, as a serving loop replays it.  The same work as the separate calls
        # (kvc_slot_mapping, kvc_store, kvc_decode) is timed beside it, and the roofline times
        # the decode alone: a graph of the kvc_decode call, replayed in a timed loop of its own
        # (an event node inside the step's graph would cost the step ~5 us of its own).
        fused_step()
        torch.cuda.synchronize()
        g_step, g_sep, g_decode = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(),
                                   torch.cuda.CUDAGraph())
        with torch.cuda.graph(g_step, stream=stream):
            fused_step()
        with torch.cuda.graph(g_sep, stream=stream):
            store_part()
            decode_part()
        with torch.cuda.graph(g_decode, stream=stream):
            decode_part()
        torch.cuda.synchronize()

        def timed_loop(graph, n):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)]
            for e0, e1 in evs:
                flush()                         # L2 flush, outside the timed events
                e0.record(stream)
                graph.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            return [a.elapsed_time(b) for a, b in evs]

        for _ in range(W):
            flush()
            g_step.replay()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        clocks = ClockSampler(torch.cuda.current_device())
        clocks.start()
        t0 = time.perf_counter()
        step_ms = timed_loop(g_step, K)
        wall = time.perf_counter() - t0
        barrier(world)
        clk = clocks.stop()
        dec_ms = timed_loop(g_decode, max(50, K // 10))
        sep_ms = timed_loop(g_sep, max(50, K // 10))
        got_headline = host_rows(out)
        total_ms = max_over_ranks(sum(step_ms), world, dev)

        step_b = decode_bytes(case) + store_bytes(case)
        value = whole_job_value(world, step_b, K, total_ms)
        dec_b = decode_bytes(case)
        achieved = dec_b / (statistics.median(dec_ms) / 1e3) / 1e9
        launches_per_step = 1 + (1 if splits > 1 else 0)

        e2e = None
        if not args.no_e2e:
            e2e = run_e2e(torch, kvc, case, d, dev, stream, flush, splits, work, max(20, K // 10))

        tiny = None
        if not args.no_legs and "tiny_decode" in args.legs:
            tiny = run_tiny(torch, kvc, args, dev, stream, flush, rank)
        append = None
        if not args.no_append:
            append = run_append(torch, kvc, args, dev, stream, flush, peaks, rank)
        legs = None
        if not args.no_legs:
            legs = run_decode_legs(torch, kvc, args, dev, stream, flush, peaks, rank)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q; no dataset, no weights)",
        "config": headline_config(case, args, world),
        "step": {"splits": splits, "chunk": chunk,
                 "timing": "CUDA events per step on the launching stream; the step is one "
                           "graph of one kvc_decode_store call; roofline from decode-only "
                           "graph replays (median)",
                 "separate_calls": {
                     "ms_per_step": round(statistics.median(sep_ms), 5),
                     "value": round(step_b / (statistics.median(sep_ms) / 1e3) / 1e9, 2),
                     "path": "kvc_slot_mapping + kvc_store + kvc_decode as one graph"}},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm"], 4),
                     "peak_source": f"of {peaks['source']} (copy bandwidth)",
                     "kernel": "paged_decode_kernel + merge_kernel (one kvc_decode call)",
                     "bytes_per_launch": dec_b,
                     "traffic": traffic_from_profile("decode_batched"),
                     "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum of one ncu "
                                       "capture (profiles/decode_batched.md), used only while "
                                       "the kernel's sources still match its sha256"},
        "gpu_launches": K * launches_per_step,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 4),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if tiny is not None:
        line["tiny_decode"] = tiny
    if append is not None:
        line["append"] = append
    if legs is not None:
        line["decode_legs"] = legs
    if args.cpu_on:
        line["cpu_baseline"] = cpu_baseline(case, got_headline, args.cpu_seconds)
    line["summary"] = summary_of(line)   # last, so that a tail of the line keeps it
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(torch, kvc, case, d, dev, stream, flush, splits, work, steps):
    """The same step through the public API with host buffers, every step inside the timed
    region: the step's inputs start in pinned host memory and its output ends there.  No copy
    is enqueued: kvc_decode_store reads the queries, tables and new keys and values straight
    from pinned host memory across the host link and writes its output into a pinned host
    tensor.  The call is issued eagerly; the same step captured as one graph is reported
    beside it."""
    names = ("q", "block_table", "context_lens", "k_new", "v_new")
    src = {name: getattr(d, name) for name in names}
    host_in = {name: t.cpu().pin_memory() for name, t in src.items()}
    out = torch.empty(case.num_seqs, case.q_heads, case.head_dim, dtype=torch.bfloat16,
                      device=dev)
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    slots = torch.empty(case.num_tokens, dtype=torch.int32, device=dev)

    def step():
        kvc.kvc_decode_store(out_host, host_in["q"], host_in["k_new"], host_in["v_new"],
                             d.k_pool, d.v_pool, host_in["block_table"],
                             host_in["context_lens"], case.max_ctx, num_splits=0,
                             workspace=work)

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    torch.cuda.synchronize()

    def timed(fn):
        times = []
        for _ in range(steps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    t_graph = timed(g.replay)
    t_eager = timed(step)
    torch.cuda.synchronize()
    kvc.kvc_decode(out, d.q, d.k_pool, d.v_pool, d.block_table, d.context_lens, case.max_ctx,
                   num_splits=0, workspace=work)
    torch.cuda.synchronize()
    assert torch.equal(out_host, out.cpu()), "host-fed output differs from device-fed output"
    h2d = sum(t.numel() * t.element_size() for t in src.values())
    d2h = out_host.numel() * out_host.element_size()
    step_b = decode_bytes(case) + store_bytes(case)
    return {"value": round(step_b / (t_eager / 1e3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(t_eager, 5), "steps": steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "graph_value": round(step_b / (t_graph / 1e3) / 1e9, 2),
            "graph_ms_per_step": round(t_graph, 5),
            "path": "kvc_decode_store reading q, block_table, context_lens, k_new and v_new "
                    "straight from pinned host memory and writing its output into pinned host "
                    "memory; no copy enqueued; issued eagerly (graph_value: the same step "
                    "captured as one graph)"}


def run_append(torch, kvc, args, dev, stream, flush, peaks, rank):
    """Append-prefill leg: KV-rewind workload, page sizes 16 and 64."""
    from workloads import config_case
    from workloads.device import to_device

    result = {}
    for P in args.append_page_sizes:
        case = config_case(4, page_size=P, num_seqs=args.append_docs,
                           seed=rank_seed(4, rank))
        d = to_device(case, dev)
        slots = torch.empty(case.num_tokens, dtype=torch.int32, device=dev)
        out = torch.empty(case.num_tokens, case.q_heads, case.head_dim, dtype=torch.bfloat16,
                          device=dev)

        def store_part():
            kvc.kvc_slot_mapping(slots, d.block_table, d.context_lens, d.q_indptr,
                                 case.page_size, max_q_len=case.max_q_len)
            kvc.kvc_store(d.k_pool, d.v_pool, d.k_new, d.v_new, slots)

        def append_part():
            kvc.kvc_append(out, d.q, d.k_pool, d.v_pool, d.block_table, d.q_indptr,
                           d.context_lens, case.max_q_len, case.max_ctx)

        store_part()
        append_part()
        torch.cuda.synchronize()
        g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            store_part()
        with torch.cuda.graph(g2, stream=stream):
            append_part()
        for _ in range(3):
            g1.replay()
            g2.replay()
        torch.cuda.synchronize()
        st_ms, ap_ms = [], []
        for _ in range(args.append_steps):
            flush()
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            g1.replay()
            e1.record(stream)
            g2.replay()
            e2.record(stream)
            e2.synchronize()
            st_ms.append(e0.elapsed_time(e1))
            ap_ms.append(e1.elapsed_time(e2))
        got_append = host_rows(out)
        bytes_, flops = append_work(case)
        t = statistics.median(ap_ms) / 1e3
        t_roof = max(flops / (peaks["bf16_sustained"] * 1e12), bytes_ / (peaks["hbm"] * 1e9))
        bound = "tensor" if flops / (peaks["bf16_sustained"] * 1e12) > bytes_ / (peaks["hbm"] * 1e9) else "hbm"
        result[f"p{P}"] = {
            "tflops": round(flops / t / 1e12, 2), "gbs": round(bytes_ / t / 1e9, 1),
            "ms": round(statistics.median(ap_ms), 4),
            "store_ms": round(statistics.median(st_ms), 4),
            "flops": flops, "bytes": bytes_, "roofline_bound": bound,
            "roofline_frac": round(t_roof / t, 4),
            "store_gbs": round(store_bytes(case) / (statistics.median(st_ms) / 1e3) / 1e9, 1),
            "gpu_launches": args.append_steps * 3,
            "traffic": (traffic_from_profile(f"append_rewind_p{P}")
                        if P in (16, 64) and args.append_docs == 1000 else None),
            "store_traffic": (traffic_from_profile("store_rewind")
                              if P == 16 and args.append_docs == 1000 else None),
        }
        del g1, g2
        # fused store + append (kvc_append_store) on the same inputs: the chunk's K/V read once
        # from k_new / v_new; the pools end as the separate store leaves them
        with torch.cuda.stream(stream):
            tf = time_graph(torch, lambda: kvc.kvc_append_store(
                out, d.q, d.k_new, d.v_new, d.k_pool, d.v_pool, d.block_table, d.q_indptr,
                d.context_lens, case.max_q_len, case.max_ctx), stream, flush,
                args.append_steps) / 1e3
        got_fused = host_rows(out)
        sep = (statistics.median(st_ms) + statistics.median(ap_ms)) / 1e3
        # kvc_append_store's plan: at pages of 64 positions or more it stores the whole chunk
        # first and runs the plain append (the chunk is then read twice)
        whole = P >= 64
        bf = store_bytes(case) + bytes_ if whole else fused_work(case)
        result[f"p{P}"]["fused_store"] = {
            "kernel": ("store_boundary_kernel (whole chunk) + paged_append_tc_kernel"
                       if whole else "store_boundary_kernel + paged_append_tc_kernel")
                      + " (kvc_append_store)",
            "ms": round(tf * 1e3, 4), "bytes": bf, "gbs": round(bf / tf / 1e9, 1),
            "separate_ms": round(sep * 1e3, 4), "speedup_vs_separate": round(sep / tf, 3),
            "gpu_launches": 2 * args.append_steps,
        }
        # the same append over INT8 pages: every slot of the bf16 pools quantised by
        # kvc_store_int8, then kvc_append_int8 (132 B per cached vector instead of 256)
        pages, _, H, D = (int(x) for x in d.k_pool.shape)
        kc = torch.empty(pages, P, H, D, dtype=torch.int8, device=dev)
        vc = torch.empty_like(kc)
        ks = torch.empty(pages, H, P, dtype=torch.float32, device=dev)
        vs = torch.empty_like(ks)
        all_slots = torch.arange(pages * P, dtype=torch.int32, device=dev)
        kvc.kvc_store_int8(kc, vc, ks, vs, d.k_pool.view(pages * P, H, D),
                           d.v_pool.view(pages * P, H, D), all_slots)
        with torch.cuda.stream(stream):
            t8 = time_graph(torch, lambda: kvc.kvc_append_int8(
                out, d.q, kc, vc, ks, vs, d.block_table, d.q_indptr, d.context_lens,
                case.max_q_len, case.max_ctx), stream, flush, args.append_steps) / 1e3
        b8 = append_work(case, int8=True)[0]
        t8_roof = max(flops / (peaks["bf16_sustained"] * 1e12), b8 / (peaks["hbm"] * 1e9))
        result[f"p{P}"]["int8"] = {
            "kernel": "paged_append_int8_kernel (kvc_append_int8)",
            "ms": round(t8 * 1e3, 4), "tflops": round(flops / t8 / 1e12, 2),
            "gbs": round(b8 / t8 / 1e9, 1), "bytes": b8,
            "roofline_frac": round(t8_roof / t8, 4), "speedup_vs_bf16": round(t / t8, 3),
            "gpu_launches": args.append_steps,
            "traffic": (traffic_from_profile("append_int8_rewind_p16")
                        if P == 16 and args.append_docs == 1000 else None),
        }
        del d, out, slots, kc, vc, ks, vs, all_slots
        torch.cuda.empty_cache()
        if args.cpu_on:
            result[f"p{P}"]["cpu_baseline"] = oracle_leg(case, got_append, "TFLOP/s",
                                                         also={"append_store": got_fused})
        del case
    result["workload"] = (f"rewind-append: {args.append_docs:,} docs x 50 new tokens over 300 "
                          "cached, 32 q / 8 kv heads, head_dim 128")
    result["peaks"] = {"hbm_gbs": peaks["hbm"], "bf16_tflops": peaks["bf16_sustained"],
                       "source": f"of {peaks['source']} (sustained bf16)"}
    return result


# ---------------------------------------------------------------------------------------
# the CPU oracle (baseline only; never the product path)
# ---------------------------------------------------------------------------------------

def _oracle_step(oracle, case, seqs, threads, k_pool, v_pool):
    """The oracle's step over sequences `seqs`: slot mapping, store of their new tokens, then
    attention gathered through the block table; returns the output rows (fp64)."""
    bt = case.block_table[seqs]
    ctx = case.context_lens[seqs]
    q_lens = case.q_lens[seqs]
    indptr = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    rows = np.concatenate([np.arange(case.q_indptr[s], case.q_indptr[s + 1]) for s in seqs])
    slots = oracle.slot_mapping(bt, ctx, indptr, case.page_size)
    oracle.store(k_pool, v_pool, case.k_new[rows], case.v_new[rows], slots)
    out, _ = oracle.attention(case.q[rows], k_pool, v_pool, bt, ctx, indptr,
                              num_threads=threads)
    return out


def _sub_bytes(case, seqs):
    per_pos = 2 * case.kv_heads * case.head_dim * 2
    row = case.kv_heads * case.head_dim * 2
    n = len(seqs)
    return (int(case.context_lens[seqs].astype(np.int64).sum()) * per_pos
            + 2 * n * case.q_heads * case.head_dim * 2 + n * (2 * row * 2 + 8))


def _sub_case_units(case, seqs, unit):
    """Work of the oracle's step over `seqs`, in the leg's unit: bytes (GB/s) or FLOPs
    (TFLOP/s) of the same definitions the GPU legs use."""
    if unit == "TFLOP/s":
        q_lens = case.q_lens[seqs].astype(np.int64)
        ctx = case.context_lens[seqs].astype(np.int64)
        pairs = int((q_lens * (ctx - q_lens) + q_lens * (q_lens + 1) // 2).sum())
        return 4 * case.head_dim * case.q_heads * pairs / 1e12
    return _sub_bytes(case, seqs) / 1e9


def parity_of(got, ref):
    """Element-wise comparison of GPU output rows with the oracle's (fp64), against the
    attention tolerance the tests hold (max abs 1e-2, mean abs 1e-3)."""
    err = np.abs(np.asarray(got, np.float64) - ref)
    mx, mean = float(err.max()), float(err.mean())
    return {"max_abs": float(f"{mx:.3e}"), "mean_abs": float(f"{mean:.3e}"),
            "elements": int(err.size), "ok": bool(mx <= 1e-2 and mean <= 1e-3)}


def oracle_leg(case, got, unit, seconds=1.0, also=None):
    """The oracle (fp64 C: slot mapping, store, attention gathered through the block table)
    on the leg's whole workload, all host cores, repeated until `seconds` have passed (at least
    once); the same oracle on one thread over the first sequences (about a second's worth,
    scaled to the same unit); and the GPU output `got` (all rows, bf16 widened) against the
    oracle's; `also` maps names to further GPU outputs of the same workload (other entry
    points), each compared with the same oracle output."""
    from oracle import oracle
    threads = len(os.sched_getaffinity(0))
    seqs = np.arange(case.num_seqs)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    t0 = time.perf_counter()
    reps = 0
    while True:
        ref = _oracle_step(oracle, case, seqs, threads, kp, vp)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = (time.perf_counter() - t0) / reps
    n1 = int(np.clip(round(case.num_seqs / max(dt * threads, 1e-9)), 1, case.num_seqs))
    few = np.arange(n1)
    kp1, vp1 = case.k_pool.copy(), case.v_pool.copy()
    t1 = time.perf_counter()
    _oracle_step(oracle, case, few, 1, kp1, vp1)
    dt1 = time.perf_counter() - t1
    del kp, vp, kp1, vp1
    return {"value": round(_sub_case_units(case, seqs, unit) / dt, 4), "unit": unit,
            "cores": threads, "kind": "oracle",
            "sample": f"the whole workload ({case.num_seqs} sequences), {reps} pass(es), "
                      f"{dt:.3f} s per pass",
            "seconds_per_pass": round(dt, 4),
            "value_1_thread": round(_sub_case_units(case, few, unit) / dt1, 4),
            "sample_1_thread": f"sequences 0-{n1 - 1} on one thread, {dt1:.2f} s",
            "parity_vs_gpu": parity_of(got, ref),
            **{f"parity_{k}": parity_of(v, ref) for k, v in (also or {}).items()}}


def cpu_baseline(case, got, seconds):
    """The headline's CPU baseline: the oracle over the full 64-sequence batch."""
    r = oracle_leg(case, got, "GB/s", seconds)
    r["sample"] += " (fp64 C oracle: slot mapping, store, gathered attention)"
    return r


def run_reference(args):
    rank, world, _ = dist_setup(args)
    if rank != 0:   # rank 0 alone times the oracle; the others wait for it and exit
        barrier(world)
        import torch.distributed as dist
        dist.destroy_process_group()
        return
    from oracle import oracle
    from workloads import config_case
    oracle.build()
    case = config_case(2)
    threads = len(os.sched_getaffinity(0))
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    # size the sample so that warmup + steps take about two minutes
    t0 = time.perf_counter()
    _oracle_step(oracle, case, np.arange(1), threads, kp, vp)
    t1 = max(time.perf_counter() - t0, 1e-4)
    n = int(np.clip(120.0 / ((args.steps + args.warmup) * t1), 1, case.num_seqs))
    seqs = np.arange(n)
    for _ in range(args.warmup):
        _oracle_step(oracle, case, seqs, threads, kp, vp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(oracle, case, seqs, threads, kp, vp)
    dt = (time.perf_counter() - t0) / args.steps
    value = _sub_bytes(case, seqs) / dt / 1e9
    sample = f"first {n} of the 64 sequences per step ({dt * 1e3:.2f} ms per step)"
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": headline_config(case, args, world),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_kvc(args)


if __name__ == "__main__":
    main()
