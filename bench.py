#!/usr/bin/env python
"""Benchmark of the paged KV-cache decode step on the 13B-shaped workload.

One step = one new token appended per sequence and a decode over every
sequence, through paged_attn_decode_append (fused append + partition kernel,
then the log-sum-exp merge kernel),
on 256 sequences x 40 heads x head_dim 128, bf16, block size 16, lengths
log-normal (median 350) clipped to [16, 2048], blocks scattered over a pool 1.2x
the live tokens.  The KV pool (2.4 GB read per step) is larger than L2, so no
flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  With N > 1 (torchrun), every rank runs its own
batch (weak scaling, no collective on the data path); the step time is the max
over ranks and the value sums all ranks' bytes.

The line checks itself: after timing, the step's output is compared with the
fp64 CPU oracle on every sequence of the batch (the oracle runs as one spawned
host process per core) and the appended rows with the new K/V bit for bit; the
result goes into "parity" and a failure ends the run with a non-zero status.
After the headline (one GPU), every other seeded workload is timed as
`--workload <name>` would time it and summarised under "workloads"
(`--no-workloads` skips them).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

# The oracle runs as one host process per core: keep numpy's BLAS (OpenBLAS) on
# one thread in each.  It reads this when numpy is first imported, which is below
# (and in the spawned processes, which inherit the environment).
os.environ["OPENBLAS_NUM_THREADS"] = "1"

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-attn decode KV GB/s (% of HBM peak), seq-tokens/s at 13B shape"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
PREFILL_SOURCES = ("paged_kv_cache_317_gb300/csrc/paged_prefill.cu",
                   "paged_kv_cache_317_gb300/csrc/tma.cuh",
                   "paged_kv_cache_317_gb300/csrc/common.cuh")
DECODE_SOURCES = ("paged_kv_cache_317_gb300/csrc/decode_partition.cuh",
                  "paged_kv_cache_317_gb300/csrc/decode_config.h",
                  "paged_kv_cache_317_gb300/csrc/common.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
# the serving loops' per-step device split is taken on every 4th step
SPLIT_NOTE = "sampled every 4th step, whose event records add host time"


# --------------------------------------------------------------- host logic
def dist_env():
    """(rank, world_size, local_rank) from torchrun's environment (1 process: 0, 1, 0)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def rank_seed(base: int, rank: int) -> int:
    """Each rank decodes its own batch: same shape, its own draw."""
    return base + 1000 * rank


def reduce_max(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def step_bytes(lens, num_heads, head_dim, block_size, elt=2, out_elt=2, partition_tokens=512):
    """Algorithmic bytes of one fused step (paged_attn_decode_append), by kernel.

    partition pass: every context K and V row once (the last one from new_k/new_v,
    the rest from the cache), q, the table entries it follows, the lengths, the
    appended rows written into the cache, and what it writes out (the output row
    of a one-partition sequence, else an fp32 partial of D floats + (m, l) per
    partition).  merge pass: the partials of split sequences, their output rows
    and the lengths.
    """
    import numpy as np
    lens = np.asarray(lens, dtype=np.int64)
    N, H, D = lens.shape[0], num_heads, head_dim
    kv = int(lens.sum()) * H * D * elt * 2
    parts = np.maximum(1, -(-lens // partition_tokens))
    split = parts > 1
    partial_bytes = int(parts[split].sum()) * H * (D + 2) * 4
    out_direct = int((~split).sum()) * H * D * out_elt
    out_merged = int(split.sum()) * H * D * out_elt
    table = int((-(-lens // block_size)).sum()) * 4
    q = N * H * D * elt
    append_write = 2 * N * H * D * elt
    partition = kv + q + table + N * 4 + out_direct + partial_bytes + append_write
    merge = partial_bytes + out_merged + N * 4
    return {"decode_partition": partition, "decode_merge": merge, "append_write": append_write,
            "kv": kv, "total": partition + merge}


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, then /proc/cpuinfo), or 'unknown'."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine() or "unknown"


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak(sustained: bool = False):
    """Dense bf16 tensor peak from MEASURED_PEAKS.json: the burst figure for a
    kernel timed alone over a short region, the sustained (power-capped) one for
    a region long enough to reach the power limit."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(path) as f:
            return float(json.load(f)[key]), f"measured {key}"
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback"


# A timed tensor-core region longer than this is compared with the sustained peak.
SUSTAINED_REGION_MS = 200.0


def gpu_uuid(dev, local_rank: int) -> str:
    """The NVML identifier of `dev` (its ordinal when the UUID is unavailable)."""
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return str(local_rank)


def source_sha(sources=DECODE_SOURCES) -> str:
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def decode_source_sha() -> str:
    return source_sha(DECODE_SOURCES)


def recorded_traffic(kernel: str, sources=DECODE_SOURCES):
    """dram bytes per launch from the last ncu capture, if the kernel is unchanged since."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[kernel]
    except Exception:
        return None
    if rec.get("source_sha") != source_sha(sources):
        return None
    return rec.get("dram_bytes_per_launch_full_size")


# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*), by the names
# nvidia-smi gives them under clocks_event_reasons.
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


def reasons_from_mask(mask: int) -> list:
    """Names of the throttle reasons set in an NVML clock-event reason mask."""
    return sorted(name for bit, name in NVML_REASONS.items() if mask & bit)


def summarize_clocks(sm, mx, reasons, source) -> dict:
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted(reasons), "samples": len(sm), "source": source}


class _Nvml:
    """Read-only NVML queries through ctypes (the driver's libnvidia-ml): SM
    clock, maximum SM clock and the active clock-event reasons of one GPU."""

    def __init__(self, uuid: str):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.lib = lib
        self.dev = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
            raise RuntimeError(f"no NVML device {uuid}")
        self._reasons = (getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                         or lib.nvmlDeviceGetCurrentClocksThrottleReasons)
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx)) != 0:   # 1 = SM clock
            raise RuntimeError("nvmlDeviceGetMaxClockInfo failed")
        self.max_mhz = float(mx.value)

    def sample(self):
        """(SM MHz, reason mask), or None if a query failed."""
        c, r = self.ct.c_uint(), self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, self.ct.byref(c)) != 0:
            return None
        if self._reasons(self.dev, self.ct.byref(r)) != 0:
            return None
        return float(c.value), int(r.value)

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clocks and throttle reasons over a timed region.  Through NVML: one
    reading when started, a thread reading about every millisecond until
    stopped, one reading when stopped (a region of a few ms still gets samples).
    Without NVML: nvidia-smi sampling every 50 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str):
        self.gpu = gpu_uuid
        self.proc = None
        self.file = None
        self.nvml = None
        self.thread = None

    def _poll(self):
        while not self.stop_flag.is_set():
            x = self.nvml.sample()
            if x is not None:
                self.rows.append(x)
            time.sleep(0.001)

    def start(self):
        import threading
        try:
            self.nvml = _Nvml(self.gpu)
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self.rows, self.stop_flag = [], threading.Event()
            x = self.nvml.sample()
            if x is not None:
                self.rows.append(x)
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.nvml is not None:
            x = self.nvml.sample()
            self.stop_flag.set()
            self.thread.join()
            if x is not None:
                self.rows.append(x)
            self.nvml.close()
            sm = [c for c, _ in self.rows]
            reasons = set()
            for _, m in self.rows:
                reasons.update(reasons_from_mask(m))
            return summarize_clocks(sm, [self.nvml.max_mhz] if sm else [], reasons, "nvml")
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0, "source": None}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        text = self.file.read()
        self.file.close()
        os.unlink(self.file.name)
        return dict(parse_clock_rows(text), source="nvidia-smi")


def parse_clock_rows(text: str) -> dict:
    """Median SM clock, max SM clock and the throttle reasons seen, from
    nvidia-smi ``--query-gpu=ClockSampler.QUERY --format=csv,noheader,nounits`` rows."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.strip().splitlines():
        r = [x.strip() for x in line.split(",")]
        try:
            sm.append(float(r[1]))
            mx.append(float(r[2]))
        except (ValueError, IndexError):
            continue
        for name, val in zip(names, r[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted(reasons), "samples": len(sm)}


def clocks_rejected(clk: dict) -> bool:
    """A timed region whose clock record shows a thermal or hardware slowdown, or SM
    clocks well below their maximum with no reason given (a leftover clock lock),
    does not count; sw_power_cap alone is normal under load and is kept."""
    reasons = set(clk.get("reasons") or [])
    if reasons & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                   "hw_power_brake_slowdown"}:
        return True
    sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    return bool(sm and mx and sm < 0.85 * mx and not reasons)


# --------------------------------------------------------------- our arm
def headline_config(b, args, world) -> dict:
    """`config` of the headline line (both arms)."""
    return {
        "workload": "13B-shaped paged decode step: append 1 token/seq + decode",
        "num_seqs_per_gpu": b.num_seqs, "num_heads": b.num_heads, "head_dim": b.head_dim,
        "block_size": b.block_size, "context_tokens_per_gpu": int(b.context_lens.sum()),
        "lengths": "lognormal(median 350, sigma 0.75) clipped to [16, 2048]",
        "pool_blocks": b.num_blocks, "partition_tokens": args.partition, "out_dtype": "bf16",
        "seed": args.seed,
        "schedule": "(sequence, partition) work items holding tokens, longest "
                    "sequences first (work_items)",
        "l2": "inputs larger than L2 (2.4 GB of K/V read per step); no flush",
        "parallelism": f"replicas x{world} (independent batches, no collective)",
    }


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    from paged_kv_cache_317_gb300 import binding as B
    from paged_kv_cache_317_gb300 import _build
    from workloads import decode_13b

    _build.build(quiet=True)
    B.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    b = decode_13b(seed=rank_seed(args.seed, rank), device=dev, block_size=args.block_size,
                   poison=False)
    N, H, D, bs = b.num_seqs, b.num_heads, b.head_dim, b.block_size
    MB = b.max_blocks_per_seq
    pt = args.partition
    bt = torch.from_numpy(b.block_tables).to(dev)
    sl = torch.from_numpy(b.context_lens).to(dev)
    # The host knows the lengths it built the tables from: it lists the (sequence,
    # partition) pairs that hold tokens, longest sequences first.
    order = torch.from_numpy(B.partition_work_items(
        b.context_lens, pt, MB, bs, order=np.argsort(-b.context_lens, kind="stable"))).to(dev)
    out = torch.empty((N, H, D), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(B.paged_attn_workspace_size(N, H, D, bs, MB, pt), dtype=torch.uint8,
                     device=dev)
    nbytes = step_bytes(b.context_lens, H, D, bs, partition_tokens=pt)
    stream = torch.cuda.current_stream(dev)
    rec = B.new_error_record(dev)

    def partition_pass():
        B.paged_attn_decode_append(b.q, b.new_k, b.new_v, b.k_cache, b.v_cache, bt, sl, b.scale,
                                   out=out, partition_tokens=pt, workspace=ws, error_record=rec,
                                   phases=1, work_items=order)

    def step():
        partition_pass()
        B.paged_attn_decode_append(b.q, b.new_k, b.new_v, b.k_cache, b.v_cache, bt, sl, b.scale,
                                   out=out, partition_tokens=pt, workspace=ws, error_record=rec,
                                   phases=2)

    K, W = args.steps, args.warmup
    for _ in range(W):
        step()
    torch.cuda.synchronize(dev)
    if B.pa_error_read(rec) != [0, 0, 0, 0]:
        raise RuntimeError(f"device error record after warm-up: {B.pa_error_read(rec)}")

    gpu_id = gpu_uuid(dev, local_rank)

    def timed(fn):
        t_start, t_end = (torch.cuda.Event(enable_timing=True),
                          torch.cuda.Event(enable_timing=True))
        clocks = ClockSampler(gpu_id)
        clocks.start()
        barrier(world)
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for _ in range(K):
            fn()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        clk = clocks.stop()
        return t_start.elapsed_time(t_end) / K, clk

    ms, clk = timed(step)
    # a region with throttled clocks on any rank is timed once more
    if reduce_max(1.0 if clocks_rejected(clk) else 0.0, world, dev) > 0:
        first = clk
        ms, clk = timed(step)
        clk = dict(clk, remeasured_after=first)
    ms_max = reduce_max(ms, world, dev)
    # The dominant kernel alone: K partition passes back to back between one pair
    # of events (no merge, no events inside the loop to disturb the launches).
    for _ in range(W):
        partition_pass()
    part_ms, part_clk = timed(partition_pass)

    # End to end through the public API: every step copies its inputs in from
    # pinned host memory and its output back out.  As in a serving loop, the
    # copies run on their own streams with two buffer sets, so step i's copies
    # overlap step i-1's kernels; each step's bytes still cross the link.
    pin = lambda t: t.detach().cpu().pin_memory()
    host_in = [pin(b.q), pin(b.new_k), pin(b.new_v), pin(bt), pin(sl), pin(order)]
    dev_in = [[torch.empty_like(t, device=dev) for t in host_in] for _ in range(2)]
    h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    d_out = [torch.empty_like(out) for _ in range(2)]
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_copied = [torch.cuda.Event() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = h_out[0].numel() * h_out[0].element_size()

    def e2e_step(i):
        j = i % 2
        h2d_stream.wait_event(done[j])                 # buffer j's last kernels have finished
        with torch.cuda.stream(h2d_stream):
            for d, h in zip(dev_in[j], host_in):
                d.copy_(h, non_blocking=True)
        in_ready[j].record(h2d_stream)
        stream.wait_event(in_ready[j])
        stream.wait_event(out_copied[j])               # d_out[j] has been read back
        q, k, v, btj, slj, oj = dev_in[j]
        B.paged_attn_decode_append(q, k, v, b.k_cache, b.v_cache, btj, slj, b.scale,
                                   out=d_out[j], partition_tokens=pt, workspace=ws,
                                   error_record=rec, work_items=oj, stream=stream)
        done[j].record(stream)
        d2h_stream.wait_event(done[j])
        with torch.cuda.stream(d2h_stream):
            h_out[j].copy_(d_out[j], non_blocking=True)
        out_copied[j].record(d2h_stream)

    for i in range(W):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_stream.wait_event(e0)
    for i in range(K):
        e2e_step(i)
    stream.wait_event(out_copied[(K - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = reduce_max(e0.elapsed_time(e1) / K, world, dev)
    if not torch.equal(h_out[(K - 1) % 2], out.cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident step's")
    if B.pa_error_read(rec) != [0, 0, 0, 0]:
        raise RuntimeError(f"device error record: {B.pa_error_read(rec)}")

    # Parity of the timed step: its output against the fp64 oracle on every
    # sequence of the batch, and the appended rows bit for bit in the cache.
    slots = torch.from_numpy(b.slot_mapping).to(dev)
    blk, row = slots // bs, slots % bs
    append_ok = (torch.equal(b.k_cache[blk, :, row, :].view(torch.int16),
                             b.new_k.view(torch.int16)) and
                 torch.equal(b.v_cache[blk, :, row, :].view(torch.int16),
                             b.new_v.view(torch.int16)))
    host = HostOracle(b, host_workers(world))
    try:
        ref, _ = host.run()
        parity = parity_report(out, ref, append_ok)
        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            cpu = oracle_timing(host, nbytes["total"], int(b.context_lens.sum()))
    finally:
        host.close()
    failed = reduce_max(0.0 if parity["ok"] else 1.0, world, dev)
    parity["max_abs_err"] = reduce_max(parity["max_abs_err"], world, dev)
    parity["ranks_checked"] = world

    total_bytes = reduce_sum(nbytes["total"], world, dev)
    tokens = reduce_sum(float(b.context_lens.sum()), world, dev)
    value = total_bytes / (ms_max * 1e-3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    achieved = nbytes["decode_partition"] / (part_ms * 1e-3) / 1e9

    # the other seeded workloads (sampling, long context, serving, ...), after the headline
    others = None
    if rank == 0 and world == 1 and not args.no_workloads:
        others = workload_summaries(args, rank, world, local_rank)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 K/V/Q; no trained weights)",
            "pct_of_hbm_peak": round(100 * value / peak, 2),
            "seq_tokens_per_s": round(tokens / (ms_max * 1e-3), 1),
            "seqs_per_s": round(world * N / (ms_max * 1e-3), 1),
            "config": headline_config(b, args, world),
            "bytes_per_step": nbytes,
            "parity": parity,
            "roofline": {
                "kernel": "paged_attn_partition_kernel", "bound": "hbm",
                "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                # the recorded capture is of the default batch (seed 2, block 16, 512)
                "traffic": (recorded_traffic("paged_attn_partition_kernel")
                            if (args.seed, args.block_size, args.partition) == (2, 16, 512)
                            else None),
                "algorithmic_bytes_per_launch": nbytes["decode_partition"],
                "avg_launch_ms": round(part_ms, 5),
                "timing": f"{K} partition passes back to back between one event pair "
                          "(rank 0)",
                "clocks": part_clk,
            },
            "e2e": {"value": round(total_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                    "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "note": "pinned H2D inputs + D2H output every step, copy streams "
                            "double-buffered against the previous step's kernels"},
            "gpu_launches": 2 * K,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        if others is not None:
            line["workloads"] = others
        print(json.dumps(line), flush=True)
    if failed > 0:
        raise SystemExit("parity check of the timed step failed: " + json.dumps(parity))


# ------------------------------------------------------- other workloads
def _time_device(fn, K, W, stream, flush=None):
    """Mean device time of fn() over K calls (after W), in ms.  With `flush`,
    L2 is flushed before every call and only the calls (replayed from a CUDA
    graph) are timed."""
    import torch
    for _ in range(W):
        fn()
    torch.cuda.synchronize()
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / K
    # The call is replayed from a CUDA graph between the two events, so that the
    # host's launch cost (which can exceed a tiny call's device time) cannot leave
    # the GPU idle inside the timed interval after the flush.
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(K):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.mean(times)


def _time_graph(fns, K, W, stream, calls_per_graph=32):
    """Mean device time per call, in ms, of the calls fns[0], fns[1], ... taken in
    turn, captured into one CUDA graph of `calls_per_graph` calls and replayed
    (after W warm-up replays) until at least K calls ran: what a serving loop
    that captures its step sees, without the host's launch cost."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for f in fns:
            f()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for j in range(calls_per_graph):
            fns[j % len(fns)]()
    for _ in range(W):
        graph.replay()
    torch.cuda.synchronize()
    reps = max(1, -(-K // calls_per_graph))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (reps * calls_per_graph)


class _Staging:
    """Per-step host inputs of a serving loop in one pinned int32 buffer per set
    (copy-on-write pairs as int64, block tables, lengths, work list,
    shared-partition records, tail starts) and one device buffer, uploaded with
    one copy, with the numbers of work items and records (device-side counts, for
    a step replayed from a CUDA graph over the lists' capacities).  The allocator
    and the planner write their outputs straight into a set's regions (views);
    two sets alternate, and a set is refilled once the copy that read it is done."""

    def __init__(self, n_seqs, max_blocks, n_items_max, record_words, dev):
        import torch
        self.sizes = {"pairs": 4 * n_seqs, "bt": n_seqs * max_blocks, "sl": n_seqs,
                      "ts": n_seqs, "cnt": 2, "it": n_items_max,
                      "rc": n_items_max * record_words}
        self.off, at = {}, 0
        for k, n in self.sizes.items():
            self.off[k] = at
            at += n + (-n) % 4           # keep every region 16-byte aligned
        self.n_seqs, self.max_blocks, self.rw = n_seqs, max_blocks, record_words
        self.host = [torch.empty(at, dtype=torch.int32).pin_memory() for _ in range(2)]
        self.host_np = [h.numpy() for h in self.host]
        self.dev = [torch.zeros(at, dtype=torch.int32, device=dev) for _ in range(2)]
        o = self.off
        # the regions whose size does not change from step to step, viewed once
        self.fixed = [(d[o["bt"]:o["bt"] + n_seqs * max_blocks].view(n_seqs, max_blocks),
                       d[o["sl"]:o["sl"] + n_seqs], d[o["ts"]:o["ts"] + n_seqs])
                      for d in self.dev]
        for d in self.dev:   # no copy-on-write pairs and no split partitions before an upload
            d[self.off["pairs"]:self.off["pairs"] + self.sizes["pairs"]] = -1
            d[self.off["ts"]:self.off["ts"] + self.sizes["ts"]] = -1
        self.done = [torch.cuda.Event() for _ in range(2)]

    def views(self, step):
        """Wait until set step % 2 may be refilled (the copy that read it two steps
        back is done); returns its host regions: tables [n, max_blocks], lengths,
        work list, records [cap, record words], tail starts."""
        j = step % 2
        self.done[j].synchronize()
        h, o, n = self.host_np[j], self.off, self.n_seqs
        return (h[o["bt"]:o["bt"] + n * self.max_blocks].reshape(n, self.max_blocks),
                h[o["sl"]:o["sl"] + n], h[o["it"]:o["it"] + self.sizes["it"]],
                h[o["rc"]:o["rc"] + self.sizes["rc"]].reshape(-1, self.rw),
                h[o["ts"]:o["ts"] + n])

    def upload(self, step, stream, pairs, n_items, n_recs, tails, pad=False):
        """Write the pairs (pad: and -1 pairs up to the capacity) and the counts
        into set step % 2 (its other regions filled through views(step)) and
        enqueue its upload; returns device views (pairs int64 [n, 2], tables,
        lengths, work list, records, tail starts or None), or None with pad (a
        captured step reads the capacity views)."""
        import numpy as np
        import torch
        j = step % 2
        h, o, n_p = self.host_np[j], self.off, len(pairs)
        if n_p:
            h[o["pairs"]:o["pairs"] + 4 * n_p].view(np.int64)[:] = pairs.ravel()
        if pad:
            h[o["pairs"] + 4 * n_p:o["pairs"] + self.sizes["pairs"]] = -1
        h[o["cnt"]] = n_items
        h[o["cnt"] + 1] = n_recs
        used = o["rc"] + n_recs * self.rw
        d = self.dev[j]
        d[:used].copy_(self.host[j][:used], non_blocking=True)
        self.done[j].record(stream)
        if pad:
            return None
        bt, sl, ts = self.fixed[j]
        return (d[o["pairs"]:o["pairs"] + 4 * n_p].view(torch.int64).view(n_p, 2), bt, sl,
                d[o["it"]:o["it"] + n_items],
                d[o["rc"]:o["rc"] + n_recs * self.rw].view(n_recs, self.rw) if n_recs else None,
                ts if tails else None)

    def capacity_views(self, j, n_items_cap, n_recs_cap):
        """Device views of set j for a captured step: pairs int64 [n_seqs, 2],
        tables, lengths, the first n_items_cap work-list entries and n_recs_cap
        records (the launches' sizes), tail starts, counts."""
        import torch
        d, o, n = self.dev[j], self.off, self.n_seqs
        return (d[o["pairs"]:o["pairs"] + 4 * n].view(torch.int64).view(n, 2),
                d[o["bt"]:o["bt"] + n * self.max_blocks].view(n, self.max_blocks),
                d[o["sl"]:o["sl"] + n], d[o["it"]:o["it"] + n_items_cap],
                d[o["rc"]:o["rc"] + n_recs_cap * self.rw].view(n_recs_cap, self.rw),
                d[o["ts"]:o["ts"] + n], d[o["cnt"]:o["cnt"] + 2])


def run_workload(args, rank, world, local_rank, emit=True):
    """Device time of one step of the other seeded workloads (decode attention,
    plus the allocator, copies and appends where the workload has them).
    Prints the line (emit) and returns it."""
    if rank != 0:
        return None
    import numpy as np
    import torch

    from paged_kv_cache_317_gb300 import binding as B
    from paged_kv_cache_317_gb300 import _build
    import workloads as WL
    import workloads.gen  # noqa: F401  (randn_rounded, _torch_gen)

    _build.build(quiet=True)
    B.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    K, W = args.steps, args.warmup
    peak, peak_kind = measured_hbm_peak()
    rec = B.new_error_record(dev)
    line = {"metric": METRIC, "unit": UNIT, "n_gpus": 1, "steps": K, "warmup": W,
            "higher_is_better": True, "vs_baseline": None, "data": "synthetic (seeded)"}
    w = args.workload
    if w in ("tiny", "long16", "long32"):
        b = (WL.tiny_decode(device=dev) if w == "tiny"
             else WL.long_context(device=dev, block_size=16 if w == "long16" else 32, poison=False))
        bt = torch.from_numpy(b.block_tables).to(dev)
        sl = torch.from_numpy(b.context_lens).to(dev)
        out = torch.empty(b.q.shape, dtype=b.q.dtype, device=dev)
        # the host schedule: partition length for the batch (512 for long context,
        # 32 for the tiny batch) and the work list, longest first
        pt = B.decode_partition_tokens(b.context_lens, b.num_heads)
        items = torch.from_numpy(B.partition_work_items(b.context_lens, pt,
                                                        b.max_blocks_per_seq,
                                                        b.block_size)).to(dev)
        ws = torch.empty(max(16, B.paged_attn_workspace_size(
            b.num_seqs, b.num_heads, b.head_dim, b.block_size, b.max_blocks_per_seq, pt)),
            dtype=torch.uint8, device=dev)
        kw = dict(out=out, partition_tokens=pt, workspace=ws, work_items=items,
                  error_record=rec)
        if b.has_append:
            fn = lambda: B.paged_attn_decode_append(b.q, b.new_k, b.new_v, b.k_cache, b.v_cache, bt,
                                                    sl, b.scale, **kw)
        else:
            fn = lambda: B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, **kw)
        flush = None
        if w == "tiny":
            # 1 GiB written between calls: more than L2, and long enough (~0.15 ms)
            # that the host has enqueued the timed call before the GPU gets to it
            scratch = torch.empty(2 ** 30, dtype=torch.uint8, device=dev)
            flush = lambda: scratch.fill_(1)
        ms = _time_device(fn, K, W, stream, flush)
        nb = step_bytes(b.context_lens, b.num_heads, b.head_dim, b.block_size,
                        partition_tokens=pt)
        total = nb["total"] - (0 if b.has_append else nb["append_write"])
        line.update(config={"workload": b.name, "num_seqs": b.num_seqs, "num_heads": b.num_heads,
                            "head_dim": b.head_dim, "block_size": b.block_size,
                            "context_tokens": int(b.context_lens.sum()),
                            "partition_tokens": pt,
                            "schedule": "host-chosen partition length and work list",
                            "timing": ("each call replayed from a CUDA graph after an L2 flush"
                                       if flush else "calls back to back between two events"),
                            "l2": "flushed between steps" if flush else "inputs larger than L2"},
                    dtype="f16" if b.dtype == torch.float16 else "bf16")
        tokens = int(b.context_lens.sum())
        value = total / (ms * 1e-3) / 1e9
    elif w == "small":
        # small decode batches: 16 sequences (13B-shaped lengths: log-normal around 350,
        # sigma 0.75, clipped to [16, 2048]), 40 heads x 128, bf16, fused append.  The
        # split-K partition length and work list come from the host schedule
        # (pa_decode_partition_tokens, pa_decode_work_items); a fixed 512 is timed
        # beside it.  Four independent batches (0.44 GB of K/V) are called in turn so
        # that each call's inputs have left L2, and the calls replay from a CUDA graph.
        import numpy as np
        H, D, bs = 40, 128, 16
        batches = []
        for j in range(4):
            lens = WL.lognormal_lengths(np.random.default_rng(args.seed * 100 + j), 16, 350.0,
                                        0.75, 16, 2048)
            batches.append(WL.random_decode_batch(args.seed * 100 + j, lens, H, D, bs,
                                                  dtype="bf16", device=dev, with_append=True,
                                                  poison=False))

        def calls(choose):
            fns, pts = [], []
            for b in batches:
                pt = B.decode_partition_tokens(b.context_lens, H) if choose else 512
                items = torch.from_numpy(B.partition_work_items(
                    b.context_lens, pt, b.max_blocks_per_seq, bs)).to(dev)
                bt = torch.from_numpy(b.block_tables).to(dev)
                sl = torch.from_numpy(b.context_lens).to(dev)
                out = torch.empty(b.q.shape, dtype=b.q.dtype, device=dev)
                ws = torch.empty(max(16, B.paged_attn_workspace_size(
                    b.num_seqs, H, D, bs, b.max_blocks_per_seq, pt)), dtype=torch.uint8,
                    device=dev)
                # the inputs are uploaded before the loop: no kernel writes them, so
                # each call may read them while the previous call's merge runs
                fns.append(lambda b=b, bt=bt, sl=sl, out=out, ws=ws, pt=pt, items=items:
                           B.paged_attn_decode_append(b.q, b.new_k, b.new_v, b.k_cache,
                                                      b.v_cache, bt, sl, b.scale, out=out,
                                                      partition_tokens=pt, workspace=ws,
                                                      error_record=rec, work_items=items,
                                                      early_inputs=True))
                pts.append(pt)
            return fns, pts

        fns, pts = calls(True)
        ms = _time_graph(fns, K, W, stream)
        fixed_ms = _time_graph(calls(False)[0], K, W, stream)
        tokens = statistics.mean(int(b.context_lens.sum()) for b in batches)
        total = statistics.mean(
            step_bytes(b.context_lens, H, D, bs, partition_tokens=p)["total"]
            for b, p in zip(batches, pts))
        value = total / (ms * 1e-3) / 1e9
        line.update(config={"workload": "small decode batches: 16 seqs, lengths lognormal("
                                        "median 350, sigma 0.75) clipped to [16, 2048], 40 "
                                        "heads x 128, bf16, block 16, fused append",
                            "batches": len(batches), "context_tokens": tokens,
                            "partition_tokens": pts,
                            "schedule": "host-chosen partition length and work list; "
                                        "early_inputs (inputs read while the previous "
                                        "call's merge runs)",
                            "timing": "CUDA graph of 32 calls, replayed",
                            "l2": "four batches in turn, 0.44 GB of K/V (inputs larger "
                                  "than L2)"},
                    dtype="bf16",
                    fixed_partition_512={"ms_per_step": round(fixed_ms, 5),
                                         "speedup_of_schedule": round(fixed_ms / ms, 3)})
    elif w == "sampling":
        plan = WL.parallel_sampling(device=dev)
        S, bs = plan.samples, plan.block_size
        alloc = B.BlockAllocator(plan.num_blocks, bs, plan.free_order)
        kc = torch.zeros((plan.num_blocks, plan.num_heads, bs, plan.head_dim), dtype=plan.dtype,
                         device=dev)
        vc = torch.zeros_like(kc)
        for k in range(plan.num_prompts):
            a, e = int(plan.prompt_offsets[k]), int(plan.prompt_offsets[k + 1])
            alloc.add(k * S, e - a)
            B.kv_cache_append(plan.prompt_k[a:e], plan.prompt_v[a:e],
                              torch.from_numpy(alloc.slots(k * S, 0, e - a)).to(dev), kc, vc)
            for s_ in range(1, S):
                alloc.fork(k * S, k * S + s_)
        ids = list(range(plan.num_seqs))
        slots, pairs = alloc.batch_append(ids)
        pairs_d = torch.from_numpy(pairs).to(dev)
        copy_ms = _time_device(lambda: B.block_copy([kc], [vc], pairs_d), 20, 3, stream)
        B.kv_cache_append(plan.tail_k[torch.from_numpy(plan.tail_offsets[:-1]).to(dev)],
                          plan.tail_v[torch.from_numpy(plan.tail_offsets[:-1]).to(dev)],
                          torch.from_numpy(slots).to(dev), kc, vc)
        rows, rslots = [], []
        for i in ids:
            for t in range(1, int(plan.tail_lens[i])):
                rows.append(int(plan.tail_offsets[i]) + t)
                rslots.append(alloc.append(i)[0])
        ri = torch.tensor(rows, device=dev)
        B.kv_cache_append(plan.tail_k[ri], plan.tail_v[ri], torch.tensor(rslots, device=dev), kc,
                          vc)
        mb = max(len(alloc.block_table(i)) for i in ids)
        tables, lens = alloc.batch_block_tables(ids, mb)
        bt, sl = torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev)
        out = torch.empty(plan.q.shape, dtype=plan.dtype, device=dev)
        fn = lambda: B.paged_attn_decode(plan.q, kc, vc, bt, sl, plan.scale, out=out,
                                         error_record=rec)
        plain_ms = _time_device(fn, K, W, stream)
        ms, sched = plain_ms, "full grid, 512-token partitions"
        if not args.no_share:
            # each prompt's full partitions read once for its 8 samples
            pt = args.serving_partition or B.decode_partition_tokens(lens, plan.num_heads)
            items, recs = B.share_plan(tables, lens, pt, bs, fused_append=False)
            it_d, rc_d = torch.from_numpy(items).to(dev), torch.from_numpy(recs).to(dev)
            ws = torch.empty(max(16, B.paged_attn_workspace_size(
                plan.num_seqs, plan.num_heads, plan.head_dim, bs, mb, pt)), dtype=torch.uint8,
                device=dev)
            fn = lambda: B.paged_attn_decode(plan.q, kc, vc, bt, sl, plan.scale, out=out,
                                             partition_tokens=pt, workspace=ws, work_items=it_d,
                                             shared_records=rc_d, error_record=rec)
            ms = _time_device(fn, K, W, stream)
            sched = (f"{len(recs)} shared-partition records + {len(items)} work items, "
                     f"{pt}-token partitions")
        nb = step_bytes(lens, plan.num_heads, plan.head_dim, bs)
        total = nb["total"] - nb["append_write"]
        st = alloc.stats()
        unique_kv = st["slots_filled"] * plan.num_heads * plan.head_dim * 4
        tokens = int(lens.sum())
        value = total / (ms * 1e-3) / 1e9
        line.update(config={"workload": "parallel sampling: 32 prompts x 8 samples, shared "
                                        "1024+U[1,15]-token prefixes, tails U[1,512]",
                            "num_seqs": plan.num_seqs, "copies": int(len(pairs)),
                            "context_tokens": tokens, "schedule": sched,
                            "l2": "inputs larger than L2"},
                    dtype="bf16", block_copy_ms=round(copy_ms, 5),
                    without_sharing_ms=round(plain_ms, 5),
                    unique_kv_bytes=unique_kv,
                    unique_kv_gbs=round(unique_kv / (ms * 1e-3) / 1e9, 1),
                    unique_kv_frac_of_peak=round(unique_kv / (ms * 1e-3) / 1e9 / peak, 4))
    elif w == "mixed":
        plan = WL.mixed_serving(device=dev)
        N, bs = plan.num_seqs, plan.block_size
        alloc = B.BlockAllocator(plan.num_blocks, bs, plan.free_order)
        kc = torch.zeros((plan.num_blocks, plan.num_heads, bs, plan.head_dim), dtype=plan.dtype,
                         device=dev)
        vc = torch.zeros_like(kc)
        slots0 = []
        for i in range(N):
            a, e = int(plan.init_offsets[i]), int(plan.init_offsets[i + 1])
            alloc.add(i, e - a)
            slots0.append(alloc.slots(i, 0, e - a))
        B.kv_cache_append(plan.init_k, plan.init_v, torch.from_numpy(np.concatenate(slots0)).to(dev),
                          kc, vc)
        ids, next_id = np.arange(N, dtype=np.int64), N     # slot -> live sequence id
        max_blocks = int(-(-(plan.init_lens.max() + plan.steps) // bs))
        tokens_all = [plan.step_tokens(s_) for s_ in range(plan.steps)]
        out = torch.empty((N, plan.num_heads, plan.head_dim), dtype=plan.dtype, device=dev)
        pt = args.serving_partition or 512
        prefix = not (args.no_share or args.no_prefix)
        ws = torch.empty(B.paged_attn_workspace_size(N, plan.num_heads, plan.head_dim, bs,
                                                     max_blocks, pt, tails=prefix),
                         dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        # per-step host inputs staged in one pinned buffer per set, one upload per step
        n_items_max = N * int(-(-max_blocks * bs // pt))
        RW = B.PA_SHARE_RECORD_WORDS
        staging = _Staging(N, max_blocks, n_items_max, RW, dev)
        graphs = None
        if not args.no_graph:
            # the device step captured once per staging set, as in the beam loop, its
            # launches sized for 2N work items and N records
            cap_items, cap_recs = 2 * N, N
            qkv = torch.empty((3,) + tuple(out.shape), dtype=plan.dtype, device=dev)
            tok_stack = torch.stack([torch.stack(t) for t in tokens_all])
            graphs = []
            for j in range(2):
                pc, btj, slj, itj, rcj, tsj, cj = staging.capacity_views(j, cap_items, cap_recs)

                def device_step(pc=pc, btj=btj, slj=slj, itj=itj, rcj=rcj, tsj=tsj, cj=cj):
                    B.block_copy([kc], [vc], pc)
                    B.paged_attn_decode_append(qkv[0], qkv[1], qkv[2], kc, vc, btj, slj,
                                               plan.scale, out=out, partition_tokens=pt,
                                               workspace=ws, error_record=rec, work_items=itj,
                                               shared_records=rcj,
                                               tail_start=tsj if prefix else None, counts=cj)
                side = torch.cuda.Stream(dev)
                side.wait_stream(stream)
                with torch.cuda.stream(side):
                    device_step()                 # counts 0, no pairs: nothing but the merge
                stream.wait_stream(side)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    device_step()
                graphs.append(g)
            torch.cuda.synchronize()
        host_s, stage_s, plan_s, lens_seen, n_shared, n_prefix = 0.0, 0.0, 0.0, 0, 0, 0
        launch_s, n_eager = 0.0, 0
        unique_seen = 0
        # per step: events before the upload, before the copies, before decode, after
        # (created before the loop: creating events costs host time every step)
        split = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
                 for _ in range(plan.steps)]
        t0 = time.perf_counter()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for s_ in range(plan.steps):
            h0 = time.perf_counter()
            fp = plan.fork_pairs[s_]
            if len(fp):   # slot b ends and continues as a fork of slot a (all distinct)
                born = np.arange(next_id, next_id + len(fp), dtype=np.int64)
                alloc.batch_free(ids[fp[:, 1]])
                alloc.batch_fork(ids[fp[:, 0]], born)
                ids[fp[:, 1]] = born
                next_id += len(fp)
            slots, pairs = alloc.batch_append(ids)
            host_s += time.perf_counter() - h0
            h1 = time.perf_counter()
            bt_h, sl_h, it_h, rc_h, ts_h = staging.views(s_)
            stage_s += time.perf_counter() - h1
            h0 = time.perf_counter()
            tables, lens = alloc.batch_block_tables(ids, max_blocks, out=(bt_h, sl_h))
            host_s += time.perf_counter() - h0
            lens_seen += int(lens.sum())
            if s_ % 10 == 0:   # tokens stored once (sampled: the call walks the pool)
                unique_seen += alloc.stats()["slots_filled"]
            q, k, v = tokens_all[s_]
            h2 = time.perf_counter()
            tails = None
            if args.no_share:
                items = B.partition_work_items(lens, pt, max_blocks, plan.block_size)
                it_h[:len(items)] = items
                recs = rc_h[:0]
            elif prefix:   # and the first chunks they share of the partition they diverge in
                items, recs, tails = B.share_plan_prefix(tables, lens, pt, plan.block_size,
                                                         fused_append=True,
                                                         out=(it_h, rc_h, ts_h))
            else:   # partitions that forked sequences still share are read once
                items, recs = B.share_plan(tables, lens, pt, plan.block_size, fused_append=True,
                                           out=(it_h, rc_h))
            plan_s += time.perf_counter() - h2
            n_shared += len(recs)
            n_prefix += int((recs[:, 1] >> 8 > 0).sum())
            evs = split[s_] if s_ % 4 == 0 else None   # the split is sampled every 4th step
            if evs:
                evs[0].record(stream)
            h1 = time.perf_counter()
            captured = (graphs is not None and len(items) <= cap_items
                        and len(recs) <= cap_recs)
            n_eager += 0 if captured else 1
            staged = staging.upload(s_, stream, pairs, len(items), len(recs), tails is not None,
                                    pad=captured)
            stage_s += time.perf_counter() - h1
            if evs:
                evs[1].record(stream)
            h3 = time.perf_counter()
            if captured:
                qkv.copy_(tok_stack[s_])
                graphs[s_ % 2].replay()
                h4 = h5 = time.perf_counter()
            else:
                pairs_d, bt_d, sl_d, it_d, rc_d, ts_d = staged
                if len(pairs):
                    B.block_copy([kc], [vc], pairs_d)
                h4 = time.perf_counter()
                if evs:
                    evs[2].record(stream)
                h5 = time.perf_counter()
                B.paged_attn_decode_append(q, k, v, kc, vc, bt_d, sl_d, plan.scale, out=out,
                                           partition_tokens=pt, workspace=ws, error_record=rec,
                                           work_items=it_d, shared_records=rc_d,
                                           tail_start=ts_d)
            launch_s += time.perf_counter() - h5 + h4 - h3
            if evs:
                evs[3].record(stream)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev1.record(stream)
        torch.cuda.synchronize()
        wall = (time.perf_counter() - t0) / plan.steps
        ms = ev0.elapsed_time(ev1) / plan.steps
        # the staged inputs of the last step gave the same output as direct uploads
        # (the fused append rewrites the same rows: idempotent)
        ref_out = torch.empty_like(out)
        if B.pa_error_read(rec) != [0, 0, 0, 0]:
            raise RuntimeError(f"device error record {B.pa_error_read(rec)}")
        B.paged_attn_decode_append(q, k, v, kc, vc, torch.from_numpy(tables).to(dev),
                                   torch.from_numpy(lens).to(dev), plan.scale, out=ref_out,
                                   partition_tokens=pt, workspace=ws, error_record=rec,
                                   work_items=torch.from_numpy(items).to(dev),
                                   shared_records=(torch.from_numpy(recs).to(dev)
                                                   if len(recs) else None),
                                   tail_start=(torch.from_numpy(tails).to(dev)
                                               if tails is not None else None))
        torch.cuda.synchronize()
        if not torch.equal(ref_out, out):
            raise RuntimeError("staged and direct inputs gave different outputs")
        seg = lambda a, c: round(statistics.mean(e[a].elapsed_time(e[c]) for e in split[::4]), 5)
        tokens = lens_seen / plan.steps
        total = tokens * plan.num_heads * plan.head_dim * 4
        value = total / (ms * 1e-3) / 1e9
        unique_kv = (unique_seen / len(range(0, plan.steps, 10)) * plan.num_heads
                     * plan.head_dim * 4)
        line.update(config={"workload": "mixed serving: 512 seqs, 70% U[32,256] / 30% "
                                        "U[1024,4096], 26 forks/step, fused append+decode",
                            "steps_run": plan.steps, "partition_tokens": pt,
                            "schedule": ("work list only" if args.no_share else
                                         f"shared partitions ({n_shared / plan.steps:.1f} "
                                         f"records per step, {n_prefix / plan.steps:.1f} "
                                         "of them prefix records) + work list"),
                            "device_step": ("copies + fused append and decode replayed from "
                                            "a CUDA graph (lists sized by device-side counts; "
                                            f"{n_eager} of {plan.steps} steps launched eagerly "
                                            "for want of room)"
                                            if graphs is not None else "eager launches"),
                            "l2": "inputs larger than L2"},
                    dtype="f16", host_allocator_ms_per_step=round(1e3 * host_s / plan.steps, 4),
                    host_staging_ms_per_step=round(1e3 * stage_s / plan.steps, 4),
                    host_plan_ms_per_step=round(1e3 * plan_s / plan.steps, 4),
                    host_launch_ms_per_step=round(1e3 * launch_s / plan.steps, 4),
                    unique_kv_bytes=round(unique_kv),
                    unique_kv_gbs=round(unique_kv / (ms * 1e-3) / 1e9, 1),
                    unique_kv_frac_of_peak=round(unique_kv / (ms * 1e-3) / 1e9 / peak, 4),
                    wall_ms_per_step=round(1e3 * wall, 4),
                    device_ms_per_step_split=(
                        {"table_uploads": seg(0, 1), "copies_append_and_decode": seg(1, 3),
                         "note": "one graph: copies, then the append fused into the decode; "
                                 + SPLIT_NOTE}
                        if graphs is not None else
                        {"table_uploads": seg(0, 1), "block_copy": seg(1, 2),
                         "append_and_decode": seg(2, 3),
                         "note": "the append is fused into the decode launch; " + SPLIT_NOTE}),
                    note="value counts K/V bytes only; device time includes copies, H2D "
                         "of tables (staged in pinned memory, two buffer sets) and the decode")
    elif w == "beam":
        # beam-search churn: each step every group keeps the survivors of a random
        # score draw (forks of their parents, the old beams end), every beam
        # appends a token (copy-on-write of shared tails) and all beams decode
        plan = WL.beam_search(device=dev, groups=64, width=4, steps=40, prompt=(500, 1500),
                              num_heads=40, head_dim=128)
        G_, Wd, H, D, bs = plan.groups, plan.width, plan.num_heads, plan.head_dim, plan.block_size
        N = G_ * Wd
        alloc = B.BlockAllocator(plan.num_blocks, bs, plan.free_order)
        kc = torch.zeros((plan.num_blocks, H, bs, D), dtype=plan.dtype, device=dev)
        vc = torch.zeros_like(kc)
        next_id, beams = 0, []
        for g in range(G_):
            a, e = int(plan.prompt_offsets[g]), int(plan.prompt_offsets[g + 1])
            root = next_id
            next_id += 1
            alloc.add(root, e - a)
            B.kv_cache_append(plan.prompt_k[a:e], plan.prompt_v[a:e],
                              torch.from_numpy(alloc.slots(root, 0, e - a)).to(dev), kc, vc)
            grp = []
            for _ in range(Wd):
                alloc.fork(root, next_id)
                grp.append(next_id)
                next_id += 1
            alloc.free(root)
            beams.append(grp)
        beams = np.asarray(beams, dtype=np.int64)                      # [groups, width]
        max_blocks = int(-(-(plan.prompt_lens.max() + plan.steps + 1) // bs))
        tokens_all = [plan.step_tokens(s_) for s_ in range(plan.steps)]
        out = torch.empty((N, H, D), dtype=plan.dtype, device=dev)
        pt = args.serving_partition or 512
        prefix = not (args.no_share or args.no_prefix)
        ws = torch.empty(B.paged_attn_workspace_size(N, H, D, bs, max_blocks, pt, tails=prefix),
                         dtype=torch.uint8, device=dev)
        n_items_max = N * int(-(-max_blocks * bs // pt))
        RW = B.PA_SHARE_RECORD_WORDS
        staging = _Staging(N, max_blocks, n_items_max, RW, dev)
        graphs = None
        if not args.no_graph:
            # the device step (copy-on-write copies, fused append + decode) captured
            # once per staging set, its launches sized for 2 N work items and N
            # records (blocks past the counts exit at once, but each costs a little);
            # each step writes its lists and their counts into the set and replays the
            # set's graph, or launches eagerly when its plan does not fit
            cap_items, cap_recs = 2 * N, N
            qkv = torch.empty((3, N, H, D), dtype=plan.dtype, device=dev)
            tok_stack = torch.stack([torch.stack(t) for t in tokens_all])
            graphs = []
            for j in range(2):
                pc, btj, slj, itj, rcj, tsj, cj = staging.capacity_views(j, cap_items, cap_recs)

                def device_step(pc=pc, btj=btj, slj=slj, itj=itj, rcj=rcj, tsj=tsj, cj=cj):
                    B.block_copy([kc], [vc], pc)
                    B.paged_attn_decode_append(qkv[0], qkv[1], qkv[2], kc, vc, btj, slj,
                                               plan.scale, out=out, partition_tokens=pt,
                                               workspace=ws, error_record=rec, work_items=itj,
                                               shared_records=rcj,
                                               tail_start=tsj if prefix else None, counts=cj)
                side = torch.cuda.Stream(dev)
                side.wait_stream(stream)
                with torch.cuda.stream(side):
                    device_step()                 # counts 0, no pairs: nothing but the merge
                stream.wait_stream(side)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    device_step()
                graphs.append(g)
            torch.cuda.synchronize()
        host_s, stage_s, plan_s, lens_seen, copies, n_shared = 0.0, 0.0, 0.0, 0, 0, 0
        n_prefix, launch_s, n_eager = 0, 0.0, 0
        unique_seen = 0
        split = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
                 for _ in range(plan.steps)]
        t0 = time.perf_counter()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for s_ in range(plan.steps):
            h0 = time.perf_counter()
            parents = np.take_along_axis(beams, plan.parents[s_], axis=1).ravel()
            children = np.arange(next_id, next_id + N, dtype=np.int64)
            next_id += N
            alloc.batch_fork(parents, children)
            alloc.batch_free(beams.ravel())
            beams = children.reshape(G_, Wd)
            ids = children
            slots, pairs = alloc.batch_append(ids)
            host_s += time.perf_counter() - h0
            h1 = time.perf_counter()
            bt_h, sl_h, it_h, rc_h, ts_h = staging.views(s_)
            stage_s += time.perf_counter() - h1
            h0 = time.perf_counter()
            tables, lens = alloc.batch_block_tables(ids, max_blocks, out=(bt_h, sl_h))
            host_s += time.perf_counter() - h0
            lens_seen += int(lens.sum())
            if s_ % 10 == 0:   # tokens stored once (sampled: the call walks the pool)
                unique_seen += alloc.stats()["slots_filled"]
            copies += len(pairs)
            q, k, v = tokens_all[s_]
            h2 = time.perf_counter()
            tails = None
            if args.no_share:
                items = B.partition_work_items(lens, pt, max_blocks, bs)
                it_h[:len(items)] = items
                recs = rc_h[:0]
            elif prefix:   # and the first chunks they share of the partition they diverge in
                items, recs, tails = B.share_plan_prefix(tables, lens, pt, bs, fused_append=True,
                                                         out=(it_h, rc_h, ts_h))
            else:   # the partitions a group's beams share are read once for the group
                items, recs = B.share_plan(tables, lens, pt, bs, fused_append=True,
                                           out=(it_h, rc_h))
            plan_s += time.perf_counter() - h2
            n_shared += len(recs)
            n_prefix += int((recs[:, 1] >> 8 > 0).sum())
            evs = split[s_] if s_ % 4 == 0 else None   # the split is sampled every 4th step
            if evs:
                evs[0].record(stream)
            h1 = time.perf_counter()
            captured = (graphs is not None and len(items) <= cap_items
                        and len(recs) <= cap_recs)
            n_eager += 0 if captured else 1
            staged = staging.upload(s_, stream, pairs, len(items), len(recs), tails is not None,
                                    pad=captured)
            stage_s += time.perf_counter() - h1
            if evs:
                evs[1].record(stream)
            h3 = time.perf_counter()
            if captured:
                qkv.copy_(tok_stack[s_])
                graphs[s_ % 2].replay()
                h4 = h5 = time.perf_counter()
            else:
                pairs_d, bt_d, sl_d, it_d, rc_d, ts_d = staged
                if len(pairs):
                    B.block_copy([kc], [vc], pairs_d)
                h4 = time.perf_counter()
                if evs:
                    evs[2].record(stream)
                h5 = time.perf_counter()
                B.paged_attn_decode_append(q, k, v, kc, vc, bt_d, sl_d, plan.scale, out=out,
                                           partition_tokens=pt, workspace=ws, error_record=rec,
                                           work_items=it_d, shared_records=rc_d,
                                           tail_start=ts_d)
            launch_s += time.perf_counter() - h5 + h4 - h3
            if evs:
                evs[3].record(stream)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev1.record(stream)
        torch.cuda.synchronize()
        wall = (time.perf_counter() - t0) / plan.steps
        ms = ev0.elapsed_time(ev1) / plan.steps
        # the staged inputs of the last step gave the same output as direct uploads
        # (the fused append rewrites the same rows: idempotent)
        ref_out = torch.empty_like(out)
        if B.pa_error_read(rec) != [0, 0, 0, 0]:
            raise RuntimeError(f"device error record {B.pa_error_read(rec)}")
        B.paged_attn_decode_append(q, k, v, kc, vc, torch.from_numpy(tables).to(dev),
                                   torch.from_numpy(lens).to(dev), plan.scale, out=ref_out,
                                   partition_tokens=pt, workspace=ws, error_record=rec,
                                   work_items=torch.from_numpy(items).to(dev),
                                   shared_records=(torch.from_numpy(recs).to(dev)
                                                   if len(recs) else None),
                                   tail_start=(torch.from_numpy(tails).to(dev)
                                               if tails is not None else None))
        torch.cuda.synchronize()
        if not torch.equal(ref_out, out):
            raise RuntimeError("staged and direct inputs gave different outputs")
        seg = lambda a, c: round(statistics.mean(e[a].elapsed_time(e[c]) for e in split[::4]), 5)
        tokens = lens_seen / plan.steps
        total = tokens * H * D * 4
        value = total / (ms * 1e-3) / 1e9
        unique_kv = unique_seen / len(range(0, plan.steps, 10)) * H * D * 4
        alloc.batch_free(beams.ravel())
        if alloc.num_free() != plan.num_blocks:
            raise RuntimeError("beam workload leaked blocks")
        line.update(config={"workload": "beam-search churn: 64 groups x 4 beams, prompts "
                                        "U[500,1500], 40 heads x 128, bf16, block 16",
                            "steps_run": plan.steps, "partition_tokens": pt,
                            "schedule": ("work list only" if args.no_share else
                                         f"shared partitions ({n_shared / plan.steps:.1f} "
                                         f"records per step, {n_prefix / plan.steps:.1f} "
                                         "of them prefix records) + work list"),
                            "device_step": ("copies + fused append and decode replayed from "
                                            "a CUDA graph (lists sized by device-side counts; "
                                            f"{n_eager} of {plan.steps} steps launched eagerly "
                                            "for want of room)"
                                            if graphs is not None else "eager launches"),
                            "l2": "inputs larger than L2"},
                    dtype="bf16", host_allocator_ms_per_step=round(1e3 * host_s / plan.steps, 4),
                    host_staging_ms_per_step=round(1e3 * stage_s / plan.steps, 4),
                    host_plan_ms_per_step=round(1e3 * plan_s / plan.steps, 4),
                    host_launch_ms_per_step=round(1e3 * launch_s / plan.steps, 4),
                    unique_kv_bytes=round(unique_kv),
                    unique_kv_gbs=round(unique_kv / (ms * 1e-3) / 1e9, 1),
                    unique_kv_frac_of_peak=round(unique_kv / (ms * 1e-3) / 1e9 / peak, 4),
                    wall_ms_per_step=round(1e3 * wall, 4),
                    copies_per_step=round(copies / plan.steps, 2),
                    device_ms_per_step_split=(
                        {"table_uploads": seg(0, 1), "copies_append_and_decode": seg(1, 3),
                         "note": "one graph: copies, then the append fused into the decode; "
                                 + SPLIT_NOTE}
                        if graphs is not None else
                        {"table_uploads": seg(0, 1), "block_copy": seg(1, 2),
                         "append_and_decode": seg(2, 3),
                         "note": "the append is fused into the decode launch; " + SPLIT_NOTE}),
                    note="value counts logical K/V bytes (beams share prefix blocks, so part "
                         "of them is served from L2)")
    elif w in ("append", "copy"):
        # the two cache kernels at sizes where bandwidth matters: the K/V rows of a
        # 16 x 512-token prefill chunk written into scattered slots, or 2000
        # copy-on-write block pairs; both are pure copies, so the measured copy
        # bandwidth is their roofline
        H, D, bs = 40, 128, 16
        g = WL.gen._torch_gen(8, dev)
        rng = np.random.default_rng(8)
        if w == "append":
            T = 16 * 512
            nb = int(1.5 * T / bs)
            kc = torch.zeros((nb, H, bs, D), dtype=torch.bfloat16, device=dev)
            vc = torch.zeros_like(kc)
            k = WL.gen.randn_rounded((T, H, D), torch.bfloat16, g, dev)
            v = WL.gen.randn_rounded((T, H, D), torch.bfloat16, g, dev)
            slots = torch.from_numpy(rng.choice(nb * bs, size=T, replace=False)).to(dev)
            fn = lambda: B.kv_cache_append(k, v, slots, kc, vc, error_record=rec)
            moved = 2 * (2 * T * H * D * 2) + T * 8        # K and V read + written, slots
            desc = f"KV append of a 16 x 512-token chunk ({T} tokens, 40 x 128, bf16) into scattered slots"
            kernel = "kv_append_kernel"
        else:
            n_pairs, nb = 2000, 6000
            kc = WL.gen.randn_rounded((nb, H, bs, D), torch.bfloat16, g, dev)
            vc = WL.gen.randn_rounded((nb, H, bs, D), torch.bfloat16, g, dev)
            pick = rng.choice(nb, size=2 * n_pairs, replace=False)
            pairs = torch.from_numpy(np.stack([pick[:n_pairs], pick[n_pairs:]], 1)).to(dev)
            fn = lambda: B.block_copy([kc], [vc], pairs, error_record=rec)
            moved = 2 * (2 * n_pairs * H * bs * D * 2) + n_pairs * 16
            desc = "copy-on-write block copy: 2000 pairs of 40 x 16 x 128 bf16 blocks (K and V)"
            kernel = "block_copy_kernel"
        ms = _time_device(fn, K, W, stream)
        value = moved / (ms * 1e-3) / 1e9
        tokens = 0
        peak, peak_kind = measured_hbm_peak()
        line.update(config={"workload": desc, "l2": "inputs larger than L2"}, dtype="bf16",
                    roofline={"kernel": kernel, "bound": "hbm", "achieved": round(value, 2),
                              "peak": peak, "unit": "GB/s", "frac": round(value / peak, 4),
                              "peak_source": f"{peak_kind} hbm_gbs", "traffic": None,
                              "algorithmic_bytes_per_launch": moved},
                    note="value = bytes read + written per launch / device time")
    elif w == "prefill":
        # chunked prefill: 16 sequences append a 512-token chunk to contexts of 512..2048
        rng = np.random.default_rng(70)
        lens = rng.integers(512, 2049, size=16)
        nq = np.full(16, 512)
        b = WL.random_decode_batch(70, lens, 40, 128, 16, dtype="bf16", device=dev, poison=False)
        g = WL.gen._torch_gen(77, dev)
        q = WL.gen.randn_rounded((int(nq.sum()), 40, 128), torch.bfloat16, g, dev)
        starts = torch.from_numpy(np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)).to(dev)
        bt = torch.from_numpy(b.block_tables).to(dev)
        sl = torch.from_numpy(b.context_lens).to(dev)
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        # longest sequences dispatched first (the host knows the lengths)
        order = torch.from_numpy(np.argsort(-lens, kind="stable").astype(np.int32)).to(dev)
        fn = lambda: B.paged_attn_prefill(q, starts, 512, b.k_cache, b.v_cache, bt, sl, b.scale,
                                          out=out, error_record=rec, seq_order=order)
        clocks = ClockSampler(gpu_uuid(dev, local_rank))
        clocks.start()
        ms = _time_device(fn, K, W, stream)
        clk = clocks.stop()
        # useful flops: 2*D per (query, visible key) for Q.K^T and again for P.V
        visible = sum(int(((lens[i] - 512) + np.arange(1, 513)).sum()) for i in range(16))
        flops = 4.0 * 128 * 40 * visible
        tflops = flops / (ms * 1e-3) / 1e12
        # a long back-to-back region runs at the power limit: compare it with the
        # sustained peak, a short one with the burst peak
        peak_tf, peak_tf_kind = measured_bf16_peak(ms * K > SUSTAINED_REGION_MS)
        tokens = int(nq.sum())
        value = (int(lens.sum()) * 40 * 128 * 4) / (ms * 1e-3) / 1e9
        line.update(config={"workload": "chunked prefill: 16 seqs x 512-token chunk on contexts "
                                        "U[512,2048], 40 heads x 128, bf16, block 16",
                            "queries": tokens, "context_tokens": int(lens.sum())},
                    dtype="bf16",
                    roofline={"kernel": "paged_prefill_kernel", "bound": "tensor",
                              "traffic": recorded_traffic("paged_prefill_kernel",
                                                          PREFILL_SOURCES),
                              "achieved": round(tflops, 2), "peak": peak_tf,
                              "unit": "TFLOP/s", "frac": round(tflops / peak_tf, 4),
                              "peak_source": peak_tf_kind, "flops_per_launch": flops,
                              "timed_region_ms": round(ms * K, 2), "clocks": clk,
                              "note": "useful flops (causal, 4*D per visible query-key pair); "
                                      "the kernel issues P.V twice (hi + lo parts)"})
    else:
        raise SystemExit(f"unknown workload {w}")
    if B.pa_error_read(rec) != [0, 0, 0, 0]:
        raise RuntimeError(f"device error record: {B.pa_error_read(rec)}")
    line.update(value=round(value, 2), ms_per_step=round(ms, 5),
                pct_of_hbm_peak=round(100 * value / peak, 2),
                peak=f"{peak} GB/s ({peak_kind} hbm_gbs)",
                seq_tokens_per_s=round(tokens / (ms * 1e-3), 1))
    if emit:
        print(json.dumps(line), flush=True)
    return line


SUMMARY_WORKLOADS = ("tiny", "small", "long16", "long32", "sampling", "mixed", "beam",
                     "prefill", "append", "copy")


def workload_summaries(args, rank, world, local_rank) -> dict:
    """The other workloads, each timed as `--workload <name>` would time it (same
    steps and warm-up), summarised for the headline line."""
    import copy
    keep = ("unique_kv_gbs", "unique_kv_frac_of_peak", "without_sharing_ms", "block_copy_ms",
            "fixed_partition_512", "device_ms_per_step_split", "dtype")
    out = {}
    for w in SUMMARY_WORKLOADS:
        a = copy.copy(args)
        a.workload = w
        line = run_workload(a, rank, world, local_rank, emit=False)
        entry = {"workload": line["config"]["workload"], "ms_per_step": line["ms_per_step"],
                 "value": line["value"], "unit": line["unit"],
                 "pct_of_hbm_peak": line["pct_of_hbm_peak"]}
        entry.update({k: line[k] for k in keep if k in line})
        if "roofline" in line:
            r = line["roofline"]
            entry["roofline"] = {k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                                   "peak_source", "clocks") if k in r}
        out[w] = entry
    return out


# --------------------------------------------------------------- oracle arms
def _oracle_sample(b, seqs):
    """Host inputs for the oracle on the listed sequences (outside any timing)."""
    import numpy as np
    import torch
    bs = b.block_size
    used = sorted({int(x) for i in seqs for x in b.block_tables[i][: -(-int(b.context_lens[i]) // bs)]})
    remap = {x: j for j, x in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=b.k_cache.device)
    to_bits = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    kc, vc = to_bits(b.k_cache.index_select(0, idx)), to_bits(b.v_cache.index_select(0, idx))
    sel = torch.tensor(seqs, device=b.q.device)
    tables = np.array([[remap[int(x)] for x in b.block_tables[i][: -(-int(b.context_lens[i]) // bs)]]
                       + [-1] * (b.max_blocks_per_seq - (-(-int(b.context_lens[i]) // bs)))
                       for i in seqs], dtype=np.int64)
    slots = np.array([remap[int(b.slot_mapping[i]) // bs] * bs + int(b.slot_mapping[i]) % bs
                      for i in seqs], dtype=np.int64)
    return dict(q=to_bits(b.q[sel]), k=to_bits(b.new_k[sel]), v=to_bits(b.new_v[sel]), kc=kc,
                vc=vc, tables=tables, lens=b.context_lens[seqs], slots=slots, bs=bs)


def _oracle_step(s, scale):
    from oracle import attention as OA
    from oracle import cache_ops as OC
    kc, vc = s["kc"].copy(), s["vc"].copy()
    OC.kv_append(kc, vc, s["k"], s["v"], s["slots"], s["bs"])
    return OA.paged_decode_attention(s["q"], kc, vc, s["tables"], s["lens"], scale, s["bs"], "bf16")


def _oracle_worker(conn, scale, block_size):
    """One host process of the oracle runner.  Receives its sequences' inputs
    once (untimed), then for every "run" computes append + decode of them with
    the oracle's own functions and sends back (outputs, seconds)."""
    s = conn.recv()
    conn.send("ready")
    while conn.recv() == "run":
        t = time.perf_counter()
        out = _oracle_step(s, scale)
        conn.send((out, time.perf_counter() - t))


def balance_groups(lens, workers: int):
    """Sequences dealt to `workers` groups, longest first, each to the group with
    the fewest tokens so far; every group sorted, empty groups dropped."""
    loads = [0] * max(1, workers)
    groups = [[] for _ in loads]
    for i in sorted(range(len(lens)), key=lambda i: (-int(lens[i]), i)):
        j = min(range(len(loads)), key=lambda j: (loads[j], j))
        groups[j].append(i)
        loads[j] += int(lens[i])
    return [sorted(g) for g in groups if g]


class HostOracle:
    """The fp64 oracle (append, then decode of every listed sequence) on several
    host processes at once, each taking a balanced share of the sequences.
    Processes are spawned, not forked: the parent holds a CUDA context.  Each
    receives its inputs before any timing; `run` then times only the oracle's
    arithmetic across all processes (wall clock, first command to last result)."""

    def __init__(self, b, workers: int, seqs=None):
        import multiprocessing as mp
        seqs = list(range(b.num_seqs)) if seqs is None else list(seqs)
        lens = b.context_lens[seqs]
        self.groups = [[seqs[k] for k in g] for g in balance_groups(lens, workers)]
        self.seqs, self.scale = seqs, b.scale
        ctx = mp.get_context("spawn")
        self.procs, self.conns = [], []
        try:
            for g in self.groups:
                a, c = ctx.Pipe()
                p = ctx.Process(target=_oracle_worker, args=(c, b.scale, b.block_size),
                                daemon=True)
                p.start()
                c.close()
                self.procs.append(p)
                self.conns.append(a)
                a.send(_oracle_sample(b, g))
            for a in self.conns:
                if self._recv(a) != "ready":
                    raise RuntimeError("oracle process did not start")
        except Exception:
            self.close()
            raise

    @staticmethod
    def _recv(conn, timeout=600.0):
        if not conn.poll(timeout):
            raise RuntimeError("oracle process gave no answer")
        return conn.recv()

    @property
    def workers(self) -> int:
        return len(self.groups)

    def run(self):
        """(fp64 outputs [n, H, D] in `seqs` order, wall seconds)."""
        import numpy as np
        t = time.perf_counter()
        for a in self.conns:
            a.send("run")
        parts = [self._recv(a) for a in self.conns]
        dt = time.perf_counter() - t
        pos = {i: k for k, i in enumerate(self.seqs)}
        out = None
        for g, (o, _) in zip(self.groups, parts):
            if out is None:
                out = np.empty((len(self.seqs),) + o.shape[1:], dtype=np.float64)
            out[[pos[i] for i in g]] = o
        return out, dt

    def close(self):
        for a in self.conns:
            try:
                a.send("stop")
            except Exception:
                pass
        for p in self.procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
        self.procs, self.conns = [], []


def host_workers(world: int) -> int:
    """Host processes one rank may use for the oracle: this host's CPUs split
    over the ranks sharing it."""
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    return max(1, n // max(1, world))


def half_ulp_bf16(x):
    """Half a bf16 ulp at |x| (8 significant bits; subnormals below 2^-126)."""
    import numpy as np
    _, e = np.frexp(np.abs(x))
    return 0.5 * np.ldexp(1.0, np.maximum(e - 1, -126) - 7)


def parity_report(out_bf16, ref, append_ok: bool) -> dict:
    """The step's bf16 output against the fp64 oracle: within 2e-3 plus half a
    bf16 ulp at the oracle's value, element by element."""
    import numpy as np
    got = out_bf16.detach().double().cpu().numpy()
    err = np.abs(got - ref)
    bound = 2e-3 + half_ulp_bf16(ref)
    bad = int((~(err <= bound)).sum())
    return {"seqs_checked": int(ref.shape[0]), "elements": int(ref.size),
            "max_abs_err": float(np.nanmax(err)) if err.size else 0.0,
            "elements_out_of_bound": bad,
            "bound": "2e-3 + half a bf16 ulp at the oracle value (bf16 output)",
            "append_bit_exact": bool(append_ok), "ok": bool(bad == 0 and append_ok),
            "oracle": "fp64 CPU oracle, append then decode, every sequence of the batch"}


def oracle_timing(host, nbytes_total: int, context_tokens: int, passes: int = 3):
    """cpu_baseline entry: mean wall time of `passes` runs of the host oracle
    over the whole batch (after the run that produced the parity reference)."""
    times = [host.run()[1] for _ in range(passes)]
    dt = statistics.mean(times)
    return {"value": round(nbytes_total / dt / 1e9, 4), "unit": UNIT, "cores": host.workers,
            "kind": "oracle", "host_cpus": os.cpu_count(), "cpu_model": host_cpu_model(),
            "sample": f"the whole batch ({len(host.seqs)} sequences, all heads, "
                      f"{context_tokens} context tokens), append + decode, over "
                      f"{host.workers} processes; mean of {passes} passes",
            "seconds": round(dt, 4)}


def run_reference(args, rank, world, local_rank):
    """The oracle arm: the fp64 CPU oracle, as it stands, timed on this host's
    cores on the headline batch (every step: append + decode of all sequences)."""
    if rank != 0:
        return
    import numpy as np
    import torch
    from workloads import decode_13b

    device = "cuda" if torch.cuda.is_available() else "cpu"
    b = decode_13b(seed=args.seed, device=device, block_size=args.block_size, poison=False)
    nb = step_bytes(b.context_lens, b.num_heads, b.head_dim, b.block_size,
                    partition_tokens=args.partition)["total"]
    host = HostOracle(b, host_workers(1))
    try:
        for _ in range(args.warmup):
            host.run()
        times = [host.run()[1] for _ in range(args.steps)]
    finally:
        host.close()
    total = sum(times)
    value = nb * args.steps / total / 1e9
    ms = 1e3 * total / args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q; no trained weights)",
        "seq_tokens_per_s": round(float(np.sum(b.context_lens)) / (ms * 1e-3), 1),
        "config": headline_config(b, args, world),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": host.workers,
                         "kind": "oracle", "host_cpus": os.cpu_count(),
                         "cpu_model": host_cpu_model(),
                         "sample": f"the whole batch ({b.num_seqs} sequences, all heads) every "
                                   f"step, over {host.workers} processes"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=2,
                    help="13B-shaped batch: seed of the lengths and values (rank r uses a "
                         "seed derived from it)")
    ap.add_argument("--block-size", type=int, default=16, help="13B-shaped batch: tokens per block")
    ap.add_argument("--partition", type=int, default=512,
                    help="13B-shaped batch: split-K partition length in tokens")
    ap.add_argument("--no-workloads", action="store_true",
                    help="13b: skip the summaries of the other workloads in the headline line")
    ap.add_argument("--no-share", action="store_true",
                    help="sampling/beam/mixed: read shared partitions once per sequence "
                         "instead of once per group")
    ap.add_argument("--no-graph", action="store_true",
                    help="beam/mixed: launch each step's copies and decode eagerly instead of "
                         "replaying them from a CUDA graph")
    ap.add_argument("--no-prefix", action="store_true",
                    help="beam/mixed: share whole partitions only, not the shared first "
                         "chunks of a partition the group's members diverge in")
    ap.add_argument("--serving-partition", type=int, default=0,
                    help="sampling/beam/mixed: split-K partition length (0: the host rule "
                         "for sampling, 512 for beam and mixed)")
    ap.add_argument("--workload", default="13b",
                    choices=["13b", "tiny", "small", "long16", "long32", "sampling", "mixed",
                             "beam", "prefill", "append", "copy"],
                    help="13b (default, the headline line) or another seeded workload")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world, local_rank)
        elif args.workload != "13b":
            run_workload(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1 and args.impl == "ours":
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
