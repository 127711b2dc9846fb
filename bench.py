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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-attn decode KV GB/s (% of HBM peak), seq-tokens/s at 13B shape"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
DECODE_SOURCES = ("paged_kv_cache_317_gb300/csrc/paged_attn_decode.cu",
                  "paged_kv_cache_317_gb300/csrc/common.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


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


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def decode_source_sha() -> str:
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """dram bytes per launch from the last ncu capture, if the kernel is unchanged since."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[kernel]
    except Exception:
        return None
    if rec.get("source_sha") != decode_source_sha():
        return None
    return rec.get("dram_bytes_per_launch_full_size")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples over an interval."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
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
        return parse_clock_rows(text)


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


# --------------------------------------------------------------- our arm
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
    b = decode_13b(seed=rank_seed(2, rank), device=dev, poison=False)
    N, H, D, bs = b.num_seqs, b.num_heads, b.head_dim, b.block_size
    MB = b.max_blocks_per_seq
    pt = 512
    bt = torch.from_numpy(b.block_tables).to(dev)
    sl = torch.from_numpy(b.context_lens).to(dev)
    slots = torch.from_numpy(b.slot_mapping).to(dev)
    out = torch.empty((N, H, D), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(B.paged_attn_workspace_size(N, H, D, bs, MB, pt), dtype=torch.uint8,
                     device=dev)
    nbytes = step_bytes(b.context_lens, H, D, bs, partition_tokens=pt)
    stream = torch.cuda.current_stream(dev)
    rec = B.new_error_record(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        B.paged_attn_decode_append(b.q, b.new_k, b.new_v, b.k_cache, b.v_cache, bt, sl, b.scale,
                                   out=out, partition_tokens=pt, workspace=ws, error_record=rec,
                                   phases=1)
        if ev is not None:
            ev[1].record(stream)
        B.paged_attn_decode_append(b.q, b.new_k, b.new_v, b.k_cache, b.v_cache, bt, sl, b.scale,
                                   out=out, partition_tokens=pt, workspace=ws, error_record=rec,
                                   phases=2)

    K, W = args.steps, args.warmup
    for _ in range(W):
        step()
    torch.cuda.synchronize(dev)
    if B.pa_error_read(rec) != [0, 0, 0, 0]:
        raise RuntimeError(f"device error record after warm-up: {B.pa_error_read(rec)}")

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local_rank)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for i in range(K):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end) / K
    part_ms = statistics.mean(a.elapsed_time(c) for a, c in evs)
    ms_max = reduce_max(ms, world, dev)

    # end to end through the public API: pinned host inputs copied in, output copied out
    pin = lambda t: t.detach().cpu().pin_memory()
    h_q, h_k, h_v = pin(b.q), pin(b.new_k), pin(b.new_v)
    h_bt, h_sl = pin(bt), pin(sl)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d_q, d_k, d_v = torch.empty_like(b.q), torch.empty_like(b.new_k), torch.empty_like(b.new_v)
    d_bt, d_sl = torch.empty_like(bt), torch.empty_like(sl)
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_bt, h_sl))
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        for d, h in ((d_q, h_q), (d_k, h_k), (d_v, h_v), (d_bt, h_bt), (d_sl, h_sl)):
            d.copy_(h, non_blocking=True)
        B.paged_attn_decode_append(d_q, d_k, d_v, b.k_cache, b.v_cache, d_bt, d_sl, b.scale,
                                   out=out, partition_tokens=pt, workspace=ws, error_record=rec)
        h_out.copy_(out, non_blocking=True)

    for _ in range(W):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = reduce_max(e0.elapsed_time(e1) / K, world, dev)
    if B.pa_error_read(rec) != [0, 0, 0, 0]:
        raise RuntimeError(f"device error record: {B.pa_error_read(rec)}")

    total_bytes = reduce_sum(nbytes["total"], world, dev)
    tokens = reduce_sum(float(b.context_lens.sum()), world, dev)
    value = total_bytes / (ms_max * 1e-3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    achieved = nbytes["decode_partition"] / (part_ms * 1e-3) / 1e9

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(b, budget_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 K/V/Q; no trained weights)",
            "pct_of_hbm_peak": round(100 * value / peak, 2),
            "seq_tokens_per_s": round(tokens / (ms_max * 1e-3), 1),
            "seqs_per_s": round(world * N / (ms_max * 1e-3), 1),
            "config": {
                "workload": "13B-shaped paged decode step: append 1 token/seq + decode",
                "num_seqs_per_gpu": N, "num_heads": H, "head_dim": D, "block_size": bs,
                "context_tokens_per_gpu": int(b.context_lens.sum()),
                "lengths": "lognormal(median 350, sigma 0.75) clipped to [16, 2048]",
                "pool_blocks": b.num_blocks, "partition_tokens": pt, "out_dtype": "bf16",
                "l2": "inputs larger than L2 (2.4 GB of K/V read per step); no flush",
                "parallelism": f"replicas x{world} (independent batches, no collective)",
            },
            "bytes_per_step": nbytes,
            "roofline": {
                "kernel": "paged_attn_partition_kernel", "bound": "hbm",
                "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                "traffic": recorded_traffic("paged_attn_partition_kernel"),
                "algorithmic_bytes_per_launch": nbytes["decode_partition"],
                "avg_launch_ms": round(part_ms, 5),
            },
            "e2e": {"value": round(total_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                    "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": 2 * K,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------- oracle arms
def _oracle_sample(b, seqs):
    """Host inputs for the oracle on the listed sequences (outside any timing)."""
    import numpy as np
    import torch
    used = sorted({int(x) for i in seqs for x in b.block_tables[i][: -(-int(b.context_lens[i]) // 16)]})
    remap = {x: j for j, x in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=b.k_cache.device)
    to_bits = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    kc, vc = to_bits(b.k_cache.index_select(0, idx)), to_bits(b.v_cache.index_select(0, idx))
    sel = torch.tensor(seqs, device=b.q.device)
    tables = np.array([[remap[int(x)] for x in b.block_tables[i][: -(-int(b.context_lens[i]) // 16)]]
                       + [-1] * (b.max_blocks_per_seq - (-(-int(b.context_lens[i]) // 16)))
                       for i in seqs], dtype=np.int64)
    slots = np.array([remap[int(b.slot_mapping[i]) // 16] * 16 + int(b.slot_mapping[i]) % 16
                      for i in seqs], dtype=np.int64)
    return dict(q=to_bits(b.q[sel]), k=to_bits(b.new_k[sel]), v=to_bits(b.new_v[sel]), kc=kc,
                vc=vc, tables=tables, lens=b.context_lens[seqs], slots=slots)


def _oracle_step(s, scale):
    from oracle import attention as OA
    from oracle import cache_ops as OC
    kc, vc = s["kc"].copy(), s["vc"].copy()
    OC.kv_append(kc, vc, s["k"], s["v"], s["slots"], 16)
    return OA.paged_decode_attention(s["q"], kc, vc, s["tables"], s["lens"], scale, 16, "bf16")


def cpu_baseline(b, budget_s=15.0):
    """The oracle, as it stands, on a bounded sample of the same batch (single thread)."""
    import numpy as np
    rng = np.random.default_rng(0)
    order = [int(i) for i in rng.permutation(b.num_seqs)]
    # size the sample from the time of the first few sequences
    probe = sorted(order[:4])
    t = time.perf_counter()
    _oracle_step(_oracle_sample(b, probe), b.scale)
    per_seq = max(1e-4, (time.perf_counter() - t) / len(probe))
    n = int(max(1, min(b.num_seqs, budget_s / per_seq)))
    seqs = sorted(order[:n])
    s = _oracle_sample(b, seqs)
    t = time.perf_counter()
    _oracle_step(s, b.scale)
    dt = time.perf_counter() - t
    nb = step_bytes(b.context_lens[seqs], b.num_heads, b.head_dim, b.block_size)
    return {"value": round(nb["total"] / dt / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} of {b.num_seqs} sequences (all heads), append + decode, "
                      f"{int(b.context_lens[seqs].sum())} context tokens, {dt:.2f} s",
            "seconds": round(dt, 3)}


def run_reference(args, rank, world, local_rank):
    """The oracle arm: the fp64 CPU oracle timed on this host on the same workload."""
    if rank != 0:
        return
    import numpy as np
    import torch
    from workloads import decode_13b

    device = "cuda" if torch.cuda.is_available() else "cpu"
    b = decode_13b(seed=2, device=device, poison=False)
    rng = np.random.default_rng(1)
    order = [int(i) for i in rng.permutation(b.num_seqs)]
    one = _oracle_sample(b, order[:1])
    t = time.perf_counter()
    _oracle_step(one, b.scale)
    per_seq = time.perf_counter() - t
    # keep (K + W) steps within about two minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(b.num_seqs, budget / max(per_seq, 1e-4))))
    groups = [order[i:i + n] for i in range(0, b.num_seqs - n + 1, n)][:4]
    samples = [_oracle_sample(b, sorted(g)) for g in groups]
    for i in range(args.warmup):
        _oracle_step(samples[i % len(samples)], b.scale)
    times, nbytes, tokens = [], 0.0, 0.0
    for i in range(args.steps):
        s = samples[i % len(samples)]
        t = time.perf_counter()
        _oracle_step(s, b.scale)
        times.append(time.perf_counter() - t)
        nbytes += step_bytes(s["lens"], b.num_heads, b.head_dim, b.block_size)["total"]
        tokens += float(np.sum(s["lens"]))
    total = sum(times)
    value = nbytes / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q)",
        "seq_tokens_per_s": round(tokens / total, 1),
        "config": {"workload": "13B-shaped paged decode step: append 1 token/seq + decode",
                   "sample_seqs_per_step": n, "of_seqs": b.num_seqs},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{n} of {b.num_seqs} sequences per step, all heads"},
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
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1 and args.impl == "ours":
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
