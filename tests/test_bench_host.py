"""CPU tests of bench.py's host logic: byte accounting, clock parsing, and the
multi-rank reductions (two gloo ranks on 127.0.0.1)."""

import os
import socket

import torch
import torch.multiprocessing as mp

import bench


def test_step_bytes_by_hand():
    # two sequences: 20 tokens (1 partition of 512) and 600 tokens (2 partitions)
    b = bench.step_bytes([20, 600], num_heads=2, head_dim=8, block_size=16, partition_tokens=512)
    kv = (20 + 600) * 2 * 8 * 2 * 2
    assert b["kv"] == kv
    partials = 2 * 2 * (8 + 2) * 4                      # 2 partitions x 2 heads of (D + m, l) fp32
    table = (2 + 38) * 4
    q = 2 * 2 * 8 * 2
    appended = 2 * 2 * 2 * 8 * 2                        # K and V rows of 2 seqs x 2 heads written
    assert b["append_write"] == appended
    assert b["decode_partition"] == kv + q + table + 2 * 4 + 1 * 2 * 8 * 2 + partials + appended
    assert b["decode_merge"] == partials + 1 * 2 * 8 * 2 + 2 * 4
    assert b["total"] == b["decode_partition"] + b["decode_merge"]


def test_clock_rows_parse_reasons_and_median():
    rows = "\n".join([
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1900, 2070, 1300.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2000, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ])
    c = bench.parse_clock_rows(rows)
    assert c == {"sm_mhz": 2000.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_rank_seeds_differ():
    assert len({bench.rank_seed(2, r) for r in range(8)}) == 8
    assert bench.rank_seed(2, 0) == 2


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    bench.barrier(w)
    mx = bench.reduce_max(1.5 + r, w)
    sm = bench.reduce_sum(10.0 * (r + 1), w)
    q.put((r, w, lr, mx, sm))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_and_sum():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 0, 2.5, 30.0), (1, 2, 1, 2.5, 30.0)]


def test_host_cpu_model_is_a_nonempty_string():
    m = bench.host_cpu_model()
    assert isinstance(m, str) and m


def test_clock_records_that_are_rejected():
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(dict(ok, reasons=["sw_power_cap"], sm_mhz=1800.0))
    assert bench.clocks_rejected(dict(ok, reasons=["hw_slowdown"]))
    assert bench.clocks_rejected(dict(ok, reasons=["sw_thermal_slowdown", "sw_power_cap"]))
    assert bench.clocks_rejected(dict(ok, sm_mhz=1200.0))          # locked low, no reason
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None,
                                      "reasons": ["nvidia-smi unavailable"]})


def test_bench_keeps_the_oracle_on_one_blas_thread():
    import subprocess
    import sys
    code = ("import bench, numpy as np; a = np.random.rand(3000, 256); "
            "[a @ a.T for _ in range(3)]; "
            "print([l for l in open('/proc/self/status') if l.startswith('Threads')][0].split()[1])")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "1"


def test_oracle_sample_follows_the_block_size():
    import numpy as np
    from oracle import attention as OA
    from oracle import cache_ops as OC
    from workloads import decode_13b
    for bs in (16, 32):
        b = decode_13b(seed=3, device="cpu", num_seqs=6, block_size=bs, poison=False)
        seqs = [0, 2, 5]
        got = bench._oracle_step(bench._oracle_sample(b, seqs), b.scale)
        # the same step on the whole pool, without the compaction
        bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()
        kc, vc = bits(b.k_cache), bits(b.v_cache)
        OC.kv_append(kc, vc, bits(b.new_k), bits(b.new_v), b.slot_mapping, bs)
        want = OA.paged_decode_attention(bits(b.q), kc, vc, b.block_tables, b.context_lens,
                                         b.scale, bs, "bf16")[seqs]
        assert np.array_equal(got, want)


def test_nvml_reason_bits_by_name():
    assert bench.reasons_from_mask(0) == []
    assert bench.reasons_from_mask(0x4 | 0x40) == ["hw_thermal_slowdown", "sw_power_cap"]
    assert bench.reasons_from_mask(0x1 | 0x8 | 0x20) == ["hw_slowdown", "sw_thermal_slowdown"]
    c = bench.summarize_clocks([2070.0, 1990.0, 2070.0], [2070.0], {"sw_power_cap"}, "nvml")
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 3, "source": "nvml"}
    assert bench.clocks_rejected(dict(c, reasons=["hw_power_brake_slowdown"]))


def test_balance_groups_cover_every_sequence_once():
    import numpy as np
    lens = np.random.default_rng(0).integers(1, 2000, size=97)
    groups = bench.balance_groups(lens, 8)
    flat = sorted(i for g in groups for i in g)
    assert flat == list(range(97))
    loads = [int(lens[g].sum()) for g in groups]
    assert max(loads) - min(loads) <= int(lens.max())       # greedy longest-first bound
    assert bench.balance_groups([5, 3], 8) == [[0], [1]]     # no empty groups


def test_host_oracle_processes_match_the_oracle_in_one_process():
    """The spawned-process runner gives exactly what the oracle gives in this
    process, sequence for sequence, on every pass."""
    import numpy as np
    from workloads import random_decode_batch
    b = random_decode_batch(41, [1, 17, 200, 513, 40, 90, 1000], 3, 64, 16, dtype="bf16",
                            device="cpu", with_append=True, poison=False)
    want = bench._oracle_step(bench._oracle_sample(b, list(range(b.num_seqs))), b.scale)
    host = bench.HostOracle(b, 3)
    try:
        assert host.workers == 3
        for _ in range(2):
            got, dt = host.run()
            assert np.array_equal(got, want) and dt > 0
    finally:
        host.close()


def test_parity_report_flags_an_element_out_of_bound():
    import numpy as np
    rng = np.random.default_rng(1)
    ref = rng.standard_normal((4, 2, 8))
    out = torch.from_numpy(ref).to(torch.bfloat16)
    r = bench.parity_report(out, ref, True)
    assert r["ok"] and r["elements_out_of_bound"] == 0 and r["seqs_checked"] == 4
    assert not bench.parity_report(out, ref, False)["ok"]      # append not bit-exact
    bad = out.clone()
    bad[2, 1, 3] += 0.05
    r = bench.parity_report(bad, ref, True)
    assert not r["ok"] and r["elements_out_of_bound"] == 1


def test_tensor_peak_for_long_regions_is_the_sustained_one(tmp_path, monkeypatch):
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    (tmp_path / "MEASURED_PEAKS.json").write_text(__import__("json").dumps(peaks))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_bf16_peak() == (1900.0, "measured bf16_tflops")
    assert bench.measured_bf16_peak(True) == (1700.0, "measured bf16_tflops_sustained")
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    assert bench.measured_bf16_peak(True)[1] == "fallback"
