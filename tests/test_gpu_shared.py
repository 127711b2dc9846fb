"""Decode over partitions that several sequences share (shared_records built by
share_plan): families of sequences forked from one prompt with private,
copy-on-write tails, checked against the oracle over each sequence's logical
tokens (PagedAttention, zeroshotmind.com page, "Sharing a prefix without copying
it")."""

import numpy as np
import pytest
import torch

from gpu_util import assert_matches_oracle
from oracle.content import LogicalSequences
from test_gpu_workloads import _oracle_logical
from workloads.gen import DTYPES, _torch_gen, randn_rounded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    from paged_kv_cache_317_gb300 import binding
    return binding


class Families:
    """Sequences forked from shared prompts, written through the library's own
    append and copy kernels; `store` holds every row ever written, in order."""

    def __init__(self, B, seed, prompts, members, tail_max, H, D, bs, dtype, fused):
        rng = np.random.default_rng(seed)
        self.H, self.D, self.bs, self.fused = H, D, bs, fused
        dt = DTYPES[dtype]
        total = int(sum(prompts) + len(prompts) * members * (tail_max + 2))
        self.store_k = randn_rounded((total, H, D), dt, _torch_gen(seed, "cuda"), "cuda")
        self.store_v = randn_rounded((total, H, D), dt, _torch_gen(seed + 1, "cuda"), "cuda")
        nb = 2 * (total // bs + len(prompts) * members + 8)
        self.alloc = B.BlockAllocator(nb, bs, rng.permutation(nb).astype(np.int32))
        self.kc = torch.full((nb, H, bs, D), float("nan"), dtype=dt, device="cuda")
        self.vc = torch.full_like(self.kc, float("nan"))
        self.content = LogicalSequences()
        self.rec = B.new_error_record()
        self.B, self.next_row, self.ids = B, 0, []
        for f, Lp in enumerate(prompts):
            root = 1000 * f
            self.alloc.add(root, Lp)
            self._write(range(self.next_row, self.next_row + Lp), self.alloc.slots(root, 0, Lp))
            self.content.add(root, range(self.next_row, self.next_row + Lp))
            self.next_row += Lp
            fam = [root]
            for s in range(1, members):
                self.alloc.fork(root, root + s)
                self.content.fork(root, root + s)
                fam.append(root + s)
            self.ids += fam
        for i in self.ids:                                  # private tails
            for _ in range(int(rng.integers(0, tail_max + 1))):
                self._append_one(i)
        self.new_rows = None
        if fused:                                           # the token this step appends
            slots, pairs = self.alloc.batch_append(self.ids)
            if len(pairs):
                B.block_copy([self.kc], [self.vc], torch.from_numpy(pairs).cuda(),
                             error_record=self.rec)
            self.new_rows = np.arange(self.next_row, self.next_row + len(self.ids))
            for i, r in zip(self.ids, self.new_rows):
                self.content.append(i, int(r))
            self.next_row += len(self.ids)
        self.q = randn_rounded((len(self.ids), H, D), dt, _torch_gen(seed + 2, "cuda"), "cuda")
        self.scale = D ** -0.5

    def _write(self, rows, slots):
        r = torch.as_tensor(list(rows), dtype=torch.long, device="cuda")
        self.B.kv_cache_append(self.store_k[r], self.store_v[r],
                               torch.as_tensor(np.asarray(slots), dtype=torch.int64).cuda(),
                               self.kc, self.vc, error_record=self.rec)

    def _append_one(self, i):
        slot, cow = self.alloc.append(i)
        if cow is not None:
            self.B.block_copy([self.kc], [self.vc],
                              torch.tensor([cow], dtype=torch.int64, device="cuda"),
                              error_record=self.rec)
        self._write([self.next_row], [slot])
        self.content.append(i, self.next_row)
        self.next_row += 1

    def tables(self, max_blocks=None):
        mb = max_blocks or max(len(self.alloc.block_table(i)) for i in self.ids)
        return self.alloc.batch_block_tables(self.ids, mb)

    def decode(self, tables, lens, pt, items=None, recs=None, out_dtype=torch.float32,
               tails=None):
        B = self.B
        kw = dict(partition_tokens=pt, error_record=self.rec, out_dtype=out_dtype)
        if tails is not None:
            kw["tail_start"] = torch.from_numpy(tails).cuda()
        if items is not None:
            kw["work_items"] = torch.from_numpy(items).cuda()
        if recs is not None:
            kw["shared_records"] = torch.from_numpy(recs).cuda()
        bt, sl = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
        if self.fused:
            nr = torch.from_numpy(self.new_rows).cuda()
            out = B.paged_attn_decode_append(self.q, self.store_k[nr], self.store_v[nr], self.kc,
                                             self.vc, bt, sl, self.scale, **kw)
        else:
            out = B.paged_attn_decode(self.q, self.kc, self.vc, bt, sl, self.scale, **kw)
        torch.cuda.synchronize()
        return out

    def check(self, out, lens, what, seqs=None):
        st_k, st_v = [(0, self.store_k)], [(0, self.store_v)]
        for n in (range(len(self.ids)) if seqs is None else seqs):
            i = self.ids[n]
            assert lens[n] == self.content.length(i)
            ref = _oracle_logical(self.q[n], self.content, i, st_k, st_v, self.scale)
            assert_matches_oracle(out[n], ref, f"{what} seq {i}")


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("dtype,D,bs", [("bf16", 128, 16), ("f16", 128, 32), ("bf16", 64, 16),
                                        ("f16", 256, 16), ("bf16", 128, 8), ("f16", 64, 8)])
def test_shared_partitions_match_oracle(B, fused, dtype, D, bs):
    fam = Families(B, 7 + D + bs, prompts=[700, 300, 1300], members=6, tail_max=150, H=4, D=D,
                   bs=bs, dtype=dtype, fused=fused)
    tables, lens = fam.tables()
    pt = 128
    items, recs = B.share_plan(tables, lens, pt, bs, fused_append=fused)
    assert len(recs) >= (700 // pt) + (300 // pt) + (1300 // pt) - 3
    out = fam.decode(tables, lens, pt, items, recs)
    assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
    fam.check(out, lens, f"shared {dtype} D{D} bs{bs} fused={fused}")


def test_shared_and_plain_paths_agree(B):
    fam = Families(B, 21, prompts=[1100, 900], members=8, tail_max=300, H=8, D=128, bs=16,
                   dtype="bf16", fused=True)
    tables, lens = fam.tables()
    items, recs = B.share_plan(tables, lens, 256, 16)
    # the cache is written by the fused append on the first call; both calls write
    # the same rows, and read the same values
    plain = fam.decode(tables, lens, 256, B.partition_work_items(lens, 256, tables.shape[1], 16))
    shared = fam.decode(tables, lens, 256, items, recs)
    again = fam.decode(tables, lens, 256, items, recs)
    assert torch.equal(shared, again)                   # repeatable bit for bit
    assert (shared - plain).abs().max().item() < 2e-3
    fam.check(shared, lens, "shared vs plain")


def test_more_than_eight_members_split_into_records(B):
    fam = Families(B, 33, prompts=[600], members=21, tail_max=40, H=2, D=128, bs=16,
                   dtype="bf16", fused=True)
    tables, lens = fam.tables()
    items, recs = B.share_plan(tables, lens, 64, 16)
    assert sorted(set(int(r[1]) for r in recs)) == [5, 8]
    out = fam.decode(tables, lens, 64, items, recs)
    assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
    fam.check(out, lens, "21 members")


def test_single_partition_members_get_their_output_directly(B):
    """With one partition per sequence (capacity = partition), a shared record
    holds the whole sequence and writes the output row itself."""
    fam = Families(B, 41, prompts=[64, 64], members=3, tail_max=0, H=2, D=64, bs=16,
                   dtype="f16", fused=False)
    tables, lens = fam.tables(max_blocks=4)
    items, recs = B.share_plan(tables, lens, 64, 16, fused_append=False)
    assert len(items) == 0 and len(recs) == 2
    assert B.paged_attn_workspace_size(len(lens), 2, 64, 16, 4, 64) == 0
    out = fam.decode(tables, lens, 64, items, recs, out_dtype=torch.float16)
    assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
    fam.check(out, lens, "direct output")


def test_bad_shared_record_is_recorded_and_skipped(B):
    fam = Families(B, 51, prompts=[400], members=4, tail_max=20, H=2, D=128, bs=16,
                   dtype="bf16", fused=False)
    tables, lens = fam.tables()
    items, recs = B.share_plan(tables, lens, 128, 16, fused_append=False)
    bad = recs.copy()
    bad[0, 3] = 99                                      # a member that does not exist
    out = torch.zeros(len(lens), 2, 128, device="cuda")
    B.paged_attn_decode(fam.q, fam.kc, fam.vc, torch.from_numpy(tables).cuda(),
                        torch.from_numpy(lens).cuda(), fam.scale, out=out, partition_tokens=128,
                        work_items=torch.from_numpy(items).cuda(),
                        shared_records=torch.from_numpy(bad).cuda(), error_record=fam.rec)
    assert B.pa_error_read(fam.rec) == [6, 1, 0, 99]
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):     # records need a work list
        B.paged_attn_decode(fam.q, fam.kc, fam.vc, torch.from_numpy(tables).cuda(),
                            torch.from_numpy(lens).cuda(), fam.scale, partition_tokens=128,
                            shared_records=torch.from_numpy(recs).cuda())


def test_long_shared_pass_eager_and_in_a_cuda_graph(B):
    """Almost all the work in shared partitions and a short per-sequence pass: the
    merge must still follow the shared pass, launched eagerly or replayed from a
    CUDA graph."""
    fam = Families(B, 61, prompts=[2000, 1600], members=12, tail_max=3, H=8, D=128, bs=16,
                   dtype="bf16", fused=True)
    tables, lens = fam.tables()
    pt = 128
    items, recs = B.share_plan(tables, lens, pt, 16)
    assert len(recs) >= 2 * 12 and len(items) <= len(lens) * 2
    eager = fam.decode(tables, lens, pt, items, recs)
    fam.check(eager, lens, "long shared pass, eager")
    bt, sl = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    it, rc = torch.from_numpy(items).cuda(), torch.from_numpy(recs).cuda()
    nr = torch.from_numpy(fam.new_rows).cuda()
    nk, nv = fam.store_k[nr], fam.store_v[nr]
    ws = torch.empty(B.paged_attn_workspace_size(len(lens), 8, 128, 16, tables.shape[1], pt),
                     dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(eager)
    step = lambda: B.paged_attn_decode_append(fam.q, nk, nv, fam.kc, fam.vc, bt, sl, fam.scale,
                                              out=out, partition_tokens=pt, workspace=ws,
                                              work_items=it, shared_records=rc,
                                              error_record=fam.rec)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        out.zero_()
        ws.fill_(0xff)                                   # stale partials would show as NaN
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]


@pytest.mark.parametrize("seed", range(16))
def test_shared_random_configuration(B, seed):
    _random_shared_case(B, seed)


@pytest.mark.parametrize("seed", range(6))
def test_shared_random_configuration_8_token_blocks(B, seed):
    """8-token blocks: each shared chunk is loaded as two 8-row boxes."""
    _random_shared_case(B, 500 + seed, block_size=8)


def _random_shared_case(B, seed, block_size=None, prefixes=False):
    rng = np.random.default_rng(7000 + seed)
    D = int(rng.choice([64, 128, 256]))
    bs = int(rng.choice([16, 32]))
    if block_size is not None:
        bs = block_size
    H = int(rng.choice([1, 2, 3, 4, 8]))
    dtype = str(rng.choice(["f16", "bf16"]))
    fused = bool(rng.integers(0, 2))
    pt = int(rng.choice([16, 64, 128, 256]))
    families = int(rng.integers(1, 4))
    prompts = [int(x) for x in rng.integers(1, 900, size=families)]
    fam = Families(B, 8000 + seed, prompts=prompts, members=int(rng.integers(1, 20)),
                   tail_max=int(rng.integers(0, 200)), H=H, D=D, bs=bs, dtype=dtype, fused=fused)
    tables, lens = fam.tables()
    order = None if seed % 3 else rng.permutation(len(lens))
    tails = None
    if prefixes:
        items, recs, tails = B.share_plan_prefix(tables, lens, pt, bs, fused_append=fused,
                                                 order=order)
    else:
        items, recs = B.share_plan(tables, lens, pt, bs, fused_append=fused, order=order)
    out_dtype = [torch.float32, torch.float16, torch.bfloat16][int(rng.integers(0, 3))]
    out = fam.decode(tables, lens, pt, items, recs, out_dtype=out_dtype, tails=tails)
    assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
    fam.check(out, lens, f"seed {seed}: D{D} bs{bs} H{H} {dtype} pt{pt} fused={fused} "
                         f"{len(recs)} records")


def test_single_member_records_match_oracle(B):
    """A record may hold one sequence (the plan never makes one, a caller may): it
    computes that sequence's partition like the per-sequence pass."""
    fam = Families(B, 91, prompts=[900, 500], members=2, tail_max=100, H=4, D=128, bs=16,
                   dtype="f16", fused=True)
    tables, lens = fam.tables()
    pt = 128
    P = -(-tables.shape[1] * 16 // pt)
    items = B.partition_work_items(lens, pt, tables.shape[1], 16)
    keep, recs = [], []
    for it in items:
        i, p = divmod(int(it), P)
        if (p + 1) * pt <= int(lens[i]) - 1 and p % 2 == 0:     # every other full partition
            r = np.full(B.PA_SHARE_RECORD_WORDS, -1, dtype=np.int32)
            r[:3] = (p, 1, i)
            recs.append(r)
        else:
            keep.append(it)
    assert len(recs) >= 4
    out = fam.decode(tables, lens, pt, np.array(keep, dtype=np.int32), np.stack(recs))
    assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
    fam.check(out, lens, "single-member records")


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("dtype,D,bs", [("bf16", 128, 16), ("f16", 64, 32), ("bf16", 256, 8),
                                        ("f16", 128, 16)])
def test_prefix_records_match_oracle(B, fused, dtype, D, bs):
    """Prompts that end inside a partition: the chunks of that partition which the
    whole family still shares are read once by a prefix record, each member's rest
    by its own item from tail_start on, and the merge adds the two."""
    fam = Families(B, 31 + D + bs, prompts=[700, 300, 1000, 1200], members=6, tail_max=150,
                   H=4, D=D, bs=bs, dtype=dtype, fused=fused)
    tables, lens = fam.tables()
    pt = 128
    items, recs, tails = B.share_plan_prefix(tables, lens, pt, bs, fused_append=fused)
    assert (recs[:, 1] >> 8).max() >= 2 and (tails >= 0).sum() >= 12
    out = fam.decode(tables, lens, pt, items, recs, tails=tails)
    assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
    fam.check(out, lens, f"prefix {dtype} D{D} bs{bs} fused={fused}")


def test_prefix_records_single_partition_sequences(B):
    """Sequences of one partition: the prefix record leaves its partial in the
    workspace (not in the output), and the merge runs for them too."""
    fam = Families(B, 77, prompts=[200, 90], members=5, tail_max=40, H=8, D=128, bs=16,
                   dtype="bf16", fused=True)
    tables, lens = fam.tables()
    pt = 256
    assert lens.max() <= pt
    items, recs, tails = B.share_plan_prefix(tables, lens, pt, 16, fused_append=True)
    assert len(recs) and (recs[:, 1] >> 8).min() >= 1
    for out_dtype in (torch.float32, torch.bfloat16):
        out = fam.decode(tables, lens, pt, items, recs, out_dtype=out_dtype, tails=tails)
        assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
        fam.check(out, lens, f"one partition, out {out_dtype}")


def test_prefix_and_whole_plans_agree(B):
    fam = Families(B, 23, prompts=[1100, 900, 650], members=8, tail_max=300, H=8, D=128,
                   bs=16, dtype="bf16", fused=False)
    tables, lens = fam.tables()
    items, recs = B.share_plan(tables, lens, 256, 16, fused_append=False)
    items2, recs2, tails = B.share_plan_prefix(tables, lens, 256, 16, fused_append=False)
    assert len(recs2) > len(recs)
    a = fam.decode(tables, lens, 256, items, recs)
    b = fam.decode(tables, lens, 256, items2, recs2, tails=tails)
    assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
    torch.testing.assert_close(a, b, rtol=2e-3, atol=2e-3)
    fam.check(b, lens, "prefix plan")


@pytest.mark.parametrize("seed", range(16))
def test_prefix_random_configuration(B, seed):
    _random_shared_case(B, 300 + seed, prefixes=True)


@pytest.mark.parametrize("seed", range(4))
def test_prefix_random_configuration_8_token_blocks(B, seed):
    _random_shared_case(B, 900 + seed, block_size=8, prefixes=True)


def test_prefix_plan_replays_from_a_cuda_graph(B):
    """The decode with prefix records captured once: new plans (other records,
    other tails) written into the same device buffers give the oracle's output."""
    fam = Families(B, 55, prompts=[800, 450], members=7, tail_max=120, H=4, D=128, bs=16,
                   dtype="f16", fused=False)
    tables, lens = fam.tables()
    pt, N, RW = 128, len(lens), B.PA_SHARE_RECORD_WORDS
    P = -(-tables.shape[1] * 16 // pt)
    it_d = torch.zeros(N * P, dtype=torch.int32, device="cuda")
    rc_d = torch.zeros((N * P, RW), dtype=torch.int32, device="cuda")
    ts_d = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    bt, sl = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    out = torch.empty((N, 4, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.paged_attn_workspace_size(N, 4, 128, 16, tables.shape[1], pt, tails=True),
                     dtype=torch.uint8, device="cuda")

    def load(items, recs, tails):
        it_d.zero_()
        it_d[:len(items)] = torch.from_numpy(items)
        rc_d[:len(recs)] = torch.from_numpy(recs)
        ts_d.copy_(torch.from_numpy(tails))
        return it_d[:len(items)], rc_d[:len(recs)]

    plans = [B.share_plan_prefix(tables, lens, pt, 16),
             B.share_plan_prefix(tables, lens, pt, 16, order=list(range(N))[::-1])]
    its, rcs = load(*plans[0])
    step = lambda: B.paged_attn_decode(fam.q, fam.kc, fam.vc, bt, sl, fam.scale, out=out,
                                       partition_tokens=pt, workspace=ws, work_items=its,
                                       shared_records=rcs, tail_start=ts_d,
                                       error_record=fam.rec)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for items, recs, tails in plans:
        assert len(items) == len(its) and len(recs) == len(rcs)
        load(items, recs, tails)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
        fam.check(out, lens, "graph replay")


def test_prefix_record_and_tail_start_that_disagree_report_an_error(B):
    """A tail_start that names another split than its prefix record, or that is not
    a multiple of 16 tokens: an error in the record, no hang, no stray writes."""
    fam = Families(B, 5, prompts=[700], members=4, tail_max=60, H=4, D=128, bs=16,
                   dtype="bf16", fused=False)
    tables, lens = fam.tables()
    items, recs, tails = B.share_plan_prefix(tables, lens, 128, 16, fused_append=False)
    s = int(np.flatnonzero(tails >= 0)[0])
    for bad in (int(tails[s]) + 16, int(tails[s]) + 3):
        if bad >= int(lens[s]):
            continue
        t = tails.copy()
        t[s] = bad
        B.pa_error_clear(fam.rec)
        fam.decode(tables, lens, 128, items, recs, tails=t)
        assert B.pa_error_read(fam.rec)[0] != 0
    B.pa_error_clear(fam.rec)
    out = fam.decode(tables, lens, 128, items, recs, tails=tails)
    assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
    fam.check(out, lens, "after the bad calls")


def test_device_counts_let_one_graph_run_plans_of_any_length(B):
    """counts (device int32 [2]) with capacity-sized lists: one captured decode
    replays plans with different numbers of work items and records (prefix plan,
    whole-partition plan, plain work list), each matching the oracle."""
    fam = Families(B, 57, prompts=[800, 450, 1200], members=6, tail_max=120, H=4, D=128,
                   bs=16, dtype="bf16", fused=False)
    tables, lens = fam.tables()
    pt, N, RW = 128, len(lens), B.PA_SHARE_RECORD_WORDS
    P = -(-tables.shape[1] * 16 // pt)
    it_d = torch.full((N * P,), -7, dtype=torch.int32, device="cuda")    # junk past the count
    rc_d = torch.full((N * P // 2, RW), -7, dtype=torch.int32, device="cuda")
    ts_d = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(2, dtype=torch.int32, device="cuda")
    bt, sl = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    out = torch.empty((N, 4, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.paged_attn_workspace_size(N, 4, 128, 16, tables.shape[1], pt, tails=True),
                     dtype=torch.uint8, device="cuda")
    plain = B.partition_work_items(lens, pt, tables.shape[1], 16)
    plans = [B.share_plan_prefix(tables, lens, pt, 16, fused_append=False),
             (*B.share_plan(tables, lens, pt, 16, fused_append=False), np.full(N, -1, np.int32)),
             (plain, np.empty((0, RW), np.int32), np.full(N, -1, np.int32))]
    assert len({len(p[0]) for p in plans}) == 2 and len({len(p[1]) for p in plans}) == 3

    def load(items, recs, tails):
        it_d[:len(items)] = torch.from_numpy(items)
        if len(recs):
            rc_d[:len(recs)] = torch.from_numpy(recs)
        ts_d.copy_(torch.from_numpy(tails))
        cnt.copy_(torch.tensor([len(items), len(recs)], dtype=torch.int32))

    step = lambda: B.paged_attn_decode(fam.q, fam.kc, fam.vc, bt, sl, fam.scale, out=out,
                                       partition_tokens=pt, workspace=ws, work_items=it_d,
                                       shared_records=rc_d, tail_start=ts_d, counts=cnt,
                                       error_record=fam.rec)
    load(*plans[0])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for k, plan in enumerate(plans + plans[::-1]):
        load(*plan)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert B.pa_error_read(fam.rec) == [0, 0, 0, 0], k
        fam.check(out, lens, f"graph replay, plan {k}")


@pytest.mark.parametrize("which", [0, 1])
def test_device_count_above_capacity_is_recorded(B, which):
    fam = Families(B, 58, prompts=[600], members=3, tail_max=50, H=4, D=128, bs=16,
                   dtype="f16", fused=False)
    tables, lens = fam.tables()
    items, recs = B.share_plan(tables, lens, 128, 16, fused_append=False)
    assert len(recs) >= 1
    n = [len(items), len(recs)]
    n[which] += 1
    B.pa_error_clear(fam.rec)
    B.paged_attn_decode(fam.q, fam.kc, fam.vc, torch.from_numpy(tables).cuda(),
                        torch.from_numpy(lens).cuda(), fam.scale, partition_tokens=128,
                        work_items=torch.from_numpy(items).cuda(),
                        shared_records=torch.from_numpy(recs).cuda(),
                        counts=torch.tensor(n, dtype=torch.int32, device="cuda"),
                        error_record=fam.rec)
    torch.cuda.synchronize()
    code, _, index, value = B.pa_error_read(fam.rec)
    assert B.STATUS[code] == "PA_ERR_BAD_SEQ_LEN" and index == -1 - which
    assert value == n[which]
    B.pa_error_clear(fam.rec)


@pytest.mark.parametrize("seed", range(6))
def test_device_counts_random_capacities(B, seed):
    """Work lists and records inside larger buffers, junk past their counts: the
    decode reads exactly the counted entries (prefix plans, fused or not)."""
    rng = np.random.default_rng(4100 + seed)
    fused = bool(seed % 2)
    fam = Families(B, 4200 + seed, prompts=[int(x) for x in rng.integers(100, 1400, 3)],
                   members=int(rng.integers(2, 10)), tail_max=int(rng.integers(0, 200)), H=4,
                   D=int(rng.choice([64, 128])), bs=16, dtype="bf16", fused=fused)
    tables, lens = fam.tables()
    pt = int(rng.choice([64, 128, 256]))
    items, recs, tails = B.share_plan_prefix(tables, lens, pt, 16, fused_append=fused)
    RW = B.PA_SHARE_RECORD_WORDS
    cap_i, cap_r = len(items) + int(rng.integers(0, 300)), len(recs) + int(rng.integers(1, 60))
    it_d = torch.full((cap_i,), -7, dtype=torch.int32, device="cuda")
    rc_d = torch.full((cap_r, RW), -7, dtype=torch.int32, device="cuda")
    it_d[:len(items)] = torch.from_numpy(items)
    if len(recs):
        rc_d[:len(recs)] = torch.from_numpy(recs)
    cnt = torch.tensor([len(items), len(recs)], dtype=torch.int32, device="cuda")
    bt, sl = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    kw = dict(partition_tokens=pt, error_record=fam.rec, work_items=it_d, shared_records=rc_d,
              tail_start=torch.from_numpy(tails).cuda(), counts=cnt)
    if fused:
        nr = torch.from_numpy(fam.new_rows).cuda()
        out = B.paged_attn_decode_append(fam.q, fam.store_k[nr], fam.store_v[nr], fam.kc,
                                         fam.vc, bt, sl, fam.scale, **kw)
    else:
        out = B.paged_attn_decode(fam.q, fam.kc, fam.vc, bt, sl, fam.scale, **kw)
    torch.cuda.synchronize()
    assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
    fam.check(out, lens, f"seed {seed}: counts inside capacities {cap_i} / {cap_r}")


def test_prefix_records_with_the_passes_called_apart(B):
    """phases=1 then phases=2 (partition passes, then the merge, as two calls on the
    same workspace) gives the single call's bits: tail rows persist between them."""
    fam = Families(B, 61, prompts=[700, 1000], members=5, tail_max=90, H=4, D=128, bs=16,
                   dtype="f16", fused=False)
    tables, lens = fam.tables()
    pt = 128
    items, recs, tails = B.share_plan_prefix(tables, lens, pt, 16, fused_append=False)
    assert (recs[:, 1] >> 8).max() > 0
    N, MB = tables.shape
    ws = torch.empty(B.paged_attn_workspace_size(N, 4, 128, 16, MB, pt, tails=True),
                     dtype=torch.uint8, device="cuda")
    args = (fam.q, fam.kc, fam.vc, torch.from_numpy(tables).cuda(),
            torch.from_numpy(lens).cuda(), fam.scale)
    kw = dict(partition_tokens=pt, workspace=ws, work_items=torch.from_numpy(items).cuda(),
              shared_records=torch.from_numpy(recs).cuda(),
              tail_start=torch.from_numpy(tails).cuda(), error_record=fam.rec)
    whole = B.paged_attn_decode(*args, **kw).clone()
    out = torch.full_like(whole, float("nan"))
    B.paged_attn_decode(*args, out=out, phases=1, **kw)
    B.paged_attn_decode(*args, out=out, phases=2, **kw)
    torch.cuda.synchronize()
    assert B.pa_error_read(fam.rec) == [0, 0, 0, 0]
    assert torch.equal(out, whole)
    fam.check(out, lens, "passes called apart")
