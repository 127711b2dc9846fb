"""Host-side decode schedule (pa_decode_partition_tokens, pa_decode_work_items):
pure host code, so it runs here without a GPU."""

import ctypes

import numpy as np
import pytest

from paged_kv_cache_317_gb300 import binding as B


def rule(lens, num_heads, heads_per_cta, num_sms):
    """The balance rule as the header states it."""
    G = heads_per_cta or (2 if num_heads % 2 == 0 else 1)
    work = int(np.sum(lens)) * (num_heads // G)
    longest = int(np.max(lens)) if len(lens) else 0
    chosen = 32
    for pt, c in ((512, 3.5), (256, 3.5), (128, 2.0), (64, 1.0)):
        if min(pt, longest) * num_sms * c <= work:
            chosen = pt
            break
    while chosen < 512 and -(-longest // chosen) > 32:   # at most 32 pieces
        chosen *= 2
    return chosen


def test_partition_choice_follows_the_balance_rule():
    rng = np.random.default_rng(0)
    for trial in range(400):
        n = int(rng.integers(1, 300))
        median = float(np.exp(rng.uniform(np.log(8), np.log(20000))))
        lens = np.clip(np.round(np.exp(np.log(median) + 0.75 * rng.standard_normal(n))), 0, 1 << 17)
        H = int(rng.choice([8, 12, 32, 40, 64, 7]))
        G = int(rng.choice([0, 1]))
        sms = int(rng.choice([1, 76, 148, 152]))
        got = B.decode_partition_tokens(lens, H, G, sms)
        assert got == rule(lens, H, G, sms), (trial, n, median, H, G, sms)


def test_partition_choice_at_the_ends():
    big = np.full(256, 350)
    assert B.decode_partition_tokens(big, 40, 0, 152) == 512      # plenty of work per SM
    assert B.decode_partition_tokens([350], 40, 0, 152) == 32     # one short sequence
    assert B.decode_partition_tokens([350] * 2, 40, 0, 152) == 64
    assert B.decode_partition_tokens([1024] * 4, 40, 0, 152) == 128
    assert B.decode_partition_tokens([], 40, 0, 152) == 512       # nothing to balance
    # a long batch keeps 512 even with one huge sequence, since the heaviest
    # block is a partition, not the sequence
    assert B.decode_partition_tokens([100000] + [300] * 255, 40, 0, 152) == 512
    # the boundary itself: work exactly 3.5 x SMs x heaviest keeps the partition
    # (7 x 512 tokens x 2 heads = 3.5 x 4 SMs x 512)
    assert B.decode_partition_tokens([512] * 7, 2, 1, 4) == 512
    assert B.decode_partition_tokens([512] * 6, 2, 1, 4) == 256
    # 128 needs only half the work per SM: 2 x 4 SMs x 128 = 1024 = 4 x 128 x 2 heads
    assert B.decode_partition_tokens([128] * 4, 2, 1, 4) == 128
    assert B.decode_partition_tokens([128] * 3, 2, 1, 4) == 64
    # 64 with c = 1: 64 x 4 SMs = 256 = 2 x 64 x 2 heads; below that, 32
    assert B.decode_partition_tokens([64] * 2, 2, 1, 4) == 64
    assert B.decode_partition_tokens([64, 63], 2, 1, 4) == 32
    # ... but the longest sequence takes at most 32 partitions
    assert B.decode_partition_tokens([1024], 8, 0, 152) == 32
    assert B.decode_partition_tokens([1025], 8, 0, 152) == 64
    assert B.decode_partition_tokens([4000], 4, 0, 152) == 128
    assert B.decode_partition_tokens([100000], 4, 0, 152) == 512


def test_partition_choice_rejects_bad_arguments():
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.decode_partition_tokens([5, -1], 40, 0, 152)
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.decode_partition_tokens([5], 40, 3, 152)                 # 3 does not divide 40
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.decode_partition_tokens([5], 32, 16, 152)                # above 8 heads per block
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.decode_partition_tokens([5], 0, 0, 152)
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.decode_partition_tokens([5], 8, 0, -1)


def _items_by_formula(lens, pt, MB, bs, order=None):
    lens = np.asarray(lens, np.int64)
    P = max(1, -(-MB * bs // pt))
    order = sorted(range(len(lens)), key=lambda i: (-lens[i], i)) if order is None else order
    return np.array([i * P + p for i in order for p in range(max(1, -(-int(lens[i]) // pt)))],
                    dtype=np.int32)


def test_work_items_match_their_definition():
    rng = np.random.default_rng(1)
    for trial in range(200):
        n = int(rng.integers(0, 60))
        bs = int(rng.choice([16, 32]))
        MB = int(rng.integers(1, 200))
        lens = rng.integers(0, MB * bs + 1, size=n)
        lens[rng.random(n) < 0.1] = 0
        pt = int(rng.choice([0, 16, 64, 128, 512, 2048]))
        order = None if trial % 3 else list(rng.permutation(n))
        got = B.partition_work_items(lens, pt, MB, bs, order=order)
        want = _items_by_formula(lens, pt or 512, MB, bs, order)
        assert got.dtype == np.int32
        assert np.array_equal(got, want), trial


def test_work_items_reject_bad_arguments():
    lib = B.load_library()
    lens = (ctypes.c_int32 * 3)(10, 40, 20)
    n = ctypes.c_int32(-1)
    buf = (ctypes.c_int32 * 8)()
    # a count query, then a buffer one short: the count comes back, nothing is written
    assert lib.pa_decode_work_items(lens, 3, 16, 4, 16, None, None, 0, ctypes.byref(n)) == 0
    assert n.value == 1 + 3 + 2
    buf[0] = 12345
    assert lib.pa_decode_work_items(lens, 3, 16, 4, 16, None, buf, 5, ctypes.byref(n)) == 1
    assert n.value == 6 and buf[0] == 12345
    assert lib.pa_decode_work_items(lens, 3, 16, 4, 16, None, buf, 8, ctypes.byref(n)) == 0
    assert list(buf[:6]) == [1 * 4 + 0, 1 * 4 + 1, 1 * 4 + 2, 2 * 4 + 0, 2 * 4 + 1, 0]
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.partition_work_items([10, 40, 20], 16, 4, 16, order=[0, 0, 2])   # not a permutation
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.partition_work_items([10, 65, 20], 16, 4, 16)                   # longer than 4 blocks
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.partition_work_items([10], 24, 4, 16)                          # not a multiple of 16
    with pytest.raises(ValueError):
        B.partition_work_items([10, 20], 16, 4, 16, order=[0])


def _plan_by_definition(tables, lens, pt, bs, fused, order=None):
    """Brute-force restatement of the share plan: records as a set of
    (partition, members), and the work list."""
    N, MB = tables.shape
    P = max(1, -(-MB * bs // pt))
    nparts = [max(1, -(-int(L) // pt)) for L in lens]
    share = [max(0, (int(L) - (1 if fused else 0)) // pt) for L in lens]
    covered, recs = set(), set()
    for p in range(max(share, default=0)):
        b0, b1 = p * pt // bs, ((p + 1) * pt - 1) // bs
        groups = {}
        for i in range(N):
            if share[i] > p:
                groups.setdefault(tuple(tables[i, b0:b1 + 1]), []).append(i)
        for grp in groups.values():
            for at in range(0, len(grp) - 1, B.PA_SHARE_MAX_MEMBERS):
                mem = tuple(grp[at:at + B.PA_SHARE_MAX_MEMBERS])
                recs.add((p, mem))
                covered.update((i, p) for i in mem)
    order = sorted(range(N), key=lambda i: (-int(lens[i]), i)) if order is None else order
    items = [i * P + p for i in order for p in range(nparts[i]) if (i, p) not in covered]
    return recs, np.array(items, dtype=np.int32)


def _records_as_set(recs):
    return {(int(r[0]), tuple(int(x) for x in r[2:2 + r[1]])) for r in recs}


def test_share_plan_matches_its_definition():
    rng = np.random.default_rng(5)
    for trial in range(150):
        bs = int(rng.choice([16, 32, 48]))        # 48: partitions cut across blocks
        pt = int(rng.choice([16, 32, 64, 128]))
        N = int(rng.integers(1, 40))
        MB = int(rng.integers(1, 24))
        # a few "prompts" whose block lists sequences copy (with private tails)
        prompts = rng.integers(0, 500, size=(4, MB)).astype(np.int32)
        tables = rng.integers(0, 500, size=(N, MB)).astype(np.int32)
        lens = rng.integers(0, MB * bs + 1, size=N)
        for i in range(N):
            if rng.random() < 0.7:
                k = int(rng.integers(0, MB + 1))
                tables[i, :k] = prompts[int(rng.integers(0, 4)), :k]
        fused = bool(rng.integers(0, 2))
        if fused:
            lens = np.maximum(lens, 1)
        order = None if trial % 4 else list(rng.permutation(N))
        items, recs = B.share_plan(tables, lens, pt, bs, fused_append=fused, order=order)
        want_recs, want_items = _plan_by_definition(tables, lens, pt, bs, fused, order)
        assert recs.shape[1] == B.PA_SHARE_RECORD_WORDS
        assert _records_as_set(recs) == want_recs, trial
        assert np.array_equal(items, want_items), trial
        for r in recs:
            assert 2 <= r[1] <= B.PA_SHARE_MAX_MEMBERS and (r[2 + r[1]:] == -1).all()


def test_share_plan_on_forked_sequences():
    """Sequences forked from one prompt by the allocator share their prompt's full
    partitions; each pair that holds tokens is computed exactly once."""
    bs, pt = 16, 64
    alloc = B.BlockAllocator(4000, bs)
    ids = []
    for k, prompt in enumerate((300, 70, 1000)):
        alloc.add(100 * k, prompt)
        for s in range(1, 21 if k == 2 else 5):          # 20 samples of the long prompt
            alloc.fork(100 * k, 100 * k + s)
            ids.append(100 * k + s)
        ids.append(100 * k)
    rng = np.random.default_rng(2)
    for _ in range(int(rng.integers(1, 40))):
        alloc.batch_append(ids)                            # one token each, copy-on-write
    for i in ids[::3]:                                     # ragged tails
        for _ in range(int(rng.integers(0, 90))):
            alloc.append(i)
    alloc.batch_append(ids)                                # the token this step appends
    MB = 80
    tables, lens = alloc.batch_block_tables(ids, MB)
    items, recs = B.share_plan(tables, lens, pt, bs, fused_append=True)
    P = -(-MB * bs // pt)
    pairs = [(int(x) // P, int(x) % P) for x in items]
    for r in recs:
        p, m = int(r[0]), int(r[1])
        mem = [int(x) for x in r[2:2 + m]]
        b0, b1 = p * pt // bs, ((p + 1) * pt - 1) // bs
        assert all((tables[i, b0:b1 + 1] == tables[mem[0], b0:b1 + 1]).all() for i in mem)
        assert all((p + 1) * pt <= lens[i] - 1 for i in mem)
        pairs += [(i, p) for i in mem]
    want = [(i, p) for i in range(len(ids)) for p in range(max(1, -(-int(lens[i]) // pt)))]
    assert sorted(pairs) == sorted(want)
    # the 21 holders of the long prompt share its 15 full partitions: 8 + 8 + 5 members each
    sizes = [int(r[1]) for r in recs]
    assert sizes.count(8) >= 30 and sizes.count(5) >= 15


def test_share_plan_rejects_bad_arguments():
    t = np.zeros((2, 4), np.int32)
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.share_plan(t, [10, 65], 16, 16)                  # longer than 4 blocks
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.share_plan(t, [10, 20], 24, 16)                  # partition not a multiple of 16
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.share_plan(t, [10, 20], 16, 16, order=[1, 1])
    with pytest.raises(ValueError):
        B.share_plan(t, [10], 16, 16)
    items, recs = B.share_plan(t, [0, 0], 16, 16)
    assert list(items) == [0, 4] and recs.shape == (0, B.PA_SHARE_RECORD_WORDS)


def test_share_plan_with_8_token_blocks_matches_its_definition():
    """8-token blocks: a 64-token partition spans 8 table entries; the plan still
    groups exactly the sequences whose slices are identical."""
    rng = np.random.default_rng(9)
    for trial in range(60):
        bs, pt = 8, int(rng.choice([16, 32, 64, 128]))
        N, MB = int(rng.integers(1, 40)), int(rng.integers(1, 48))
        prompts = rng.integers(0, 500, size=(4, MB)).astype(np.int32)
        tables = rng.integers(0, 500, size=(N, MB)).astype(np.int32)
        lens = rng.integers(0, MB * bs + 1, size=N)
        for i in range(N):
            if rng.random() < 0.7:
                k = int(rng.integers(0, MB + 1))
                tables[i, :k] = prompts[int(rng.integers(0, 4)), :k]
        fused = bool(rng.integers(0, 2))
        if fused:
            lens = np.maximum(lens, 1)
        items, recs = B.share_plan(tables, lens, pt, bs, fused_append=fused)
        want_recs, want_items = _plan_by_definition(tables, lens, pt, bs, fused)
        assert _records_as_set(recs) == want_recs, trial
        assert np.array_equal(items, want_items), trial


def _prefix_plan_by_definition(tables, lens, pt, bs, fused, order=None):
    """The prefix step restated: (prefix records as a set of (p, m, c, members),
    tail_start), on top of the whole-partition plan."""
    N, MB = tables.shape
    full, items = _plan_by_definition(tables, lens, pt, bs, fused, order)
    covered = {(i, p) for p, mem in full for i in mem}
    nparts = [max(1, -(-int(L) // pt)) for L in lens]
    tails = np.full(N, -1, dtype=np.int32)
    recs = set()
    max_chunks = pt // 16 - 1
    if max_chunks >= 1:
        for p in range(max(nparts, default=0)):
            start = p * pt
            cand = [i for i in range(N) if tails[i] < 0 and p < nparts[i]
                    and (i, p) not in covered and int(lens[i]) - 1 - start >= 16]
            groups = {}
            for i in sorted(cand, key=lambda i: (int(tables[i, start // bs]), i)):
                groups.setdefault(int(tables[i, start // bs]), []).append(i)
            for grp in groups.values():
                for at in range(0, len(grp) - 1, B.PA_SHARE_MAX_MEMBERS):
                    mem = grp[at:at + B.PA_SHARE_MAX_MEMBERS]
                    c = min([max_chunks] + [(int(lens[i]) - 1 - start) // 16 for i in mem])
                    same = 0
                    while same < c:
                        t0 = start + 16 * same
                        blocks = range(t0 // bs, (t0 + 15) // bs + 1)
                        if any(tables[i, b] != tables[mem[0], b] for i in mem for b in blocks):
                            break
                        same += 1
                    if same < 1:
                        continue
                    recs.add((p, len(mem), same, tuple(mem)))
                    for i in mem:
                        tails[i] = start + 16 * same
    return full, recs, items, tails


def _random_family_tables(rng, bs):
    pt = int(rng.choice([32, 64, 128, 256]))
    N, MB = int(rng.integers(2, 40)), int(rng.integers(2, 24))
    prompts = rng.integers(0, 500, size=(4, MB)).astype(np.int32)
    tables = rng.integers(0, 500, size=(N, MB)).astype(np.int32)
    lens = rng.integers(0, MB * bs + 1, size=N)
    for i in range(N):
        if rng.random() < 0.8:
            k = int(rng.integers(0, MB + 1))
            tables[i, :k] = prompts[int(rng.integers(0, 4)), :k]
    return pt, tables, lens


@pytest.mark.parametrize("bs", [8, 16, 32, 48])
def test_share_plan_prefix_matches_its_definition(bs):
    rng = np.random.default_rng(11 + bs)
    for trial in range(80):
        pt, tables, lens = _random_family_tables(rng, bs)
        fused = bool(rng.integers(0, 2))
        if fused:
            lens = np.maximum(lens, 1)
        order = None if trial % 3 else list(rng.permutation(len(lens)))
        items, recs, tails = B.share_plan_prefix(tables, lens, pt, bs, fused_append=fused,
                                                 order=order)
        full, want_pre, want_items, want_tails = _prefix_plan_by_definition(
            tables, lens, pt, bs, fused, order)
        whole = {(int(r[0]), tuple(int(x) for x in r[2:2 + (r[1] & 255)])) for r in recs
                 if r[1] >> 8 == 0}
        pre = {(int(r[0]), int(r[1]) & 255, int(r[1]) >> 8,
                tuple(int(x) for x in r[2:2 + (r[1] & 255)])) for r in recs if r[1] >> 8}
        assert whole == full, trial
        assert pre == want_pre, trial
        assert np.array_equal(items, want_items), trial
        assert np.array_equal(tails, want_tails), trial
        # without prefixes the plan is the whole-partition one, tails all -1
        items0, recs0 = B.share_plan(tables, lens, pt, bs, fused_append=fused, order=order)
        assert np.array_equal(items0, items) and _records_as_set(recs0) == full


def test_share_plan_prefix_covers_every_token_once_on_forked_sequences():
    """Beams forked from prompts, diverging at different steps: every token of every
    sequence is read exactly once, by a whole-partition record, a prefix record
    (over blocks every member's table names alike) or the sequence's own item."""
    bs, pt = 16, 128
    alloc = B.BlockAllocator(6000, bs)
    rng = np.random.default_rng(4)
    ids = []
    for k, prompt in enumerate((300, 700, 1000, 77)):
        alloc.add(100 * k, prompt)
        for s in range(1, 5):
            alloc.fork(100 * k, 100 * k + s)
            ids.append(100 * k + s)
        ids.append(100 * k)
    for step in range(30):                                 # fork / free churn per step
        if step % 3 == 0:
            for k in range(4):
                par, child = 100 * k, 1000 + 10 * step + k
                alloc.fork(par, child)
                ids.append(child)
        alloc.batch_append(ids)
    MB = 90
    tables, lens = alloc.batch_block_tables(ids, MB)
    items, recs, tails = B.share_plan_prefix(tables, lens, pt, bs, fused_append=True)
    assert (tails >= 0).sum() > 0 and any(r[1] >> 8 for r in recs)
    P = -(-MB * bs // pt)
    seen = [np.zeros(int(L), dtype=np.int32) for L in lens]
    for x in items:
        i, p = int(x) // P, int(x) % P
        a = int(tails[i]) if tails[i] >= 0 and tails[i] // pt == p else p * pt
        seen[i][a:min(int(lens[i]), (p + 1) * pt)] += 1
    for r in recs:
        p, m, c = int(r[0]), int(r[1]) & 255, int(r[1]) >> 8
        mem = [int(x) for x in r[2:2 + m]]
        end = (p + 1) * pt if c == 0 else p * pt + 16 * c
        blocks = slice(p * pt // bs, (end - 1) // bs + 1)
        assert all((tables[i, blocks] == tables[mem[0], blocks]).all() for i in mem)
        for i in mem:
            assert end <= int(lens[i]) - 1                 # the appended token stays private
            if c:
                assert tails[i] == end
            seen[i][p * pt:end] += 1
    assert all((s == 1).all() for s in seen)


def test_plan_and_tables_fill_caller_buffers_in_place():
    """out= buffers (a pinned staging buffer in a serving loop) get the same plan
    and tables as fresh arrays; the results are views of them."""
    bs, pt = 16, 128
    alloc = B.BlockAllocator(800, bs)
    ids = []
    for k, n in enumerate((300, 520, 90)):
        alloc.add(10 * k, n)
        ids.append(10 * k)
        for s in range(1, 4):
            alloc.fork(10 * k, 10 * k + s)
            ids.append(10 * k + s)
    for _ in range(20):
        alloc.batch_append(ids)
    MB = 48
    want_t, want_l = alloc.batch_block_tables(ids, MB)
    buf = np.full(len(ids) * (MB + 1) + 8, 7, dtype=np.int32)
    bt, sl = buf[:len(ids) * MB].reshape(len(ids), MB), buf[len(ids) * MB:len(ids) * (MB + 1)]
    t, l = alloc.batch_block_tables(ids, MB, out=(bt, sl))
    assert np.shares_memory(t, buf) and np.array_equal(t, want_t) and np.array_equal(l, want_l)
    assert (buf[len(ids) * (MB + 1):] == 7).all()
    with pytest.raises(ValueError):
        alloc.batch_block_tables(ids, MB, out=(bt[:, :-1], sl))
    with pytest.raises(ValueError):
        alloc.batch_block_tables(ids, MB, out=(bt.astype(np.int64), sl))
    P = -(-MB * bs // pt)
    it = np.empty(len(ids) * P, np.int32)
    rc = np.empty((len(ids) * P // 2, B.PA_SHARE_RECORD_WORDS), np.int32)
    ts = np.empty(len(ids), np.int32)
    for fn, out, n_out in ((B.share_plan_prefix, (it, rc, ts), 3), (B.share_plan, (it, rc), 2)):
        want = fn(want_t, want_l, pt, bs)
        got = fn(t, l, pt, bs, out=out)
        assert len(got) == n_out
        for g, w, o in zip(got, want, out):
            assert np.shares_memory(g, o) and np.array_equal(g, w)
    with pytest.raises(ValueError):
        B.share_plan_prefix(t, l, pt, bs, out=(it, rc, ts[:-1]))
    with pytest.raises(ValueError):
        B.share_plan(t, l, pt, bs, out=(it, rc[:, :-1]))
    with pytest.raises(B.PagedKVError):
        B.share_plan(t, l, pt, bs, out=(it[:3], rc))        # too little room


def test_share_plan_with_many_distinct_slices_behind_one_first_block():
    """Many sequences that share only a partition's first block (a short common
    prompt) and differ after it: no whole records, and the plan takes one sort per
    partition, not one pass per distinct slice."""
    import time
    N, MB, bs, pt = 30000, 64, 16, 512
    rng = np.random.default_rng(8)
    tables = rng.permutation(N * MB).astype(np.int32).reshape(N, MB) + 10
    tables[:, 0] = 3                                   # every table's first block alike
    lens = np.full(N, MB * bs)
    t0 = time.perf_counter()
    items, recs = B.share_plan(tables, lens, pt, bs, fused_append=True)
    took = time.perf_counter() - t0
    assert len(recs) == 0 and len(items) == N * (MB * bs // pt)
    assert took < 0.5, took                        # one pass per slice took seconds
    items, recs, tails = B.share_plan_prefix(tables, lens, pt, bs, fused_append=True)
    assert (recs[:, 1] >> 8 == 1).all() and len(recs) == N // 8 and (tails == 16).all()
