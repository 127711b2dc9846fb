"""CPU tests of the C ABI: the library loads, exports every function the header
declares, rejects malformed arguments on the host, and its host allocator
matches the oracle's allocator model operation for operation."""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle.allocator_model import AllocatorError, BlockAllocatorModel

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")


def declared_functions():
    names = []
    for fn in os.listdir(HEADER_DIR):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, re.M):
            if m.group(1) not in ("defined",):
                names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for required in ("paged_attn_decode", "kv_cache_append", "block_copy",
                     "paged_attn_workspace_size", "pa_alloc_create", "pa_seq_append"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    from paged_kv_cache_317_gb300.binding import STATUS
    assert lib.pa_version() == 3
    import re
    from paged_kv_cache_317_gb300 import binding
    hdr = open(os.path.join(HEADER_DIR, "pagedkv.h")).read()
    assert int(re.search(r"#define PAGEDKV_VERSION (\d+)", hdr).group(1)) == binding.ABI_VERSION == 3
    for code in STATUS:
        assert lib.pa_status_string(code)
    assert lib.pa_status_string(999) == b"unknown status"


def test_workspace_size_arithmetic(lib):
    # 256 seqs, 40 heads, D 128, capacity 129 blocks * 16 = 2064 tokens -> 5 partitions of 512
    rows = 256 * 40 * 5
    assert lib.paged_attn_workspace_size(256, 40, 128, 16, 129, 0) == rows * 128 * 4 + rows * 8
    # the whole capacity fits one partition: no workspace
    assert lib.paged_attn_workspace_size(4, 8, 64, 16, 32, 512) == 0
    assert lib.paged_attn_workspace_size(4, 8, 64, 16, 33, 512) == 4 * 8 * 2 * (64 * 4 + 8)


def test_decode_rejects_bad_arguments_on_the_host(lib):
    from paged_kv_cache_317_gb300.binding import STATUS_CODE
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its checks first
    INV, UNS = STATUS_CODE["PA_ERR_INVALID_ARG"], STATUS_CODE["PA_ERR_UNSUPPORTED"]

    def call(**kw):
        a = dict(q=p, k=p, v=p, bt=p, sl=p, N=4, H=8, D=64, bs=16, MB=4, B=64, scale=0.125,
                 dt=0, out=p, odt=2, pt=0, ws=None, wsb=0)
        a.update(kw)
        return lib.paged_attn_decode(a["q"], a["k"], a["v"], a["bt"], a["sl"], a["N"], a["H"],
                                     a["D"], a["bs"], a["MB"], a["B"], a["scale"], a["dt"],
                                     a["out"], a["odt"], a["pt"], a["ws"], a["wsb"], None, None)

    assert call(D=96) == UNS
    assert call(bs=24) == UNS                                # neither 8 nor a multiple of 16
    assert call(bs=4) == UNS
    assert call(dt=2) == UNS
    assert call(odt=7) == UNS
    assert call(q=None) == INV
    assert call(q=ctypes.c_void_p((1 << 20) + 8)) == INV      # not 16-byte aligned
    assert call(pt=100) == INV                                # not a multiple of 16
    assert call(MB=64) == INV                                 # needs a workspace, none given
    assert call(H=0) == INV
    assert call(scale=float("nan")) == INV
    assert call(N=65536) == INV                               # more sequences than a call takes
    assert call(N=0) == 0                                     # nothing to do


def test_append_and_copy_reject_bad_arguments(lib):
    p = ctypes.c_void_p(1 << 20)
    assert lib.kv_cache_append(p, p, p, 4, p, p, 8, 60, 16, 64, 0, None, None) == 2  # D % 8
    assert lib.kv_cache_append(p, p, p, -1, p, p, 8, 64, 16, 64, 0, None, None) == 1
    assert lib.kv_cache_append(p, p, p, 0, p, p, 8, 64, 16, 64, 0, None, None) == 0
    arr = (ctypes.c_void_p * 1)(1 << 20)
    assert lib.block_copy(arr, arr, 0, p, 1, 8, 64, 16, 64, 0, None, None) == 1
    assert lib.block_copy(arr, arr, 129, p, 1, 8, 64, 16, 64, 0, None, None) == 1
    assert lib.block_copy(arr, arr, 1, p, 0, 8, 64, 16, 64, 0, None, None) == 0


def test_allocator_create_rejects_non_permutations(lib):
    bad = (ctypes.c_int32 * 3)(0, 0, 1)
    assert not lib.pa_alloc_create(3, 4, bad)
    assert not lib.pa_alloc_create(0, 4, None)
    h = lib.pa_alloc_create(3, 4, (ctypes.c_int32 * 3)(2, 0, 1))
    assert h
    lib.pa_alloc_destroy(h)


def _same_state(cpp, model):
    for s in model.tables:
        assert cpp.block_table(s) == model.tables[s]
        assert cpp.length(s) == model.lens[s]
    for b in range(model.num_blocks):
        assert cpp.refcount(b) == model.refcount[b]
    assert cpp.num_free() == len(model.free)
    assert cpp.num_seqs() == len(model.tables)


@pytest.mark.parametrize("seed", range(6))
def test_cpp_allocator_matches_the_model(lib, seed):
    from paged_kv_cache_317_gb300.binding import BlockAllocator, PagedKVError
    rng = np.random.default_rng(100 + seed)
    nb, bs = 120, int(rng.choice([1, 4, 16]))
    order = rng.permutation(nb)
    cpp, model = BlockAllocator(nb, bs, order), BlockAllocatorModel(nb, bs, order)
    next_id = 0
    for _ in range(600):
        live = list(model.tables)
        op = int(rng.integers(0, 5))
        if op == 0 or not live:
            n = int(rng.integers(0, 30))
            try:
                model.add(next_id, n)
                ok = True
            except AllocatorError:
                ok = False
            if ok:
                cpp.add(next_id, n)
            else:
                with pytest.raises(PagedKVError):
                    cpp.add(next_id, n)
            next_id += 1
        elif op == 1:
            p = live[int(rng.integers(len(live)))]
            model.fork(p, next_id)
            cpp.fork(p, next_id)
            next_id += 1
        elif op in (2, 3):
            s = live[int(rng.integers(len(live)))]
            try:
                expect = model.append(s)
            except AllocatorError:
                expect = None
            if expect is None:
                with pytest.raises(PagedKVError):
                    cpp.append(s)
            else:
                assert cpp.append(s) == expect
        else:
            s = live[int(rng.integers(len(live)))]
            model.free_seq(s)
            cpp.free(s)
        cpp.check()
    _same_state(cpp, model)


def test_batch_append_matches_sequential_appends(lib):
    from paged_kv_cache_317_gb300.binding import BlockAllocator
    bs = 16
    cpp, model = BlockAllocator(400, bs), BlockAllocatorModel(400, bs)
    for s, n in enumerate([1029, 16, 33, 0]):
        cpp.add(s, n)
        model.add(s, n)
    for child in range(4, 11):                       # 7 forks of the partly filled prompt
        cpp.fork(0, child)
        model.fork(0, child)
    seqs = [0, 4, 5, 6, 7, 8, 9, 10, 1, 2, 3, 2]     # sequence 2 twice
    slots, pairs = cpp.batch_append(seqs)
    want = [model.append(s) for s in seqs]
    assert slots.tolist() == [w[0] for w in want]
    assert [tuple(p) for p in pairs.tolist()] == [w[1] for w in want if w[1] is not None]
    assert len(pairs) == 7                           # 8 holders of one partial block
    tables, lens = cpp.batch_block_tables(list(range(11)), 70)
    for s in range(11):
        assert tables[s, : len(model.tables[s])].tolist() == model.tables[s]
        assert (tables[s, len(model.tables[s]):] == -1).all()
        assert lens[s] == model.lens[s]
    cpp.check()


def test_batch_append_is_all_or_nothing_when_out_of_blocks(lib):
    from paged_kv_cache_317_gb300.binding import BlockAllocator, PagedKVError
    cpp = BlockAllocator(3, 4)
    cpp.add(0, 4)
    cpp.add(1, 4)                                    # one block left, two appends need two
    before = (cpp.block_table(0), cpp.block_table(1), cpp.num_free())
    with pytest.raises(PagedKVError) as e:
        cpp.batch_append([0, 1])
    assert e.value.name == "PA_ERR_OOM"
    assert (cpp.block_table(0), cpp.block_table(1), cpp.num_free()) == before


def test_allocator_error_codes(lib):
    from paged_kv_cache_317_gb300.binding import BlockAllocator, PagedKVError
    a = BlockAllocator(4, 4)
    a.add(1, 3)
    for fn, args, name in ((a.add, (1, 2), "PA_ERR_SEQ_EXISTS"), (a.fork, (9, 2), "PA_ERR_NO_SEQ"),
                           (a.free, (9,), "PA_ERR_NO_SEQ"), (a.add, (2, 100), "PA_ERR_OOM")):
        with pytest.raises(PagedKVError) as e:
            fn(*args)
        assert e.value.name == name
    assert a.slots(1, 0, 3).tolist() == [a.block_table(1)[0] * 4 + i for i in range(3)]


def test_fused_append_rejects_missing_rows(lib):
    p = ctypes.c_void_p(1 << 20)
    assert lib.paged_attn_decode_append(p, None, p, p, p, p, p, 4, 8, 64, 16, 4, 64, 0.125, 0, p,
                                        2, 0, None, 0, None, None, None) == 1
    assert lib.paged_attn_decode_append(p, p, ctypes.c_void_p((1 << 20) + 4), p, p, p, p, 4, 8, 64,
                                        16, 4, 64, 0.125, 0, p, 2, 0, None, 0, None, None,
                                        None) == 1


def test_partition_work_items_cover_each_partition_once():
    from paged_kv_cache_317_gb300.binding import partition_work_items
    lens = np.array([5, 0, 1024, 1025, 512, 3000, 513])
    MB, bs, pt = 200, 16, 512
    P = -(-MB * bs // pt)
    items = partition_work_items(lens, pt, MB, bs)
    assert items.dtype == np.int32
    seen = sorted((int(i) // P, int(i) % P) for i in items)
    want = sorted((i, p) for i, L in enumerate(lens) for p in range(max(1, -(-int(L) // pt))))
    assert seen == want
    # longest sequences first, partitions of a sequence in order
    seqs = [int(i) // P for i in items]
    order = list(dict.fromkeys(seqs))
    assert order == sorted(range(len(lens)), key=lambda i: (-lens[i], i))
    # automatic partition length (0) means 512; an explicit order is followed
    assert np.array_equal(partition_work_items(lens, 0, MB, bs), items)
    mine = partition_work_items(lens, 256, MB, bs, order=[6, 0, 1, 2, 3, 4, 5])
    assert int(mine[0]) // (-(-MB * bs // 256)) == 6


def test_decode_opts_layout_matches_the_header():
    """The ctypes mirror of pa_decode_opts has the header's field order and size."""
    from paged_kv_cache_317_gb300.binding import pa_decode_opts
    hdr = open(os.path.join(HEADER_DIR, "pagedkv.h")).read()
    body = hdr[hdr.index("typedef struct pa_decode_opts {"):hdr.index("} pa_decode_opts;")]
    names = [ln.strip().rstrip(";").split()[-1].lstrip("*") for ln in body.splitlines()[1:]
             if ln.strip()]
    assert names == [f[0] for f in pa_decode_opts._fields_]
    # size and offsets as a C compiler lays the header's struct out
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    prog = ("#include <stdio.h>\n#include <stddef.h>\n#include \"pagedkv.h\"\n"
            "int main(void) { printf(\"%zu" + " %zu" * len(names) + "\\n\", sizeof(pa_decode_opts)"
            + "".join(f", offsetof(pa_decode_opts, {n})" for n in names) + "); return 0; }\n")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        open(src, "w").write(prog)
        subprocess.run([cc, "-I", HEADER_DIR, src, "-o", exe], check=True)
        got = [int(x) for x in subprocess.run([exe], capture_output=True, text=True,
                                              check=True).stdout.split()]
    assert got == [ctypes.sizeof(pa_decode_opts)] + [getattr(pa_decode_opts, n).offset
                                                      for n in names]


def test_batch_fork_and_free_match_single_calls(lib):
    from paged_kv_cache_317_gb300.binding import BlockAllocator
    rng = np.random.default_rng(11)
    order = rng.permutation(600).astype(np.int32)
    one, many = BlockAllocator(600, 16, order), BlockAllocator(600, 16, order)
    model = BlockAllocatorModel(600, 16, order)
    for s in range(6):
        n = int(rng.integers(1, 300))
        for a in (one, many, model):
            a.add(s, n)
    next_id = 6
    live = list(range(6))
    for step in range(30):
        parents = [int(rng.choice(live)) for _ in range(5)]
        children = list(range(next_id, next_id + 5))
        next_id += 5
        parents[3] = children[1]                     # a child forked earlier in the batch
        for p, c in zip(parents, children):
            one.fork(p, c)
            model.fork(p, c)
        many.batch_fork(parents, children)
        live += children
        gone = [int(x) for x in rng.choice(live, size=4, replace=False)]
        for g in gone:
            one.free(g)
            model.free_seq(g)
        many.batch_free(gone)
        live = [x for x in live if x not in gone]
        for a in (one, many, model):
            a.append(live[0])
        for s in live:
            assert many.block_table(s) == one.block_table(s) == model.tables[s]
        assert many.num_free() == one.num_free()
    many.check()
    _same_state(many, model)


def test_batch_fork_and_free_are_all_or_nothing(lib):
    from paged_kv_cache_317_gb300.binding import BlockAllocator, PagedKVError
    cpp = BlockAllocator(50, 16)
    cpp.add(0, 40)
    cpp.add(1, 20)
    before = (cpp.num_seqs(), cpp.num_free(), cpp.refcount(cpp.block_table(0)[0]))
    for parents, children, code in (([0, 7], [2, 3], "PA_ERR_NO_SEQ"),       # missing parent
                                    ([0, 1], [2, 2], "PA_ERR_SEQ_EXISTS"),   # repeated child
                                    ([0, 1], [2, 1], "PA_ERR_SEQ_EXISTS")):  # existing child
        with pytest.raises(PagedKVError) as e:
            cpp.batch_fork(parents, children)
        assert e.value.name == code
        assert (cpp.num_seqs(), cpp.num_free(), cpp.refcount(cpp.block_table(0)[0])) == before
    for seqs in ([0, 9], [1, 1]):                                            # missing / twice
        with pytest.raises(PagedKVError) as e:
            cpp.batch_free(seqs)
        assert e.value.name == "PA_ERR_NO_SEQ"
        assert (cpp.num_seqs(), cpp.num_free()) == before[:2]
    cpp.batch_free([0, 1])
    assert cpp.num_seqs() == 0 and cpp.num_free() == 50


def test_beam_churn_reuses_sequences_exactly(lib):
    """Whole-batch fork/free rounds (beam search) recycle the allocator's freed
    sequence records; tables, lengths and refcounts follow the model exactly, and
    a refused batch changes nothing."""
    from paged_kv_cache_317_gb300.binding import BlockAllocator, PagedKVError
    rng = np.random.default_rng(12)
    order = rng.permutation(3000).astype(np.int32)
    alloc, model = BlockAllocator(3000, 16, order), BlockAllocatorModel(3000, 16, order)
    beams, next_id = [], 0
    for g in range(8):
        n = int(rng.integers(20, 200))
        alloc.add(next_id, n)
        model.add(next_id, n)
        beams.append(next_id)
        next_id += 1
    for step in range(40):
        parents = [int(rng.choice(beams)) for _ in beams]
        children = list(range(next_id, next_id + len(beams)))
        next_id += len(beams)
        alloc.batch_fork(parents, children)
        for p, c in zip(parents, children):
            model.fork(p, c)
        alloc.batch_free(beams)
        for b in beams:
            model.free_seq(b)
        beams = children
        for b in beams:
            for _ in range(int(rng.integers(0, 20))):
                assert alloc.append(b) == model.append(b)
        for b in beams:
            assert alloc.block_table(b) == model.tables[b]
            assert alloc.length(b) == model.lens[b]
        alloc.check()
        _same_state(alloc, model)
    # refused batches leave everything as it was
    before = {b: alloc.block_table(b) for b in beams}
    free_before = alloc.num_free()
    with pytest.raises(PagedKVError, match="SEQ_EXISTS"):
        alloc.batch_fork([beams[0], beams[1]], [next_id, next_id])          # child twice
    with pytest.raises(PagedKVError, match="SEQ_EXISTS"):
        alloc.batch_fork([beams[0]], [beams[1]])                            # child exists
    with pytest.raises(PagedKVError, match="NO_SEQ"):
        alloc.batch_fork([next_id + 1, beams[0]], [next_id, next_id + 1])   # parent only later
    with pytest.raises(PagedKVError, match="NO_SEQ"):
        alloc.batch_free([beams[0], beams[0]])                              # listed twice
    with pytest.raises(PagedKVError, match="NO_SEQ"):
        alloc.batch_free([beams[0], next_id + 5])                           # unknown id
    assert alloc.num_free() == free_before
    assert {b: alloc.block_table(b) for b in beams} == before
    alloc.batch_free(beams)
    assert alloc.num_free() == 3000


def test_prefill_rejects_bad_arguments_on_the_host(lib):
    from paged_kv_cache_317_gb300.binding import STATUS_CODE
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its checks first
    INV, UNS = STATUS_CODE["PA_ERR_INVALID_ARG"], STATUS_CODE["PA_ERR_UNSUPPORTED"]

    def call(**kw):
        a = dict(q=p, qs=p, T=64, mq=64, k=p, v=p, bt=p, sl=p, N=4, H=8, D=128, bs=16, MB=4,
                 B=64, scale=0.125, dt=1, out=p, odt=2)
        a.update(kw)
        return lib.paged_attn_prefill(a["q"], a["qs"], a["T"], a["mq"], a["k"], a["v"], a["bt"],
                                      a["sl"], a["N"], a["H"], a["D"], a["bs"], a["MB"], a["B"],
                                      a["scale"], a["dt"], a["out"], a["odt"], None, None)

    assert call(D=96) == UNS
    assert call(bs=24) == UNS
    assert call(dt=2) == UNS
    assert call(odt=7) == UNS
    assert call(qs=None) == INV
    assert call(out=ctypes.c_void_p((1 << 20) + 8)) == INV    # not 16-byte aligned
    assert call(scale=0.0) == INV
    assert call(scale=float("inf")) == INV
    assert call(B=1 << 24, H=128) == INV                      # cache rows >= 2^31
    # 2^20 sequences x 64 heads x 16 query tiles = 2^30 items: too many
    assert call(N=1 << 20, H=64, mq=2048, B=8) == INV
    assert call(N=0) == 0 and call(T=0) == 0 and call(mq=0) == 0   # nothing to do
