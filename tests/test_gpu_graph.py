"""The decode step as a CUDA graph: the C-ABI calls allocate nothing when given a
workspace, never synchronise, and keep all per-step state in device memory, so a
serving loop can capture a step once and replay it with new inputs written into
the same buffers."""

import numpy as np
import pytest
import torch

from gpu_util import assert_matches_oracle, bits, oracle_decode
from workloads import random_decode_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    from paged_kv_cache_317_gb300 import binding
    return binding


def _step(B, st):
    """One device step: copy-on-write copies (padded), then fused append + decode."""
    B.block_copy([st["kc"]], [st["vc"]], st["pairs"], error_record=st["rec"])
    B.paged_attn_decode_append(st["q"], st["nk"], st["nv"], st["kc"], st["vc"], st["bt"],
                               st["sl"], st["scale"], out=st["out"], out_dtype=torch.bfloat16,
                               workspace=st["ws"], error_record=st["rec"],
                               seq_order=st["order"])


def test_decode_step_replays_from_a_cuda_graph(B):
    lens = [5, 900, 33, 1500, 64, 700, 2, 1100, 513, 1024]
    H, D, bs = 8, 128, 16
    base = random_decode_batch(21, lens, H, D, bs, dtype="bf16", device="cuda",
                               with_append=True, pool_factor=2.0, poison=False)
    N, MB = len(lens), base.max_blocks_per_seq
    used = {int(x) for x in base.block_tables[base.block_tables >= 0]}
    spare = [x for x in range(base.num_blocks) if x not in used]
    st = {
        "kc": base.k_cache.clone(), "vc": base.v_cache.clone(),
        "q": base.q.clone(), "nk": base.new_k.clone(), "nv": base.new_v.clone(),
        "bt": torch.from_numpy(base.block_tables).cuda(),
        "sl": torch.from_numpy(base.context_lens).cuda(),
        "order": torch.from_numpy(np.argsort(-base.context_lens, kind="stable")
                                  .astype(np.int32)).cuda(),
        "pairs": torch.full((4, 2), -1, dtype=torch.int64, device="cuda"),
        "out": torch.empty((N, H, D), dtype=torch.bfloat16, device="cuda"),
        "ws": torch.empty(B.paged_attn_workspace_size(N, H, D, bs, MB, 0), dtype=torch.uint8,
                          device="cuda"),
        "rec": B.new_error_record(), "scale": base.scale,
    }
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _step(B, st)                       # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(B, st)
    rng = np.random.default_rng(5)
    for it in range(3):
        # new inputs for this step, written into the captured buffers
        g = torch.Generator(device="cuda").manual_seed(100 + it)
        st["q"].copy_(torch.randn(st["q"].shape, generator=g, device="cuda").to(torch.bfloat16))
        st["nk"].copy_(torch.randn(st["nk"].shape, generator=g, device="cuda").to(torch.bfloat16))
        st["nv"].copy_(torch.randn(st["nv"].shape, generator=g, device="cuda").to(torch.bfloat16))
        n_pairs = it % 3                   # 0, 1 or 2 real copies, the rest padding
        pairs = np.full((4, 2), -1, dtype=np.int64)
        for k in range(n_pairs):
            pairs[k] = (rng.choice(sorted(used)), spare[4 * it + k])
        st["pairs"].copy_(torch.from_numpy(pairs))
        # eager reference on copies of the same state
        ref = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in st.items()}
        ref["rec"] = B.new_error_record()
        _step(B, ref)
        graph.replay()
        torch.cuda.synchronize()
        assert B.pa_error_read(st["rec"]) == [0, 0, 0, 0]
        assert torch.equal(st["out"].view(torch.int16), ref["out"].view(torch.int16))
        assert np.array_equal(bits(st["kc"]), bits(ref["kc"]))
        assert np.array_equal(bits(st["vc"]), bits(ref["vc"]))
    # and the replayed step is the oracle's step
    base.k_cache.copy_(st["kc"])
    base.v_cache.copy_(st["vc"])
    base.q.copy_(st["q"])
    base.new_k.copy_(st["nk"])
    base.new_v.copy_(st["nv"])
    assert_matches_oracle(st["out"], oracle_decode(base), "graph replay")
