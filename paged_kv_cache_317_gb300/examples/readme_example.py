"""Using the library from Python: a prompt, a fork that shares its blocks, one
decode step with copy-on-write and the fused append + decode (run it as a script
on a CUDA device)."""

import torch
from paged_kv_cache_317_gb300 import binding as pa

# caches [num_blocks, heads, block_size, head_dim]; one layer
H, D, bs, nblk = 8, 128, 16, 1024
kc = torch.zeros(nblk, H, bs, D, dtype=torch.bfloat16, device="cuda")
vc = torch.zeros_like(kc)

alloc = pa.BlockAllocator(nblk, bs)            # host free list + reference counts
alloc.add(0, 100)                              # sequence 0: a 100-token prompt
k = torch.randn(100, H, D, dtype=torch.bfloat16, device="cuda")
pa.kv_cache_append(k, k, torch.from_numpy(alloc.slots(0, 0, 100)).cuda(), kc, vc)
alloc.fork(0, 1)                               # sequence 1 shares every block of 0

slots, pairs = alloc.batch_append([0, 1])      # next token of each; copy-on-write pairs
if len(pairs):
    pa.block_copy([kc], [vc], torch.from_numpy(pairs).cuda())
tables, lens = alloc.batch_block_tables([0, 1], max_blocks=64)
q = torch.randn(2, H, D, dtype=torch.bfloat16, device="cuda")
new = torch.randn(2, H, D, dtype=torch.bfloat16, device="cuda")
pt = pa.decode_partition_tokens(lens, H)       # split-K length for this batch (host rule)
items = pa.partition_work_items(lens, pt, 64, bs)   # (sequence, partition) work list
out = pa.paged_attn_decode_append(q, new, new, kc, vc, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(lens).cuda(), scale=D ** -0.5,
                                  partition_tokens=pt, work_items=torch.from_numpy(items).cuda())
