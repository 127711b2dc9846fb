"""Seeded generators for the five decode workloads and for ad-hoc test batches.

Values are N(0,1) drawn in fp32 from a seeded ``torch.Generator`` on the
requested device and rounded to nearest-even into the storage dtype, in the
order q, k pool, v pool, new k, new v.  Structure (lengths, physical placement,
forks) comes from ``numpy.random.default_rng(seed)``.  The same seed on the same
device gives the same tensors; CPU and CUDA generators give different streams,
so a test draws once and hands the same tensors to both sides.

Every slot of a pool that holds no live token is filled with NaN, so that a
kernel reading a slot it should have masked produces NaN in its output.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}
_DRAW_CHUNK = 1 << 26  # fp32 elements drawn per call (256 MB)


def _torch_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def randn_rounded(shape, dtype: torch.dtype, gen: torch.Generator, device) -> torch.Tensor:
    """N(0,1) in fp32, rounded to ``dtype``; drawn in fixed-size chunks."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _DRAW_CHUNK):
        e = min(n, s + _DRAW_CHUNK)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32).to(dtype)
    return out


def default_scale(head_dim: int) -> float:
    """1/sqrt(head_dim), rounded to fp32 (the value both sides receive)."""
    return float(np.float32(1.0 / math.sqrt(head_dim)))


def lognormal_lengths(rng: np.random.Generator, n: int, median: float, sigma: float,
                      lo: int, hi: int) -> np.ndarray:
    z = rng.standard_normal(n)
    return np.clip(np.round(np.exp(math.log(median) + sigma * z)), lo, hi).astype(np.int64)


@dataclass
class DecodeBatch:
    """One decode step over a paged pool whose blocks are scattered at random.

    ``context_lens[i]`` is the number of tokens sequence ``i`` attends over.
    With an append, the cache holds ``context_lens[i] - 1`` of them and the
    step writes the last one (``new_k``/``new_v``) at ``slot_mapping[i]``;
    that slot is NaN until the append writes it.
    """

    name: str
    seed: int
    num_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: torch.dtype
    context_lens: np.ndarray       # int32 [N]
    block_tables: np.ndarray       # int32 [N, MB]; -1 past a sequence's blocks
    q: torch.Tensor                # [N, H, D]
    k_cache: torch.Tensor          # [B, H, bs, D]
    v_cache: torch.Tensor          # [B, H, bs, D]
    scale: float
    new_k: Optional[torch.Tensor] = None   # [N, H, D]
    new_v: Optional[torch.Tensor] = None
    slot_mapping: Optional[np.ndarray] = None  # int64 [N]

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def has_append(self) -> bool:
        return self.new_k is not None

    @property
    def cached_lens(self) -> np.ndarray:
        """Tokens in the cache before the step's append."""
        return self.context_lens - (1 if self.has_append else 0)

    def to(self, device) -> "DecodeBatch":
        d = dict(self.__dict__)
        for k in ("q", "k_cache", "v_cache", "new_k", "new_v"):
            if d[k] is not None:
                d[k] = d[k].to(device)
        return DecodeBatch(**d)


def _build_scattered(name: str, seed: int, rng: np.random.Generator, gen: torch.Generator,
                     context_lens, num_heads: int, head_dim: int, block_size: int,
                     dtype: torch.dtype, device, with_append: bool,
                     num_blocks: Optional[int] = None, pool_factor: float = 1.2,
                     poison: bool = True) -> DecodeBatch:
    lens = np.asarray(context_lens, dtype=np.int64)
    n = lens.shape[0]
    need = -(-lens // block_size)
    if num_blocks is None:
        num_blocks = max(int(math.ceil(pool_factor * lens.sum() / block_size)), int(need.sum()), 1)
    if need.sum() > num_blocks:
        raise ValueError(f"{name}: pool of {num_blocks} blocks cannot hold {need.sum()}")
    mb = max(1, int(need.max()) if n else 1)
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.full((n, mb), -1, np.int32)
    start = 0
    for i in range(n):
        tables[i, : need[i]] = perm[start : start + need[i]]
        start += int(need[i])

    H, D = num_heads, head_dim
    q = randn_rounded((n, H, D), dtype, gen, device)
    k_cache = randn_rounded((num_blocks, H, block_size, D), dtype, gen, device)
    v_cache = randn_rounded((num_blocks, H, block_size, D), dtype, gen, device)
    new_k = new_v = slots = None
    cached = lens - (1 if with_append else 0)
    if with_append:
        if (lens < 1).any():
            raise ValueError("an appended token needs context_lens >= 1")
        new_k = randn_rounded((n, H, D), dtype, gen, device)
        new_v = randn_rounded((n, H, D), dtype, gen, device)
        pos = cached
        slots = (tables[np.arange(n), pos // block_size].astype(np.int64) * block_size
                 + pos % block_size)
    if poison:
        live = np.zeros((num_blocks, block_size), dtype=bool)
        for i in range(n):
            for j in range(int(need[i])):
                rows = int(min(block_size, max(0, cached[i] - j * block_size)))
                live[tables[i, j], :rows] = True
        dead = torch.from_numpy(~live).to(device)[:, None, :, None]
        k_cache.masked_fill_(dead, float("nan"))
        v_cache.masked_fill_(dead, float("nan"))
    return DecodeBatch(name=name, seed=seed, num_heads=H, head_dim=D, block_size=block_size,
                       num_blocks=num_blocks, dtype=dtype, context_lens=lens.astype(np.int32),
                       block_tables=tables, q=q, k_cache=k_cache, v_cache=v_cache,
                       scale=default_scale(D), new_k=new_k, new_v=new_v, slot_mapping=slots)


def random_decode_batch(seed: int, context_lens, num_heads: int, head_dim: int, block_size: int,
                        dtype="f16", device="cpu", with_append: bool = False,
                        num_blocks: Optional[int] = None, pool_factor: float = 1.2,
                        poison: bool = True, name: str = "random") -> DecodeBatch:
    """A batch with the given lengths and a seeded scattered placement."""
    rng = np.random.default_rng(seed)
    gen = _torch_gen(seed, device)
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    return _build_scattered(name, seed, rng, gen, context_lens, num_heads, head_dim, block_size,
                            dt, device, with_append, num_blocks, pool_factor, poison)


def tiny_decode(seed: int = 1, device="cpu", with_append: bool = True) -> DecodeBatch:
    """4 sequences, 8 heads, head_dim 64, block 16, fp16, lengths U[1,200], pool of 64 blocks."""
    rng = np.random.default_rng(seed)
    gen = _torch_gen(seed, device)
    lens = rng.integers(1, 201, size=4)
    return _build_scattered("tiny", seed, rng, gen, lens, 8, 64, 16, torch.float16, device,
                            with_append, num_blocks=64)


def decode_13b(seed: int = 2, device="cuda", num_seqs: int = 256, block_size: int = 16,
               with_append: bool = True, sigma: float = 0.75, dtype="bf16",
               poison: bool = True) -> DecodeBatch:
    """13B-shaped decode: 40 heads x 128, lengths log-normal (median 350) clipped to [16, 2048],
    pool 1.2x the live tokens, blocks shuffled; one appended token per sequence."""
    rng = np.random.default_rng(seed)
    gen = _torch_gen(seed, device)
    lens = lognormal_lengths(rng, num_seqs, 350.0, sigma, 16, 2048)
    return _build_scattered("decode_13b", seed, rng, gen, lens, 40, 128, block_size,
                            DTYPES[dtype], device, with_append, poison=poison)


def long_context(seed: int = 4, device="cuda", block_size: int = 16, num_seqs: int = 32,
                 seq_len: int = 16384, num_heads: int = 40, poison: bool = True) -> DecodeBatch:
    """Long-context decode: every sequence ``seq_len`` tokens, scattered over a 1.2x pool."""
    rng = np.random.default_rng(seed)
    gen = _torch_gen(seed, device)
    lens = np.full(num_seqs, seq_len, dtype=np.int64)
    return _build_scattered("long_context", seed, rng, gen, lens, num_heads, 128, block_size,
                            torch.bfloat16, device, False, poison=poison)


# ---------------------------------------------------------------------------
# Parallel sampling: prompts shared by several samples, then private tails.
# ---------------------------------------------------------------------------

@dataclass
class SamplingPlan:
    """``num_prompts`` prompts, each held once and shared by ``samples`` sequences.

    Sequence ``k * samples + s`` is sample ``s`` of prompt ``k``.  Its tokens are
    prompt ``k``'s tokens followed by its own ``tail_lens`` tokens.  Token
    values live in two stores: prompt tokens (prompt ``k`` at rows
    ``prompt_offsets[k]:prompt_offsets[k+1]``) and tail tokens (sequence ``i``
    at ``tail_offsets[i]:tail_offsets[i+1]``).  ``free_order`` is the order in
    which an allocator hands out the pool's blocks.
    """

    seed: int
    num_prompts: int
    samples: int
    num_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    num_blocks: int
    prompt_lens: np.ndarray
    prompt_offsets: np.ndarray
    tail_lens: np.ndarray
    tail_offsets: np.ndarray
    q: torch.Tensor
    prompt_k: torch.Tensor
    prompt_v: torch.Tensor
    tail_k: torch.Tensor
    tail_v: torch.Tensor
    free_order: np.ndarray
    scale: float

    @property
    def num_seqs(self) -> int:
        return self.num_prompts * self.samples


def parallel_sampling(seed: int = 3, device="cuda", num_prompts: int = 32, samples: int = 8,
                      prefix: int = 1024, partial_prefix: bool = True, max_tail: int = 512,
                      num_heads: int = 40, head_dim: int = 128, block_size: int = 16,
                      dtype="bf16") -> SamplingPlan:
    """Parallel sampling with shared prompts.  Prompt ``k`` has ``prefix + p_k`` tokens with
    ``p_k ~ U[1, 15]`` (so its last block is partly filled and the first divergent write
    copies it), or exactly ``prefix`` tokens when ``partial_prefix`` is False.  Tails are
    U[1, max_tail]."""
    rng = np.random.default_rng(seed)
    gen = _torch_gen(seed, device)
    pad = rng.integers(1, 16, size=num_prompts) if partial_prefix else np.zeros(num_prompts, np.int64)
    prompt_lens = (prefix + pad).astype(np.int64)
    tail_lens = rng.integers(1, max_tail + 1, size=num_prompts * samples).astype(np.int64)
    bs = block_size
    need = int((-(-prompt_lens // bs)).sum() + (1 + (tail_lens + bs) // bs + 1).sum())
    num_blocks = int(math.ceil(1.2 * need))
    free_order = rng.permutation(num_blocks).astype(np.int32)
    dt = DTYPES[dtype]
    H, D = num_heads, head_dim
    q = randn_rounded((num_prompts * samples, H, D), dt, gen, device)
    pk = randn_rounded((int(prompt_lens.sum()), H, D), dt, gen, device)
    pv = randn_rounded((int(prompt_lens.sum()), H, D), dt, gen, device)
    tk = randn_rounded((int(tail_lens.sum()), H, D), dt, gen, device)
    tv = randn_rounded((int(tail_lens.sum()), H, D), dt, gen, device)
    return SamplingPlan(seed=seed, num_prompts=num_prompts, samples=samples, num_heads=H,
                        head_dim=D, block_size=bs, dtype=dt, num_blocks=num_blocks,
                        prompt_lens=prompt_lens,
                        prompt_offsets=np.concatenate([[0], np.cumsum(prompt_lens)]),
                        tail_lens=tail_lens,
                        tail_offsets=np.concatenate([[0], np.cumsum(tail_lens)]),
                        q=q, prompt_k=pk, prompt_v=pv, tail_k=tk, tail_v=tv,
                        free_order=free_order, scale=default_scale(D))


# ---------------------------------------------------------------------------
# Mixed serving: bimodal lengths, one token per step, forks every step.
# ---------------------------------------------------------------------------

@dataclass
class MixedServingPlan:
    """A batch of ``num_seqs`` sequences run for ``steps`` decode steps.

    Batch slot ``b`` starts with ``init_lens[b]`` tokens, stored at rows
    ``init_offsets[b]:init_offsets[b+1]`` of ``init_k``/``init_v``.  At step
    ``s``, for each pair ``(a, b)`` in ``fork_pairs[s]``, the sequence in slot
    ``b`` ends and is replaced by a fork of the sequence in slot ``a``; then
    every slot appends one token and the batch decodes.  ``step_tokens(s)``
    gives that step's q, new k and new v.
    """

    seed: int
    num_seqs: int
    num_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    steps: int
    num_blocks: int
    init_lens: np.ndarray
    init_offsets: np.ndarray
    init_k: torch.Tensor
    init_v: torch.Tensor
    fork_pairs: np.ndarray          # int64 [steps, F, 2]
    free_order: np.ndarray
    scale: float
    device: str = "cuda"

    def step_tokens(self, step: int, device=None):
        device = self.device if device is None else device
        gen = _torch_gen(self.seed * 1_000_003 + 7919 * (step + 1), device)
        shape = (self.num_seqs, self.num_heads, self.head_dim)
        q = randn_rounded(shape, self.dtype, gen, device)
        k = randn_rounded(shape, self.dtype, gen, device)
        v = randn_rounded(shape, self.dtype, gen, device)
        return q, k, v


def mixed_serving(seed: int = 5, device="cuda", num_seqs: int = 512, steps: int = 100,
                  fork_frac: float = 0.05, short=(32, 256), long=(1024, 4096),
                  long_frac: float = 0.3, num_heads: int = 32, head_dim: int = 128,
                  block_size: int = 16, dtype="f16") -> MixedServingPlan:
    rng = np.random.default_rng(seed)
    gen = _torch_gen(seed, device)
    n_long = int(round(long_frac * num_seqs))
    is_long = np.zeros(num_seqs, dtype=bool)
    is_long[:n_long] = True
    rng.shuffle(is_long)
    lens = np.where(is_long, rng.integers(long[0], long[1] + 1, size=num_seqs),
                    rng.integers(short[0], short[1] + 1, size=num_seqs)).astype(np.int64)
    forks = int(math.ceil(fork_frac * num_seqs))
    pairs = np.zeros((steps, forks, 2), dtype=np.int64)
    for s in range(steps):
        pick = rng.choice(num_seqs, size=2 * forks, replace=False)
        pairs[s, :, 0] = pick[:forks]
        pairs[s, :, 1] = pick[forks:]
    bs = block_size
    num_blocks = int(math.ceil(1.2 * (-(-(lens + steps) // bs)).sum()))
    free_order = rng.permutation(num_blocks).astype(np.int32)
    dt = DTYPES[dtype]
    total = int(lens.sum())
    ik = randn_rounded((total, num_heads, head_dim), dt, gen, device)
    iv = randn_rounded((total, num_heads, head_dim), dt, gen, device)
    return MixedServingPlan(seed=seed, num_seqs=num_seqs, num_heads=num_heads, head_dim=head_dim,
                            block_size=bs, dtype=dt, steps=steps, num_blocks=num_blocks,
                            init_lens=lens, init_offsets=np.concatenate([[0], np.cumsum(lens)]),
                            init_k=ik, init_v=iv, fork_pairs=pairs, free_order=free_order,
                            scale=default_scale(head_dim), device=str(device))


# ---------------------------------------------------------------------------
# Beam-search-style churn: survivors chosen by random scores (no model).
# ---------------------------------------------------------------------------

@dataclass
class BeamPlan:
    """``groups`` beam groups of ``width`` beams, run for ``steps`` steps.

    Group ``g`` starts as one prompt of ``prompt_lens[g]`` tokens (rows
    ``prompt_offsets[g]:prompt_offsets[g+1]`` of ``prompt_k``/``prompt_v``)
    held by all ``width`` beams.  At step ``s`` new beam ``j`` of group ``g``
    continues old beam ``parents[s, g, j]`` (the survivors of a random score
    draw standing in for a model) and every beam appends one token;
    ``step_tokens(s)`` gives that step's q, k, v as ``[groups * width, H, D]``.
    """

    seed: int
    groups: int
    width: int
    steps: int
    num_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    num_blocks: int
    prompt_lens: np.ndarray
    prompt_offsets: np.ndarray
    prompt_k: torch.Tensor
    prompt_v: torch.Tensor
    parents: np.ndarray           # int64 [steps, groups, width]
    free_order: np.ndarray
    scale: float
    device: str = "cuda"

    def step_tokens(self, step: int, device=None):
        device = self.device if device is None else device
        gen = _torch_gen(self.seed * 7_000_003 + 104729 * (step + 1), device)
        shape = (self.groups * self.width, self.num_heads, self.head_dim)
        return tuple(randn_rounded(shape, self.dtype, gen, device) for _ in range(3))


def beam_search(seed: int = 6, device="cuda", groups: int = 16, width: int = 4,
                steps: int = 40, prompt=(100, 400), num_heads: int = 8, head_dim: int = 128,
                block_size: int = 16, dtype="bf16") -> BeamPlan:
    rng = np.random.default_rng(seed)
    gen = _torch_gen(seed, device)
    lens = rng.integers(prompt[0], prompt[1] + 1, size=groups).astype(np.int64)
    parents = np.zeros((steps, groups, width), dtype=np.int64)
    for s in range(steps):
        for g in range(groups):
            # width x width candidate scores; the best `width` survive
            scores = rng.random((width, width))
            best = np.argsort(-scores, axis=None, kind="stable")[:width]
            parents[s, g] = np.sort(best // width)
    bs = block_size
    # worst case: every beam private (prompt copied per beam) plus its steps
    need = int((width * (-(-(lens + steps + 1) // bs) + 1)).sum())
    num_blocks = int(math.ceil(1.2 * need))
    free_order = rng.permutation(num_blocks).astype(np.int32)
    dt = DTYPES[dtype]
    total = int(lens.sum())
    pk = randn_rounded((total, num_heads, head_dim), dt, gen, device)
    pv = randn_rounded((total, num_heads, head_dim), dt, gen, device)
    return BeamPlan(seed=seed, groups=groups, width=width, steps=steps, num_heads=num_heads,
                    head_dim=head_dim, block_size=bs, dtype=dt, num_blocks=num_blocks,
                    prompt_lens=lens, prompt_offsets=np.concatenate([[0], np.cumsum(lens)]),
                    prompt_k=pk, prompt_v=pv, parents=parents, free_order=free_order,
                    scale=default_scale(head_dim), device=str(device))
