"""Seeded synthetic inputs for the paged decode path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no attention, no pool bookkeeping), so both the CUDA path
and the CPU oracle can be fed from it.  The pages evaluate on no dataset: every
workload here is synthetic, shaped like the five workloads the library is
measured on (tiny fp32 check, 7B-shaped MHA fp16, 8B-shaped GQA bf16, parallel
sampling with copy-on-write, shared-prefix mixed batch).

Conventions
-----------
* Lengths, placements and op scripts come from ``numpy.random.default_rng``.
* Q/K/V values are N(0, 1) drawn in float32 and rounded to the storage dtype.
  On a CUDA device they are drawn with a seeded ``torch.Generator`` on that
  device so multi-GB caches need no host generation; on the CPU with numpy.
* Block tables are padded with ``-1`` past each sequence's last logical block,
  so any read beyond ``ceil(ctx / 16)`` entries is an out-of-range block id.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16
SEED_BASE = 1000          # workload i uses seed SEED_BASE + i


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def uniform_lengths(n: int, lo: int, hi: int, gen: np.random.Generator) -> np.ndarray:
    return gen.integers(lo, hi + 1, size=n).astype(np.int32)


def log_uniform_lengths(n: int, lo: int, hi: int, gen: np.random.Generator) -> np.ndarray:
    """``clip(round(exp(U(ln lo, ln hi))), lo, hi)``."""
    x = np.exp(gen.uniform(math.log(lo), math.log(hi), size=n))
    return np.clip(np.rint(x), lo, hi).astype(np.int32)


def lognormal_lengths(n: int, median: float, sigma: float, lo: int, hi: int,
                      gen: np.random.Generator) -> np.ndarray:
    x = gen.lognormal(mean=math.log(median), sigma=sigma, size=n)
    return np.clip(np.rint(x), lo, hi).astype(np.int32)


def num_blocks_for(lengths) -> np.ndarray:
    return (np.asarray(lengths, dtype=np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE


def pool_size(lengths, slack: float = 0.10) -> int:
    """Pool sized to the blocks the lengths need plus ``slack`` free."""
    return int(math.ceil((1.0 + slack) * int(num_blocks_for(lengths).sum())))


def disjoint_tables(lengths, num_blocks: int, gen: np.random.Generator,
                    max_blocks: int | None = None) -> np.ndarray:
    """Random disjoint placement: a seeded permutation of the pool, dealt out in
    order, ``ceil(len / 16)`` blocks per sequence.  Returns int32
    ``[num_seqs, max_blocks]`` padded with -1."""
    need = num_blocks_for(lengths)
    if max_blocks is None:
        max_blocks = max(1, int(need.max()) if len(need) else 1)
    if int(need.sum()) > num_blocks:
        raise ValueError("pool too small for these lengths")
    perm = gen.permutation(num_blocks).astype(np.int32)
    tables = np.full((len(need), max_blocks), -1, dtype=np.int32)
    at = 0
    for i, count in enumerate(need):
        tables[i, :count] = perm[at:at + count]
        at += int(count)
    return tables


def normal(shape, dtype, seed: int, device="cpu"):
    """N(0, 1) float32 values rounded to ``dtype`` (a torch dtype)."""
    import torch
    device = torch.device(device)
    if device.type == "cuda":
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)
    values = np.random.default_rng(seed).standard_normal(size=shape, dtype=np.float32)
    return torch.from_numpy(values).to(dtype)


# --------------------------------------------------------------------------
# The five workloads
# --------------------------------------------------------------------------
@dataclass
class DecodeBatch:
    """Shapes and host-side integer inputs of one decode-attention batch."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                      # "f32" | "f16" | "bf16"
    context_lens: np.ndarray        # int32 [B]
    block_tables: np.ndarray        # int32 [B, max_blocks], -1 padded
    num_blocks: int
    num_layers: int = 1
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def new_token_slots(self) -> np.ndarray:
        """Slot of each sequence's newest token (position ctx-1), int64."""
        pos = self.context_lens.astype(np.int64) - 1
        blocks = self.block_tables[np.arange(self.num_seqs), pos // BLOCK_SIZE].astype(np.int64)
        return blocks * BLOCK_SIZE + pos % BLOCK_SIZE


def tiny(seed: int = SEED_BASE + 1) -> DecodeBatch:
    """4 sequences, lengths U{1..100}, 4/4 heads, d=64, fp32, 64-block pool in
    random order."""
    gen = rng(seed)
    lens = uniform_lengths(4, 1, 100, gen)
    tables = disjoint_tables(lens, 64, gen, max_blocks=7)
    return DecodeBatch("tiny", 4, 4, 64, "f32", lens, tables, 64, seed=seed)


def mha_7b(seed: int = SEED_BASE + 2, batch: int = 64) -> DecodeBatch:
    """7B-shaped MHA: 32/32 heads, d=128, fp16, lengths log-uniform [16, 2048],
    pool = blocks needed + 10 %, 32 layers (32 separate caches)."""
    gen = rng(seed)
    lens = log_uniform_lengths(batch, 16, 2048, gen)
    nb = pool_size(lens)
    tables = disjoint_tables(lens, nb, gen, max_blocks=2048 // BLOCK_SIZE)
    return DecodeBatch("mha_7b_fp16", 32, 32, 128, "f16", lens, tables, nb,
                       num_layers=32, seed=seed)


def gqa_8b(seed: int = SEED_BASE + 3, batch: int = 128, fixed_long: int = 4) -> DecodeBatch:
    """8B-shaped GQA: 32/8 heads, d=128, bf16, ``batch - fixed_long`` lengths
    log-uniform [128, 8192] plus ``fixed_long`` sequences of exactly 8192."""
    gen = rng(seed)
    lens = np.concatenate([log_uniform_lengths(batch - fixed_long, 128, 8192, gen),
                           np.full(fixed_long, 8192, dtype=np.int32)])
    nb = pool_size(lens)
    tables = disjoint_tables(lens, nb, gen, max_blocks=8192 // BLOCK_SIZE)
    return DecodeBatch("gqa_8b_bf16", 32, 8, 128, "bf16", lens, tables, nb, seed=seed)


def prefill_8b(seed: int = SEED_BASE + 6, batch: int = 16, chunk: int = 512,
               layers: int = 8) -> DecodeBatch:
    """Chunked prefill, 8B-shaped GQA (32/8 heads, d=128, bf16): ``batch``
    sequences, each a ``chunk``-token piece of its prompt on top of a cached
    prefix log-uniform in [16, 8192] tokens.  ``context_lens`` counts the chunk;
    ``extra["query_lens"]`` holds the chunk lengths.  ``layers`` separate layer
    caches."""
    gen = rng(seed)
    prefix = log_uniform_lengths(batch, 16, 8192, gen)
    lens = (prefix + chunk).astype(np.int32)
    nb = pool_size(lens)
    tables = disjoint_tables(lens, nb, gen)
    return DecodeBatch("prefill_8b_bf16", 32, 8, 128, "bf16", lens, tables, nb,
                       num_layers=layers, seed=seed,
                       extra={"query_lens": np.full(batch, chunk, dtype=np.int32)})


@dataclass
class SamplingScript:
    """Parallel sampling with copy-on-write: ``prompts`` prompts of
    ``prompt_len + shared_extra[p]`` tokens, each forked into ``branches``
    branches, then ``steps`` decode steps in which every branch appends one
    token.  ``shared_extra`` (U{1..15}) makes every prompt end inside a
    partially filled block, which the first divergent append copies."""
    prompts: int
    prompt_len: int
    branches: int
    steps: int
    shared_extra: np.ndarray
    initial_order: np.ndarray
    num_blocks: int
    seed: int


def sampling_cow(seed: int = SEED_BASE + 4, prompts: int = 32, prompt_len: int = 1024,
                 branches: int = 4, steps: int = 256, zero_extra: bool = False) -> SamplingScript:
    gen = rng(seed)
    extra = (np.zeros(prompts, dtype=np.int32) if zero_extra
             else uniform_lengths(prompts, 1, 15, gen))
    prompt_blocks = int(num_blocks_for(prompt_len + extra).sum())
    cow_blocks = prompts * (branches - 1)
    decode_blocks = prompts * branches * (steps // BLOCK_SIZE + 2)
    nb = int(math.ceil(1.1 * (prompt_blocks + cow_blocks + decode_blocks)))
    order = gen.permutation(nb).astype(np.int32)
    return SamplingScript(prompts, prompt_len, branches, steps, extra, order, nb, seed)


@dataclass
class PrefixScript:
    """Shared-prefix mixed batch: one ``prefix_len``-token system prefix held by
    every request, then per-request suffixes of heavy-tailed length."""
    prefix_len: int
    suffix_lens: np.ndarray
    initial_order: np.ndarray
    num_blocks: int
    num_layers: int
    seed: int


def prefix_mix(seed: int = SEED_BASE + 5, requests: int = 100, prefix_len: int = 1024,
               median: float = 512.0, sigma: float = 1.0, max_suffix: int = 16384,
               num_layers: int = 32) -> PrefixScript:
    gen = rng(seed)
    suffix = lognormal_lengths(requests, median, sigma, 1, max_suffix, gen)
    need = int(num_blocks_for([prefix_len])[0]) + int(num_blocks_for(suffix).sum()) + requests
    nb = int(math.ceil(1.1 * need))
    order = gen.permutation(nb).astype(np.int32)
    return PrefixScript(prefix_len, suffix, order, nb, num_layers, seed)
