"""Oracle for the device-side steps of paged decode: attention, append, copy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): plain numpy, float64
arithmetic, loops written the way the pages describe the computation, no
blocking, fusion or reordering beyond what the definition states.

Sources (page title, section):

* "vLLM: treating the KV cache as virtual memory", section "破除误解"
  (misconception 2): PagedAttention is *not* a new attention formula; it is
  still scaled dot-product attention, only the K/V layout changed -- a logical
  block number is translated through a block table to a physical block, one
  indirection per block, like a CPU walking a page table.
* "留书阁 / knowledge-20" page, section "注意力计算的改写" (attention
  rewrite): the contiguous reference ``softmax(Q K^T / sqrt(d_k)) V`` and the
  per-block walk over ``block_table[request]`` reading 16-token K/V blocks.
  The printed per-block pseudo-code never defines its running maximum and
  never rescales the output when the maximum changes, so as printed it is not
  softmax; we take the plain definition (two passes: max, then exp/sum) which
  the first page states is unchanged.
* Same page, section "PagedAttention：虚实分离，按需取用": logical block 0 ->
  physical 37 holds tokens 0-15, logical block 1 -> physical 12 holds tokens
  16-31, ... so token t lives at physical ``block_table[t // 16]``, offset
  ``t % 16``.  A slot number is therefore ``physical * 16 + offset``.
* "Lazy Allocation 与 Copy-on-Write 在 LLM 推理系统中的应用" (OS-lab
  appendix), section 2.1: each decode step reads all earlier K/V and appends
  the new token's K/V; sections 4.3-4.4: a shared block is copied whole before
  the writer's first write into it.

Layout (our reading; the pages only give a conceptual ``kv_cache[block, 0|1]``
of shape ``[block_size, heads, d]``): separate ``k_cache`` and ``v_cache`` of
shape ``[num_blocks, num_kv_heads, 16, head_dim]``.  ``test_oracle_attention``
checks that the page-3 conceptual layout gives the same result.

GQA head mapping (the pages name GQA but do not fix the mapping): query head
``h`` reads KV head ``h // (num_q_heads // num_kv_heads)`` -- contiguous groups,
the convention ``torch.nn.functional.scaled_dot_product_attention(...,
enable_gqa=True)`` uses; a pin checks the two agree.
"""

from __future__ import annotations

import numpy as np

BLOCK_SIZE = 16


def gather_sequence(cache: np.ndarray, block_table, context_len: int) -> np.ndarray:
    """Return one sequence's keys (or values) as a contiguous float64 buffer.

    ``cache`` is ``[num_blocks, num_kv_heads, block_size, head_dim]`` (16 on the
    device; the OS-lab worked example uses 4); the result is
    ``[context_len, num_kv_heads, head_dim]``.  Walks the block table one
    logical block at a time (page-3 "注意力计算的改写": ``for block_idx,
    physical_block_id in enumerate(block_table[request_id])``) and copies the
    tokens of that block that lie below ``context_len``.
    """
    num_kv_heads, block_size, head_dim = cache.shape[1], cache.shape[2], cache.shape[3]
    out = np.empty((context_len, num_kv_heads, head_dim), dtype=np.float64)
    num_logical = (context_len + block_size - 1) // block_size
    for logical in range(num_logical):
        physical = int(block_table[logical])
        first = logical * block_size
        count = min(block_size, context_len - first)
        # cache[physical] is [heads, 16, d]; tokens are its middle axis.
        out[first:first + count] = np.transpose(
            cache[physical, :, :count, :], (1, 0, 2)).astype(np.float64)
    return out


def attention_one(q: np.ndarray, keys: np.ndarray, values: np.ndarray,
                  scale: float) -> np.ndarray:
    """Scaled dot-product attention of one query vector over a contiguous context.

    ``q``: ``[d]``; ``keys``, ``values``: ``[ctx, d]`` (float64).  Computes
    ``s_t = scale * q . k_t``, ``p = exp(s - max s)``, ``o = sum_t p_t v_t /
    sum_t p_t``.  An empty context (``ctx == 0``) gives the zero vector (the
    pages are silent on it; we choose zeros rather than NaN).
    """
    if keys.shape[0] == 0:
        return np.zeros(values.shape[1], dtype=np.float64)
    scores = scale * (keys @ q.astype(np.float64))
    weights = np.exp(scores - scores.max())
    return (weights @ values) / weights.sum()


def paged_attention_decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                           block_tables, context_lens, scale: float,
                           seqs=None, heads=None) -> np.ndarray:
    """Decode attention of each sequence's single new query over its paged K/V.

    ``q``: ``[num_seqs, num_q_heads, d]``; caches ``[num_blocks, num_kv_heads,
    16, d]``; ``block_tables``: ``[num_seqs, max_blocks]`` int; ``context_lens``:
    ``[num_seqs]``.  Returns float64 ``[num_seqs, num_q_heads, d]``.

    ``seqs`` / ``heads`` restrict the work to a sample (other rows stay NaN),
    so full-size workloads can be checked one output at a time.
    """
    num_seqs, num_q_heads, head_dim = q.shape
    num_kv_heads = k_cache.shape[1]
    group = num_q_heads // num_kv_heads
    out = np.full((num_seqs, num_q_heads, head_dim), np.nan, dtype=np.float64)
    seq_list = range(num_seqs) if seqs is None else seqs
    head_list = range(num_q_heads) if heads is None else heads
    for b in seq_list:
        ctx = int(context_lens[b])
        keys = gather_sequence(k_cache, block_tables[b], ctx)
        values = gather_sequence(v_cache, block_tables[b], ctx)
        for h in head_list:
            kv_head = h // group
            out[b, h] = attention_one(q[b, h].astype(np.float64),
                                      keys[:, kv_head, :], values[:, kv_head, :],
                                      scale)
    return out


def chunk_positions(context_len: int, query_len: int) -> range:
    """Token positions of a sequence's newest ``query_len`` tokens.

    A prefill chunk is the last ``query_len`` tokens of the sequence's
    ``context_len`` (their K/V already stored in the cache): positions
    ``context_len - query_len .. context_len - 1``.
    """
    return range(context_len - query_len, context_len)


def causal_prefix(buf: np.ndarray, position: int) -> np.ndarray:
    """The tokens a query at ``position`` attends: 0 .. position inclusive."""
    return buf[:position + 1]


def paged_attention_prefill(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                            block_tables, context_lens, query_start, scale: float,
                            rows=None) -> np.ndarray:
    """Chunked-prefill attention over the paged cache.

    OS-lab appendix, section 2.1: prefill writes the K/V of every prompt token
    into the cache; "vLLM: treating the KV cache as virtual memory", section
    "KV 的体积从哪来，页表如何把它切开": chunked prefill cuts a long prompt's
    computation into pieces run between decode steps.  Each query attends, as
    in any causal Transformer, over itself and the tokens before it.

    ``q``: ``[total_q, num_q_heads, d]``; the query rows of sequence ``b`` are
    ``query_start[b] .. query_start[b + 1] - 1`` (``T_b`` rows), the queries of
    its newest ``T_b`` tokens (``chunk_positions``), whose K/V are in the cache
    already, so ``T_b <= context_lens[b]``.  Query row ``i`` of sequence ``b``
    at position ``p`` attends over tokens ``0 .. p`` of the sequence
    (``causal_prefix``).  ``T_b = 1`` for every sequence is decode.  Returns
    float64 ``[total_q, num_q_heads, d]``; ``rows`` restricts the work to a
    sample of query rows (the others stay NaN).
    """
    total_q, num_q_heads, head_dim = q.shape
    num_kv_heads = k_cache.shape[1]
    group = num_q_heads // num_kv_heads
    out = np.full((total_q, num_q_heads, head_dim), np.nan, dtype=np.float64)
    wanted = None if rows is None else set(int(r) for r in rows)
    for b in range(len(context_lens)):
        first, last = int(query_start[b]), int(query_start[b + 1])
        ctx, query_len = int(context_lens[b]), last - first
        if query_len <= 0:
            continue
        if query_len > ctx:
            raise ValueError(f"sequence {b}: {query_len} queries but only {ctx} tokens")
        if wanted is not None and not any(first <= r < last for r in wanted):
            continue
        keys = gather_sequence(k_cache, block_tables[b], ctx)
        values = gather_sequence(v_cache, block_tables[b], ctx)
        for i, position in enumerate(chunk_positions(ctx, query_len)):
            row = first + i
            if wanted is not None and row not in wanted:
                continue
            k_seen = causal_prefix(keys, position)
            v_seen = causal_prefix(values, position)
            for h in range(num_q_heads):
                kv_head = h // group
                out[row, h] = attention_one(q[row, h].astype(np.float64),
                                            k_seen[:, kv_head, :], v_seen[:, kv_head, :], scale)
    return out


def attention_lse(q: np.ndarray, keys: np.ndarray, scale: float) -> float:
    """Natural-log sum-exp of the scores of one query (used by split tests)."""
    if keys.shape[0] == 0:
        return -np.inf
    scores = scale * (keys @ q.astype(np.float64))
    top = scores.max()
    return float(top + np.log(np.exp(scores - top).sum()))


def kv_append(k: np.ndarray, v: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
              slot_mapping) -> None:
    """Write each new token's K/V rows into its paged slot, in place.

    ``k``, ``v``: ``[num_tokens, num_kv_heads, d]``; ``slot_mapping[i]`` is
    ``physical_block * 16 + offset`` (page-3 block-table example).  A negative
    slot marks a padding token and is skipped (our reading).  Arrays may be any
    dtype, including ``uint16`` views of 16-bit floats, so the copy is exact.
    """
    block_size = k_cache.shape[2]
    for i, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        block, offset = slot // block_size, slot % block_size
        k_cache[block, :, offset, :] = k[i]
        v_cache[block, :, offset, :] = v[i]


def block_copy(k_caches, v_caches, src_dst_pairs) -> None:
    """Copy whole physical blocks ``src -> dst`` in every layer, in pair order.

    OS-lab appendix section 4.4: on a write into a block whose refcount is 2,
    the writer gets a fresh copy of the block; the copy covers every slot of
    the block (all 16 tokens, every KV head) and, because each layer keeps its
    own cache, every layer.
    """
    for src, dst in src_dst_pairs:
        src, dst = int(src), int(dst)
        for k_cache, v_cache in zip(k_caches, v_caches):
            k_cache[dst] = k_cache[src]
            v_cache[dst] = v_cache[src]


def block_swap(src_k_caches, src_v_caches, dst_k_caches, dst_v_caches, pairs) -> None:
    """Copy whole blocks between two tiers, in every layer, in pair order.

    "vLLM: treating the KV cache as virtual memory", section
    "调度：词一级的进入与退出": a preempted sequence's KV moves to host memory
    block by block and comes back later.  ``pairs[i] = (src, dst)``:
    ``dst_cache[dst] = src_cache[src]`` for K and V of every layer.
    """
    for src, dst in pairs:
        src, dst = int(src), int(dst)
        for sk, sv, dk, dv in zip(src_k_caches, src_v_caches, dst_k_caches, dst_v_caches):
            dk[dst] = sk[src]
            dv[dst] = sv[src]
