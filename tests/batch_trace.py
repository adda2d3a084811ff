"""A continuous-batching trace applied to paged KV caches.

The batcher (``batching.ContinuousBatcher``) runs a request stream over the
native pool with the prefix cache and a host tier; each step's ordered device
operations (swap-in, copy-on-write copies, token appends, swap-out) are applied
to caches.  ``HostTiers`` applies them with the oracle's copies to host
arrays; the GPU test applies the same operations with the device kernels and
keeps a ``HostTiers`` beside them as the mirror.

Every token's K/V is a fixed function of (layer, K or V, token id, position),
so a sequence's cache content is known in closed form: whatever path its
blocks took (prefix-cache hits, eviction and recomputation, a trip through
host memory), gathering its table must give exactly those rows.

Sources: "留书阁 / knowledge-20" page, continuous-batching passage (the
scheduler refills the batch every step); "vLLM: treating the KV cache as
virtual memory", sections "调度：词一级的进入与退出" (preempted KV goes to host
memory and back) and "碎片从哪里来" (hot prefixes stay cached); "第 6 章
缓存管理", section "缓存放不下的时候" (evict least recently used, recompute).
"""

from __future__ import annotations

import numpy as np
import torch

import oracle.attention as oa

BS = 16
LAYERS, HQ, HKV, D = 2, 8, 2, 64


def kv_rows(layer: int, kind: int, tokens, positions) -> np.ndarray:
    """bf16 bit patterns ([n, HKV, D] uint16) of the K (kind 0) or V (kind 1)
    rows of the given tokens at the given positions."""
    t = np.asarray(tokens, dtype=np.float64)[:, None, None]
    p = np.asarray(positions, dtype=np.float64)[:, None, None]
    h = np.arange(HKV, dtype=np.float64)[None, :, None]
    j = np.arange(D, dtype=np.float64)[None, None, :]
    x = np.sin(t * 0.7071067 + p * 0.3183098 + h * 1.618034 + j * 0.5772157
               + layer * 2.7182818 + kind * 1.4142136)
    bf = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    return bf.view(torch.int16).numpy().view(np.uint16)


def bits_to_float(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def request_stream(seed: int, n_requests: int, vocab: int = 5_000):
    """Requests on three shared system prompts (48, 100 and 200 tokens) with
    lognormal suffixes (median 24, clipped to [1, 120]) and U{16..96} new
    tokens; returns (prompt, max_new_tokens) pairs."""
    gen = np.random.default_rng(seed)
    systems = [list(range(100_000 * (k + 1), 100_000 * (k + 1) + n))
               for k, n in enumerate((48, 100, 200))]
    reqs = []
    for _ in range(n_requests):
        sfx = int(np.clip(round(np.exp(gen.normal(np.log(24), 1.0))), 1, 120))
        prompt = systems[int(gen.integers(3))] + [int(x) for x in gen.integers(0, vocab, sfx)]
        reqs.append((prompt, int(gen.integers(16, 97))))
    return reqs


def next_token(req) -> int:
    """The token a request generates next: a function of the request and how
    many it has generated, so a recomputed request replays the same ids."""
    return (req.rid * 7919 + req.generated * 104729) % 5_000


class HostTiers:
    """Device-tier and host-tier caches as host arrays (bf16 bit patterns),
    written only through the oracle's copy functions."""

    def __init__(self, num_blocks: int, num_host_blocks: int):
        shape = (num_blocks, HKV, BS, D)
        hshape = (max(num_host_blocks, 1), HKV, BS, D)
        # unused slots hold a pattern no token row produces
        self.k = [np.full(shape, 0x7FC1, dtype=np.uint16) for _ in range(LAYERS)]
        self.v = [np.full(shape, 0x7FC2, dtype=np.uint16) for _ in range(LAYERS)]
        self.hk = [np.full(hshape, 0x7FC3, dtype=np.uint16) for _ in range(LAYERS)]
        self.hv = [np.full(hshape, 0x7FC4, dtype=np.uint16) for _ in range(LAYERS)]

    def apply(self, op) -> None:
        kind = op[0]
        if kind == "swap_in":
            oa.block_swap(self.hk, self.hv, self.k, self.v, op[2])
        elif kind == "swap_out":
            oa.block_swap(self.k, self.v, self.hk, self.hv, op[2])
        else:
            pairs, entries = op[1], op[2]
            oa.block_copy(self.k, self.v, pairs)
            if entries:
                toks = [e[2] for e in entries]
                pos = [e[3] for e in entries]
                slots = [e[1] for e in entries]
                for layer in range(LAYERS):
                    oa.kv_append(kv_rows(layer, 0, toks, pos), kv_rows(layer, 1, toks, pos),
                                 self.k[layer], self.v[layer], slots)


def sequence_tokens(req) -> list:
    """Token ids of a running request's sequence: its prompt, then what it
    generated."""
    return list(req.prompt) + [(req.rid * 7919 + g * 104729) % 5_000
                               for g in range(req.generated)]


def check_running_contents(batcher, pool, tiers: HostTiers) -> int:
    """Every running sequence's table gathers exactly its tokens' rows, in
    every layer, K and V.  Returns the number of tokens checked."""
    checked = 0
    for req in batcher.running:
        table, ctx = pool.block_table(req.seq)
        toks = sequence_tokens(req)
        assert ctx == len(toks), (req.rid, ctx, len(toks))
        pos = np.arange(ctx)
        for layer in range(LAYERS):
            for kind, cache in ((0, tiers.k[layer]), (1, tiers.v[layer])):
                got = cache[np.asarray(table)[pos // BS], :, pos % BS, :]
                want = kv_rows(layer, kind, toks, pos)
                assert np.array_equal(got, want), (
                    f"request {req.rid} (seq {req.seq}) layer {layer} kind {kind}: "
                    f"{int((got != want).any(axis=(1, 2)).sum())} of {ctx} rows wrong")
        checked += ctx
    return checked


class RekeyWatch:
    """Finds prefix-cache hits served by a physical block that earlier held
    another block's content (it was evicted, reused, then keyed again)."""

    def __init__(self):
        self.content = {}      # block -> (token ids, start position) of its keyed content
        self.rekeyed_hits = 0

    def admitted(self, batcher, pool, rep) -> None:
        by_rid = {r.rid: r for r in batcher.running}
        for rid, seq, hit in rep.admitted:
            req = by_rid.get(rid)
            if req is None:
                continue
            table, _ = pool.block_table(seq)
            for lb in range(hit // BS):
                ident = (tuple(req.prompt[:(lb + 1) * BS]), lb)
                old = self.content.get(table[lb])
                if old is not None and old != ident:
                    self.rekeyed_hits += 1
                self.content[table[lb]] = ident

    def filled(self, batcher, pool) -> None:
        """Record the content of every full block of the running sequences."""
        for req in batcher.running:
            table, ctx = pool.block_table(req.seq)
            toks = sequence_tokens(req)
            for lb in range(ctx // BS):
                self.content[table[lb]] = (tuple(toks[:(lb + 1) * BS]), lb)


class ShortPool:
    """The native pool, except that the first ``shorts`` prompt appends of
    more than 40 tokens stop 7 tokens early, as a pool that ran out of blocks
    would.  The batcher then frees the sequence and requeues the request; the
    full blocks the partial append wrote stay in the prefix cache, and the
    request's next admission hits them."""

    def __init__(self, pool, shorts: int):
        self._pool = pool
        self.shorts = shorts

    def append_tokens(self, seqs, tokens):
        seqs, tokens = list(seqs), list(tokens)
        if self.shorts > 0 and len(seqs) > 40 and len(set(seqs)) == 1:
            self.shorts -= 1
            slots, pairs, done = self._pool.append_tokens(seqs[:-7], tokens[:-7])
            return slots, pairs, done
        return self._pool.append_tokens(seqs, tokens)

    def __getattr__(self, name):
        return getattr(self._pool, name)


def run_trace(seed: int, num_blocks: int, host_blocks: int, n_requests: int, max_steps: int,
              apply_op, after_step=None, max_running: int = 32, short_admissions: int = 0):
    """Drive one request stream through the batcher on the native pool.

    ``apply_op(op)`` is called for each device operation in order;
    ``after_step(step, batcher, pool, report)`` after each step;
    ``short_admissions`` prompt appends are cut short (``ShortPool``).
    Returns (batcher, pool, statistics)."""
    from pagedattention_decode_attention_gb300 import BlockPool
    from pagedattention_decode_attention_gb300.batching import ContinuousBatcher
    pool = BlockPool(num_blocks, BS, np.random.default_rng(seed).permutation(num_blocks))
    pool.enable_prefix_cache()
    pool.set_host_blocks(host_blocks, np.random.default_rng(seed + 1).permutation(host_blocks))
    if short_admissions:
        pool = ShortPool(pool, short_admissions)
    batcher = ContinuousBatcher(pool, BS, max_running=max_running)
    pending = request_stream(seed, n_requests)
    arrivals = np.random.default_rng(seed + 2).integers(0, 4, size=max_steps)
    watch = RekeyWatch()
    stats = dict(steps=0, swap_out=0, swap_in=0, requeued=0, cow=0, aborted_admissions=0)
    for step in range(max_steps):
        for _ in range(int(arrivals[step])):
            if pending:
                batcher.submit(*pending.pop(0))
        rep = batcher.step(next_token)
        for op in rep.ops:
            apply_op(op)
        watch.admitted(batcher, pool, rep)
        watch.filled(batcher, pool)
        stats["steps"] += 1
        stats["swap_out"] += len(rep.swap_out)
        stats["swap_in"] += len(rep.swap_in)
        stats["requeued"] += len(rep.requeued)
        stats["cow"] += len(rep.cow_pairs)
        stats["aborted_admissions"] += len(rep.aborted)
        if after_step is not None:
            after_step(step, batcher, pool, rep)
        if not pending and batcher.idle:
            break
    st = pool.stats()
    stats.update(evictions=st["evictions"], prefix_hit_tokens=st["prefix_hit_tokens"],
                 rekeyed_hits=watch.rekeyed_hits)
    return batcher, pool, stats
