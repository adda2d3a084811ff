"""Iteration-level (continuous) batching over a block pool.

"留书阁 / knowledge-20" page, section on continuous batching: after every
decode step the scheduler retires finished sequences and fills their places
from the waiting queue, and a new request only needs blocks from the pool, not
a contiguous region.  "vLLM: treating the KV cache as virtual memory", section
"调度：词一级的进入与退出": a sequence can be preempted (its KV swapped to host
memory, block by block) and resumed later; section "碎片从哪里来": requests
sharing a system prompt hit the prefix cache.

This driver exercises the pool the way a serving loop does -- admissions with
prefix-cache hits, one token per running sequence per step, retirements,
preemption by swapping out, resumption by swapping in -- and reports what the
device kernels would need each step (slots, copy-on-write pairs, swap pairs),
also as one ordered list of device operations.  A prompt's appends, and a
step's appends for all running sequences, each go to the pool in one
``append_tokens`` call.  It only calls pool methods, so the native pool and a
model pool with the same methods can be driven by the same script and
compared step by step.

Policy (ours; the pages leave it to the product): first-come first-served
admission while the pool can hold the prompt's uncached blocks plus one; when
a running sequence needs a block and none is left, the most recently admitted
running sequence is preempted (swapped out if the host tier has room, else
freed and requeued for recomputation); swapped sequences resume first-in
first-out as soon as their blocks fit.
"""

from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field


@dataclass
class Request:
    rid: int
    prompt: list
    max_new_tokens: int
    seq: int = -1
    generated: int = 0
    hit_tokens: int = 0


@dataclass
class StepReport:
    """What one step asked of the device path."""
    admitted: list = field(default_factory=list)     # (request id, seq, prefix-hit tokens)
    slots: list = field(default_factory=list)        # (seq, slot) of every token appended
    cow_pairs: list = field(default_factory=list)    # (src, dst) block copies
    swap_out: list = field(default_factory=list)     # (seq, [(device, host), ...])
    swap_in: list = field(default_factory=list)      # (seq, [(host, device), ...])
    retired: list = field(default_factory=list)      # request ids
    requeued: list = field(default_factory=list)     # request ids freed for recomputation
    aborted: list = field(default_factory=list)      # (request id, seq): prompt did not fit
    # The same work as an ordered list of device operations, in the order the
    # device must apply them:
    #   ("swap_in", seq, [(host, device), ...])
    #   ("append", [(src, dst), ...], [(seq, slot, token, position), ...]):
    #       the block copies first, then every token's K/V into its slot
    #   ("swap_out", seq, [(device, host), ...])
    # Order matters: a block freed by a swap-out can be handed to a later
    # append of the same step.
    ops: list = field(default_factory=list)


class ContinuousBatcher:
    def __init__(self, pool, block_size: int, max_running: int = 256):
        """``pool``: a block pool with the native pool's methods; its
        ``append_tokens`` reports how many appends fit before it ran out of
        blocks."""
        self.pool = pool
        self.bs = block_size
        self.max_running = max_running
        self.waiting: deque[Request] = deque()
        self.swapped: deque[Request] = deque()
        self.running: list[Request] = []
        self.next_rid = 0

    def submit(self, prompt, max_new_tokens: int) -> int:
        rid = self.next_rid
        self.next_rid += 1
        self.waiting.append(Request(rid, [int(t) for t in prompt], int(max_new_tokens)))
        return rid

    def _free_blocks(self) -> int:
        st = self.pool.stats()
        return st["free_blocks"] + st.get("evictable_blocks", 0)

    def _preempt(self, rep: StepReport) -> bool:
        """Preempt the most recently admitted running sequence."""
        if not self.running:
            return False
        victim = self.running.pop()
        st = self.pool.stats()
        table, _ = self.pool.block_table(victim.seq)
        if st["host_free_blocks"] >= len(table):
            try:
                pairs = self.pool.swap_out(victim.seq)
            except Exception:  # noqa: BLE001  (shared or pinned blocks cannot leave)
                pairs = None
            if pairs is not None:
                moved = [tuple(int(x) for x in p) for p in pairs]
                rep.swap_out.append((victim.seq, moved))
                rep.ops.append(("swap_out", victim.seq, moved))
                self.swapped.append(victim)
                return True
        self.pool.free_seq(victim.seq)
        victim.seq, victim.generated = -1, 0
        rep.requeued.append(victim.rid)
        self.waiting.appendleft(victim)
        return True

    def step(self, next_token) -> StepReport:
        """One decode step: resume, admit, append a token per running sequence
        (``next_token(request)`` gives its id), retire the finished."""
        rep = StepReport()
        # resume swapped sequences first, in order
        while self.swapped and len(self.running) < self.max_running:
            req = self.swapped[0]
            table, _ = self.pool.block_table(req.seq)
            if self._free_blocks() < len(table) + 1:
                break
            pairs = [tuple(int(x) for x in p) for p in self.pool.swap_in(req.seq)]
            rep.swap_in.append((req.seq, pairs))
            rep.ops.append(("swap_in", req.seq, pairs))
            self.running.append(self.swapped.popleft())
        # admit waiting requests while their uncached blocks fit
        while self.waiting and len(self.running) < self.max_running and not self.swapped:
            req = self.waiting[0]
            need = -(-len(req.prompt) // self.bs) + 1
            if self._free_blocks() < need:
                break
            seq, hit = self.pool.new_seq_with_prompt(req.prompt)
            req.seq, req.hit_tokens = seq, hit
            rest = req.prompt[hit:]
            slots, pairs, done = self.pool.append_tokens([seq] * len(rest), rest)
            # Reported even when the prompt does not fit after all: every block
            # the partial append filled was keyed into the prefix cache and
            # stays there after the sequence is freed, so its K/V must be
            # written for a later request that hits it.
            rep.slots.extend((seq, int(s)) for s in slots)
            rep.cow_pairs.extend((int(a), int(b)) for a, b in pairs)
            rep.ops.append(("append", [(int(a), int(b)) for a, b in pairs],
                            [(seq, int(s), rest[j], hit + j) for j, s in enumerate(slots)]))
            if done < len(rest):                         # cached blocks were evicted meanwhile
                rep.aborted.append((req.rid, seq))
                self.pool.free_seq(seq)
                req.seq = -1
                break
            self.waiting.popleft()
            self.running.append(req)
            rep.admitted.append((req.rid, seq, hit))
        # one new token for every running sequence, in one pool call; where
        # the pool runs out, preempt and go on from the sequence that failed
        i = 0
        while i < len(self.running):
            batch = self.running[i:]
            tokens = [next_token(r) for r in batch]
            slots, pairs, done = self.pool.append_tokens([r.seq for r in batch], tokens)
            entries = []
            for r, s, t in zip(batch[:done], slots, tokens):
                entries.append((r.seq, int(s), t, len(r.prompt) + r.generated))
                r.generated += 1
                rep.slots.append((r.seq, int(s)))
            rep.cow_pairs.extend((int(a), int(b)) for a, b in pairs)
            rep.ops.append(("append", [(int(a), int(b)) for a, b in pairs], entries))
            i += done
            if i < len(self.running):
                req = self.running[i]
                if not self._preempt(rep) or req not in self.running:
                    if req in self.running:              # nothing left to preempt
                        raise RuntimeError("pool too small for one sequence")
        # retire the finished
        for req in [r for r in self.running if r.generated >= r.max_new_tokens]:
            self.running.remove(req)
            self.pool.free_seq(req.seq)
            rep.retired.append(req.rid)
        return rep

    @property
    def idle(self) -> bool:
        return not (self.waiting or self.swapped or self.running)
