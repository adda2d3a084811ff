"""Pure-Python model of the paged-KV block pool.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It restates the
bookkeeping the pages describe, step by step, so the native pool can be checked
against it operation by operation:

* fixed-size physical blocks in one global pool with a free list; a finished
  sequence returns its blocks to the free list ("vLLM: treating the KV cache as
  virtual memory", section "碎片从哪里来"; "留书阁 / knowledge-20" page,
  section "PagedAttention：虚实分离，按需取用");
* lazy allocation: a physical block is taken only when generation reaches the
  first slot of a new logical block (OS-lab appendix, section 3.3; same
  page-3 section: "after the first 16 tokens are full, take the next block");
* reference counts: sharing a block increments its count, finishing a holder
  decrements it, the block goes back to the free list only at zero ("第 6 章
  缓存管理", section "块表长什么样");
* fork copies the block table, not the data, and bumps every refcount
  (page 2, section "碎片从哪里来"; OS-lab appendix, section 4.3);
* copy-on-write: appending into a block whose refcount is above one first
  moves the writer onto a fresh private copy (source refcount - 1, copy
  refcount 1); the last remaining holder writes in place (OS-lab appendix,
  section 4.4; page 3, section "写时复制与前缀缓存");
* prefix sharing: a new request's table starts with the first
  ``ceil(n / block_size)`` entries of another request's table (page 4, section
  "块表长什么样": a 200-token shared prefix gives 13 shared entries);
* pinning: a prefix-cache block stays out of the free list even at refcount
  zero (page 2, section "碎片从哪里来": hot prefixes are kept outside the free
  list);
* prefix caching: a full block is keyed by its content -- the key of the block
  before it and its 16 token ids -- so a later request whose prompt starts
  with the same blocks reuses them instead of recomputing them (page 2,
  section "碎片从哪里来": the prefix cache keeps hot prefixes outside the free
  list so the next request with the same system prompt hits them; page 4,
  section "缓存放不下的时候": when memory is full, evict in least-recently-used
  order and recompute on the next use);
* swapping: a preempted sequence's KV moves to host memory block by block and
  comes back later ("vLLM: treating the KV cache as virtual memory", section
  "调度：词一级的进入与退出"; "第 6 章 缓存管理", section "缓存放不下的时候":
  spill cold cache to CPU memory).  Host blocks have their own free list.

Policy choices the pages leave open (both implementations follow them so their
tables can be compared bit for bit):

* the free list is a stack (LIFO); it starts as ``initial_order`` with
  ``initial_order[0]`` handed out first;
* freeing a sequence releases its blocks from the last logical block to the
  first;
* sequence ids count up from 0 and are never reused;
* the host tier is a second LIFO stack (``host_initial_order[0]`` first); a
  sequence swaps out only when none of its blocks is shared or pinned (a
  shared block still has a reader on the device); swapping out takes a host
  block per logical block in order, then releases the device blocks last to
  first; swapping in is the mirror image; a swapped sequence cannot append,
  fork, share or pin until it is swapped back in;
* prefix cache: the key hash is 64-bit FNV-1a over the parent key (8 bytes,
  little-endian; 0 for a sequence's first block) then the 16 token ids (int32,
  little-endian); a lookup also compares the parent block and the token ids,
  so equal hashes never alias different content.  A prompt reuses its longest
  run of leading full cached blocks, but leaves at least one token to compute
  (whose logits the caller needs).  A block is keyed when an append fills it,
  unless its key is already cached.  A keyed block whose refcount drops to
  zero goes to the back of an LRU list instead of the free list; allocation
  takes the free list first and evicts the front of the LRU list (dropping its
  key) only when the free list is empty; a hit on an LRU block takes it back
  out.
"""

from __future__ import annotations

from collections import OrderedDict
from dataclasses import dataclass, field

_FNV_OFFSET = 0xCBF29CE484222325
_FNV_PRIME = 0x100000001B3
_MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """64-bit FNV-1a (Fowler-Noll-Vo): start from the offset basis, for each
    byte xor it in, then multiply by the FNV prime modulo 2^64."""
    h = _FNV_OFFSET
    for byte in data:
        h ^= byte
        h = (h * _FNV_PRIME) & _MASK64
    return h


def block_key_hash(parent_hash: int, tokens) -> int:
    """Prefix-cache key hash of a full block: FNV-1a over the parent hash
    (8 bytes LE) and the token ids (int32 LE each)."""
    data = int(parent_hash & _MASK64).to_bytes(8, "little")
    data += b"".join(int(t & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens)
    return fnv1a64(data)


class NoBlocks(Exception):
    """The pool has no free block left (page 4, "缓存放不下的时候": reject)."""


@dataclass
class _Seq:
    table: list = field(default_factory=list)
    ctx: int = 0
    swapped: bool = False           # table holds host blocks
    tokens: list | None = None      # token ids, when known (prefix cache)
    hashes: list = field(default_factory=list)   # key hash of each keyed-or-full block


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int = 16, initial_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if initial_order is None else [int(x) for x in initial_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("initial_order must be a permutation of range(num_blocks)")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = list(reversed(order))          # top of the stack is the end
        self.refcount = [0] * num_blocks
        self.pinned = [False] * num_blocks
        self.seqs: dict[int, _Seq] = {}
        self.next_id = 0
        self.cow_copies = 0
        self.num_host_blocks = 0
        self.host_free: list[int] = []
        self.prefix_cache = False
        self.cache: dict[int, int] = {}            # key hash -> block
        self.key = [None] * num_blocks             # block -> (hash, parent block, tokens)
        self.lru: OrderedDict[int, None] = OrderedDict()   # evictable keyed blocks, oldest first
        self.hit_tokens = 0
        self.evictions = 0

    def enable_prefix_cache(self, on: bool = True) -> None:
        if self.seqs:
            raise ValueError("enable the prefix cache before the first sequence")
        self.prefix_cache = bool(on)

    def set_host_blocks(self, num_host_blocks: int, initial_order=None) -> None:
        """Give the pool a host tier of ``num_host_blocks`` blocks (swap space)."""
        if num_host_blocks < 0 or any(s.swapped for s in self.seqs.values()):
            raise ValueError("bad host block count, or sequences are swapped out")
        order = (list(range(num_host_blocks)) if initial_order is None
                 else [int(x) for x in initial_order])
        if sorted(order) != list(range(num_host_blocks)):
            raise ValueError("initial_order must be a permutation of range(num_host_blocks)")
        self.num_host_blocks = num_host_blocks
        self.host_free = list(reversed(order))

    # -- internal -----------------------------------------------------------
    def _available(self) -> int:
        return len(self.free) + len(self.lru)

    def _alloc(self) -> int:
        if self.free:
            block = self.free.pop()
        elif self.lru:
            block, _ = self.lru.popitem(last=False)      # least recently used
            del self.cache[self.key[block][0]]
            self.key[block] = None
            self.evictions += 1
        else:
            raise NoBlocks()
        self.refcount[block] = 1
        return block

    def _to_idle(self, block: int) -> None:
        """A block nobody holds: evictable when keyed, else free."""
        if self.key[block] is not None:
            self.lru[block] = None
        else:
            self.free.append(block)

    def _release(self, block: int) -> None:
        self.refcount[block] -= 1
        if self.refcount[block] == 0 and not self.pinned[block]:
            self._to_idle(block)

    def _seq(self, seq_id: int) -> _Seq:
        if seq_id not in self.seqs:
            raise KeyError(seq_id)
        return self.seqs[seq_id]

    def _resident(self, seq_id: int) -> _Seq:
        seq = self._seq(seq_id)
        if seq.swapped:
            raise ValueError("sequence is swapped out")
        return seq

    # -- operations ---------------------------------------------------------
    def new_seq(self) -> int:
        seq_id = self.next_id
        self.next_id += 1
        self.seqs[seq_id] = _Seq()
        return seq_id

    def append_slot(self, seq_id: int):
        """Reserve the slot of the sequence's next token.

        Returns ``(slot, cow)`` where ``slot = physical * block_size + offset``
        and ``cow`` is ``(src, dst)`` when a copy-on-write happened, else None.
        """
        seq = self._resident(seq_id)
        logical, offset = divmod(seq.ctx, self.block_size)
        cow = None
        if offset == 0:
            block = self._alloc()
            seq.table.append(block)
        else:
            block = seq.table[logical]
            if self.refcount[block] > 1:
                fresh = self._alloc()
                self.refcount[block] -= 1
                seq.table[logical] = fresh
                cow = (block, fresh)
                self.cow_copies += 1
                block = fresh
        seq.ctx += 1
        if seq.tokens is not None:
            seq.tokens = None          # the content of the new slot is unknown
        return block * self.block_size + offset, cow

    def new_seq_with_prompt(self, tokens):
        """A new sequence for a prompt: its longest run of leading full blocks
        found in the prefix cache is reused (refcount + 1).  Returns
        ``(seq_id, hit_tokens)``; the caller appends the remaining prompt tokens
        with ``append_token``."""
        tokens = [int(t) for t in tokens]
        seq_id = self.new_seq()
        seq = self.seqs[seq_id]
        seq.tokens = []
        if not self.prefix_cache:
            return seq_id, 0
        bs = self.block_size
        limit = (len(tokens) - 1) // bs if tokens else 0
        parent_hash, parent_block = 0, -1
        for i in range(limit):
            chunk = tokens[i * bs:(i + 1) * bs]
            h = block_key_hash(parent_hash, chunk)
            block = self.cache.get(h)
            if block is None or self.key[block][1] != parent_block or self.key[block][2] != tuple(chunk):
                break
            if self.refcount[block] == 0 and block in self.lru:
                del self.lru[block]
            self.refcount[block] += 1
            seq.table.append(block)
            seq.hashes.append(h)
            seq.tokens += chunk
            seq.ctx += bs
            parent_hash, parent_block = h, block
        self.hit_tokens += seq.ctx
        return seq_id, seq.ctx

    def append_token(self, seq_id: int, token: int):
        """``append_slot`` for a token whose id is known: a block it fills is
        keyed into the prefix cache.  Returns ``(slot, cow)``."""
        seq = self._resident(seq_id)
        known = seq.tokens
        slot, cow = self.append_slot(seq_id)
        if known is None:
            return slot, cow
        known.append(int(token))
        seq.tokens = known
        bs = self.block_size
        if self.prefix_cache and seq.ctx % bs == 0:
            i = seq.ctx // bs - 1
            parent_hash = seq.hashes[i - 1] if i > 0 else 0
            parent_block = seq.table[i - 1] if i > 0 else -1
            chunk = tuple(known[i * bs:(i + 1) * bs])
            h = block_key_hash(parent_hash, chunk)
            seq.hashes.append(h)
            block = seq.table[i]
            if h not in self.cache and self.key[block] is None:
                self.cache[h] = block
                self.key[block] = (h, parent_block, chunk)
        return slot, cow

    def append_tokens(self, seqs, tokens):
        """``append_token(seqs[i], tokens[i])`` for every i in order, stopping
        where the pool runs out of blocks.  Returns (slots, copy pairs, number
        of appends made), the native pool's batched form."""
        slots, pairs, done = [], [], 0
        for seq_id, token in zip(seqs, tokens):
            try:
                slot, cow = self.append_token(int(seq_id), int(token))
            except NoBlocks:
                break
            slots.append(slot)
            if cow is not None:
                pairs.append(cow)
            done += 1
        return slots, pairs, done

    def fork(self, parent_id: int) -> int:
        parent = self._resident(parent_id)
        child_id = self.new_seq()
        child = self.seqs[child_id]
        child.table = list(parent.table)
        child.ctx = parent.ctx
        child.tokens = None if parent.tokens is None else list(parent.tokens)
        child.hashes = list(parent.hashes)
        for block in child.table:
            self.refcount[block] += 1
        return child_id

    def share_prefix(self, src_id: int, dst_id: int, num_tokens: int) -> None:
        src, dst = self._resident(src_id), self._resident(dst_id)
        if dst.ctx != 0 or dst.table:
            raise ValueError("destination must be an empty sequence")
        if num_tokens <= 0 or num_tokens > src.ctx:
            raise ValueError("num_tokens must be in 1..src context length")
        count = -(-num_tokens // self.block_size)
        dst.table = list(src.table[:count])
        dst.ctx = num_tokens
        dst.tokens = None if src.tokens is None else list(src.tokens[:num_tokens])
        dst.hashes = list(src.hashes[:num_tokens // self.block_size])
        for block in dst.table:
            self.refcount[block] += 1

    def pin(self, seq_id: int, num_tokens: int) -> None:
        seq = self._resident(seq_id)
        if num_tokens < 0 or num_tokens > seq.ctx:
            raise ValueError("num_tokens must be in 0..context length")
        for block in seq.table[:-(-num_tokens // self.block_size)]:
            self.pinned[block] = True

    def unpin(self, block: int) -> None:
        if not self.pinned[block]:
            raise ValueError("block is not pinned")
        self.pinned[block] = False
        if self.refcount[block] == 0:
            self._to_idle(block)

    def free_seq(self, seq_id: int) -> None:
        seq = self._seq(seq_id)
        for block in reversed(seq.table):
            if seq.swapped:
                self.host_free.append(block)
            else:
                self._release(block)
        del self.seqs[seq_id]

    def swap_out(self, seq_id: int):
        """Move a sequence's blocks to the host tier.  Returns the copy pairs
        ``(device_block, host_block)`` in logical order (copy them before the
        device blocks are written again)."""
        seq = self._resident(seq_id)
        if any(self.refcount[b] != 1 or self.pinned[b] for b in seq.table):
            raise ValueError("a shared or pinned block cannot be swapped out")
        if len(seq.table) > len(self.host_free):
            raise NoBlocks()
        host = [self.host_free.pop() for _ in seq.table]
        pairs = list(zip(seq.table, host))
        for block in reversed(seq.table):
            self._release(block)
        seq.table = host
        seq.swapped = True
        return pairs

    def swap_in(self, seq_id: int):
        """Bring a swapped sequence back.  Returns the copy pairs
        ``(host_block, device_block)`` in logical order."""
        seq = self._seq(seq_id)
        if not seq.swapped:
            raise ValueError("sequence is not swapped out")
        if len(seq.table) > self._available():
            raise NoBlocks()
        dev = [self._alloc() for _ in seq.table]
        pairs = list(zip(seq.table, dev))
        for block in reversed(seq.table):
            self.host_free.append(block)
        seq.table = dev
        seq.swapped = False
        return pairs

    def is_swapped(self, seq_id: int) -> bool:
        return self._seq(seq_id).swapped

    # -- queries ------------------------------------------------------------
    def block_table(self, seq_id: int):
        seq = self._seq(seq_id)
        return list(seq.table), seq.ctx

    def stats(self) -> dict:
        live = self.seqs.values()
        return {
            "num_blocks": self.num_blocks,
            "free_blocks": len(self.free),
            "used_blocks": sum(1 for rc in self.refcount if rc > 0),
            "pinned_blocks": sum(1 for p in self.pinned if p),
            "shared_blocks": sum(1 for rc in self.refcount if rc > 1),
            "cow_copies": self.cow_copies,
            "live_seqs": len(self.seqs),
            "tokens": sum(s.ctx for s in live),
            "internal_frag_slots": sum(len(s.table) * self.block_size - s.ctx for s in live),
            "host_blocks": self.num_host_blocks,
            "host_free_blocks": len(self.host_free),
            "swapped_seqs": sum(1 for s in live if s.swapped),
            "cached_blocks": len(self.cache),
            "evictable_blocks": len(self.lru),
            "prefix_hit_tokens": self.hit_tokens,
            "evictions": self.evictions,
        }
