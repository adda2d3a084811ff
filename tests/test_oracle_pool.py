"""Pins for the Python block-pool model against the pages' worked examples and
the bookkeeping invariants the pages state."""

import numpy as np
import pytest

import oracle.attention as oa
from oracle.pool import BlockPool, NoBlocks
from tests.conftest import golden


def prefill(pool, seq, n):
    slots = []
    for _ in range(n):
        slot, cow = pool.append_slot(seq)
        assert cow is None
        slots.append(slot)
    return slots


def test_oslab_cow_example_block4():
    """OS-lab appendix 4.4 with real data: tokens are written through slots,
    the copy is applied through the block-copy oracle, and each branch reads
    its own fourth token afterwards."""
    g = golden("cow_examples.json")["oslab_block4"]
    bs = g["block_size"]
    vocab = {w: i + 1 for i, w in enumerate(g["prefix_tokens"] + ["fathers", "mothers"])}
    pool = BlockPool(8, block_size=bs)
    cache_k = np.zeros((8, 1, bs, 1))
    cache_v = np.zeros((8, 1, bs, 1))

    def write(slot, word):
        blk, off = divmod(slot, bs)
        cache_k[blk, 0, off, 0] = vocab[word]

    a1 = pool.new_seq()
    for w in g["prefix_tokens"]:
        slot, _ = pool.append_slot(a1)
        write(slot, w)
    a2 = pool.fork(a1)
    table, _ = pool.block_table(a1)
    assert pool.refcount[table[0]] == g["block0_refcount_after_fork"]
    assert pool.refcount[table[1]] == g["block1_refcount_after_fork"]

    slot, cow = pool.append_slot(a1)                 # A1 writes 'fathers'
    assert cow is not None and cow[0] == table[1]
    oa.block_copy([cache_k], [cache_v], [cow])
    write(slot, "fathers")
    assert pool.cow_copies == g["a1_copies"]
    assert pool.refcount[table[1]] == g["block1_refcount_after_a1_write"]

    slot, cow = pool.append_slot(a2)                 # A2 writes 'mothers' in place
    assert cow is None and slot // bs == table[1]
    write(slot, "mothers")
    assert pool.cow_copies == g["a1_copies"] + g["a2_copies"]

    inv = {i: w for w, i in vocab.items()}
    for seq, expect in ((a1, g["a1_block1_contents"]), (a2, g["a2_block1_contents"])):
        t, ctx = pool.block_table(seq)
        got = oa.gather_sequence(cache_k, t, ctx)[:, 0, 0]
        assert [inv[int(x)] for x in got[4:8]] == expect
        assert [inv[int(x)] for x in got[:4]] == g["prefix_tokens"][:4]
    # block 0 stayed shared, never copied
    assert pool.block_table(a1)[0][0] == pool.block_table(a2)[0][0]
    assert pool.refcount[table[0]] == 2


def test_beam_cow_example():
    g = golden("cow_examples.json")["beam4"]
    pool = BlockPool(64)
    beam0 = pool.new_seq()
    prefill(pool, beam0, 100)                        # first 100 tokens shared
    beams = [beam0] + [pool.fork(beam0) for _ in range(g["beams"] - 1)]
    shared = pool.block_table(beam0)[0][-1]          # partially filled last block
    assert pool.refcount[shared] == g["shared_refcount"]
    _, cow = pool.append_slot(beams[0])
    assert cow[0] == shared
    assert pool.refcount[shared] == g["after_first_write"]["shared_refcount"]
    assert pool.refcount[cow[1]] == g["after_first_write"]["copy_refcount"]
    # the other beams copy in turn until the last holder writes in place
    copies = [pool.append_slot(b)[1] for b in beams[1:]]
    assert [c is not None for c in copies] == [True, True, False]
    assert pool.refcount[shared] == 1


def test_share_prefix_example():
    g = golden("cow_examples.json")["share_200_of_500"]
    pool = BlockPool(128)
    r1 = pool.new_seq()
    prefill(pool, r1, g["first_tokens"])
    t1, _ = pool.block_table(r1)
    assert len(t1) == g["first_blocks"]
    assert all(pool.refcount[b] == g["refcount_before"] for b in t1)
    r2 = pool.new_seq()
    pool.share_prefix(r1, r2, g["shared_tokens"])
    t2, ctx2 = pool.block_table(r2)
    assert len(t2) == g["shared_entries"] and t2 == t1[:g["shared_entries"]]
    assert ctx2 == g["shared_tokens"]
    assert all(pool.refcount[b] == g["refcount_shared"] for b in t2)
    # r2's first append lands in the shared, partially used 13th block -> CoW
    _, cow = pool.append_slot(r2)
    assert cow is not None and cow[0] == t1[12]
    free_before = len(pool.free)
    pool.free_seq(r1)
    assert all(pool.refcount[b] == g["refcount_after_one_ends"] for b in t2[:12])
    # r1's private blocks (20 of them, plus the 13th it kept) went back
    assert len(pool.free) == free_before + (32 - 12)
    pool.free_seq(r2)
    assert len(pool.free) == 128 and all(rc == 0 for rc in pool.refcount)


def test_slot_example_lazy_allocation():
    """OS-lab 3.2 requests A (10 slots) and B (5 slots): under lazy paged
    allocation each holds one 16-slot block instead of 2048 / 512 slots."""
    g = golden("fragmentation.json")
    pool = BlockPool(8)
    a, b = pool.new_seq(), pool.new_seq()
    prefill(pool, a, g["request_A"]["used"])
    prefill(pool, b, g["request_B"]["used"])
    s = pool.stats()
    assert s["used_blocks"] == 2
    assert s["internal_frag_slots"] == (16 - 10) + (16 - 5)


def test_lazy_allocation_at_block_boundary():
    pool = BlockPool(4)
    s = pool.new_seq()
    used = []
    for t in range(33):
        pool.append_slot(s)
        used.append(pool.stats()["used_blocks"])
    assert used[0] == 1 and used[15] == 1 and used[16] == 2 and used[31] == 2 and used[32] == 3


def test_exhaustion_raises_and_leaves_state():
    pool = BlockPool(2)
    s = pool.new_seq()
    prefill(pool, s, 20)
    c = pool.fork(s)
    before = (list(pool.free), list(pool.refcount), pool.block_table(c))
    with pytest.raises(NoBlocks):
        pool.append_slot(c)                           # needs a CoW copy, none free
    assert (list(pool.free), list(pool.refcount), pool.block_table(c)) == before


def test_pinned_prefix_stays_out_of_free_list():
    pool = BlockPool(16)
    owner = pool.new_seq()
    prefill(pool, owner, 32)
    pool.pin(owner, 32)
    reqs = [pool.new_seq() for _ in range(3)]
    for r in reqs:
        pool.share_prefix(owner, r, 32)
    pool.free_seq(owner)
    prefix = pool.block_table(reqs[0])[0]
    assert all(pool.refcount[b] == 3 for b in prefix)
    for r in reqs:
        pool.free_seq(r)
    assert all(pool.refcount[b] == 0 for b in prefix)
    assert not any(b in pool.free for b in prefix)
    assert pool.stats()["pinned_blocks"] == 2
    for b in prefix:
        pool.unpin(b)
    assert len(pool.free) == 16


def random_ops(pool, gen, n_ops):
    """Random fork / append / share / free mix; checks invariants as it goes."""
    live = []
    log = []
    for _ in range(n_ops):
        op = gen.integers(0, 10)
        try:
            if op < 2 or not live:
                s = pool.new_seq()
                live.append(s)
                log.append(("new", s))
            elif op < 7:
                s = live[gen.integers(len(live))]
                log.append(("append", s, pool.append_slot(s)))
            elif op < 8:
                s = live[gen.integers(len(live))]
                c = pool.fork(s)
                live.append(c)
                log.append(("fork", s, c))
            elif op < 9:
                src = live[gen.integers(len(live))]
                ctx = pool.block_table(src)[1]
                if ctx > 0:
                    d = pool.new_seq()
                    live.append(d)
                    n = int(gen.integers(1, ctx + 1))
                    pool.share_prefix(src, d, n)
                    log.append(("share", src, d, n))
            else:
                s = live.pop(gen.integers(len(live)))
                pool.free_seq(s)
                log.append(("free", s))
        except NoBlocks:
            log.append(("noblocks",))
        check_invariants(pool)
    return log


def check_invariants(pool):
    # a block is free iff refcount 0 and not pinned; no duplicates on the list
    assert len(set(pool.free)) == len(pool.free)
    for b in range(pool.num_blocks):
        on_free = b in pool.free
        assert on_free == (pool.refcount[b] == 0 and not pool.pinned[b])
    # sum of refcounts == total table entries over live sequences
    assert sum(pool.refcount) == sum(len(s.table) for s in pool.seqs.values())
    for s in pool.seqs.values():
        assert len(s.table) == -(-s.ctx // pool.block_size)


def test_random_ops_keep_invariants():
    gen = np.random.default_rng(123)
    pool = BlockPool(40, initial_order=gen.permutation(40))
    log = random_ops(pool, gen, 1500)
    assert any(e[0] == "noblocks" for e in log)
    assert any(e[0] == "append" and e[2][1] is not None for e in log)


def test_write_never_lands_in_shared_block():
    """After append_slot returns, the block written holds refcount 1."""
    gen = np.random.default_rng(7)
    pool = BlockPool(64)
    seqs = [pool.new_seq()]
    prefill(pool, seqs[0], 21)
    for _ in range(5):
        seqs.append(pool.fork(seqs[gen.integers(len(seqs))]))
    for _ in range(200):
        s = seqs[gen.integers(len(seqs))]
        slot, _ = pool.append_slot(s)
        assert pool.refcount[slot // 16] == 1


def test_swap_out_and_in_keep_the_sequence():
    """Swapping (vLLM-VM, section "调度：词一级的进入与退出"): the device blocks
    go back to the free list, the sequence keeps its length and its logical
    order, and coming back it gets device blocks again."""
    pool = BlockPool(10, 16, list(range(10)))
    pool.set_host_blocks(6, list(range(6)))
    a = pool.new_seq()
    for _ in range(40):
        pool.append_slot(a)
    dev_table, ctx = pool.block_table(a)
    pairs = pool.swap_out(a)
    assert [d for d, _ in pairs] == dev_table
    assert all(pool.refcount[b] == 0 for b in dev_table)
    assert pool.stats()["free_blocks"] == 10 and pool.stats()["host_free_blocks"] == 3
    assert pool.block_table(a) == ([h for _, h in pairs], ctx) and pool.is_swapped(a)
    back = pool.swap_in(a)
    assert [h for h, _ in back] == [h for _, h in pairs]
    table, ctx2 = pool.block_table(a)
    assert ctx2 == ctx and len(table) == len(dev_table) and not pool.is_swapped(a)
    assert all(pool.refcount[b] == 1 for b in table)
    assert pool.stats()["host_free_blocks"] == 6
    pool.append_slot(a)                          # resident again: appends work
    assert pool.block_table(a)[1] == ctx + 1


def test_swap_refuses_shared_and_pinned_blocks():
    import pytest
    pool = BlockPool(10, 16)
    pool.set_host_blocks(10)
    a = pool.new_seq()
    for _ in range(20):
        pool.append_slot(a)
    b = pool.fork(a)
    with pytest.raises(ValueError):
        pool.swap_out(a)                         # a reader remains on the device
    pool.free_seq(b)
    pool.pin(a, 16)
    with pytest.raises(ValueError):
        pool.swap_out(a)
    c = pool.new_seq()
    pool.append_slot(c)
    pool.swap_out(c)
    for op in (lambda: pool.append_slot(c), lambda: pool.fork(c), lambda: pool.pin(c, 0)):
        with pytest.raises(ValueError):
            op()
    pool.free_seq(c)                             # host block goes back
    assert pool.stats()["host_free_blocks"] == 10


# ------------------------------------------------------------- prefix cache
def test_fnv1a64_published_vectors():
    """The hash the prefix cache keys blocks with, against the FNV-1a 64-bit
    test vectors of its authors."""
    from oracle.pool import fnv1a64
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def _prompt_pool(num_blocks=64):
    pool = BlockPool(num_blocks, 16)
    pool.enable_prefix_cache()
    return pool


def _run_prompt(pool, tokens):
    seq, hit = pool.new_seq_with_prompt(tokens)
    for t in tokens[hit:]:
        pool.append_token(seq, t)
    return seq, hit


def test_prefix_cache_share_200_of_500():
    """Page 4, section "块表长什么样": a 500-token request, then one whose first
    200 tokens are the same.  Content-keyed caching serves the 12 full shared
    blocks (192 tokens); the 13th, partly shared block is recomputed (sharing
    it as a partial block is what share_prefix does instead)."""
    pool = _prompt_pool()
    system = list(range(1000, 1200))
    first = system + list(range(300))
    s1, hit1 = _run_prompt(pool, first)
    assert hit1 == 0 and len(pool.block_table(s1)[0]) == 32
    second = system + list(range(5000, 5100))
    s2, hit2 = _run_prompt(pool, second)
    assert hit2 == 192
    t1, t2 = pool.block_table(s1)[0], pool.block_table(s2)[0]
    assert t2[:12] == t1[:12] and t2[12] != t1[12]
    assert all(pool.refcount[b] == 2 for b in t1[:12])
    assert pool.stats()["prefix_hit_tokens"] == 192


def test_prefix_cache_hot_system_prompt_survives_its_request():
    """Page 2, section "碎片从哪里来": the prefix cache keeps a hot prefix
    outside the free list, so the next request with the same system prompt
    hits it even after the first one finished."""
    pool = _prompt_pool()
    system = list(range(64))                     # 4 full blocks
    a, _ = _run_prompt(pool, system + [7, 8, 9])
    blocks = pool.block_table(a)[0][:4]
    pool.free_seq(a)
    assert all(pool.refcount[b] == 0 for b in blocks)
    assert pool.stats()["evictable_blocks"] >= 4 and pool.stats()["cached_blocks"] >= 4
    b, hit = _run_prompt(pool, system + [1, 2])
    assert hit == 64 and pool.block_table(b)[0][:4] == blocks
    # at least one token is always left to compute
    c, hit_c = _run_prompt(pool, system)
    assert hit_c == 48


def test_prefix_cache_evicts_least_recently_used():
    """Page 4, section "缓存放不下的时候": when memory is full, evict in
    least-recently-used order."""
    pool = _prompt_pool(num_blocks=9)
    seqs = [_run_prompt(pool, [100 * p + i for i in range(33)])[0] for p in range(3)]
    assert pool.stats()["free_blocks"] == 0 and pool.stats()["cached_blocks"] == 6
    tables = [pool.block_table(s)[0] for s in seqs]
    for s in (seqs[1], seqs[0], seqs[2]):        # each releases its blocks last to first
        pool.free_seq(s)
    # LRU order now: seq 1 block 1, seq 1 block 0, seq 0 block 1, ...; the
    # three partial (unkeyed) blocks are on the free list
    d = pool.new_seq()
    for _ in range(4 * 16):                      # 3 free blocks, then one eviction
        pool.append_slot(d)
    assert pool.stats()["evictions"] == 1
    assert tables[1][1] in pool.block_table(d)[0]
    s0, hit0 = pool.new_seq_with_prompt([i for i in range(33)])
    s1, hit1 = pool.new_seq_with_prompt([100 + i for i in range(33)])
    assert hit0 == 32 and pool.block_table(s0)[0] == tables[0][:2]
    assert hit1 == 16 and pool.block_table(s1)[0] == tables[1][:1]


def test_prefix_cache_equal_hashes_do_not_alias(monkeypatch):
    """Keys compare the parent block and the token ids as well as the hash, so
    even a total hash collision never serves another prompt's blocks."""
    import oracle.pool as op
    monkeypatch.setattr(op, "block_key_hash", lambda parent, tokens: 42)
    pool = _prompt_pool()
    _run_prompt(pool, list(range(40)))
    s, hit = _run_prompt(pool, list(range(500, 540)))
    assert hit == 0
    # only the first block could be keyed (a key is never duplicated), and it
    # still serves the prompt that really owns it
    s2, hit2 = _run_prompt(pool, list(range(40)))
    assert hit2 == 16
