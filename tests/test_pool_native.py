"""The native (C++) block pool against the Python pool model and the pages'
worked examples (CPU only: the pool touches no device memory)."""

import os

import numpy as np
import pytest

from oracle.pool import BlockPool as ModelPool, NoBlocks
from tests.conftest import golden


@pytest.fixture(scope="module", autouse=True)
def built():
    from pagedattention_decode_attention_gb300 import build, capi
    if not os.path.exists(capi.LIB_PATH):
        build.build()


def native(num_blocks, block_size=16, initial_order=None):
    from pagedattention_decode_attention_gb300 import BlockPool
    return BlockPool(num_blocks, block_size, initial_order)


def is_no_blocks(exc):
    from pagedattention_decode_attention_gb300.capi import PA_ERR_NO_BLOCKS, PagedAttnError
    return isinstance(exc, PagedAttnError) and exc.status == PA_ERR_NO_BLOCKS


def replay(pool, ops, is_native):
    """Apply an op script; return every observable result."""
    out = []
    for op in ops:
        kind = op[0]
        try:
            if kind == "new":
                out.append(("new", pool.new_seq()))
            elif kind == "append":
                slot, cow = pool.append_slot(op[1])
                out.append(("append", slot, None if cow is None else tuple(int(x) for x in cow)))
            elif kind == "tokens":
                slots, pairs, done = pool.append_tokens(op[1], op[2])
                out.append(("tokens", [int(x) for x in slots],
                            [tuple(int(v) for v in p) for p in pairs], done))
            elif kind == "fork":
                out.append(("fork", pool.fork(op[1])))
            elif kind == "share":
                pool.share_prefix(op[1], op[2], op[3])
                out.append(("share",))
            elif kind == "free":
                pool.free_seq(op[1])
                out.append(("free",))
            elif kind == "pin":
                pool.pin(op[1], op[2])
                out.append(("pin",))
            elif kind in ("swapout", "swapin"):
                pairs = pool.swap_out(op[1]) if kind == "swapout" else pool.swap_in(op[1])
                out.append((kind, [tuple(int(x) for x in p) for p in pairs]))
        except Exception as e:  # noqa: BLE001
            if isinstance(e, NoBlocks) or (is_native and is_no_blocks(e)):
                out.append(("noblocks",))
            else:
                raise
    return out


def _can_swap_out(model, s):
    table, _ = model.block_table(s)
    return (all(model.refcount[b] == 1 and not model.pinned[b] for b in table)
            and len(table) <= len(model.host_free))


def random_script(gen, n_ops, model, swaps=False):
    """Random op script, generated against the model pool so every op is legal
    (with ``swaps``, sequences also move to and from the host tier)."""
    ops, live = [], []
    for _ in range(n_ops):
        r = gen.integers(0, 22 if swaps else 20)
        if r < 3 or not live:
            ops.append(("new",))
            live.append(model.new_seq())
            continue
        s = live[gen.integers(len(live))]
        if model.is_swapped(s):
            if r < 20 and len(model.block_table(s)[0]) <= len(model.free):
                ops.append(("swapin", s))
                model.swap_in(s)
            elif r >= 20:
                live.remove(s)
                ops.append(("free", s))
                model.free_seq(s)
            continue
        if r >= 20:
            if _can_swap_out(model, s):
                ops.append(("swapout", s))
                model.swap_out(s)
            continue
        if r < 12:
            ops.append(("append", s))
            try:
                model.append_slot(s)
            except NoBlocks:
                pass
        elif r < 14:                                  # a batch over resident sequences
            resident = [x for x in live if not model.is_swapped(x)]
            k = int(gen.integers(1, 7))
            seqs = [resident[int(i)] for i in gen.integers(len(resident), size=k)]
            toks = [int(t) for t in gen.integers(0, 50_000, size=k)]
            ops.append(("tokens", seqs, toks))
            model.append_tokens(seqs, toks)
        elif r < 16:
            ops.append(("fork", s))
            live.append(model.fork(s))
        elif r < 17:
            ctx = model.block_table(s)[1]
            if ctx:
                d = model.new_seq()
                live.append(d)
                n = int(gen.integers(1, ctx + 1))
                ops += [("new",), ("share", s, d, n)]
                model.share_prefix(s, d, n)
        elif r < 18:
            ctx = model.block_table(s)[1]
            n = int(gen.integers(0, ctx + 1))
            ops.append(("pin", s, n))
            model.pin(s, n)
        else:
            live.remove(s)
            ops.append(("free", s))
            model.free_seq(s)
    return ops


@pytest.mark.parametrize("seed,num_blocks,block_size", [(1, 48, 16), (2, 30, 4), (3, 200, 16)])
def test_native_matches_model_on_random_scripts(seed, num_blocks, block_size):
    gen = np.random.default_rng(seed)
    order = gen.permutation(num_blocks)
    script = random_script(gen, 3000, ModelPool(num_blocks, block_size, order))
    model = ModelPool(num_blocks, block_size, order)
    nat = native(num_blocks, block_size, order)
    assert replay(nat, script, True) == replay(model, script, False)
    for s in model.seqs:
        assert nat.block_table(s) == model.block_table(s)
    for b in range(num_blocks):
        assert nat.refcount(b) == model.refcount[b]
    assert nat.stats() == model.stats()


@pytest.mark.parametrize("seed,num_blocks,host_blocks", [(4, 64, 40), (5, 120, 300)])
def test_native_matches_model_with_swapping(seed, num_blocks, host_blocks):
    gen = np.random.default_rng(seed)
    order = gen.permutation(num_blocks)
    horder = gen.permutation(host_blocks)
    m0 = ModelPool(num_blocks, 16, order)
    m0.set_host_blocks(host_blocks, horder)
    script = random_script(gen, 3000, m0, swaps=True)
    assert any(op[0] == "swapout" for op in script) and any(op[0] == "swapin" for op in script)
    model = ModelPool(num_blocks, 16, order)
    model.set_host_blocks(host_blocks, horder)
    nat = native(num_blocks, 16, order)
    nat.set_host_blocks(host_blocks, horder)
    assert replay(nat, script, True) == replay(model, script, False)
    for s in model.seqs:
        assert nat.block_table(s) == model.block_table(s)
        assert nat.is_swapped(s) == model.is_swapped(s)
    for b in range(num_blocks):
        assert nat.refcount(b) == model.refcount[b]
    assert nat.stats() == model.stats()


def test_native_swap_refusals():
    from pagedattention_decode_attention_gb300.capi import (PA_ERR_INVALID_ARG, PA_ERR_NO_BLOCKS,
                                                            PagedAttnError)
    pool = native(8)
    pool.set_host_blocks(2)
    a = pool.new_seq()
    for _ in range(40):                      # 3 blocks
        pool.append_slot(a)
    with pytest.raises(PagedAttnError) as e:
        pool.swap_out(a)                     # 3 blocks, 2 host blocks
    assert e.value.status == PA_ERR_NO_BLOCKS
    b = pool.fork(a)
    pool.set_host_blocks(8)
    with pytest.raises(PagedAttnError) as e:
        pool.swap_out(a)                     # shared with the fork
    assert e.value.status == PA_ERR_INVALID_ARG
    pool.free_seq(b)
    pairs = pool.swap_out(a)
    assert pairs.shape == (3, 2) and pool.stats()["free_blocks"] == 8
    for op in (lambda: pool.append_slot(a), lambda: pool.fork(a), lambda: pool.pin(a, 1)):
        with pytest.raises(PagedAttnError) as e:
            op()
        assert e.value.status == PA_ERR_INVALID_ARG
    back = pool.swap_in(a)
    assert [tuple(p) for p in back[:, ::-1].tolist()] != [] and pool.block_table(a)[1] == 40
    assert back[:, 0].tolist() == pairs[:, 1].tolist()     # the same host blocks come back


def test_batched_append_matches_single():
    gen = np.random.default_rng(9)
    a, b = native(64), native(64)
    seqs = [a.new_seq() for _ in range(4)]
    [b.new_seq() for _ in range(4)]
    for _ in range(21):
        for s in seqs:
            a.append_slot(s)
            b.append_slot(s)
    kids_a = [a.fork(s) for s in seqs]
    kids_b = [b.fork(s) for s in seqs]
    order = np.array(seqs + kids_a, dtype=np.int32)[gen.permutation(8)]
    slots, pairs = a.append_slots(order)
    single = [b.append_slot(int(s)) for s in order]
    assert slots.tolist() == [s for s, _ in single]
    assert [tuple(p) for p in pairs.tolist()] == [c for _, c in single if c is not None]
    assert kids_a == kids_b



def test_append_tokens_matches_model_through_exhaustion():
    """The batched token append against the pool model, prefix cache on: a
    prompt in one call, a fork, then alternating appends that copy the shared
    partial block and run the pool dry part way through the batch.  Slots,
    copy pairs, the count made, the tables and the cache keys agree; a second
    prompt with the same tokens hits the blocks the appends keyed."""
    order = np.random.default_rng(5).permutation(12)
    nat, mod = native(12, 4, order), ModelPool(12, 4, order)
    for pool in (nat, mod):
        pool.enable_prefix_cache()
    prompt = list(range(100, 110))                         # 2 full blocks + 2 tokens
    out = []
    for pool in (nat, mod):
        a, _ = pool.new_seq_with_prompt(prompt)              # nothing cached yet
        r0 = pool.append_tokens([a] * len(prompt), prompt)
        b = pool.fork(a)
        seqs = [a, b] * 20
        toks = [200 + i for i in range(len(seqs))]
        r1 = pool.append_tokens(seqs, toks)
        tables = [pool.block_table(s) for s in (a, b)]
        pool.free_seq(a)
        pool.free_seq(b)
        c, hit = pool.new_seq_with_prompt(prompt + [200, 202, 204])
        out.append((r0, r1, tables, hit, pool.stats()))
    (n0, n1, nt, nh, nst), (m0, m1, mt, mh, mst) = out
    for n, m in ((n0, m0), (n1, m1)):
        assert list(n[0]) == list(m[0])
        assert [tuple(p) for p in n[1].tolist()] == [tuple(p) for p in m[1]]
        assert n[2] == m[2]
    assert n0[2] == len(prompt) and len(n0[1]) == 0
    assert 0 < n1[2] < 40 and len(n1[1]) == 1                # ran dry part way; one copy
    assert [(list(t), c) for t, c in nt] == [(list(t), c) for t, c in mt]
    assert nh == mh == 12                                  # 3 keyed blocks of 4 (a's)
    for k in ("free_blocks", "cached_blocks", "evictable_blocks", "cow_copies"):
        assert nst[k] == mst[k], k


def test_append_tokens_empty_and_bad_arguments():
    pool = native(4, 4)
    s = pool.new_seq()
    slots, pairs, done = pool.append_tokens([], [])
    assert (len(slots), len(pairs), done) == (0, 0, 0)
    with pytest.raises(ValueError):
        pool.append_tokens([s, s], [1])
    from pagedattention_decode_attention_gb300.capi import PagedAttnError
    with pytest.raises(PagedAttnError):
        pool.append_tokens([s, 999], [1, 2])                # unknown sequence: not a short count

def test_native_oslab_cow_example():
    g = golden("cow_examples.json")["oslab_block4"]
    pool = native(8, block_size=4)
    a1 = pool.new_seq()
    for _ in g["prefix_tokens"]:
        pool.append_slot(a1)
    a2 = pool.fork(a1)
    table, _ = pool.block_table(a1)
    assert pool.refcount(table[1]) == g["block1_refcount_after_fork"]
    _, cow = pool.append_slot(a1)
    assert cow[0] == table[1]
    assert pool.refcount(table[1]) == g["block1_refcount_after_a1_write"]
    slot, cow = pool.append_slot(a2)
    assert cow is None and slot // 4 == table[1]
    assert pool.stats()["cow_copies"] == g["a1_copies"] + g["a2_copies"]


def test_native_share_example():
    g = golden("cow_examples.json")["share_200_of_500"]
    pool = native(128)
    r1 = pool.new_seq()
    for _ in range(g["first_tokens"]):
        pool.append_slot(r1)
    assert len(pool.block_table(r1)[0]) == g["first_blocks"]
    r2 = pool.new_seq()
    pool.share_prefix(r1, r2, g["shared_tokens"])
    t2, _ = pool.block_table(r2)
    assert len(t2) == g["shared_entries"]
    assert all(pool.refcount(b) == g["refcount_shared"] for b in t2)
    pool.free_seq(r1)
    assert all(pool.refcount(b) == g["refcount_after_one_ends"] for b in t2)
    pool.free_seq(r2)
    assert pool.stats()["free_blocks"] == 128


def test_native_errors():
    from pagedattention_decode_attention_gb300.capi import (PA_ERR_INVALID_ARG, PA_ERR_NO_BLOCKS,
                                                            PA_ERR_NOT_FOUND, PagedAttnError)
    with pytest.raises(PagedAttnError) as e:
        native(4, initial_order=[0, 1, 1, 2])
    assert e.value.status == PA_ERR_INVALID_ARG
    pool = native(1)
    s = pool.new_seq()
    for _ in range(16):
        pool.append_slot(s)
    with pytest.raises(PagedAttnError) as e:
        pool.append_slot(s)
    assert e.value.status == PA_ERR_NO_BLOCKS
    with pytest.raises(PagedAttnError) as e:
        pool.free_seq(99)
    assert e.value.status == PA_ERR_NOT_FOUND
    pool.free_seq(s)
    with pytest.raises(PagedAttnError) as e:
        pool.free_seq(s)                    # double free of a sequence
    assert e.value.status == PA_ERR_NOT_FOUND


# ------------------------------------------------- bench batches, both pools
def test_bench_pool_batches_match_the_model():
    """The bench's pool-built workloads (the prefix mix and the sampling
    divergence) give the same tables, lengths and groups from the native pool
    and from the oracle's model of it (the reference arm uses the model)."""
    import bench
    for name in ("prefix_8b", "sampling_8b"):
        native, model = bench.make_batch(name, 0), bench.make_batch(name, 0, model_pool=True)
        assert np.array_equal(native.block_tables, model.block_tables)
        assert np.array_equal(native.context_lens, model.context_lens)
        for key in ("group_start", "group_blocks"):
            if key in native.extra:
                assert np.array_equal(native.extra[key], model.extra[key])


def test_sampling_divergence_pairs_and_groups():
    """The divergence of 32 prompts forked 4 ways: 3 copy-on-write pairs per
    prompt, distinct destinations, no destination another pair's source; each
    group's members share exactly the prompt's whole blocks."""
    import bench
    from pagedattention_decode_attention_gb300 import workloads as wl
    script = wl.sampling_cow()
    pool = native(script.num_blocks, 16, script.initial_order)
    branches, pairs = bench.cow_divergence(pool, script)
    assert len(branches) == script.prompts * script.branches
    assert pairs.shape == (script.prompts * (script.branches - 1), 2)
    assert len(set(pairs[:, 1])) == len(pairs)
    assert not set(pairs[:, 0]) & set(pairs[:, 1])
    batch = bench.sampling_batch(script)
    whole = (script.prompt_len + script.shared_extra) // 16
    assert np.array_equal(batch.extra["group_blocks"], whole.astype(np.int32))
    assert np.array_equal(batch.extra["group_start"],
                          np.arange(0, len(branches) + 1, script.branches))
