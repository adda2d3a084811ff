"""Pins for the oracle's three copy steps: kv_append, block_copy, block_swap
(CPU only).

The copies are exact, so every pin is a closed form.  Each cache cell holds a
distinct integer tag computed from (tier, layer, K/V, block, head, slot,
column); the expected cache after an operation is written out from the tag
formula and the operation's definition, never by calling the oracle again:

* kv_append -- "留书阁 / knowledge-20" page, section "PagedAttention：虚实分离"
  (token t of a sequence lives at physical ``block_table[t // 16]``, offset
  ``t % 16``) and the OS-lab appendix, section 2.1 (each decode step writes
  the new token's K/V).  Negative slots are padding (our reading).
* block_copy -- OS-lab appendix, sections 4.3-4.4: a shared block is copied
  whole (every slot, every KV head, K and V, every layer) before the writer's
  first write; pairs apply in order.
* block_swap -- "vLLM: treating the KV cache as virtual memory", section
  "调度：词一级的进入与退出": a preempted sequence's KV moves to host memory
  block by block and comes back; the same whole-block copy, between two tiers.

The mutation tests at the bottom plant plausible mistakes in these oracle
functions (on the CPU) and require that some pin catches each one.
"""

import numpy as np
import pytest

import oracle.attention as oa

BS = 16
LAYERS, HKV, D = 3, 2, 4


def tags(tier, layer, kind, num_blocks):
    """Distinct int64 tag for every cell of one [num_blocks, HKV, 16, D] cache."""
    b, h, s, c = np.meshgrid(np.arange(num_blocks), np.arange(HKV), np.arange(BS),
                             np.arange(D), indexing="ij")
    return (((((tier * LAYERS + layer) * 2 + kind) * 1000 + b) * HKV + h) * BS + s) * D + c


def tier_caches(tier, num_blocks):
    k = [tags(tier, l, 0, num_blocks) for l in range(LAYERS)]
    v = [tags(tier, l, 1, num_blocks) for l in range(LAYERS)]
    return k, v


# --------------------------------------------------------------------------
# block_swap
# --------------------------------------------------------------------------
def check_swap_moves_listed_blocks():
    """dst[d] holds exactly src[s]'s cells for each listed pair, K and V, in
    every layer; every other block of both tiers is untouched."""
    nd, nh = 9, 7
    pairs = [(4, 0), (0, 6), (8, 3), (2, 2)]
    sk, sv = tier_caches(0, nd)
    dk, dv = tier_caches(1, nh)
    oa.block_swap(sk, sv, dk, dv, pairs)
    dst_of = {d: s for s, d in pairs}
    for l in range(LAYERS):
        for kind, (src, dst) in enumerate(((sk[l], dk[l]), (sv[l], dv[l]))):
            if not np.array_equal(src, tags(0, l, kind, nd)):
                return False
            want_src = tags(0, l, kind, nd)
            want_dst = tags(1, l, kind, nh)
            for d, s in dst_of.items():
                want_dst[d] = want_src[s]
            if not np.array_equal(dst, want_dst):
                return False
    return True


def check_swap_round_trip():
    """Out to the host tier, the device blocks overwritten, back into other
    device blocks: each block's cells are back, under its new id."""
    nd, nh = 10, 6
    dk, dv = tier_caches(0, nd)
    hk, hv = tier_caches(1, nh)
    out_pairs = [(1, 5), (7, 0), (3, 2)]
    oa.block_swap(dk, dv, hk, hv, out_pairs)
    for l in range(LAYERS):           # the freed device blocks are reused
        for blk in (1, 7, 3):
            dk[l][blk] = -1
            dv[l][blk] = -1
    new_dev = {5: 9, 0: 4, 2: 1}       # host block -> new device block
    oa.block_swap(hk, hv, dk, dv, [(h, d) for h, d in new_dev.items()])
    back = {1: 9, 7: 4, 3: 1}          # old device block -> new device block
    for l in range(LAYERS):
        for kind, cache in enumerate((dk[l], dv[l])):
            orig = tags(0, l, kind, nd)
            for old, new in back.items():
                if not np.array_equal(cache[new], orig[old]):
                    return False
    return True


def check_swap_pair_order():
    """Pairs apply in order: with a repeated destination the later pair wins
    (the device kernel requires distinct destinations; the oracle's
    definition is sequential)."""
    sk, sv = tier_caches(0, 4)
    dk, dv = tier_caches(1, 4)
    oa.block_swap(sk, sv, dk, dv, [(1, 2), (3, 2)])
    return all(np.array_equal(dk[l][2], tags(0, l, 0, 4)[3]) and
               np.array_equal(dv[l][2], tags(0, l, 1, 4)[3]) for l in range(LAYERS))


def check_swap_empty():
    sk, sv = tier_caches(0, 3)
    dk, dv = tier_caches(1, 3)
    oa.block_swap(sk, sv, dk, dv, np.zeros((0, 2), dtype=np.int64))
    return all(np.array_equal(dk[l], tags(1, l, 0, 3)) and np.array_equal(dv[l], tags(1, l, 1, 3))
               for l in range(LAYERS))


# --------------------------------------------------------------------------
# block_copy
# --------------------------------------------------------------------------
def check_copy_moves_listed_blocks():
    nb = 8
    pairs = [(1, 4), (2, 5), (1, 6)]
    k, v = tier_caches(0, nb)
    oa.block_copy(k, v, pairs)
    for l in range(LAYERS):
        for kind, cache in enumerate((k[l], v[l])):
            want = tags(0, l, kind, nb)
            for s, d in pairs:
                want[d] = tags(0, l, kind, nb)[s]
            if not np.array_equal(cache, want):
                return False
    return True


def check_copy_pair_order():
    """In order: (1 -> 2) then (2 -> 3) leaves block 1's cells in block 3."""
    k, v = tier_caches(0, 5)
    oa.block_copy(k, v, [(1, 2), (2, 3)])
    return all(np.array_equal(k[l][3], tags(0, l, 0, 5)[1]) and
               np.array_equal(v[l][3], tags(0, l, 1, 5)[1]) for l in range(LAYERS))


# --------------------------------------------------------------------------
# kv_append
# --------------------------------------------------------------------------
def check_append_slots():
    """Token i lands at block slot // 16, row slot % 16, all heads and columns;
    negative slots write nothing; nothing else changes."""
    nb = 6
    slots = [0, 17, 95, -1, 40]
    kc, vc = tags(0, 0, 0, nb), tags(0, 0, 1, nb)
    k = -(np.arange(len(slots) * HKV * D).reshape(len(slots), HKV, D) + 1)
    v = k - 10_000
    oa.kv_append(k, v, kc, vc, slots)
    want_k, want_v = tags(0, 0, 0, nb), tags(0, 0, 1, nb)
    for i, slot in enumerate(slots):
        if slot >= 0:
            want_k[slot // BS, :, slot % BS, :] = k[i]
            want_v[slot // BS, :, slot % BS, :] = v[i]
    return np.array_equal(kc, want_k) and np.array_equal(vc, want_v)


def check_append_page_table_example():
    """The page's table [37, 12, ...]: token 20 (logical block 1, offset 4)
    goes to physical block 12, row 4."""
    kc = np.zeros((40, HKV, BS, D), dtype=np.int64)
    vc = np.zeros_like(kc)
    table = [37, 12]
    t = 20
    k = np.full((1, HKV, D), 7)
    oa.kv_append(k, k + 1, kc, vc, [table[t // BS] * BS + t % BS])
    return (np.all(kc[12, :, 4] == 7) and np.all(vc[12, :, 4] == 8)
            and np.count_nonzero(kc) == HKV * D and np.count_nonzero(vc) == HKV * D)


ALL_CHECKS = [check_swap_moves_listed_blocks, check_swap_round_trip, check_swap_pair_order,
              check_swap_empty, check_copy_moves_listed_blocks, check_copy_pair_order,
              check_append_slots, check_append_page_table_example]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_copy_pin(check):
    assert check()


def test_tags_are_distinct():
    every = np.concatenate([tags(t, l, kind, 10).ravel() for t in (0, 1)
                            for l in range(LAYERS) for kind in (0, 1)])
    assert len(np.unique(every)) == every.size


# --------------------------------------------------------------------------
# mutation tests: plant a plausible mistake, some pin must fail
# --------------------------------------------------------------------------
def _swap_src_dst_exchanged(sk, sv, dk, dv, pairs):
    for s, d in pairs:
        for a, b, c, e in zip(sk, sv, dk, dv):
            c[int(s)] = a[int(d)] if int(d) < len(a) else c[int(s)]
            e[int(s)] = b[int(d)] if int(d) < len(b) else e[int(s)]


def _swap_k_only(sk, sv, dk, dv, pairs):
    for s, d in pairs:
        for a, c in zip(sk, dk):
            c[int(d)] = a[int(s)]


def _swap_layer0_only(sk, sv, dk, dv, pairs):
    for s, d in pairs:
        dk[0][int(d)] = sk[0][int(s)]
        dv[0][int(d)] = sv[0][int(s)]


def _swap_reverse_order(sk, sv, dk, dv, pairs):
    for s, d in list(pairs)[::-1]:
        for a, b, c, e in zip(sk, sv, dk, dv):
            c[int(d)] = a[int(s)]
            e[int(d)] = b[int(s)]


def _swap_kv_crossed(sk, sv, dk, dv, pairs):
    for s, d in pairs:
        for a, b, c, e in zip(sk, sv, dk, dv):
            c[int(d)] = b[int(s)]
            e[int(d)] = a[int(s)]


def _swap_first_head_only(sk, sv, dk, dv, pairs):
    for s, d in pairs:
        for a, b, c, e in zip(sk, sv, dk, dv):
            c[int(d), 0] = a[int(s), 0]
            e[int(d), 0] = b[int(s), 0]


def _swap_moves_instead_of_copy(sk, sv, dk, dv, pairs):
    for s, d in pairs:
        for a, b, c, e in zip(sk, sv, dk, dv):
            c[int(d)] = a[int(s)]
            e[int(d)] = b[int(s)]
            a[int(s)] = 0
            b[int(s)] = 0


def _copy_reverse_order(k_caches, v_caches, pairs):
    for s, d in list(pairs)[::-1]:
        for k, v in zip(k_caches, v_caches):
            k[int(d)] = k[int(s)]
            v[int(d)] = v[int(s)]


def _copy_first_slot_only(k_caches, v_caches, pairs):
    for s, d in pairs:
        for k, v in zip(k_caches, v_caches):
            k[int(d), :, 0] = k[int(s), :, 0]
            v[int(d), :, 0] = v[int(s), :, 0]


def _append_offset_block_swapped(k, v, kc, vc, slots):
    for i, slot in enumerate(slots):
        if slot >= 0 and slot % BS < kc.shape[0] and slot // BS < BS:
            kc[slot % BS, :, slot // BS, :] = k[i]
            vc[slot % BS, :, slot // BS, :] = v[i]


def _append_padding_not_skipped(k, v, kc, vc, slots):
    for i, slot in enumerate(slots):
        kc[int(slot) // BS, :, int(slot) % BS, :] = k[i]
        vc[int(slot) // BS, :, int(slot) % BS, :] = v[i]


MUTANTS = {
    "swap_src_dst_exchanged": ("block_swap", _swap_src_dst_exchanged),
    "swap_k_only": ("block_swap", _swap_k_only),
    "swap_layer0_only": ("block_swap", _swap_layer0_only),
    "swap_reverse_order": ("block_swap", _swap_reverse_order),
    "swap_kv_crossed": ("block_swap", _swap_kv_crossed),
    "swap_first_head_only": ("block_swap", _swap_first_head_only),
    "swap_moves_instead_of_copy": ("block_swap", _swap_moves_instead_of_copy),
    "copy_reverse_order": ("block_copy", _copy_reverse_order),
    "copy_first_slot_only": ("block_copy", _copy_first_slot_only),
    "append_offset_block_swapped": ("kv_append", _append_offset_block_swapped),
    "append_padding_not_skipped": ("kv_append", _append_padding_not_skipped),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(oa, attr, fn)
    failed = []
    for check in ALL_CHECKS:
        try:
            ok = check()
        except Exception:
            ok = False
        if not ok:
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
