"""Pins for the attention / append / copy oracle (CPU only).

Each ``check_*`` function pins the oracle to something other than itself: a
library routine (torch's fp64 scaled-dot-product attention, scipy's
logsumexp), a closed form, an invariant, or a worked example printed on the
pages.  The mutation tests at the bottom plant plausible mistakes in the oracle
(on the CPU) and require that some check catches each one.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle.attention as oa
from tests.conftest import golden

BS = 16


# --------------------------------------------------------------------------
# case construction (scatter through slot numbers, not through the oracle)
# --------------------------------------------------------------------------
def make_case(seed, lens, num_q_heads, num_kv_heads, head_dim, num_blocks=None):
    gen = np.random.default_rng(seed)
    lens = [int(x) for x in lens]
    need = [-(-n // BS) for n in lens]
    if num_blocks is None:
        num_blocks = sum(need) + 5
    q = gen.standard_normal((len(lens), num_q_heads, head_dim))
    keys = [gen.standard_normal((n, num_kv_heads, head_dim)) for n in lens]
    values = [gen.standard_normal((n, num_kv_heads, head_dim)) for n in lens]
    perm = gen.permutation(num_blocks)
    tables = np.full((len(lens), max(1, max(need))), -1, dtype=np.int64)
    at = 0
    for i, c in enumerate(need):
        tables[i, :c] = perm[at:at + c]
        at += c
    # Unused slots hold noise, so reading a wrong slot changes the answer.
    k_slots = gen.standard_normal((num_blocks * BS, num_kv_heads, head_dim))
    v_slots = gen.standard_normal((num_blocks * BS, num_kv_heads, head_dim))
    for i, n in enumerate(lens):
        t = np.arange(n)
        slots = tables[i, t // BS] * BS + t % BS
        k_slots[slots] = keys[i]
        v_slots[slots] = values[i]
    # slot-major [NB*16, H, d] -> [NB, H, 16, d]
    k_cache = k_slots.reshape(num_blocks, BS, num_kv_heads, head_dim).transpose(0, 2, 1, 3).copy()
    v_cache = v_slots.reshape(num_blocks, BS, num_kv_heads, head_dim).transpose(0, 2, 1, 3).copy()
    return dict(q=q, keys=keys, values=values, tables=tables, k_cache=k_cache,
                v_cache=v_cache, lens=np.array(lens), scale=1.0 / math.sqrt(head_dim))


def run_oracle(case):
    return oa.paged_attention_decode(case["q"], case["k_cache"], case["v_cache"],
                                     case["tables"], case["lens"], case["scale"])


# --------------------------------------------------------------------------
# checks (each returns True when the oracle agrees with the pin)
# --------------------------------------------------------------------------
def check_block_table_example():
    """Page-3 block-table example: token t sits at physical block[t // 16],
    offset t % 16 (token 20 of request A is physical 12, offset 4)."""
    g = golden("block_table_example.json")
    table = g["table"]
    num_blocks = max(table) + 1
    # Cache whose every slot stores its own (physical, offset) pair.
    cache = np.zeros((num_blocks, 1, BS, 2))
    for p in range(num_blocks):
        for off in range(BS):
            cache[p, 0, off] = (p, off)
    got = oa.gather_sequence(cache, table, 48)
    return all(tuple(got[t, 0]) == (phys, off) for t, phys, off in g["token_to_physical"])


def check_sdpa(seed=0, lens=(1, 15, 16, 17, 33, 100), hq=8, hkv=2, d=16):
    """Equality with torch's fp64 scaled_dot_product_attention on the unpaged
    contiguous K/V (the pages: the formula is unchanged, only the layout)."""
    case = make_case(seed, lens, hq, hkv, d)
    got = run_oracle(case)
    for b, n in enumerate(case["lens"]):
        qt = torch.from_numpy(case["q"][b]).reshape(1, hq, 1, d)
        kt = torch.from_numpy(case["keys"][b]).permute(1, 0, 2).unsqueeze(0)
        vt = torch.from_numpy(case["values"][b]).permute(1, 0, 2).unsqueeze(0)
        ref = F.scaled_dot_product_attention(qt, kt, vt, scale=case["scale"],
                                             enable_gqa=True).reshape(hq, d).numpy()
        if not np.allclose(got[b], ref, rtol=1e-12, atol=1e-12):
            return False
    return True


def check_ctx_one():
    """One token of context: the output is that token's value row exactly."""
    case = make_case(1, [1, 1], 4, 4, 8)
    got = run_oracle(case)
    return all(np.array_equal(got[b], case["values"][b][0]) for b in range(2))


def check_equal_keys_mean():
    """All keys equal: every weight is equal, the output is the mean of V."""
    case = make_case(2, [37], 4, 2, 8)
    kc = case["k_cache"]
    for t in range(37):
        kc[case["tables"][0, t // BS], :, t % BS, :] = kc[case["tables"][0, 0], :, 0, :]
    got = run_oracle(case)
    mean = case["values"][0].mean(axis=0)          # [Hkv, d]
    expect = np.repeat(mean, 2, axis=0)            # q-head h reads kv-head h // 2
    return np.allclose(got[0], expect, rtol=0, atol=1e-13)


def check_zero_query_mean():
    case = make_case(3, [50], 2, 2, 8)
    case["q"][:] = 0.0
    got = run_oracle(case)
    return np.allclose(got[0], case["values"][0].mean(axis=0), rtol=0, atol=1e-13)


def check_dominant_score():
    """One key aligned with q and a score ~1e3 above the rest: softmax is a
    one-hot at that token (needs the max subtraction to avoid overflow)."""
    case = make_case(4, [40], 1, 1, 4)
    q = np.array([1.0, 0.0, 0.0, 0.0]) * 64.0
    case["q"][0, 0] = q
    case["scale"] = 1.0
    kc = case["k_cache"]
    hot = 23
    for t in range(40):
        row = np.zeros(4)
        row[1] = t                                  # orthogonal to q
        kc[case["tables"][0, t // BS], 0, t % BS] = row
    kc[case["tables"][0, hot // BS], 0, hot % BS] = np.array([20.0, 0, 0, 0])
    got = run_oracle(case)
    return np.all(np.isfinite(got)) and np.allclose(got[0, 0], case["values"][0][hot, 0], atol=1e-12)


def check_two_token_logistic():
    """Two tokens: weights are the logistic function of the score gap."""
    case = make_case(5, [2], 1, 1, 8)
    k = case["keys"][0][:, 0]
    v = case["values"][0][:, 0]
    s = case["scale"] * (k @ case["q"][0, 0])
    w0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
    expect = w0 * v[0] + (1.0 - w0) * v[1]
    return np.allclose(run_oracle(case)[0, 0], expect, rtol=1e-13, atol=1e-13)


def check_permutation_invariance(seed=6):
    """Relabelling physical blocks (cache'[pi(i)] = cache[i], table' = pi o
    table) leaves the output bit-identical."""
    case = make_case(seed, [5, 16, 31, 70], 4, 2, 8)
    base = run_oracle(case)
    nb = case["k_cache"].shape[0]
    pi = np.random.default_rng(seed + 100).permutation(nb)
    k2 = np.empty_like(case["k_cache"])
    v2 = np.empty_like(case["v_cache"])
    k2[pi] = case["k_cache"]
    v2[pi] = case["v_cache"]
    t2 = np.where(case["tables"] >= 0, pi[np.maximum(case["tables"], 0)], -1)
    moved = oa.paged_attention_decode(case["q"], k2, v2, t2, case["lens"], case["scale"])
    return np.array_equal(base, moved)


def check_gqa_equals_repeated_mha():
    """GQA equals MHA over KV heads repeated group-size times."""
    case = make_case(7, [9, 40], 8, 2, 8)
    got = run_oracle(case)
    k_rep = np.repeat(case["k_cache"], 4, axis=1)
    v_rep = np.repeat(case["v_cache"], 4, axis=1)
    mha = oa.paged_attention_decode(case["q"], k_rep, v_rep, case["tables"],
                                    case["lens"], case["scale"])
    return np.allclose(got, mha, rtol=0, atol=0)


def check_page3_layout():
    """The page-3 conceptual layout kv_cache[block, 0|1] of shape [16, heads, d]
    holds the same tokens as separate [block, heads, 16, d] caches."""
    case = make_case(8, [3, 29], 4, 4, 8)
    nb = case["k_cache"].shape[0]
    kv = np.zeros((nb, 2, BS, 4, 8))
    kv[:, 0] = case["k_cache"].transpose(0, 2, 1, 3)
    kv[:, 1] = case["v_cache"].transpose(0, 2, 1, 3)
    # gather the page-3 way: K_block = kv_cache[physical, 0] -> [16, heads, d]
    for b, n in enumerate(case["lens"]):
        ks = []
        for logical in range(-(-int(n) // BS)):
            ks.append(kv[case["tables"][b, logical], 0])
        ks = np.concatenate(ks)[:n]
        if not np.array_equal(ks, oa.gather_sequence(case["k_cache"], case["tables"][b], int(n))):
            return False
    return True


def check_lse_scipy():
    case = make_case(9, [45], 2, 2, 8)
    keys = case["keys"][0][:, 0]
    got = oa.attention_lse(case["q"][0, 0], keys, case["scale"])
    return math.isclose(got, logsumexp(case["scale"] * keys @ case["q"][0, 0]), rel_tol=1e-13)


def check_split_merge_identity():
    """Splitting the context in two and merging with log-sum-exp weights gives
    the unsplit result (the identity a split-K kernel relies on; the pages'
    'multiply-add per block, then reduce across blocks')."""
    case = make_case(10, [77], 1, 1, 8)
    q = case["q"][0, 0]
    k = case["keys"][0][:, 0]
    v = case["values"][0][:, 0]
    full = oa.attention_one(q, k, v, case["scale"])
    parts = [(oa.attention_one(q, k[a:b], v[a:b], case["scale"]),
              oa.attention_lse(q, k[a:b], case["scale"])) for a, b in ((0, 32), (32, 77))]
    top = max(l for _, l in parts)
    w = [math.exp(l - top) for _, l in parts]
    merged = sum(wi * o for wi, (o, _) in zip(w, parts)) / sum(w)
    return np.allclose(full, merged, rtol=1e-13, atol=1e-13)


def check_ctx_zero():
    case = make_case(11, [0, 3], 2, 2, 8)
    got = run_oracle(case)
    return np.array_equal(got[0], np.zeros_like(got[0])) and np.all(np.isfinite(got[1]))


ALL_CHECKS = [check_block_table_example, check_sdpa, check_ctx_one, check_equal_keys_mean,
              check_zero_query_mean, check_dominant_score, check_two_token_logistic,
              check_permutation_invariance, check_gqa_equals_repeated_mha, check_page3_layout,
              check_lse_scipy, check_split_merge_identity, check_ctx_zero]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    assert check()


def test_sdpa_more_shapes():
    assert check_sdpa(seed=21, lens=(3, 64, 65, 130), hq=4, hkv=4, d=64)
    assert check_sdpa(seed=22, lens=(250,), hq=32, hkv=8, d=128)


# --------------------------------------------------------------------------
# kv_append / block_copy
# --------------------------------------------------------------------------
def test_kv_append_page_example_slots():
    """Slots follow the page-3 table example: token 20 of a request whose
    table is [37, 12, 88] goes to slot 12 * 16 + 4."""
    g = golden("block_table_example.json")
    nb = max(g["table"]) + 1
    kc = np.zeros((nb, 2, BS, 4), dtype=np.float32)
    vc = np.zeros_like(kc)
    tokens = [t for t, _, _ in g["token_to_physical"]]
    slots = [g["table"][t // BS] * BS + t % BS for t in tokens]
    k = np.arange(len(tokens) * 8, dtype=np.float32).reshape(len(tokens), 2, 4) + 1
    oa.kv_append(k, -k, kc, vc, slots)
    for i, (t, phys, off) in enumerate(g["token_to_physical"]):
        assert np.array_equal(kc[phys, :, off], k[i])
        assert np.array_equal(vc[phys, :, off], -k[i])
    # nothing else was written
    assert np.count_nonzero(kc) == k.size


def test_kv_append_skips_negative_slots_and_is_bit_exact():
    kc = np.zeros((4, 2, BS, 8), dtype=np.uint16)
    vc = np.zeros_like(kc)
    k = np.random.default_rng(0).integers(1, 65535, size=(3, 2, 8)).astype(np.uint16)
    oa.kv_append(k, k, kc, vc, [5, -1, 63])
    assert np.array_equal(kc[0, :, 5], k[0]) and np.array_equal(kc[3, :, 15], k[2])
    assert np.count_nonzero(kc) == np.count_nonzero(k[[0, 2]])


def test_block_copy_all_layers_all_slots():
    gen = np.random.default_rng(1)
    ks = [gen.standard_normal((6, 2, BS, 4)) for _ in range(3)]
    vs = [gen.standard_normal((6, 2, BS, 4)) for _ in range(3)]
    k0 = [x.copy() for x in ks]
    oa.block_copy(ks, vs, [(1, 4), (2, 5)])
    for layer in range(3):
        assert np.array_equal(ks[layer][4], ks[layer][1])
        assert np.array_equal(vs[layer][5], vs[layer][2])
        for blk in (0, 1, 2, 3):
            assert np.array_equal(ks[layer][blk], k0[layer][blk])


# --------------------------------------------------------------------------
# mutation tests: plant a plausible mistake in the oracle, some check must fail
# --------------------------------------------------------------------------
def _mut_gqa_modulo(q, k_cache, v_cache, block_tables, context_lens, scale, seqs=None, heads=None):
    num_seqs, hq, d = q.shape
    hkv = k_cache.shape[1]
    out = np.full((num_seqs, hq, d), np.nan)
    for b in range(num_seqs):
        ctx = int(context_lens[b])
        keys = oa.gather_sequence(k_cache, block_tables[b], ctx)
        values = oa.gather_sequence(v_cache, block_tables[b], ctx)
        for h in range(hq):
            out[b, h] = oa.attention_one(q[b, h], keys[:, h % hkv], values[:, h % hkv], scale)
    return out


def _mut_gather_swapped(cache, block_table, context_len):
    hk, d = cache.shape[1], cache.shape[3]
    out = np.empty((context_len, hk, d))
    for t in range(context_len):
        out[t] = cache[int(block_table[t % BS]) if t % BS < len(block_table) else 0, :, t // BS, :]
    return out


def _mut_gather_drop_tail(cache, block_table, context_len):
    hk, d = cache.shape[1], cache.shape[3]
    full = (context_len // BS) * BS
    out = np.zeros((context_len, hk, d))
    for logical in range(context_len // BS):
        out[logical * BS:(logical + 1) * BS] = np.transpose(cache[int(block_table[logical])], (1, 0, 2))
    return out[:max(full, 1)] if context_len else out


def _mut_no_scale(q, keys, values, scale):
    if keys.shape[0] == 0:
        return np.zeros(values.shape[1])
    s = keys @ q
    w = np.exp(s - s.max())
    return (w @ values) / w.sum()


def _mut_no_max(q, keys, values, scale):
    if keys.shape[0] == 0:
        return np.zeros(values.shape[1])
    with np.errstate(over="ignore", invalid="ignore"):
        w = np.exp(scale * (keys @ q))
        return (w @ values) / w.sum()


def _mut_swap_kv(q, keys, values, scale):
    if keys.shape[0] == 0:
        return np.zeros(values.shape[1])
    s = scale * (values @ q)
    w = np.exp(s - s.max())
    return (w @ keys) / w.sum()


def _mut_no_normalise(q, keys, values, scale):
    if keys.shape[0] == 0:
        return np.zeros(values.shape[1])
    s = scale * (keys @ q)
    w = np.exp(s - s.max())
    return w @ values


def _mut_off_by_one_block(cache, block_table, context_len):
    hk, d = cache.shape[1], cache.shape[3]
    out = np.empty((context_len, hk, d))
    for t in range(context_len):
        logical = (t + 1) // BS if (t + 1) // BS < -(-context_len // BS) else t // BS
        out[t] = cache[int(block_table[logical]), :, t % BS, :]
    return out


MUTANTS = {
    "gqa_modulo": ("paged_attention_decode", _mut_gqa_modulo),
    "gather_block_offset_swapped": ("gather_sequence", _mut_gather_swapped),
    "gather_drops_partial_block": ("gather_sequence", _mut_gather_drop_tail),
    "gather_off_by_one_block": ("gather_sequence", _mut_off_by_one_block),
    "missing_scale": ("attention_one", _mut_no_scale),
    "missing_max_subtraction": ("attention_one", _mut_no_max),
    "keys_values_swapped": ("attention_one", _mut_swap_kv),
    "missing_normalisation": ("attention_one", _mut_no_normalise),
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
