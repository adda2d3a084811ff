"""Pins for the chunked-prefill oracle (``oracle.attention.paged_attention_prefill``).

Each pin checks the oracle against something other than itself:
* torch's float64 ``scaled_dot_product_attention`` with an explicit causal
  mask (bottom-right aligned: the chunk is the sequence's newest tokens) on
  contiguous K/V that the test scatters into a paged cache itself;
* the last query row of a chunk is the decode of the whole context, and a
  chunk of one token is decode (decode is chunked prefill with T = 1);
* causality: changing the K/V of tokens after a query's position does not
  change that query's output, changing the token at its position does;
* block-placement invariance;
and planted mistakes (mask off by one, top-left mask alignment, wrong query
offsets, attending one token too few) must each fail at least one pin.
"""

import numpy as np
import pytest
import torch

import oracle.attention as oa

BS = 16


def _scatter(contig, gen, extra_blocks=5):
    """Paged cache + table holding one sequence's contiguous [ctx, Hkv, d]."""
    ctx, hkv, d = contig.shape
    nblk = (ctx + BS - 1) // BS
    nb = nblk + extra_blocks
    cache = gen.standard_normal((nb, hkv, BS, d))          # garbage in unused slots
    table = gen.permutation(nb)[:nblk]
    for t in range(ctx):
        cache[table[t // BS], :, t % BS, :] = contig[t]
    return cache, table


def _case(seed, lens, qlens, hq=4, hkv=2, d=16):
    gen = np.random.default_rng(seed)
    ks, vs = [], []
    for ctx in lens:
        ks.append(gen.standard_normal((ctx, hkv, d)))
        vs.append(gen.standard_normal((ctx, hkv, d)))
    # one shared pool: sequences' blocks placed disjointly
    nblks = [(c + BS - 1) // BS for c in lens]
    nb = sum(nblks) + 7
    kc = gen.standard_normal((nb, hkv, BS, d))
    vc = gen.standard_normal((nb, hkv, BS, d))
    perm = gen.permutation(nb)
    mb = max(nblks) if nblks else 1
    tables = -np.ones((len(lens), mb), dtype=np.int64)
    at = 0
    for b, ctx in enumerate(lens):
        tables[b, :nblks[b]] = perm[at:at + nblks[b]]
        at += nblks[b]
        for t in range(ctx):
            kc[tables[b, t // BS], :, t % BS] = ks[b][t]
            vc[tables[b, t // BS], :, t % BS] = vs[b][t]
    qs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int64)
    q = gen.standard_normal((int(qs[-1]), hq, d))
    return dict(q=q, kc=kc, vc=vc, tables=tables, lens=np.array(lens), qs=qs, ks=ks, vs=vs,
                scale=1.0 / np.sqrt(d), hq=hq, hkv=hkv)


def _sdpa_reference(c):
    """torch float64 SDPA per sequence on the contiguous K/V, explicit mask."""
    out = np.zeros(c["q"].shape)
    for b, ctx in enumerate(c["lens"]):
        first, last = int(c["qs"][b]), int(c["qs"][b + 1])
        qlen = last - first
        if qlen == 0:
            continue
        q = torch.from_numpy(c["q"][first:last]).permute(1, 0, 2)           # [Hq, T, d]
        k = torch.from_numpy(c["ks"][b]).permute(1, 0, 2)                  # [Hkv, ctx, d]
        v = torch.from_numpy(c["vs"][b]).permute(1, 0, 2)
        rows = torch.arange(qlen)[:, None] + (ctx - qlen)
        mask = torch.arange(ctx)[None, :] <= rows                          # bottom-right causal
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=mask, scale=c["scale"], enable_gqa=True)
        out[first:last] = o.permute(1, 0, 2).numpy()
    return out


def _oracle(c, **kw):
    return oa.paged_attention_prefill(c["q"], c["kc"], c["vc"], c["tables"], c["lens"], c["qs"],
                                      c["scale"], **kw)


CASES = [
    (1, [40, 17, 5, 64], [8, 17, 1, 20]),      # chunk = whole prompt, partial chunk, decode
    (2, [100, 33], [33, 1]),                   # chunk crossing block boundaries
    (3, [16, 48, 7], [16, 16, 0]),             # block-aligned chunks, an idle sequence
]


def check_matches_sdpa():
    for seed, lens, qlens in CASES:
        c = _case(seed, lens, qlens)
        if not np.allclose(_oracle(c), _sdpa_reference(c), atol=1e-12, rtol=1e-12):
            return False
    return True


def check_last_row_is_decode():
    c = _case(4, [70, 23, 45], [12, 23, 5])
    pre = _oracle(c)
    last_rows = c["qs"][1:] - 1
    dec = oa.paged_attention_decode(c["q"][last_rows], c["kc"], c["vc"], c["tables"], c["lens"],
                                    c["scale"])
    return np.allclose(pre[last_rows], dec, atol=1e-12)


def check_one_token_chunks_are_decode():
    c = _case(5, [9, 31, 64], [1, 1, 1])
    dec = oa.paged_attention_decode(c["q"], c["kc"], c["vc"], c["tables"], c["lens"], c["scale"])
    return np.allclose(_oracle(c), dec, atol=1e-12)


def check_causality():
    c = _case(6, [50], [20])
    base = _oracle(c)
    row = 3                                       # position 50 - 20 + 3 = 33
    later = c["kc"].copy()
    for t in range(34, 50):                       # every token after position 33
        later[c["tables"][0, t // BS], :, t % BS] += 5.0
    moved_later = oa.paged_attention_prefill(c["q"], later, c["vc"], c["tables"], c["lens"],
                                             c["qs"], c["scale"])
    at_pos = c["kc"].copy()
    at_pos[c["tables"][0, 33 // BS], :, 33 % BS] += 5.0
    moved_at = oa.paged_attention_prefill(c["q"], at_pos, c["vc"], c["tables"], c["lens"], c["qs"],
                                          c["scale"])
    return (np.array_equal(moved_later[row], base[row])
            and not np.allclose(moved_at[row], base[row]))


def check_placement_invariance():
    c = _case(7, [60, 30], [10, 30])
    base = _oracle(c)
    pi = np.random.default_rng(8).permutation(c["kc"].shape[0])
    kc2, vc2 = np.empty_like(c["kc"]), np.empty_like(c["vc"])
    kc2[pi], vc2[pi] = c["kc"], c["vc"]
    t2 = np.where(c["tables"] >= 0, pi[np.maximum(c["tables"], 0)], -1)
    moved = oa.paged_attention_prefill(c["q"], kc2, vc2, t2, c["lens"], c["qs"], c["scale"])
    return np.array_equal(base, moved)


ALL_CHECKS = [check_matches_sdpa, check_last_row_is_decode, check_one_token_chunks_are_decode,
              check_causality, check_placement_invariance]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_prefill_pin(check):
    assert check()


def test_rows_sample_matches_full():
    c = _case(9, [80, 20], [16, 20])
    full = _oracle(c)
    sample = _oracle(c, rows=[0, 15, 17, 35])
    assert np.array_equal(sample[[0, 15, 17, 35]], full[[0, 15, 17, 35]])
    assert np.isnan(sample[1]).all()


def test_chunk_longer_than_context_is_refused():
    c = _case(10, [5], [5])
    c["qs"] = np.array([0, 6])
    c["q"] = np.zeros((6, c["hq"], 16))
    with pytest.raises(ValueError):
        _oracle(c)


# ----------------------------------------------------------- planted mistakes
def _mut_positions_shifted(context_len, query_len):
    return range(context_len - query_len + 1, context_len + 1)


def _mut_positions_top_left(context_len, query_len):
    return range(0, query_len)


def _mut_prefix_short(buf, position):
    return buf[:position]


def _mut_prefix_long(buf, position):
    return buf[:position + 2]


MUTANTS = {
    "mask_shifted_by_one": ("chunk_positions", _mut_positions_shifted),
    "mask_top_left_aligned": ("chunk_positions", _mut_positions_top_left),
    "attends_one_token_too_few": ("causal_prefix", _mut_prefix_short),
    "attends_one_token_too_many": ("causal_prefix", _mut_prefix_long),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_prefill_pins_catch_planted_mistake(name, monkeypatch):
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
