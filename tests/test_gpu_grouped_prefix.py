"""GPU parity of the grouped shared-prefix decode
(``pa_paged_attention_decode_grouped_prefix``): groups of sequences, each
sharing its own prefix (forked sampling branches, requests on one of several
system prompts), give the same result as decode attention (oracle:
``oracle.attention.paged_attention_decode``) with each group's shared blocks
read once for the group."""

import numpy as np
import pytest
import torch

import oracle.attention as oa
from pagedattention_decode_attention_gb300 import workloads as wl
from tests.gpu_helpers import TORCH_DTYPES, assert_attention_close, to_f32_numpy

pytestmark = pytest.mark.gpu


def pa():
    import pagedattention_decode_attention_gb300 as m
    return m


# Groups as ("share", prefix tokens, suffix lengths): requests on a pinned
# system prompt; or ("fork", prompt tokens, branch appends): a prompt forked
# into len(appends) branches that then diverge (the partial last block is
# copied for all but its last holder, so the whole blocks stay shared).
GROUPS = [("share", 1024, [0, 5, 300]),
          ("share", 0, [40, 17]),           # nothing shared: the suffix decode does it all
          ("fork", 100, [1, 1, 20, 3]),
          ("share", 48, [1]),
          ("share", 160, [16, 17, 900, 2]),
          ("fork", 512, [1, 16]),
          ("share", 64, [3, 1, 2, 50, 7, 9])]   # more members than one shared unit holds


def grouped_batch(groups, hq, hkv, d, dtype, seed, dev):
    """Tables from the pool; returns q, caches, tables, lengths, group_start,
    group_prefix_blocks (numpy)."""
    need = sum(t // 16 + 1 + sum(-(-s // 16) + 1 for s in sfx) for _, t, sfx in groups) + 16
    pool = pa().BlockPool(need, 16, np.random.default_rng(seed).permutation(need))
    seqs, starts, shared = [], [0], []
    for kind, tokens, tails in groups:
        root = pool.new_seq()
        for _ in range(tokens):
            pool.append_slot(root)
        if kind == "share":
            if tokens:
                pool.pin(root, tokens)
            members = []
            for n in tails:
                s = pool.new_seq()
                if tokens:
                    pool.share_prefix(root, s, tokens)
                for _ in range(n):
                    pool.append_slot(s)
                members.append(s)
        else:
            members = [root] + [pool.fork(root) for _ in tails[1:]]
            for s, n in zip(members, tails):
                for _ in range(n):
                    pool.append_slot(s)
        seqs += members
        starts.append(len(seqs))
        shared.append(tokens // 16)
    rows = [pool.block_table(s) for s in seqs]
    mb = max(len(t) for t, _ in rows)
    tables = np.full((len(rows), mb), -1, dtype=np.int32)
    for i, (t, _) in enumerate(rows):
        tables[i, :len(t)] = t
    lens = np.array([c for _, c in rows], dtype=np.int32)
    # the declared prefixes really are shared
    for g in range(len(groups)):
        a, b = starts[g], starts[g + 1]
        assert all((tables[i, :shared[g]] == tables[a, :shared[g]]).all() for i in range(a, b))
    dt = TORCH_DTYPES[dtype]
    q = wl.normal((len(seqs), hq, d), dt, seed * 10 + 1, dev)
    kc = wl.normal((need, hkv, 16, d), dt, seed * 10 + 2, dev)
    vc = wl.normal((need, hkv, 16, d), dt, seed * 10 + 3, dev)
    return (q, kc, vc, tables, lens, np.array(starts, dtype=np.int32),
            np.array(shared, dtype=np.int32))


def on(dev, *arrays):
    return [torch.from_numpy(a).to(dev) for a in arrays]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("heads", [(8, 8), (32, 8), (16, 2)], ids=["g1", "g4", "g8"])
def test_grouped_prefix_matches_oracle(gpu, dtype, head_dim, heads):
    hq, hkv = heads
    q, kc, vc, tables, lens, gs, gb = grouped_batch(GROUPS, hq, hkv, head_dim, dtype,
                                                    seed=500 + hq + head_dim, dev=gpu)
    bt, cl, gs_d, gb_d = on(gpu, tables, lens, gs, gb)
    scale = 1.0 / np.sqrt(head_dim)
    out = pa().paged_attention_decode_grouped_prefix(q, kc, vc, bt, cl, gs_d, gb_d, scale)
    pa().check_status()
    ref = oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc), tables,
                                    lens, scale)
    assert_attention_close(out, ref, TORCH_DTYPES[dtype])


def test_grouped_prefix_one_group_equals_shared_prefix(gpu):
    """One group over the whole batch is the single-prefix cascade."""
    groups = [("share", 1024, [0, 1, 15, 16, 17, 100, 300, 513, 900, 2, 64])]
    q, kc, vc, tables, lens, gs, gb = grouped_batch(groups, 32, 8, 128, "bf16", seed=520,
                                                    dev=gpu)
    bt, cl, gs_d, gb_d = on(gpu, tables, lens, gs, gb)
    scale = 1.0 / np.sqrt(128)
    got = pa().paged_attention_decode_grouped_prefix(q, kc, vc, bt, cl, gs_d, gb_d, scale)
    single = pa().paged_attention_decode_shared_prefix(q, kc, vc, bt, cl, 64, scale)
    pa().check_status()
    ref = oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc), tables,
                                    lens, scale)
    assert_attention_close(got, ref, torch.bfloat16)
    assert_attention_close(single, ref, torch.bfloat16)


@pytest.mark.parametrize("dtype,head_dim", [("bf16", 128), ("f16", 64)])
def test_grouped_prefix_one_plan_serves_every_layer(gpu, dtype, head_dim):
    """grouped_prefix_plan once, then the run on three layers' caches and
    queries: each is bit-identical to the one-shot call on that layer and
    matches the oracle."""
    dt = TORCH_DTYPES[dtype]
    q0, kc0, vc0, tables, lens, gs, gb = grouped_batch(GROUPS, 32, 8, head_dim, dtype, seed=530,
                                                       dev=gpu)
    layers = [(q0, kc0, vc0)] + [(wl.normal(q0.shape, dt, 540 + 3 * i, gpu),
                                  wl.normal(kc0.shape, dt, 541 + 3 * i, gpu),
                                  wl.normal(vc0.shape, dt, 542 + 3 * i, gpu)) for i in range(2)]
    bt, cl, gs_d, gb_d = on(gpu, tables, lens, gs, gb)
    scale = 1.0 / np.sqrt(head_dim)
    n = pa().grouped_prefix_workspace_size(len(lens), 32, 8, head_dim, tables.shape[1])
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=gpu)
    pa().grouped_prefix_plan(bt, cl, gs_d, gb_d, 32, 8, head_dim, scale, dt, ws)
    runs = [pa().paged_attention_decode_grouped_prefix_run(q, kc, vc, bt, gs_d, gb_d, scale,
                                                           ws).clone()
            for q, kc, vc in layers]
    pa().check_status()
    for (q, kc, vc), got in zip(layers, runs):
        whole = pa().paged_attention_decode_grouped_prefix(q, kc, vc, bt, cl, gs_d, gb_d, scale)
        pa().check_status()
        assert torch.equal(got, whole)
        ref = oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc),
                                        tables, lens, scale)
        assert_attention_close(got, ref, dt)


def test_grouped_prefix_mismatched_table_sets_bounds_status(gpu):
    q, kc, vc, tables, lens, gs, gb = grouped_batch(GROUPS, 8, 8, 64, "f16", seed=550, dev=gpu)
    tables = tables.copy()
    a = gs[4]                                        # group 4 shares 10 blocks
    tables[a + 1, 3] = tables[a + 1, 11]             # its second member no longer shares block 3
    bt, cl, gs_d, gb_d = on(gpu, tables, lens, gs, gb)
    pa().paged_attention_decode_grouped_prefix(q, kc, vc, bt, cl, gs_d, gb_d, 0.125)
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()


@pytest.mark.parametrize("case", ["last_start", "prefix_past_context", "unsorted"])
def test_grouped_prefix_bad_groups_set_status(gpu, case):
    q, kc, vc, tables, lens, gs, gb = grouped_batch(GROUPS, 8, 8, 64, "f16", seed=560, dev=gpu)
    gs, gb = gs.copy(), gb.copy()
    if case == "last_start":
        gs[-1] -= 1                                  # does not end at num_seqs
    elif case == "prefix_past_context":
        gb[0] = 70                                   # beyond a member's 1024 tokens
    else:
        gs[2], gs[3] = gs[3], gs[2]
    bt, cl, gs_d, gb_d = on(gpu, tables, lens, gs, gb)
    pa().paged_attention_decode_grouped_prefix(q, kc, vc, bt, cl, gs_d, gb_d, 0.125)
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()


def test_grouped_prefix_run_without_plan_sets_status(gpu):
    q, kc, vc, tables, lens, gs, gb = grouped_batch(GROUPS, 32, 8, 128, "bf16", seed=570,
                                                    dev=gpu)
    bt, gs_d, gb_d = on(gpu, tables, gs, gb)
    n = pa().grouped_prefix_workspace_size(len(lens), 32, 8, 128, tables.shape[1])
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=gpu)
    pa().paged_attention_decode_grouped_prefix_run(q, kc, vc, bt, gs_d, gb_d, 1.0 / np.sqrt(128),
                                                   ws)
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()


def test_grouped_prefix_rejects_fp32_and_bad_group_count(gpu):
    q, kc, vc, tables, lens, gs, gb = grouped_batch(GROUPS[:2], 8, 8, 64, "f16", seed=580,
                                                    dev=gpu)
    bt, cl, gs_d, gb_d = on(gpu, tables, lens, gs, gb)
    with pytest.raises(pa().PagedAttnError):
        pa().paged_attention_decode_grouped_prefix(q.float(), kc.float(), vc.float(), bt, cl,
                                                   gs_d, gb_d, 0.125)
    with pytest.raises(ValueError):                  # group_start one entry short
        pa().paged_attention_decode_grouped_prefix(q, kc, vc, bt, cl, gs_d[:-1], gb_d, 0.125)


@pytest.mark.parametrize("dtype,head_dim", [("bf16", 128), ("f16", 64)])
def test_grouped_prefix_append_run_equals_append_then_run(gpu, dtype, head_dim):
    """The fused grouped run stores each sequence's new row past its group's
    prefix and attends it: caches and output bit-identical to kv_append
    followed by the run; the oracle over the updated caches agrees."""
    dt = TORCH_DTYPES[dtype]
    q, kc, vc, tables, lens, gs, gb = grouped_batch(GROUPS, 32, 8, head_dim, dtype, seed=590,
                                                    dev=gpu)
    first_private = np.repeat(gb.astype(np.int64) * 16, np.diff(gs))
    pos = lens.astype(np.int64) - 1
    slots = tables[np.arange(len(lens)), pos // 16].astype(np.int64) * 16 + pos % 16
    slots[pos < first_private] = -1          # nothing past the prefix: no new token there
    slots_d = torch.from_numpy(slots).to(gpu)
    k_new = wl.normal((len(lens), 8, head_dim), dt, 591, gpu)
    v_new = wl.normal((len(lens), 8, head_dim), dt, 592, gpu)
    bt, cl, gs_d, gb_d = on(gpu, tables, lens, gs, gb)
    scale = 1.0 / np.sqrt(head_dim)
    n = pa().grouped_prefix_workspace_size(len(lens), 32, 8, head_dim, tables.shape[1])
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=gpu)
    kc2, vc2 = kc.clone(), vc.clone()
    pa().grouped_prefix_plan(bt, cl, gs_d, gb_d, 32, 8, head_dim, scale, dt, ws)
    pa().kv_append(k_new, v_new, kc, vc, slots_d)
    ref = pa().paged_attention_decode_grouped_prefix_run(q, kc, vc, bt, gs_d, gb_d, scale,
                                                         ws).clone()
    got = pa().paged_attention_decode_grouped_prefix_append_run(q, k_new, v_new, slots_d, kc2,
                                                                vc2, bt, gs_d, gb_d, scale, ws)
    pa().check_status()
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    assert torch.equal(got, ref)
    want = oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc), tables,
                                     lens, scale)
    assert_attention_close(got, want, dt)
