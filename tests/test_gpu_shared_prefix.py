"""GPU parity of the shared-prefix decode (``pa_paged_attention_decode_shared_prefix``):
the same result as decode attention (oracle: ``oracle.attention.paged_attention_decode``),
with the shared blocks read once for the whole batch."""

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


def shared_batch(prefix_tokens, suffixes, hq, hkv, d, dtype, seed, dev):
    """Tables from the pool: a pinned prefix sequence, every request shares its
    blocks and appends its own suffix."""
    nb = prefix_tokens // 16 + sum(-(-s // 16) for s in suffixes) + 8
    pool = pa().BlockPool(nb, 16, np.random.default_rng(seed).permutation(nb))
    root = pool.new_seq()
    for _ in range(prefix_tokens):
        pool.append_slot(root)
    pool.pin(root, prefix_tokens)
    seqs = []
    for n in suffixes:
        s = pool.new_seq()
        pool.share_prefix(root, s, prefix_tokens)
        for _ in range(n):
            pool.append_slot(s)
        seqs.append(s)
    mb = max(len(pool.block_table(s)[0]) for s in seqs)
    tables, lens = pool.tables(seqs, mb)
    dt = TORCH_DTYPES[dtype]
    q = wl.normal((len(seqs), hq, d), dt, seed * 10 + 1, dev)
    kc = wl.normal((nb, hkv, 16, d), dt, seed * 10 + 2, dev)
    vc = wl.normal((nb, hkv, 16, d), dt, seed * 10 + 3, dev)
    return q, kc, vc, tables, lens


SUFFIXES = [0, 1, 15, 16, 17, 100, 300, 513, 900, 2, 64]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("heads", [(8, 8), (32, 8), (16, 2)], ids=["g1", "g4", "g8"])
def test_shared_prefix_matches_oracle(gpu, dtype, head_dim, heads):
    hq, hkv = heads
    q, kc, vc, tables, lens = shared_batch(1024, SUFFIXES, hq, hkv, head_dim, dtype,
                                           seed=300 + hq + head_dim, dev=gpu)
    out = pa().paged_attention_decode_shared_prefix(
        q, kc, vc, torch.from_numpy(tables).to(gpu), torch.from_numpy(lens).to(gpu), 1024 // 16,
        1.0 / np.sqrt(head_dim))
    pa().check_status()
    ref = oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc), tables,
                                    lens, 1.0 / np.sqrt(head_dim))
    assert_attention_close(out, ref, TORCH_DTYPES[dtype])


def test_shared_prefix_small_batch_and_short_prefix(gpu):
    """Few queries over a 48-token prefix (the prefix phase then splits)."""
    q, kc, vc, tables, lens = shared_batch(48, [5, 0, 40], 32, 8, 128, "bf16", seed=41, dev=gpu)
    bt, cl = torch.from_numpy(tables).to(gpu), torch.from_numpy(lens).to(gpu)
    out = pa().paged_attention_decode_shared_prefix(q, kc, vc, bt, cl, 3, 1.0 / np.sqrt(128))
    plain = pa().paged_attention_decode(q, kc, vc, bt, cl, 1.0 / np.sqrt(128))
    pa().check_status()
    ref = oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc), tables,
                                    lens, 1.0 / np.sqrt(128))
    assert_attention_close(out, ref, torch.bfloat16)
    assert_attention_close(plain, ref, torch.bfloat16)


def test_shared_prefix_mismatched_table_sets_bounds_status(gpu):
    q, kc, vc, tables, lens = shared_batch(64, [10, 20], 8, 8, 64, "f16", seed=43, dev=gpu)
    tables = tables.copy()
    tables[1, 2] = tables[1, 4]                      # sequence 1 no longer shares block 2
    pa().paged_attention_decode_shared_prefix(
        q, kc, vc, torch.from_numpy(tables).to(gpu), torch.from_numpy(lens).to(gpu), 4, 0.125)
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()


@pytest.mark.parametrize("dtype,head_dim,prefix", [("bf16", 128, 1024), ("f16", 64, 1024),
                                                   ("bf16", 128, 0), ("f32", 128, 1024)])
def test_shared_prefix_one_plan_serves_every_layer(gpu, dtype, head_dim, prefix):
    """shared_prefix_plan once, then the run on three layers' caches and
    queries: each is bit-identical to the one-shot call on that layer and
    matches the oracle (prefix 0 is the plain decode's plan and run)."""
    dt = TORCH_DTYPES[dtype]
    q0, kc0, vc0, tables, lens = shared_batch(1024, SUFFIXES, 32, 8, head_dim, dtype, seed=350,
                                              dev=gpu)
    layers = [(q0, kc0, vc0)] + [(wl.normal(q0.shape, dt, 360 + 3 * i, gpu),
                                  wl.normal(kc0.shape, dt, 361 + 3 * i, gpu),
                                  wl.normal(vc0.shape, dt, 362 + 3 * i, gpu)) for i in range(2)]
    bt, cl = torch.from_numpy(tables).to(gpu), torch.from_numpy(lens).to(gpu)
    mb = tables.shape[1]
    scale = 1.0 / np.sqrt(head_dim)
    n = pa().shared_prefix_workspace_size(len(SUFFIXES), 32, 8, head_dim, mb)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=gpu)
    pa().shared_prefix_plan(cl, prefix // 16, 32, 8, head_dim, mb, scale, dt, ws)
    runs = [pa().paged_attention_decode_shared_prefix_run(q, kc, vc, bt, cl, prefix // 16, scale,
                                                          ws).clone()
            for q, kc, vc in layers]
    pa().check_status()
    for (q, kc, vc), got in zip(layers, runs):
        whole = pa().paged_attention_decode_shared_prefix(q, kc, vc, bt, cl, prefix // 16, scale)
        pa().check_status()
        assert torch.equal(got, whole)
        ref = oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc),
                                        tables, lens, scale)
        assert_attention_close(got, ref, dt)


def test_shared_prefix_run_without_plan_sets_status(gpu):
    q, kc, vc, tables, lens = shared_batch(256, [5, 40, 100], 32, 8, 128, "bf16", seed=45,
                                           dev=gpu)
    bt, cl = torch.from_numpy(tables).to(gpu), torch.from_numpy(lens).to(gpu)
    n = pa().shared_prefix_workspace_size(3, 32, 8, 128, tables.shape[1])
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=gpu)
    pa().paged_attention_decode_shared_prefix_run(q, kc, vc, bt, cl, 16, 1.0 / np.sqrt(128), ws)
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()


@pytest.mark.parametrize("heads", [(8, 8), (32, 8), (16, 2)], ids=["g1", "g4", "g8"])
def test_shared_prefix_split_with_partial_tiles(gpu, heads):
    """A 63-block prefix: the prefix phase's splits are 7 or 8 blocks, so a
    split's last 128-token tile is partial and the tokens past its last block
    (the next split's) must not count."""
    hq, hkv = heads
    q, kc, vc, tables, lens = shared_batch(1008, SUFFIXES, hq, hkv, 128, "bf16", seed=47 + hq,
                                           dev=gpu)
    bt, cl = torch.from_numpy(tables).to(gpu), torch.from_numpy(lens).to(gpu)
    out = pa().paged_attention_decode_shared_prefix(q, kc, vc, bt, cl, 63, 1.0 / np.sqrt(128))
    pa().check_status()
    ref = oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc), tables,
                                    lens, 1.0 / np.sqrt(128))
    assert_attention_close(out, ref, torch.bfloat16)


def new_token_inputs(q, kc, tables, lens, first_private, seed, dev):
    """Each sequence's newest token as the step's new row: its slot (-1 where
    the token lies inside the shared blocks: copy-on-write never appends
    there) and random K/V rows."""
    pos = lens.astype(np.int64) - 1
    slots = tables[np.arange(len(lens)), pos // 16].astype(np.int64) * 16 + pos % 16
    slots[pos < first_private] = -1
    hkv, d = kc.shape[1], kc.shape[3]
    k_new = wl.normal((len(lens), hkv, d), kc.dtype, seed, dev)
    v_new = wl.normal((len(lens), hkv, d), kc.dtype, seed + 1, dev)
    return k_new, v_new, torch.from_numpy(slots).to(dev)


@pytest.mark.parametrize("dtype,head_dim", [("bf16", 128), ("f16", 64)])
def test_shared_prefix_append_run_equals_append_then_run(gpu, dtype, head_dim):
    """The fused run stores the new rows and attends them: caches and output
    bit-identical to kv_append followed by the run, and the oracle over the
    updated caches agrees."""
    dt = TORCH_DTYPES[dtype]
    q, kc, vc, tables, lens = shared_batch(1024, SUFFIXES, 32, 8, head_dim, dtype, seed=370,
                                           dev=gpu)
    k_new, v_new, slots = new_token_inputs(q, kc, tables, lens, 1024, 380, gpu)
    bt, cl = torch.from_numpy(tables).to(gpu), torch.from_numpy(lens).to(gpu)
    mb, scale = tables.shape[1], 1.0 / np.sqrt(head_dim)
    n = pa().shared_prefix_workspace_size(len(lens), 32, 8, head_dim, mb)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=gpu)
    kc2, vc2 = kc.clone(), vc.clone()
    pa().shared_prefix_plan(cl, 64, 32, 8, head_dim, mb, scale, dt, ws)
    pa().kv_append(k_new, v_new, kc, vc, slots)
    ref = pa().paged_attention_decode_shared_prefix_run(q, kc, vc, bt, cl, 64, scale, ws).clone()
    got = pa().paged_attention_decode_shared_prefix_append_run(q, k_new, v_new, slots, kc2, vc2,
                                                               bt, cl, 64, scale, ws)
    pa().check_status()
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    assert torch.equal(got, ref)
    want = oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc), tables,
                                     lens, scale)
    assert_attention_close(got, want, dt)


def test_shared_prefix_append_into_the_prefix_sets_bounds_status(gpu):
    """A new token with nothing past the prefix would be written into a
    shared block: refused through the status word."""
    q, kc, vc, tables, lens = shared_batch(256, [0, 5, 40], 32, 8, 128, "bf16", seed=390,
                                           dev=gpu)
    k_new, v_new, slots = new_token_inputs(q, kc, tables, lens, 0, 391, gpu)  # every slot set
    bt, cl = torch.from_numpy(tables).to(gpu), torch.from_numpy(lens).to(gpu)
    n = pa().shared_prefix_workspace_size(3, 32, 8, 128, tables.shape[1])
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=gpu)
    pa().shared_prefix_plan(cl, 16, 32, 8, 128, tables.shape[1], 0.125, torch.bfloat16, ws)
    pa().paged_attention_decode_shared_prefix_append_run(q, k_new, v_new, slots, kc, vc, bt, cl,
                                                         16, 0.125, ws)
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()
