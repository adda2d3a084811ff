"""The seeded synthetic inputs (CPU): every workload has the shapes, length
distributions and block placement its recipe states, and the same seed gives
the same batch."""

import math

import numpy as np
import pytest

from pagedattention_decode_attention_gb300 import workloads as wl


def check_tables(batch):
    """Tables hold ceil(len / 16) blocks per sequence, -1 after them, and the
    used entries are distinct physical blocks of the pool."""
    used = []
    for b, ctx in enumerate(batch.context_lens):
        n = -(-int(ctx) // 16)
        row = batch.block_tables[b]
        assert (row[:n] >= 0).all() and (row[:n] < batch.num_blocks).all()
        assert (row[n:] == -1).all()
        used.extend(row[:n].tolist())
    assert len(used) == len(set(used)), "a physical block is used twice"


def test_log_uniform_lengths_follow_the_reading():
    """clip(round(exp(U(ln lo, ln hi))), lo, hi): inside the range, median near
    sqrt(lo * hi), and uniform in log space (equal mass per decade)."""
    gen = np.random.default_rng(0)
    x = wl.log_uniform_lengths(200_000, 16, 2048, gen)
    assert x.min() >= 16 and x.max() <= 2048 and x.dtype == np.int32
    assert abs(np.median(x) / math.sqrt(16 * 2048) - 1) < 0.02
    lo, hi = np.mean(x < 181), np.mean(x >= 181)          # split at sqrt(16 * 2048)
    assert abs(lo - hi) < 0.01


def test_lognormal_lengths_follow_the_reading():
    gen = np.random.default_rng(1)
    x = wl.lognormal_lengths(200_000, 512.0, 1.0, 1, 16384, gen)
    assert x.min() >= 1 and x.max() <= 16384
    assert abs(np.median(x) / 512 - 1) < 0.02
    assert abs(np.std(np.log(x)) - 1.0) < 0.02


def test_tiny_workload():
    b = wl.tiny()
    assert (b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim, b.dtype) == (4, 4, 4, 64, "f32")
    assert b.num_blocks == 64 and b.context_lens.min() >= 1 and b.context_lens.max() <= 100
    check_tables(b)


def test_mha_7b_workload():
    b = wl.mha_7b()
    assert (b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim, b.dtype, b.num_layers) == \
        (64, 32, 32, 128, "f16", 32)
    assert b.context_lens.min() >= 16 and b.context_lens.max() <= 2048
    need = int(wl.num_blocks_for(b.context_lens).sum())
    assert b.num_blocks == math.ceil(1.1 * need)              # blocks needed + 10 % free
    check_tables(b)


def test_gqa_8b_workload():
    b = wl.gqa_8b()
    assert (b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim, b.dtype) == (128, 32, 8, 128, "bf16")
    assert (b.context_lens[-4:] == 8192).all()                 # 124 log-uniform + 4 fixed
    assert b.context_lens[:-4].min() >= 128 and b.context_lens[:-4].max() <= 8192
    check_tables(b)


def test_prefill_8b_workload():
    b = wl.prefill_8b()
    q = b.extra["query_lens"]
    assert b.num_seqs == 16 and (q == 512).all() and b.num_layers == 8
    prefix = b.context_lens - q
    assert prefix.min() >= 16 and prefix.max() <= 8192
    check_tables(b)


def test_prefix_mix_and_sampling_scripts():
    p = wl.prefix_mix()
    assert p.prefix_len == 1024 and len(p.suffix_lens) == 100
    assert p.suffix_lens.min() >= 1 and p.suffix_lens.max() <= 16384
    assert sorted(p.initial_order) == list(range(p.num_blocks))
    s = wl.sampling_cow()
    assert (s.prompts, s.prompt_len, s.branches, s.steps) == (32, 1024, 4, 256)
    assert s.shared_extra.min() >= 1 and s.shared_extra.max() <= 15   # a partial last block
    assert (wl.sampling_cow(zero_extra=True).shared_extra == 0).all()
    assert sorted(s.initial_order) == list(range(s.num_blocks))


def test_new_token_slots_are_the_last_positions():
    b = wl.gqa_8b()
    slots = b.new_token_slots()
    for i in (0, 17, 127):
        pos = int(b.context_lens[i]) - 1
        assert slots[i] == int(b.block_tables[i, pos // 16]) * 16 + pos % 16


@pytest.mark.parametrize("make", [wl.tiny, wl.mha_7b, wl.gqa_8b, wl.prefill_8b])
def test_same_seed_same_batch(make):
    a, b = make(), make()
    assert np.array_equal(a.context_lens, b.context_lens)
    assert np.array_equal(a.block_tables, b.block_tables)
    c = make(seed=12345)
    assert not np.array_equal(a.block_tables, c.block_tables)
