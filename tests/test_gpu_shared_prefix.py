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
