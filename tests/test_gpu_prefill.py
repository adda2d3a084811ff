"""GPU parity of chunked-prefill attention (``pa_paged_attention_prefill``).

Expected values come from ``oracle.attention.paged_attention_prefill`` on
host copies of the same seeded inputs; tolerances are the attention ones of
``tests/gpu_helpers.py``.
"""

import numpy as np
import pytest
import torch

import oracle.attention as oa
from pagedattention_decode_attention_gb300 import workloads as wl
from tests.gpu_helpers import TORCH_DTYPES, assert_attention_close, custom_batch, to_f32_numpy

pytestmark = pytest.mark.gpu


def pa():
    import pagedattention_decode_attention_gb300 as m
    return m


def prefill_inputs(lens, qlens, hq, hkv, d, dtype, seed, dev):
    """Paged caches for the sequences' full contexts, their chunk queries."""
    batch = custom_batch(lens, hq, hkv, d, dtype, seed=seed)
    dt = TORCH_DTYPES[dtype]
    shape = (batch.num_blocks, hkv, 16, d)
    kc = wl.normal(shape, dt, seed * 10 + 2, dev)
    vc = wl.normal(shape, dt, seed * 10 + 3, dev)
    qs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = wl.normal((int(qs[-1]), hq, d), dt, seed * 10 + 1, dev)
    return batch, q, kc, vc, qs


def run_prefill(batch, q, kc, vc, qs, dev, workspace=None, out=None):
    out = pa().paged_attention_prefill(
        q, kc, vc, torch.from_numpy(batch.block_tables).to(dev),
        torch.from_numpy(batch.context_lens).to(dev), torch.from_numpy(qs).to(dev), batch.scale,
        out=out, workspace=workspace)
    pa().check_status()
    return out


def oracle_prefill(batch, q, kc, vc, qs, rows=None):
    return oa.paged_attention_prefill(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc),
                                      batch.block_tables, batch.context_lens, qs, batch.scale,
                                      rows=rows)


# whole prompts, partial chunks over a cached prefix, decode rows, an idle
# sequence, chunks crossing blocks and a long prefix with a short chunk
LENS = [40, 17, 300, 1, 530, 2000, 64, 900]
QLENS = [40, 17, 37, 1, 1, 9, 0, 128]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("heads", [(8, 8), (32, 8), (16, 2)], ids=["g1", "g4", "g8"])
def test_prefill_matches_oracle(gpu, dtype, head_dim, heads):
    hq, hkv = heads
    batch, q, kc, vc, qs = prefill_inputs(LENS, QLENS, hq, hkv, head_dim, dtype,
                                          seed=60 + hq + head_dim, dev=gpu)
    out = run_prefill(batch, q, kc, vc, qs, gpu)
    assert_attention_close(out, oracle_prefill(batch, q, kc, vc, qs), TORCH_DTYPES[dtype])


@pytest.mark.parametrize("head_dim", [64, 128])
def test_prefill_fp32_matches_oracle(gpu, head_dim):
    batch, q, kc, vc, qs = prefill_inputs([33, 70, 5], [33, 20, 1], 6, 2, head_dim, "f32",
                                          seed=81, dev=gpu)
    out = run_prefill(batch, q, kc, vc, qs, gpu)
    assert_attention_close(out, oracle_prefill(batch, q, kc, vc, qs), torch.float32)


def test_prefill_long_context_short_chunks_splits(gpu):
    """Few query blocks over long contexts: the plan splits the KV range and
    the splits are merged; the answer must not depend on it."""
    batch, q, kc, vc, qs = prefill_inputs([12345, 7000], [3, 16], 32, 8, 128, "bf16", seed=83,
                                          dev=gpu)
    out = run_prefill(batch, q, kc, vc, qs, gpu)
    assert_attention_close(out, oracle_prefill(batch, q, kc, vc, qs), torch.bfloat16)


def test_prefill_long_chunk_sampled_rows(gpu):
    """A 2048-token chunk after a 2048-token prefix, 4 sequences: sampled rows."""
    lens, qlens = [4096, 2048, 3000, 2100], [2048, 2048, 1000, 77]
    batch, q, kc, vc, qs = prefill_inputs(lens, qlens, 32, 8, 128, "bf16", seed=85, dev=gpu)
    out = run_prefill(batch, q, kc, vc, qs, gpu)
    rows = sorted(set([0, 1, 15, 16, 17, 2047, 2048, 2049, 4095, 4096, 4500, 5095, 5096, 5172]
                      + list(np.random.default_rng(1).integers(0, int(qs[-1]), 24))))
    ref = oracle_prefill(batch, q, kc, vc, qs, rows=rows)
    assert_attention_close(out, ref, torch.bfloat16, rows=rows)


def test_prefill_one_token_chunks_match_decode(gpu):
    """T = 1 for every sequence is decode: both kernels agree with the oracle."""
    lens = [1, 16, 17, 300, 2000]
    batch, q, kc, vc, qs = prefill_inputs(lens, [1] * 5, 32, 8, 128, "f16", seed=87, dev=gpu)
    out = run_prefill(batch, q, kc, vc, qs, gpu)
    dec = pa().paged_attention_decode(q, kc, vc, torch.from_numpy(batch.block_tables).to(gpu),
                                      torch.from_numpy(batch.context_lens).to(gpu), batch.scale)
    pa().check_status()
    ref = oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc),
                                    batch.block_tables, batch.context_lens, batch.scale)
    assert_attention_close(out, ref, torch.float16)
    assert_attention_close(dec, ref, torch.float16)


def test_prefill_placement_invariance_is_bit_exact(gpu):
    batch, q, kc, vc, qs = prefill_inputs([100, 260], [60, 200], 16, 4, 128, "bf16", seed=89,
                                          dev=gpu)
    base = run_prefill(batch, q, kc, vc, qs, gpu).clone()
    pi = torch.from_numpy(np.random.default_rng(5).permutation(batch.num_blocks)).to(gpu)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    bt = torch.from_numpy(batch.block_tables).to(gpu)
    bt2 = torch.where(bt >= 0, pi[bt.clamp(min=0).long()].int(), bt).contiguous()
    moved = pa().paged_attention_prefill(q, kc2, vc2, bt2,
                                         torch.from_numpy(batch.context_lens).to(gpu),
                                         torch.from_numpy(qs).to(gpu), batch.scale)
    pa().check_status()
    assert torch.equal(base, moved)


def test_prefill_workspace_reused_without_init(gpu):
    batch, q, kc, vc, qs = prefill_inputs([5000, 90], [7, 90], 32, 8, 128, "f16", seed=91,
                                          dev=gpu)
    ws = pa().alloc_prefill_workspace(2, int(qs[-1]), 32, 8, 128, gpu)
    ws.fill_(0xCD)
    outs = [run_prefill(batch, q, kc, vc, qs, gpu, workspace=ws).clone() for _ in range(3)]
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    assert_attention_close(outs[0], oracle_prefill(batch, q, kc, vc, qs), torch.float16)


def test_prefill_chunk_longer_than_context_sets_bounds_status(gpu):
    batch, q, kc, vc, qs = prefill_inputs([20, 30], [20, 30], 8, 8, 64, "bf16", seed=93, dev=gpu)
    qs_bad = np.array([0, 20, 50], dtype=np.int32)
    cl = torch.from_numpy(np.array([20, 25], dtype=np.int32)).to(gpu)   # 30 queries, 25 tokens
    out = torch.zeros_like(q)
    pa().paged_attention_prefill(q, kc, vc, torch.from_numpy(batch.block_tables).to(gpu), cl,
                                 torch.from_numpy(qs_bad).to(gpu), batch.scale, out=out)
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()
    assert torch.count_nonzero(out[20:]) == 0                       # skipped sequence
    ref = oracle_prefill(batch, q[:20], kc, vc, np.array([0, 20, 20], dtype=np.int32))
    assert_attention_close(out[:20], ref[:20], torch.bfloat16)


@pytest.mark.parametrize("dtype,head_dim", [("bf16", 128), ("f16", 128), ("bf16", 64), ("f32", 128)])
def test_prefill_one_plan_serves_every_layer(gpu, dtype, head_dim):
    """prefill_plan once, then paged_attention_prefill_run on three layers'
    caches and queries: each is bit-identical to the one-shot call on that
    layer and matches the oracle."""
    dt = TORCH_DTYPES[dtype]
    batch = custom_batch(LENS, 32, 8, head_dim, dtype, seed=95)
    qs = np.concatenate([[0], np.cumsum(QLENS)]).astype(np.int32)
    shape = (batch.num_blocks, 8, 16, head_dim)
    layers = [(wl.normal((int(qs[-1]), 32, head_dim), dt, 950 + 3 * i, gpu),
               wl.normal(shape, dt, 951 + 3 * i, gpu), wl.normal(shape, dt, 952 + 3 * i, gpu))
              for i in range(3)]
    bt = torch.from_numpy(batch.block_tables).to(gpu)
    cl = torch.from_numpy(batch.context_lens).to(gpu)
    qsd = torch.from_numpy(qs).to(gpu)
    ws = pa().alloc_prefill_workspace(len(LENS), int(qs[-1]), 32, 8, head_dim, gpu)
    pa().prefill_plan(cl, qsd, int(qs[-1]), 32, 8, head_dim, batch.max_blocks, batch.scale, dt, ws)
    runs = [pa().paged_attention_prefill_run(q, kc, vc, bt, cl, qsd, batch.scale, ws).clone()
            for q, kc, vc in layers]
    pa().check_status()
    for (q, kc, vc), got in zip(layers, runs):
        whole = run_prefill(batch, q, kc, vc, qs, gpu)
        assert torch.equal(got, whole)
        assert_attention_close(got, oracle_prefill(batch, q, kc, vc, qs), dt)


def test_prefill_run_without_plan_sets_status(gpu):
    batch, q, kc, vc, qs = prefill_inputs([300, 90], [64, 90], 32, 8, 128, "bf16", seed=97,
                                          dev=gpu)
    ws = pa().alloc_prefill_workspace(2, int(qs[-1]), 32, 8, 128, gpu)
    ws.zero_()
    out = torch.zeros_like(q)
    pa().paged_attention_prefill_run(q, kc, vc, torch.from_numpy(batch.block_tables).to(gpu),
                                     torch.from_numpy(batch.context_lens).to(gpu),
                                     torch.from_numpy(qs).to(gpu), batch.scale, ws, out=out)
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()
    assert torch.count_nonzero(out) == 0
    # a plan makes the same workspace usable
    pa().prefill_plan(torch.from_numpy(batch.context_lens).to(gpu), torch.from_numpy(qs).to(gpu),
                      int(qs[-1]), 32, 8, 128, batch.max_blocks, batch.scale, torch.bfloat16, ws)
    got = pa().paged_attention_prefill_run(q, kc, vc, torch.from_numpy(batch.block_tables).to(gpu),
                                           torch.from_numpy(batch.context_lens).to(gpu),
                                           torch.from_numpy(qs).to(gpu), batch.scale, ws)
    pa().check_status()
    assert_attention_close(got, oracle_prefill(batch, q, kc, vc, qs), torch.bfloat16)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_split_merge_with_mixed_tiles(gpu, dtype):
    """Few query blocks over long contexts: the plan splits their KV ranges and
    the kernel merges the splits; query blocks with one and with two 128-row
    tiles interleave, which exercises the merge's phase bookkeeping."""
    lens, qlens = [9000, 5000, 300, 4100], [300, 20, 290, 33]
    batch, q, kc, vc, qs = prefill_inputs(lens, qlens, 32, 8, 128, dtype, seed=99, dev=gpu)
    out = run_prefill(batch, q, kc, vc, qs, gpu)
    again = run_prefill(batch, q, kc, vc, qs, gpu)
    assert torch.equal(out, again)            # the counters reset between runs
    assert_attention_close(out, oracle_prefill(batch, q, kc, vc, qs), TORCH_DTYPES[dtype])


@pytest.mark.parametrize("heads", [(32, 8), (8, 8)], ids=["g4", "g1"])
def test_prefill_one_and_two_tile_items_alternate(gpu, heads):
    """Enough query blocks not to split, with items of one 128-row query tile
    (whose S alternates between the two S buffers) and of two tiles mixed in
    the work list, over contexts of 3 to 24 KV tiles (odd and even counts):
    the buffers change hands between the two kinds of item."""
    hq, hkv = heads
    g = hq // hkv
    # rows = chunk * G: one tile (<= 128), two tiles, two with a partial second
    chunks = [max(1, 100 // g), 256 // g, 132 // g, max(1, 20 // g), 360 // g, 64 // g,
              max(1, 120 // g), 200 // g] * 2
    rng = np.random.default_rng(123)
    lens = [int(c + rng.integers(300, 3000)) for c in chunks]
    batch, q, kc, vc, qs = prefill_inputs(lens, chunks, hq, hkv, 128, "bf16", seed=124, dev=gpu)
    out = run_prefill(batch, q, kc, vc, qs, gpu)
    again = run_prefill(batch, q, kc, vc, qs, gpu)
    assert torch.equal(out, again)
    assert_attention_close(out, oracle_prefill(batch, q, kc, vc, qs), torch.bfloat16)
