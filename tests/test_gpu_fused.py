"""GPU parity of the fused append + attention entry point.

``paged_attention_decode_append_run`` must equal ``kv_append`` followed by
``paged_attention_decode_run`` bit for bit (outputs and both whole caches), and
match the oracle (its own append into host copies of the caches, then its
attention) within the attention tolerance of ``tests/gpu_helpers.py``.
"""

import numpy as np
import pytest
import torch

import oracle.attention as oa
from pagedattention_decode_attention_gb300 import workloads as wl
from tests.gpu_helpers import (TORCH_DTYPES, assert_attention_close, custom_batch, decode_inputs,
                               to_f32_numpy)

pytestmark = pytest.mark.gpu

LENS = [1, 2, 15, 16, 17, 31, 100, 511, 512, 513, 1100, 2000, 4100]


def pa():
    import pagedattention_decode_attention_gb300 as m
    return m


def new_rows(batch, dev, seed):
    dt = TORCH_DTYPES[batch.dtype]
    shape = (batch.num_seqs, batch.num_kv_heads, batch.head_dim)
    return wl.normal(shape, dt, seed, dev), wl.normal(shape, dt, seed + 1, dev)


def unfused(batch, q, kc, vc, bt, cl, kn, vn, slots):
    kc, vc = kc.clone(), vc.clone()
    ws = pa().alloc_workspace(batch.num_seqs, batch.num_q_heads, batch.num_kv_heads,
                              batch.head_dim, batch.max_blocks, q.device)
    pa().kv_append(kn, vn, kc, vc, slots)
    pa().paged_attention_decode_plan(cl, batch.num_q_heads, batch.num_kv_heads, batch.head_dim,
                                     batch.max_blocks, ws)
    out = pa().paged_attention_decode_run(q, kc, vc, bt, cl, batch.scale, ws)
    return out, kc, vc


def fused(batch, q, kc, vc, bt, cl, kn, vn, slots):
    kc, vc = kc.clone(), vc.clone()
    ws = pa().alloc_workspace(batch.num_seqs, batch.num_q_heads, batch.num_kv_heads,
                              batch.head_dim, batch.max_blocks, q.device)
    ws.fill_(0x5A)                                   # garbage: the plan initialises it
    pa().paged_attention_decode_plan(cl, batch.num_q_heads, batch.num_kv_heads, batch.head_dim,
                                     batch.max_blocks, ws)
    out = pa().paged_attention_decode_append_run(q, kn, vn, slots, kc, vc, bt, cl, batch.scale, ws)
    return out, kc, vc


def oracle_fused(batch, q, kc, vc, kn, vn, slots):
    """Oracle: append into float32 host copies of the caches, then attend."""
    hk, hv = to_f32_numpy(kc).copy(), to_f32_numpy(vc).copy()
    oa.kv_append(to_f32_numpy(kn), to_f32_numpy(vn), hk, hv, slots)
    return oa.paged_attention_decode(to_f32_numpy(q), hk, hv, batch.block_tables,
                                     batch.context_lens, batch.scale)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("heads", [(8, 8), (32, 8), (16, 2)], ids=["g1", "g4", "g8"])
def test_fused_equals_append_then_run(gpu, dtype, head_dim, heads):
    hq, hkv = heads
    batch = custom_batch(LENS, hq, hkv, head_dim, dtype, seed=700 + hq + head_dim)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    kn, vn = new_rows(batch, gpu, 900 + hq)
    slots_np = batch.new_token_slots()
    slots = torch.from_numpy(slots_np).to(gpu)
    o1, k1, v1 = unfused(batch, q, kc, vc, bt, cl, kn, vn, slots)
    o2, k2, v2 = fused(batch, q, kc, vc, bt, cl, kn, vn, slots)
    pa().check_status()
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(o1, o2)
    assert_attention_close(o2, oracle_fused(batch, q, kc, vc, kn, vn, slots_np),
                           TORCH_DTYPES[dtype])


def test_fused_padding_slots_and_empty_sequence(gpu):
    """A negative slot stores nothing and attends the cache as it is; a
    sequence with no context still has its new row stored, and a zero output."""
    lens = [0, 40, 700, 16, 0, 3]
    batch = custom_batch(lens, 32, 8, 128, "bf16", seed=41)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    kn, vn = new_rows(batch, gpu, 77)
    slots_np = np.where(batch.context_lens > 0, 0, -1).astype(np.int64)
    pos = np.maximum(batch.context_lens.astype(np.int64) - 1, 0)
    tab = batch.block_tables[np.arange(batch.num_seqs), pos // 16].astype(np.int64)
    slots_np = np.where(batch.context_lens > 0, tab * 16 + pos % 16, -1)
    slots_np[2] = -1                                 # padding: no new token for sequence 2
    free = sorted(set(range(batch.num_blocks)) - set(batch.block_tables[batch.block_tables >= 0]))
    slots_np[4] = free[0] * 16 + 5                   # empty sequence with a new token
    slots = torch.from_numpy(slots_np).to(gpu)
    o1, k1, v1 = unfused(batch, q, kc, vc, bt, cl, kn, vn, slots)
    o2, k2, v2 = fused(batch, q, kc, vc, bt, cl, kn, vn, slots)
    pa().check_status()
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(o1, o2)
    assert torch.count_nonzero(o2[0]) == 0 and torch.count_nonzero(o2[4]) == 0
    assert torch.equal(k2[free[0], :, 5], kn[4])
    assert_attention_close(o2, oracle_fused(batch, q, kc, vc, kn, vn, slots_np), torch.bfloat16)


def test_fused_one_plan_many_layers(gpu):
    """One plan, then a fused call per layer on separate caches."""
    batch = custom_batch(LENS, 32, 8, 128, "f16", seed=43)
    ws = pa().alloc_workspace(batch.num_seqs, 32, 8, 128, batch.max_blocks, gpu)
    bt = torch.from_numpy(batch.block_tables).to(gpu)
    cl = torch.from_numpy(batch.context_lens).to(gpu)
    slots_np = batch.new_token_slots()
    slots = torch.from_numpy(slots_np).to(gpu)
    pa().paged_attention_decode_plan(cl, 32, 8, 128, batch.max_blocks, ws)
    layers = []
    for layer in range(3):
        q, kc, vc, _, _ = decode_inputs(batch, gpu, seed_offset=layer)
        kn, vn = new_rows(batch, gpu, 300 + 2 * layer)
        ref = oracle_fused(batch, q, kc, vc, kn, vn, slots_np)
        out = pa().paged_attention_decode_append_run(q, kn, vn, slots, kc, vc, bt, cl,
                                                     batch.scale, ws)
        layers.append((out, ref))
    pa().check_status()
    for out, ref in layers:
        assert_attention_close(out, ref, torch.float16)


@pytest.mark.parametrize("case", ["out_of_range", "not_last_position"])
def test_fused_bad_slot_sets_bounds_status(gpu, case):
    batch = custom_batch([40, 300], 8, 8, 64, "bf16", seed=45)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    kn, vn = new_rows(batch, gpu, 11)
    slots_np = batch.new_token_slots()
    if case == "out_of_range":
        slots_np[1] = batch.num_blocks * 16
    else:
        slots_np[1] -= 1                             # the slot of the token before the last
    before = kc.clone()
    fused(batch, q, kc, vc, bt, cl, kn, vn, torch.from_numpy(slots_np).to(gpu))
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()
    assert torch.equal(kc, before)                   # fused() worked on clones
