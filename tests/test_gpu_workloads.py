"""The five workloads end to end on the GPU, checked against the oracle.

Every oracle input comes from the seeded generators: the oracle keeps its own
host copies of the caches, written through ``oracle.attention.kv_append`` /
``block_copy`` from the generator's K/V values and the Python pool model's
slots, and is compared bit for bit with the device caches that the CUDA path
wrote.  Attention outputs are compared within the stated tolerance on every
sequence at small sizes and on sampled sequences at full size.
"""

import numpy as np
import pytest
import torch

import oracle.attention as oa
from oracle.pool import BlockPool as ModelPool
from pagedattention_decode_attention_gb300 import workloads as wl
from tests.gpu_helpers import (TORCH_DTYPES, assert_attention_close, decode_inputs, oracle_decode,
                               to_f32_numpy)

pytestmark = pytest.mark.gpu


def pa():
    import pagedattention_decode_attention_gb300 as m
    return m


class Mirror:
    """Device caches + the oracle's host caches, kept in lock step."""

    def __init__(self, num_layers, num_blocks, hkv, d, dtype, device, seed):
        dt = TORCH_DTYPES[dtype]
        self.dt, self.device = dt, device
        self.k = [wl.normal((num_blocks, hkv, 16, d), dt, seed + 2 * i, device) for i in range(num_layers)]
        self.v = [wl.normal((num_blocks, hkv, 16, d), dt, seed + 2 * i + 1, device) for i in range(num_layers)]
        self.hk = [to_f32_numpy(t) for t in self.k]
        self.hv = [to_f32_numpy(t) for t in self.v]

    def append(self, layer, k, v, slots_np):
        pa().kv_append(k, v, self.k[layer], self.v[layer], torch.from_numpy(slots_np).to(self.device))
        oa.kv_append(to_f32_numpy(k), to_f32_numpy(v), self.hk[layer], self.hv[layer], slots_np)

    def copy(self, pairs_np):
        if len(pairs_np) == 0:
            return
        pa().block_copy(self.k, self.v, torch.from_numpy(pairs_np).to(self.device))
        oa.block_copy(self.hk, self.hv, pairs_np)

    def assert_equal(self):
        for layer in range(len(self.k)):
            assert np.array_equal(to_f32_numpy(self.k[layer]), self.hk[layer])
            assert np.array_equal(to_f32_numpy(self.v[layer]), self.hv[layer])


def both_append(native, model, seqs):
    slots, pairs = native.append_slots(seqs)
    ms, mp = [], []
    for s in seqs:
        slot, cow = model.append_slot(int(s))
        ms.append(slot)
        if cow is not None:
            mp.append(cow)
    assert slots.tolist() == ms
    assert [tuple(p) for p in pairs.tolist()] == mp
    return slots, pairs


def tables_of(native, model, seqs, max_blocks):
    tab, lens = native.tables(seqs, max_blocks)
    for i, s in enumerate(seqs):
        t, ctx = model.block_table(s)
        assert tab[i, :len(t)].tolist() == t and lens[i] == ctx
    return tab, lens


def decode_and_check(mirror, layer, q, tab, lens, scale, seqs_check=None):
    dev = mirror.device
    out = pa().paged_attention_decode(q, mirror.k[layer], mirror.v[layer],
                                      torch.from_numpy(tab).to(dev), torch.from_numpy(lens).to(dev),
                                      scale)
    pa().check_status()
    ref = oa.paged_attention_decode(to_f32_numpy(q), mirror.hk[layer], mirror.hv[layer], tab, lens,
                                    scale, seqs=seqs_check)
    assert_attention_close(out, ref, mirror.dt, rows=seqs_check)
    return out


# --------------------------------------------------------------- workload 1
def test_tiny_workload_with_append_and_cow(gpu):
    """4 sequences, lengths U{1..100}, 4/4 heads, d=64, fp32, 64-block pool in
    random order; one kv_append step and one copy-on-write block copy."""
    batch = wl.tiny()
    order = wl.rng(batch.seed + 7).permutation(batch.num_blocks)
    native, model = pa().BlockPool(batch.num_blocks, 16, order), ModelPool(batch.num_blocks, 16, order)
    seqs = [native.new_seq() for _ in range(4)]
    [model.new_seq() for _ in range(4)]
    mir = Mirror(1, batch.num_blocks, 4, 64, "f32", gpu, batch.seed * 10)
    # prefill every sequence to its drawn length
    order_tokens = np.concatenate([np.full(int(n), s, dtype=np.int32)
                                   for s, n in zip(seqs, batch.context_lens)])
    slots, pairs = both_append(native, model, order_tokens)
    assert len(pairs) == 0
    t = len(order_tokens)
    mir.append(0, wl.normal((t, 4, 64), torch.float32, 1, gpu), wl.normal((t, 4, 64), torch.float32, 2, gpu), slots)
    # one decode step: one new token per sequence, then attention over ctx + 1
    slots, _ = both_append(native, model, np.array(seqs, dtype=np.int32))
    mir.append(0, wl.normal((4, 4, 64), torch.float32, 3, gpu), wl.normal((4, 4, 64), torch.float32, 4, gpu), slots)
    tab, lens = tables_of(native, model, seqs, 8)
    decode_and_check(mir, 0, wl.normal((4, 4, 64), torch.float32, 5, gpu), tab, lens, batch.scale)
    # fork a sequence whose last block is partly filled; the child's append copies it
    parent = next(s for s, n in zip(seqs, lens) if n % 16 != 0)
    child = native.fork(parent)
    assert model.fork(parent) == child
    slots, pairs = both_append(native, model, np.array([child], dtype=np.int32))
    assert len(pairs) == 1
    mir.copy(pairs)
    mir.append(0, wl.normal((1, 4, 64), torch.float32, 6, gpu), wl.normal((1, 4, 64), torch.float32, 7, gpu), slots)
    mir.assert_equal()
    all_seqs = seqs + [child]
    tab, lens = tables_of(native, model, all_seqs, 8)
    decode_and_check(mir, 0, wl.normal((5, 4, 64), torch.float32, 8, gpu), tab, lens, batch.scale)


# --------------------------------------------------------------- workloads 2, 3
def sample_rows(lens, n, seed):
    order = np.argsort(lens)
    pick = set(order[-4:].tolist()) | set(order[:2].tolist())
    gen = np.random.default_rng(seed)
    pick |= set(gen.choice(len(lens), size=min(n, len(lens)), replace=False).tolist())
    return sorted(pick)


def test_mha_7b_full_size_sampled(gpu):
    """Batch 64, 32/32 heads, d=128, fp16, log-uniform lengths; two of the 32
    layer caches, the same launch the benchmark times."""
    batch = wl.mha_7b()
    rows = sample_rows(batch.context_lens, 8, 1)
    for layer in range(2):
        q, kc, vc, bt, cl = decode_inputs(batch, gpu, seed_offset=layer)
        out = pa().paged_attention_decode(q, kc, vc, bt, cl, batch.scale)
        pa().check_status()
        assert_attention_close(out, oracle_decode(batch, q, kc, vc, seqs=rows), torch.float16, rows=rows)


def test_gqa_8b_full_size_sampled_then_append(gpu):
    """Batch 128 (124 log-uniform [128, 8192] + 4 x 8192), 32/8 heads, d=128,
    bf16; then kv_append of one new token per sequence, bit-exact."""
    batch = wl.gqa_8b()
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    out = pa().paged_attention_decode(q, kc, vc, bt, cl, batch.scale)
    pa().check_status()
    rows = sample_rows(batch.context_lens, 10, 2)
    assert_attention_close(out, oracle_decode(batch, q, kc, vc, seqs=rows), torch.bfloat16, rows=rows)
    slots = batch.new_token_slots()
    k = wl.normal((128, 8, 128), torch.bfloat16, 91, gpu)
    v = wl.normal((128, 8, 128), torch.bfloat16, 92, gpu)
    ref_k, ref_v = kc.cpu(), vc.cpu()
    pa().kv_append(k, v, kc, vc, torch.from_numpy(slots).to(gpu))
    pa().check_status()
    bits = lambda t: t.view(torch.int16).numpy()  # noqa: E731  (exact 16-bit copies)
    oa.kv_append(bits(k.cpu()), bits(v.cpu()), bits(ref_k), bits(ref_v), slots)
    assert torch.equal(kc.cpu(), ref_k) and torch.equal(vc.cpu(), ref_v)


# --------------------------------------------------------------- workload 4
def run_sampling(gpu, script, check_every_step=True, check_rows=4):
    hq, hkv, d = 32, 8, 128
    nb = script.num_blocks
    native = pa().BlockPool(nb, 16, script.initial_order)
    model = ModelPool(nb, 16, script.initial_order)
    mir = Mirror(1, nb, hkv, d, "bf16", gpu, script.seed * 10)
    prompts = []
    for p in range(script.prompts):
        s = native.new_seq()
        assert model.new_seq() == s
        prompts.append(s)
    toks = np.concatenate([np.full(script.prompt_len + int(script.shared_extra[i]), s, dtype=np.int32)
                           for i, s in enumerate(prompts)])
    slots, pairs = both_append(native, model, toks)
    assert len(pairs) == 0
    t = len(toks)
    mir.append(0, wl.normal((t, hkv, d), torch.bfloat16, 11, gpu), wl.normal((t, hkv, d), torch.bfloat16, 12, gpu), slots)
    branches = []
    for s in prompts:
        kids = [native.fork(s) for _ in range(script.branches - 1)]
        assert [model.fork(s) for _ in range(script.branches - 1)] == kids
        branches += [s] + kids
    prefix_block = native.block_table(prompts[0])[0][0]
    assert native.refcount(prefix_block) == script.branches
    branches = np.array(branches, dtype=np.int32)
    max_blocks = -(-(script.prompt_len + 16 + script.steps) // 16)
    total_pairs = 0
    gen = np.random.default_rng(script.seed)
    for step in range(script.steps):
        slots, pairs = both_append(native, model, branches)
        total_pairs += len(pairs)
        mir.copy(pairs)                       # copies first, then the new rows
        n = len(branches)
        mir.append(0, wl.normal((n, hkv, d), torch.bfloat16, 1000 + 2 * step, gpu),
                   wl.normal((n, hkv, d), torch.bfloat16, 1001 + 2 * step, gpu), slots)
        if step == 0:
            mir.assert_equal()
        if check_every_step or step == script.steps - 1:
            tab, lens = tables_of(native, model, branches.tolist(), max_blocks)
            rows = sorted(gen.choice(n, size=check_rows, replace=False).tolist())
            q = wl.normal((n, hq, d), torch.bfloat16, 5000 + step, gpu)
            decode_and_check(mir, 0, q, tab, lens, 1.0 / np.sqrt(d), seqs_check=rows)
    mir.assert_equal()
    return total_pairs


def test_parallel_sampling_cow_full(gpu):
    """32 prompts of 1024 (+1..15 shared) tokens forked 4 ways, 256 decode steps
    with per-branch appends, attention verified every step."""
    script = wl.sampling_cow()
    pairs = run_sampling(gpu, script)
    assert pairs == script.prompts * (script.branches - 1)


def test_parallel_sampling_no_partial_block_no_copy(gpu):
    """Prompts that end exactly on a block boundary never copy."""
    script = wl.sampling_cow(prompts=4, steps=20, zero_extra=True)
    assert run_sampling(gpu, script) == 0


# --------------------------------------------------------------- workload 5
def test_prefix_mix_full(gpu):
    """1024-token shared prefix (64 blocks, refcount 100, pinned) + 100
    heavy-tailed suffixes; GQA 32/8, d=128, bf16, 32 layer caches; one decode
    step over all layers.  Two layers are mirrored and checked against the
    oracle on sampled sequences; all 32 layers run."""
    sc = wl.prefix_mix()
    hq, hkv, d = 32, 8, 128
    nb = sc.num_blocks
    native, model = pa().BlockPool(nb, 16, sc.initial_order), ModelPool(nb, 16, sc.initial_order)
    owner = native.new_seq()
    assert model.new_seq() == owner
    pre = np.full(sc.prefix_len, owner, dtype=np.int32)
    pre_slots, _ = both_append(native, model, pre)
    native.pin(owner, sc.prefix_len)
    model.pin(owner, sc.prefix_len)
    reqs = []
    for _ in range(len(sc.suffix_lens)):
        r = native.new_seq()
        assert model.new_seq() == r
        native.share_prefix(owner, r, sc.prefix_len)
        model.share_prefix(owner, r, sc.prefix_len)
        reqs.append(r)
    native.free_seq(owner)
    model.free_seq(owner)
    prefix_blocks = native.block_table(reqs[0])[0][:64]
    assert all(native.refcount(b) == len(reqs) for b in prefix_blocks)
    assert native.stats()["pinned_blocks"] == 64
    suf = np.concatenate([np.full(int(n), r, dtype=np.int32) for r, n in zip(reqs, sc.suffix_lens)])
    suf_slots, pairs = both_append(native, model, suf)
    assert len(pairs) == 0                      # suffixes start on a fresh block
    step_slots, pairs = both_append(native, model, np.array(reqs, dtype=np.int32))
    assert len(pairs) == 0
    max_blocks = -(-(sc.prefix_len + int(sc.suffix_lens.max()) + 1) // 16)
    tab, lens = tables_of(native, model, reqs, max_blocks)
    mirrored = {0: None, sc.num_layers - 1: None}
    rows = sample_rows(lens, 6, 5)
    all_slots = np.concatenate([pre_slots, suf_slots, step_slots])
    tt = len(all_slots)
    for layer in range(sc.num_layers):
        dt = torch.bfloat16
        k = wl.normal((tt, hkv, d), dt, 100 + 3 * layer, gpu)
        v = wl.normal((tt, hkv, d), dt, 101 + 3 * layer, gpu)
        q = wl.normal((len(reqs), hq, d), dt, 102 + 3 * layer, gpu)
        if layer in mirrored:
            mir = Mirror(1, nb, hkv, d, "bf16", gpu, 7000 + layer)
            mir.append(0, k, v, all_slots)
            mir.assert_equal()
            decode_and_check(mir, 0, q, tab, lens, 1.0 / np.sqrt(d), seqs_check=rows)
            del mir
        else:
            kc = torch.empty((nb, hkv, 16, d), dtype=dt, device=gpu)
            vc = torch.empty_like(kc)
            pa().kv_append(k, v, kc, vc, torch.from_numpy(all_slots).to(gpu))
            out = pa().paged_attention_decode(q, kc, vc, torch.from_numpy(tab).to(gpu),
                                              torch.from_numpy(lens).to(gpu), 1.0 / np.sqrt(d))
            pa().check_status()
            assert torch.isfinite(out.float()).all()
