"""GPU parity of block swapping between the device caches and page-locked host
caches (``pa_block_swap``), alone and driven by the pool's swap_out / swap_in.

Copies are checked bit for bit against ``oracle.attention.block_swap``; the
preempt-and-resume test checks that a sequence's attention output is
unchanged by a round trip through host memory while its device blocks were
reused by another sequence.
"""

import numpy as np
import pytest
import torch

import oracle.attention as oa
from pagedattention_decode_attention_gb300 import workloads as wl
from tests.gpu_helpers import TORCH_DTYPES

pytestmark = pytest.mark.gpu


def pa():
    import pagedattention_decode_attention_gb300 as m
    return m


def as_bits(t):
    """Host numpy view that compares bit patterns (16-bit floats as int16)."""
    t = t.cpu()
    return t.numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_block_swap_bit_exact(gpu, dtype):
    dt = TORCH_DTYPES[dtype]
    layers, nb, nh, hkv, d = 3, 40, 25, 8, 128
    dk = [wl.normal((nb, hkv, 16, d), dt, 10 + i, gpu) for i in range(layers)]
    dv = [wl.normal((nb, hkv, 16, d), dt, 20 + i, gpu) for i in range(layers)]
    hk = [wl.normal((nh, hkv, 16, d), dt, 30 + i, gpu).cpu().pin_memory() for i in range(layers)]
    hv = [wl.normal((nh, hkv, 16, d), dt, 40 + i, gpu).cpu().pin_memory() for i in range(layers)]
    gen = np.random.default_rng(3)
    out_pairs = np.stack([gen.choice(nb, 12, replace=False), gen.choice(nh, 12, replace=False)], 1)
    ref_hk = [as_bits(t).copy() for t in hk]
    ref_hv = [as_bits(t).copy() for t in hv]
    oa.block_swap([as_bits(t) for t in dk], [as_bits(t) for t in dv], ref_hk, ref_hv, out_pairs)
    pa().block_swap(dk, dv, hk, hv, torch.from_numpy(out_pairs).to(gpu), pa().PA_SWAP_OUT)
    pa().check_status()
    for got, ref in zip(hk + hv, ref_hk + ref_hv):
        assert np.array_equal(as_bits(got), ref)
    in_pairs = np.stack([gen.choice(nh, 9, replace=False), gen.choice(nb, 9, replace=False)], 1)
    ref_dk = [as_bits(t).copy() for t in dk]
    ref_dv = [as_bits(t).copy() for t in dv]
    oa.block_swap([as_bits(t) for t in hk], [as_bits(t) for t in hv], ref_dk, ref_dv, in_pairs)
    pa().block_swap(dk, dv, hk, hv, torch.from_numpy(in_pairs).to(gpu), pa().PA_SWAP_IN)
    pa().check_status()
    for got, ref in zip(dk + dv, ref_dk + ref_dv):
        assert np.array_equal(as_bits(got), ref)


def test_preempt_and_resume_keeps_attention(gpu):
    """Pool-driven round trip: sequence x is swapped out, its device blocks
    are reused (and overwritten) by a new sequence, x comes back into other
    blocks, and its attention output is bit-identical to before."""
    layers, nb, nh, hq, hkv, d = 2, 24, 16, 16, 4, 128
    dt = torch.bfloat16
    pool = pa().BlockPool(nb, 16, np.random.default_rng(5).permutation(nb))
    pool.set_host_blocks(nh, np.random.default_rng(6).permutation(nh))
    dk = [torch.zeros((nb, hkv, 16, d), dtype=dt, device=gpu) for _ in range(layers)]
    dv = [torch.zeros_like(dk[0]) for _ in range(layers)]
    hk = [torch.zeros((nh, hkv, 16, d), dtype=dt).pin_memory() for _ in range(layers)]
    hv = [torch.zeros_like(hk[0]).pin_memory() for _ in range(layers)]
    seqs = [pool.new_seq() for _ in range(3)]
    lens = [70, 33, 100]

    def fill(seq, n, seed):
        slots = np.array([pool.append_slot(seq)[0] for _ in range(n)], dtype=np.int64)
        for i in range(layers):
            k = wl.normal((n, hkv, d), dt, seed + 2 * i, gpu)
            v = wl.normal((n, hkv, d), dt, seed + 2 * i + 1, gpu)
            pa().kv_append(k, v, dk[i], dv[i], torch.from_numpy(slots).to(gpu))

    for s, n in zip(seqs, lens):
        fill(s, n, 100 * s + 7)
    q = wl.normal((1, hq, d), dt, 99, gpu)

    def attend(seq):
        tab, ctx = pool.tables([seq], 8)
        bt, cl = torch.from_numpy(tab).to(gpu), torch.from_numpy(ctx).to(gpu)
        return [pa().paged_attention_decode(q, dk[i], dv[i], bt, cl, 1.0 / np.sqrt(d)).clone()
                for i in range(layers)]

    x = seqs[1]
    before = attend(x)
    out_pairs = pool.swap_out(x)
    pa().block_swap(dk, dv, hk, hv, torch.from_numpy(out_pairs).to(gpu), pa().PA_SWAP_OUT)
    y = pool.new_seq()                            # takes x's freed blocks and overwrites them
    fill(y, 48, 555)
    assert set(pool.block_table(y)[0]) & set(out_pairs[:, 0].tolist())
    in_pairs = pool.swap_in(x)
    pa().block_swap(dk, dv, hk, hv, torch.from_numpy(in_pairs).to(gpu), pa().PA_SWAP_IN)
    after = attend(x)
    pa().check_status()
    assert not np.array_equal(pool.block_table(x)[0], out_pairs[:, 0])   # moved blocks
    for a, b in zip(before, after):
        assert torch.equal(a, b)


def test_block_swap_rejects_pageable_host_memory_and_bad_ids(gpu):
    dk = [torch.zeros((4, 2, 16, 64), dtype=torch.float16, device=gpu)]
    dv = [torch.zeros_like(dk[0])]
    pageable = [torch.zeros((4, 2, 16, 64), dtype=torch.float16)]
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device=gpu)
    with pytest.raises(ValueError):
        pa().block_swap(dk, dv, pageable, pageable, pairs, pa().PA_SWAP_OUT)
    hk = [t.pin_memory() for t in pageable]
    hv = [t.clone().pin_memory() for t in pageable]
    bad = torch.tensor([[0, 4]], dtype=torch.int64, device=gpu)     # host block 4 of 4
    pa().block_swap(dk, dv, hk, hv, bad, pa().PA_SWAP_OUT)
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()


# ------------------------------------------------------- prepared caches
def test_layer_caches_copy_and_swap_repeated(gpu):
    """One LayerCaches object serves many copy-on-write copies and a swap
    round trip; every result equals the oracle's, bit for bit."""
    dt, nb, hkv, d, layers = torch.bfloat16, 40, 8, 128, 6
    dk = [wl.normal((nb, hkv, 16, d), dt, 300 + i, gpu) for i in range(layers)]
    dv = [wl.normal((nb, hkv, 16, d), dt, 400 + i, gpu) for i in range(layers)]
    rk, rv = [as_bits(t).copy() for t in dk], [as_bits(t).copy() for t in dv]
    caches = pa().LayerCaches(dk, dv)
    assert (caches.num_layers, caches.num_blocks, caches.num_kv_heads, caches.head_dim) == \
        (layers, nb, hkv, d)
    steps = [np.array([[1, 20], [2, 21]]), np.array([[20, 30], [7, 3], [39, 0]]),
             np.array([[5, 6]])]
    for pairs in steps:
        oa.block_copy(rk, rv, pairs)
        caches.block_copy(torch.from_numpy(pairs.astype(np.int64)).to(gpu))
    hk = [torch.zeros((8, hkv, 16, d), dtype=dt).pin_memory() for _ in range(layers)]
    hv = [torch.zeros((8, hkv, 16, d), dtype=dt).pin_memory() for _ in range(layers)]
    host = pa().LayerCaches(hk, hv, host=True)
    hrk, hrv = [as_bits(t).copy() for t in hk], [as_bits(t).copy() for t in hv]
    out = np.array([[20, 0], [3, 5], [39, 7]])
    inn = np.array([[0, 11], [7, 12]])
    oa.block_swap(rk, rv, hrk, hrv, out)
    caches.block_swap(host, torch.from_numpy(out.astype(np.int64)).to(gpu), pa().PA_SWAP_OUT)
    oa.block_swap(hrk, hrv, rk, rv, inn)
    caches.block_swap(host, torch.from_numpy(inn.astype(np.int64)).to(gpu), pa().PA_SWAP_IN)
    pa().check_status()
    for got, want in zip(dk + dv + hk + hv, rk + rv + hrk + hrv):
        assert np.array_equal(as_bits(got), want)


def test_layer_caches_rejects_mismatches(gpu):
    k = [torch.zeros((4, 2, 16, 64), dtype=torch.float16, device=gpu) for _ in range(2)]
    with pytest.raises(ValueError):
        pa().LayerCaches(k, k[:1])                                    # layer counts differ
    with pytest.raises(ValueError):
        pa().LayerCaches(k, [k[0], torch.zeros((4, 2, 16, 128), dtype=torch.float16,
                                               device=gpu)])         # shapes differ
    with pytest.raises(ValueError):
        pa().LayerCaches([t.cpu() for t in k], [t.cpu() for t in k], host=True)   # pageable
    caches = pa().LayerCaches(k, k)
    with pytest.raises(ValueError):
        caches.block_copy(torch.tensor([[0, 1]], dtype=torch.int32, device=gpu))
    host = pa().LayerCaches([torch.zeros((4, 2, 16, 64), dtype=torch.float16).pin_memory()],
                            [torch.zeros((4, 2, 16, 64), dtype=torch.float16).pin_memory()],
                            host=True)
    with pytest.raises(ValueError):                                   # one host layer, two device
        caches.block_swap(host, torch.tensor([[0, 1]], dtype=torch.int64, device=gpu),
                          pa().PA_SWAP_OUT)
    with pytest.raises(ValueError):
        host.block_copy(torch.tensor([[0, 1]], dtype=torch.int64, device=gpu))
