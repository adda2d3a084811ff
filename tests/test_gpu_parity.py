"""GPU parity: the sm_103a kernels, called through the C ABI, against the oracle.

Tolerances are in ``tests/gpu_helpers.py``: fp32 max-abs 1e-5; fp16/bf16
``1e-2 + 2e-2 |oracle|`` element-wise; kv_append and block_copy bit-exact over
the whole cache tensors.
"""

import numpy as np
import pytest
import torch

import oracle.attention as oa
from oracle.pool import BlockPool as ModelPool
from tests.gpu_helpers import (TORCH_DTYPES, assert_attention_close, custom_batch, decode_inputs,
                               oracle_decode, to_f32_numpy)

pytestmark = pytest.mark.gpu


def pa():
    import pagedattention_decode_attention_gb300 as m
    return m


def run_decode(batch, q, kc, vc, bt, cl):
    out = pa().paged_attention_decode(q, kc, vc, bt, cl, batch.scale)
    pa().check_status()
    return out


# ------------------------------------------------------------- attention
LENS_SMALL = [1, 15, 16, 17, 100, 511, 512, 513, 1100, 2000]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("heads", [(4, 4), (8, 4), (32, 8), (16, 2)], ids=["g1", "g2", "g4", "g8"])
def test_decode_matches_oracle(gpu, dtype, head_dim, heads):
    hq, hkv = heads
    batch = custom_batch(LENS_SMALL, hq, hkv, head_dim, dtype, seed=hq * 131 + head_dim)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    out = run_decode(batch, q, kc, vc, bt, cl)
    assert_attention_close(out, oracle_decode(batch, q, kc, vc), TORCH_DTYPES[dtype])


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("heads", [(4, 4), (6, 2)])
def test_decode_fp32_matches_oracle(gpu, head_dim, heads):
    batch = custom_batch([1, 7, 16, 33, 300], heads[0], heads[1], head_dim, "f32", seed=5)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    out = run_decode(batch, q, kc, vc, bt, cl)
    assert_attention_close(out, oracle_decode(batch, q, kc, vc), torch.float32)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_placement_invariance_is_bit_exact(gpu, dtype):
    """Relabelling physical blocks leaves the GPU output bit-identical."""
    batch = custom_batch([3, 40, 700, 1500], 32, 8, 128, dtype, seed=77)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    base = run_decode(batch, q, kc, vc, bt, cl).clone()
    pi = torch.from_numpy(np.random.default_rng(3).permutation(batch.num_blocks)).to(gpu)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    bt2 = torch.where(bt >= 0, pi[bt.clamp(min=0).long()].int(), bt)
    moved = run_decode(batch, q, kc2, vc2, bt2.contiguous(), cl)
    assert torch.equal(base, moved)


def test_empty_and_full_contexts(gpu):
    """ctx = 0 gives zero rows; ctx = max_blocks * 16 reads every table entry."""
    mb = 40
    batch = custom_batch([0, mb * 16, 0, 5, mb * 16 - 1], 16, 4, 128, "bf16", seed=8, max_blocks=mb)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    out = pa().paged_attention_decode(q, kc, vc, bt, cl, batch.scale,
                                      out=torch.full_like(q, float("nan")))
    pa().check_status()
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
    assert_attention_close(out, oracle_decode(batch, q, kc, vc), torch.bfloat16)


def test_single_sequence_long_context(gpu):
    """One sequence of 12,345 tokens: many splits merged by the last CTA."""
    batch = custom_batch([12345], 32, 8, 128, "bf16", seed=12)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    out = run_decode(batch, q, kc, vc, bt, cl)
    assert_attention_close(out, oracle_decode(batch, q, kc, vc), torch.bfloat16)


def test_repeated_calls_reuse_workspace(gpu):
    batch = custom_batch([900, 2100, 33], 32, 8, 128, "f16", seed=13)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    ws = pa().alloc_workspace(3, 32, 8, 128, batch.max_blocks, gpu)
    ws.fill_(0xAB)                                   # garbage: the call needs no init
    outs = [pa().paged_attention_decode(q, kc, vc, bt, cl, batch.scale, workspace=ws).clone()
            for _ in range(3)]
    pa().check_status()
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    assert_attention_close(outs[0], oracle_decode(batch, q, kc, vc), torch.float16)


def test_bad_table_entry_sets_bounds_status(gpu):
    batch = custom_batch([40, 40], 8, 8, 64, "bf16", seed=14)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    bt[1, 1] = batch.num_blocks + 5
    pa().paged_attention_decode(q, kc, vc, bt, cl, batch.scale)
    with pytest.raises(pa().PagedAttnError) as e:
        pa().check_status()
    assert e.value.status == 5
    pa().check_status()                              # cleared by the read


def test_context_beyond_table_sets_bounds_status(gpu):
    batch = custom_batch([20], 4, 4, 64, "f16", seed=15)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    cl[0] = batch.max_blocks * 16 + 1
    out = pa().paged_attention_decode(q, kc, vc, bt, cl, batch.scale)
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()
    assert torch.isfinite(out.float()).all()


# ------------------------------------------------------------- kv_append
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_kv_append_bit_exact_whole_cache(gpu, dtype):
    dt = TORCH_DTYPES[dtype]
    nb, hkv, d, t = 50, 8, 128, 300
    gen = np.random.default_rng(21)
    slots = gen.choice(nb * 16, size=t, replace=False).astype(np.int64)
    slots[::17] = -1                                 # padding tokens
    from pagedattention_decode_attention_gb300 import workloads as wl
    kc = wl.normal((nb, hkv, 16, d), dt, 1, gpu)
    vc = wl.normal((nb, hkv, 16, d), dt, 2, gpu)
    k = wl.normal((t, hkv, d), dt, 3, gpu)
    v = wl.normal((t, hkv, d), dt, 4, gpu)
    ref_k, ref_v = kc.cpu().clone(), vc.cpu().clone()
    oa.kv_append(k.cpu().numpy() if dt == torch.float32 else k.cpu().view(torch.int16).numpy(),
                 v.cpu().numpy() if dt == torch.float32 else v.cpu().view(torch.int16).numpy(),
                 ref_k.numpy() if dt == torch.float32 else ref_k.view(torch.int16).numpy(),
                 ref_v.numpy() if dt == torch.float32 else ref_v.view(torch.int16).numpy(), slots)
    pa().kv_append(k, v, kc, vc, torch.from_numpy(slots).to(gpu))
    pa().check_status()
    assert torch.equal(kc.cpu(), ref_k) and torch.equal(vc.cpu(), ref_v)


def test_kv_append_out_of_range_slot(gpu):
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device=gpu)
    vc = torch.zeros_like(kc)
    k = torch.ones((2, 2, 64), dtype=torch.bfloat16, device=gpu)
    pa().kv_append(k, k, kc, vc, torch.tensor([3, 4 * 16], dtype=torch.int64, device=gpu))
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()
    assert torch.count_nonzero(kc) == 2 * 64 and kc[0, :, 3].eq(1).all()


# ------------------------------------------------------------ block_copy
# A block is 2048 16-byte chunks in bf16 8 x 128 (one batch of eight per
# thread), 4096 in f32 (two batches) and 384 in f16 3 x 64 (a ragged batch).
@pytest.mark.parametrize("dtype,hkv,d", [("bf16", 8, 128), ("f32", 8, 128), ("f16", 3, 64)])
def test_block_copy_bit_exact_all_layers(gpu, dtype, hkv, d):
    dt = TORCH_DTYPES[dtype]
    from pagedattention_decode_attention_gb300 import workloads as wl
    layers = [(wl.normal((30, hkv, 16, d), dt, 10 + i, gpu),
               wl.normal((30, hkv, 16, d), dt, 50 + i, gpu)) for i in range(5)]
    pairs = np.array([[1, 20], [2, 21], [7, 3], [29, 0]], dtype=np.int64)
    ref = [(k.cpu().clone(), v.cpu().clone()) for k, v in layers]
    as_np = (lambda t: t.numpy()) if dt == torch.float32 else (lambda t: t.view(torch.int16).numpy())
    oa.block_copy([as_np(k) for k, _ in ref], [as_np(v) for _, v in ref], pairs)
    pa().block_copy([k for k, _ in layers], [v for _, v in layers],
                    torch.from_numpy(pairs).to(gpu))
    pa().check_status()
    for (k, v), (rk, rv) in zip(layers, ref):
        assert torch.equal(k.cpu(), rk) and torch.equal(v.cpu(), rv)


def test_block_copy_bad_pair_is_skipped(gpu):
    kc = torch.arange(4 * 2 * 16 * 64, dtype=torch.float32, device=gpu).reshape(4, 2, 16, 64)
    vc = kc.clone()
    before = kc.clone()
    pa().block_copy([kc], [vc], torch.tensor([[0, 9]], dtype=torch.int64, device=gpu))
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()
    assert torch.equal(kc, before)


# ------------------------------------------------------- plan once, run many
def test_one_plan_serves_many_runs(gpu):
    """A plan followed by several runs (one per layer) gives, bit for bit, what
    the combined call gives for each layer."""
    batch = custom_batch([5, 530, 1300, 16, 2049], 32, 8, 128, "bf16", seed=31)
    ws = pa().alloc_workspace(5, 32, 8, 128, batch.max_blocks, gpu)
    _, _, _, bt, cl = decode_inputs(batch, gpu)
    pa().paged_attention_decode_plan(cl, 32, 8, 128, batch.max_blocks, ws)
    for layer in range(4):
        q, kc, vc, _, _ = decode_inputs(batch, gpu, seed_offset=layer)
        got = pa().paged_attention_decode_run(q, kc, vc, bt, cl, batch.scale, ws).clone()
        ref = pa().paged_attention_decode(q, kc, vc, bt, cl, batch.scale)
        pa().check_status()
        assert torch.equal(got, ref)
        if layer == 0:
            assert_attention_close(got, oracle_decode(batch, q, kc, vc), torch.bfloat16)
        # re-plan on a separate workspace does not disturb this one
        pa().paged_attention_decode_plan(cl, 32, 8, 128, batch.max_blocks,
                                         pa().alloc_workspace(5, 32, 8, 128, batch.max_blocks, gpu))


def test_run_without_plan_is_refused_on_device(gpu):
    batch = custom_batch([40, 70], 8, 8, 64, "f16", seed=32)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    ws = pa().alloc_workspace(2, 8, 8, 64, batch.max_blocks, gpu)
    ws.zero_()
    out = torch.full_like(q, 7.0)
    pa().paged_attention_decode_run(q, kc, vc, bt, cl, batch.scale, ws, out=out)
    with pytest.raises(pa().PagedAttnError) as e:
        pa().check_status()
    assert e.value.status == 1
    assert torch.all(out == 7.0)                     # nothing was written
    # a plan for other shapes is refused as well
    pa().paged_attention_decode_plan(cl, 8, 4, 64, batch.max_blocks, ws)
    pa().paged_attention_decode_run(q, kc, vc, bt, cl, batch.scale, ws, out=out)
    with pytest.raises(pa().PagedAttnError):
        pa().check_status()


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_unused_slots_holding_nan_do_not_leak(gpu, dtype):
    """Slots past the context in each sequence's last block hold NaN / Inf; the
    output must still match the oracle (which never reads them)."""
    batch = custom_batch([1, 7, 15, 17, 31, 100, 529], 16, 4, 128, dtype, seed=33)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    for b, n in enumerate(batch.context_lens):
        last = int(batch.block_tables[b, (int(n) - 1) // 16])
        off = int(n) % 16
        if off:
            kc[last, :, off:] = float("nan")
            vc[last, :, off:] = float("inf")
    out = run_decode(batch, q, kc, vc, bt, cl)
    assert_attention_close(out, oracle_decode(batch, q, kc, vc), TORCH_DTYPES[dtype])
