"""The decode step exactly as the benchmark times it, at full size, against the
oracle.

One plan from the context lengths, then per layer one fused launch that
appends each sequence's new K/V row at its slot and attends over the cache
including it (OS-lab appendix, section 2.1: each decode step appends the new
token's K/V, then reads all earlier K/V).  Three separate layer caches, the
benchmark's shapes and seeds:

* 7B-shaped MHA: 64 sequences, 32/32 heads, d=128, fp16, lengths log-uniform
  in [16, 2048];
* 8B-shaped GQA: 128 sequences (124 log-uniform in [128, 8192] + 4 x 8192),
  32/8 heads, d=128, bf16.

Every layer's caches are compared bit for bit with host mirrors written by
``oracle.attention.kv_append``; the outputs of sampled sequences (the longest
four, the shortest two and ten drawn at random), every head, are compared with
``oracle.attention.paged_attention_decode`` within the attention tolerance.  A
second step over the same inputs must give bit-identical outputs.
"""

import numpy as np
import pytest
import torch

import oracle.attention as oa
from pagedattention_decode_attention_gb300 import workloads as wl
from tests.gpu_helpers import TORCH_DTYPES, assert_attention_close

pytestmark = pytest.mark.gpu

LAYERS = 3


def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    return t.view(torch.int16).numpy()


def _sample_rows(lens, n, seed):
    order = np.argsort(lens, kind="stable")
    pick = set(order[-4:].tolist()) | set(order[:2].tolist())
    gen = np.random.default_rng(seed)
    pick |= set(gen.choice(len(lens), size=min(n, len(lens)), replace=False).tolist())
    return sorted(pick)


def _compact(bits_k, bits_v, tables, rows, dt):
    """The sampled rows' blocks only (a relabelling of physical blocks, which
    leaves attention unchanged), widened exactly to float32."""
    sub = tables[rows]
    blocks = np.unique(sub[sub >= 0])
    remap = np.full(int(tables.max()) + 1, -1, dtype=np.int64)
    remap[blocks] = np.arange(len(blocks))
    tab = np.where(sub >= 0, remap[np.maximum(sub, 0)], -1)
    widen = lambda b: torch.from_numpy(b[blocks]).view(dt).float().numpy()  # noqa: E731
    return widen(bits_k), widen(bits_v), tab


@pytest.mark.parametrize("name", ["mha_7b", "gqa_8b"])
def test_benched_step_full_size(gpu, name):
    import pagedattention_decode_attention_gb300 as pa
    batch = getattr(wl, name)()
    dt = TORCH_DTYPES[batch.dtype]
    b, hq, hkv, d, nb = (batch.num_seqs, batch.num_q_heads, batch.num_kv_heads, batch.head_dim,
                         batch.num_blocks)
    s = batch.seed * 1000
    kc = [wl.normal((nb, hkv, 16, d), dt, s + 4 * i, gpu) for i in range(LAYERS)]
    vc = [wl.normal((nb, hkv, 16, d), dt, s + 4 * i + 1, gpu) for i in range(LAYERS)]
    q = wl.normal((LAYERS, b, hq, d), dt, s + 7, gpu)
    k_new = wl.normal((LAYERS, b, hkv, d), dt, s + 8, gpu)
    v_new = wl.normal((LAYERS, b, hkv, d), dt, s + 9, gpu)
    out = torch.full((LAYERS, b, hq, d), float("nan"), dtype=dt, device=gpu)
    tables = torch.from_numpy(batch.block_tables).to(gpu)
    lens = torch.from_numpy(batch.context_lens).to(gpu)
    slots_np = batch.new_token_slots()
    slots = torch.from_numpy(slots_np).to(gpu)
    ws = pa.alloc_workspace(b, hq, hkv, d, batch.max_blocks, gpu)

    mirror_k = [_bits(t) for t in kc]
    mirror_v = [_bits(t) for t in vc]

    plan = pa.prepare_decode_plan(lens, hq, hkv, d, batch.max_blocks, ws)
    calls = [pa.prepare_decode_append_run(q[i], k_new[i], v_new[i], slots, kc[i], vc[i], tables,
                                          lens, batch.scale, ws, out[i]) for i in range(LAYERS)]
    plan()
    for call in calls:
        call()
    pa.check_status()
    first = out.clone()

    rows = _sample_rows(batch.context_lens, 10, batch.seed)
    for i in range(LAYERS):
        oa.kv_append(_bits(k_new[i]), _bits(v_new[i]), mirror_k[i], mirror_v[i], slots_np)
        assert np.array_equal(_bits(kc[i]), mirror_k[i]), f"layer {i}: K cache differs"
        assert np.array_equal(_bits(vc[i]), mirror_v[i]), f"layer {i}: V cache differs"
        kf, vf, tab = _compact(mirror_k[i], mirror_v[i], batch.block_tables, rows, dt)
        want = oa.paged_attention_decode(q[i, rows].float().cpu().numpy(), kf, vf, tab,
                                         batch.context_lens[rows], batch.scale)
        assert_attention_close(out[i, rows], want, dt)
    assert 8192 in batch.context_lens[rows].tolist() or name == "mha_7b"

    # the benchmark repeats the step; the same inputs give the same bits
    plan()
    for call in calls:
        call()
    pa.check_status()
    assert torch.equal(out, first)
