"""Randomised batches for the grouped shared-prefix decode: group structures
(forked prompts whose branches diverge, requests on shared system prompts,
groups with nothing shared), member counts below and above one shared unit's
capacity, own suffixes from none to many blocks, every head grouping and
head_dim, with the step's new K/V rows stored and attended in the same run.
The caches must equal the oracle's kv_append of the same rows bit for bit,
and the outputs the oracle's attention over them within the attention
tolerance ("第 6 章 缓存管理", section 块表长什么样; OS-lab appendix, sections
2.1 and 4.3)."""

import numpy as np
import pytest
import torch

import oracle.attention as oa
from pagedattention_decode_attention_gb300 import workloads as wl
from tests.gpu_helpers import TORCH_DTYPES, assert_attention_close, to_f32_numpy
from tests.test_gpu_grouped_prefix import grouped_batch, on

pytestmark = pytest.mark.gpu

HEADS = [(8, 8), (16, 8), (32, 8), (16, 2), (8, 4)]


def random_groups(gen):
    groups = []
    for _ in range(int(gen.integers(1, 9))):
        members = int(gen.integers(1, 13))
        if gen.random() < 0.5:
            # a prompt forked into `members` branches, each appending a few tokens
            groups.append(("fork", int(gen.integers(1, 700)),
                           [int(x) for x in gen.integers(1, 40, members)]))
        else:
            # requests on a shared system prompt (possibly empty)
            tokens = int(gen.choice([0, 16, 48, 160, 512, 1024]))
            tails = [int(x) for x in gen.integers(0, 300, members)]
            if tokens == 0:
                tails = [max(1, t) for t in tails]
            groups.append(("share", tokens, tails))
    return groups


@pytest.mark.parametrize("seed", range(8))
def test_random_grouped_batches_with_append(gpu, seed):
    import pagedattention_decode_attention_gb300 as pa
    gen = np.random.default_rng(7000 + seed)
    hq, hkv = HEADS[int(gen.integers(len(HEADS)))]
    d = int(gen.choice([64, 128]))
    dtype = str(gen.choice(["bf16", "f16"]))
    dt = TORCH_DTYPES[dtype]
    groups = random_groups(gen)
    q, kc, vc, tables, lens, gs, gb = grouped_batch(groups, hq, hkv, d, dtype, seed=7100 + seed,
                                                    dev=gpu)
    b = len(lens)
    # each sequence's new token is its last one; a sequence with nothing past
    # its group's shared blocks has none (copy-on-write never appends there)
    first_private = np.repeat(gb.astype(np.int64) * 16, np.diff(gs))
    pos = lens.astype(np.int64) - 1
    slots = tables[np.arange(b), pos // 16].astype(np.int64) * 16 + pos % 16
    slots[pos < first_private] = -1
    slots[gen.random(b) < 0.15] = -1           # padding rows: nothing stored for them
    k_new = wl.normal((b, hkv, d), dt, 7200 + seed, gpu)
    v_new = wl.normal((b, hkv, d), dt, 7300 + seed, gpu)
    host_k, host_v = to_f32_numpy(kc), to_f32_numpy(vc)
    oa.kv_append(to_f32_numpy(k_new), to_f32_numpy(v_new), host_k, host_v, slots)

    bt, cl, gs_d, gb_d = on(gpu, tables, lens, gs, gb)
    scale = 1.0 / np.sqrt(d)
    n = pa.grouped_prefix_workspace_size(b, hq, hkv, d, tables.shape[1])
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=gpu)
    pa.grouped_prefix_plan(bt, cl, gs_d, gb_d, hq, hkv, d, scale, dt, ws)
    out = pa.paged_attention_decode_grouped_prefix_append_run(
        q, k_new, v_new, torch.from_numpy(slots).to(gpu), kc, vc, bt, gs_d, gb_d, scale, ws)
    pa.check_status()
    assert np.array_equal(to_f32_numpy(kc), host_k)
    assert np.array_equal(to_f32_numpy(vc), host_v)
    want = oa.paged_attention_decode(to_f32_numpy(q), host_k, host_v, tables, lens, scale)
    assert_attention_close(out, want, dt)
    # a second run on the same plan (the step's next layer) gives the same bits
    again = pa.paged_attention_decode_grouped_prefix_append_run(
        q, k_new, v_new, torch.from_numpy(slots).to(gpu), kc, vc, bt, gs_d, gb_d, scale, ws)
    pa.check_status()
    assert torch.equal(out, again)
