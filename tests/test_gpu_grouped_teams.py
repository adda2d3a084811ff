"""The grouped decode merges a sequence's splits in one of two ways inside its
attention launch: in teams, when every chunk of a group takes its members' own
blocks into its last shared split and has at most four splits (the splits of
each (chunk, KV head) then run on four warps of one CTA and are merged in
shared memory), or else through a queue of ready merges that warps out of work
take.  Each batch below is made to take one of the two ways (the plan's
choice is read from the workspace header), with the step's new K/V rows stored
and attended in the same run; caches must equal the oracle's kv_append bit for
bit and the outputs the oracle's attention within the attention tolerance
("第 6 章 缓存管理", section 块表长什么样; OS-lab appendix, sections 2.1 and
4.3: forked tables point at the same blocks)."""

import numpy as np
import pytest
import torch

import oracle.attention as oa
from pagedattention_decode_attention_gb300 import workloads as wl
from tests.gpu_helpers import TORCH_DTYPES, assert_attention_close, to_f32_numpy
from tests.test_gpu_grouped_prefix import grouped_batch, on

pytestmark = pytest.mark.gpu

HEADER_TEAM = 8  # workspace header word: 4 when the plan placed teams, else 0


def forks(gen, groups, members, prompt):
    """Forked prompts whose branches each append a few tokens."""
    return [("fork", prompt, [int(x) for x in gen.integers(1, 20, members)])
            for _ in range(groups)]


CASES = {
    # (head grouping, groups) -> expected team word
    "teams-64-blocks": ((32, 8), lambda g: forks(g, 6, 4, 1024), 4),
    "teams-g1": ((8, 8), lambda g: forks(g, 5, 3, 1000), 4),
    "teams-g8": ((16, 2), lambda g: forks(g, 7, 2, 700), 4),
    "teams-one-split": ((32, 8), lambda g: forks(g, 4, 4, 40), 4),
    "teams-mixed-members": ((32, 8), lambda g: forks(g, 3, 4, 900) + forks(g, 3, 1, 500)
                            + forks(g, 2, 2, 300), 4),
    # six members of one prompt with G = 1: more than a chunk absorbs
    "queue-big-chunk": ((8, 8), lambda g: forks(g, 2, 6, 800) + forks(g, 2, 3, 600), 0),
    # a suffix too long to absorb
    "queue-long-suffix": ((32, 8), lambda g: forks(g, 3, 4, 600)
                          + [("share", 512, [1, 400])], 0),
}


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("case", sorted(CASES))
def test_grouped_merges_in_teams_or_queue(gpu, case, head_dim):
    import pagedattention_decode_attention_gb300 as pa
    (hq, hkv), make, want_team = CASES[case]
    seed = 8000 + sorted(CASES).index(case) * 10 + head_dim
    gen = np.random.default_rng(seed)
    dtype = "bf16" if head_dim == 128 else "f16"
    dt = TORCH_DTYPES[dtype]
    groups = make(gen)
    q, kc, vc, tables, lens, gs, gb = grouped_batch(groups, hq, hkv, head_dim, dtype,
                                                    seed=seed + 1, dev=gpu)
    b = len(lens)
    first_private = np.repeat(gb.astype(np.int64) * 16, np.diff(gs))
    pos = lens.astype(np.int64) - 1
    slots = tables[np.arange(b), pos // 16].astype(np.int64) * 16 + pos % 16
    slots[pos < first_private] = -1
    k_new = wl.normal((b, hkv, head_dim), dt, seed + 2, gpu)
    v_new = wl.normal((b, hkv, head_dim), dt, seed + 3, gpu)
    host_k, host_v = to_f32_numpy(kc), to_f32_numpy(vc)
    oa.kv_append(to_f32_numpy(k_new), to_f32_numpy(v_new), host_k, host_v, slots)

    bt, cl, gs_d, gb_d = on(gpu, tables, lens, gs, gb)
    scale = 1.0 / np.sqrt(head_dim)
    n = pa.grouped_prefix_workspace_size(b, hq, hkv, head_dim, tables.shape[1])
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=gpu)
    pa.grouped_prefix_plan(bt, cl, gs_d, gb_d, hq, hkv, head_dim, scale, dt, ws)
    sl = torch.from_numpy(slots).to(gpu)
    out = pa.paged_attention_decode_grouped_prefix_append_run(q, k_new, v_new, sl, kc, vc, bt,
                                                              gs_d, gb_d, scale, ws)
    pa.check_status()
    assert int(ws[:64].view(torch.int32)[HEADER_TEAM]) == want_team
    assert np.array_equal(to_f32_numpy(kc), host_k)
    assert np.array_equal(to_f32_numpy(vc), host_v)
    want = oa.paged_attention_decode(to_f32_numpy(q), host_k, host_v, tables, lens, scale)
    assert_attention_close(out, want, dt)
    # the next layer's run on the same plan: same bits (the run leaves the
    # workspace's counters and queue as it found them)
    again = pa.paged_attention_decode_grouped_prefix_append_run(q, k_new, v_new, sl, kc, vc, bt,
                                                                gs_d, gb_d, scale, ws)
    pa.check_status()
    assert torch.equal(out, again)
