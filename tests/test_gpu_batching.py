"""The continuous-batching driver's trace on the device: every step's ordered
operations (swap-in, copy-on-write copies, token appends, swap-out) run on
the device kernels (``pa_block_swap``, ``pa_block_copy``, ``pa_kv_append``)
while the oracle applies the same operations to host mirrors; then decode
attention runs over every running sequence.

Checked at every step:
* the device caches (both tiers, every layer, K and V) equal the mirrors bit
  for bit;
* every running sequence's table gathers exactly its tokens' K/V rows (a
  closed form: each row is a fixed function of token id and position), so a
  prefix-cache hit, an evicted-and-re-keyed block, a recomputed request and a
  trip through host memory all read the right data;
* decode attention on the device matches the oracle within the attention
  tolerance.

Sources: "留书阁 / knowledge-20" page, continuous-batching passage; "vLLM:
treating the KV cache as virtual memory", sections "调度：词一级的进入与退出"
and "碎片从哪里来"; "第 6 章 缓存管理", section "缓存放不下的时候".
"""

import numpy as np
import pytest
import torch

import oracle.attention as oa
from pagedattention_decode_attention_gb300 import workloads as wl
from tests import batch_trace as bt
from tests.gpu_helpers import assert_attention_close

pytestmark = pytest.mark.gpu

MAX_BLOCKS = 32


def _device_tensor(bits: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    return t.to(device) if device is not None else t.pin_memory()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("seed,num_blocks,host_blocks", [(11, 40, 12), (13, 48, 16)])
def test_batcher_trace_on_device(gpu, seed, num_blocks, host_blocks):
    import pagedattention_decode_attention_gb300 as pa
    mirror = bt.HostTiers(num_blocks, host_blocks)
    dk = [_device_tensor(a, gpu) for a in mirror.k]
    dv = [_device_tensor(a, gpu) for a in mirror.v]
    hk = [_device_tensor(a, None) for a in mirror.hk]
    hv = [_device_tensor(a, None) for a in mirror.hv]
    dev = pa.LayerCaches(dk, dv)
    host = pa.LayerCaches(hk, hv, host=True)
    scale = 1.0 / np.sqrt(bt.D)

    def apply(op):
        kind = op[0]
        if kind in ("swap_in", "swap_out"):
            pairs = torch.tensor(op[2], dtype=torch.int64, device=gpu).reshape(-1, 2)
            if pairs.shape[0]:
                dev.block_swap(host, pairs,
                               pa.PA_SWAP_IN if kind == "swap_in" else pa.PA_SWAP_OUT)
        else:
            pairs, entries = op[1], op[2]
            if pairs:
                dev.block_copy(torch.tensor(pairs, dtype=torch.int64, device=gpu))
            if entries:
                toks = [e[2] for e in entries]
                pos = [e[3] for e in entries]
                slots = torch.tensor([e[1] for e in entries], dtype=torch.int64, device=gpu)
                for layer in range(bt.LAYERS):
                    k = _device_tensor(bt.kv_rows(layer, 0, toks, pos), gpu)
                    v = _device_tensor(bt.kv_rows(layer, 1, toks, pos), gpu)
                    pa.kv_append(k, v, dk[layer], dv[layer], slots)
        mirror.apply(op)

    decoded = []

    def after(step, batcher, pool, rep):
        pa.check_status()
        for got, want in zip(dk + dv, mirror.k + mirror.v):
            assert np.array_equal(_bits(got), want), f"device tier differs at step {step}"
        for got, want in zip(hk + hv, mirror.hk + mirror.hv):
            assert np.array_equal(_bits(got), want), f"host tier differs at step {step}"
        bt.check_running_contents(batcher, pool, mirror)
        seqs = [r.seq for r in batcher.running]
        if not seqs:
            return
        tab, lens = pool.tables(seqs, MAX_BLOCKS)
        bt_dev = torch.from_numpy(tab).to(gpu)
        cl_dev = torch.from_numpy(lens).to(gpu)
        q = wl.normal((len(seqs), bt.HQ, bt.D), torch.bfloat16, 50_000 + step, gpu)
        q_host = q.float().cpu().numpy()
        for layer in range(bt.LAYERS):
            out = pa.paged_attention_decode(q, dk[layer], dv[layer], bt_dev, cl_dev, scale)
            pa.check_status()
            want = oa.paged_attention_decode(q_host, bt.bits_to_float(mirror.k[layer]),
                                             bt.bits_to_float(mirror.v[layer]), tab, lens, scale)
            assert_attention_close(out, want, torch.bfloat16)
        decoded.append(len(seqs))

    batcher, pool, stats = bt.run_trace(seed, num_blocks, host_blocks, 40, 3000, apply, after,
                                        short_admissions=6)
    assert batcher.idle, stats
    assert sum(decoded) > 0
    assert stats["prefix_hit_tokens"] > 0 and stats["evictions"] > 0, stats
    assert stats["swap_out"] > 0 and stats["swap_in"] > 0 and stats["requeued"] > 0, stats
    assert stats["rekeyed_hits"] > 0 and stats["aborted_admissions"] > 0, stats
