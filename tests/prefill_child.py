"""Chunked-prefill parity checks run in a child process (the kernel choice,
PA_PREFILL_TC, is read once per process).  ``python -m tests.prefill_child
[quick]``; exit status 0 means every check passed."""

import sys

import numpy as np
import torch

import oracle.attention as oa
from pagedattention_decode_attention_gb300 import workloads as wl
from tests.gpu_helpers import TORCH_DTYPES, assert_attention_close, custom_batch, to_f32_numpy


def check(lens, qlens, hq, hkv, d, dtype, seed, rows=None):
    import pagedattention_decode_attention_gb300 as pa
    dev = torch.device("cuda", 0)
    batch = custom_batch(lens, hq, hkv, d, dtype, seed=seed)
    dt = TORCH_DTYPES[dtype]
    kc = wl.normal((batch.num_blocks, hkv, 16, d), dt, seed * 10 + 2, dev)
    vc = wl.normal((batch.num_blocks, hkv, 16, d), dt, seed * 10 + 3, dev)
    qs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = wl.normal((int(qs[-1]), hq, d), dt, seed * 10 + 1, dev)
    outs = []
    ws = pa.alloc_prefill_workspace(len(lens), int(qs[-1]), hq, hkv, d, dev)
    for _ in range(2):  # twice on one workspace: the counters reset
        outs.append(pa.paged_attention_prefill(
            q, kc, vc, torch.from_numpy(batch.block_tables).to(dev),
            torch.from_numpy(batch.context_lens).to(dev), torch.from_numpy(qs).to(dev),
            batch.scale, workspace=ws).clone())
    pa.check_status()
    ref = oa.paged_attention_prefill(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc),
                                     batch.block_tables, batch.context_lens, qs, batch.scale,
                                     rows=rows)
    assert torch.equal(outs[0], outs[1])
    assert_attention_close(outs[0], ref, dt, rows=rows)


def main(quick: bool) -> int:
    lens = [40, 17, 300, 1, 530, 2000, 64, 900]
    qlens = [40, 17, 37, 1, 1, 9, 0, 128]
    check(lens, qlens, 32, 8, 128, "bf16", 71)
    if quick:
        return 0
    for hq, hkv in ((8, 8), (16, 8), (16, 2)):
        for dtype in ("bf16", "f16"):
            check(lens, qlens, hq, hkv, 128, dtype, 72 + hq)
    check(lens, qlens, 32, 8, 64, "bf16", 80)                 # head_dim 64: the mma.sync path
    check([12345, 7000], [3, 16], 32, 8, 128, "bf16", 81)
    lens2, qlens2 = [4096, 2048, 3000, 2100], [2048, 2048, 1000, 77]
    rows = sorted(set([0, 1, 15, 16, 127, 128, 2047, 2048, 4095, 4096, 5095, 5096, 5172]
                      + list(np.random.default_rng(1).integers(0, sum(qlens2), 24))))
    check(lens2, qlens2, 32, 8, 128, "bf16", 82, rows=rows)
    return 0


if __name__ == "__main__":
    sys.exit(main(len(sys.argv) > 1 and sys.argv[1] == "quick"))
