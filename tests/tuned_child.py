"""Parity checks run in a child process under non-default kernel tuning.

The attention library reads its tuning variables (PA_DECODE_*) once per
process, so each configuration gets a fresh interpreter; the parent test
(``test_gpu_tuning.py``) sets the variables and runs ``python -m
tests.tuned_child``.  Exit status 0 means every check passed.
"""

import sys

import torch

from tests.gpu_helpers import (TORCH_DTYPES, assert_attention_close, custom_batch, decode_inputs,
                               oracle_decode)


def main() -> int:
    import pagedattention_decode_attention_gb300 as pa
    dev = torch.device("cuda", 0)
    lens = [1, 15, 16, 17, 100, 511, 512, 513, 1100, 2000, 4100]
    cases = [(lens, 4, 4, 128, "f16"), (lens, 32, 8, 128, "bf16"), (lens, 16, 2, 64, "bf16"),
             ([12345], 32, 8, 128, "bf16"), ([0, 3, 700], 8, 8, 64, "f16")]
    for i, (ls, hq, hkv, d, dt) in enumerate(cases):
        batch = custom_batch(ls, hq, hkv, d, dt, seed=500 + i)
        q, kc, vc, bt, cl = decode_inputs(batch, dev)
        ref = oracle_decode(batch, q, kc, vc)
        ws = pa.alloc_workspace(batch.num_seqs, hq, hkv, d, batch.max_blocks, dev)
        outs = []
        for _ in range(2):  # twice on one workspace: the counters must reset
            outs.append(pa.paged_attention_decode(q, kc, vc, bt, cl, batch.scale,
                                                  workspace=ws).clone())
        pa.check_status()
        for o in outs:
            assert_attention_close(o, ref, TORCH_DTYPES[dt])
        assert torch.equal(outs[0], outs[1])
    # the grouped decode's plan under the same split, tail and piece settings
    import numpy as np

    import oracle.attention as oa
    from tests.gpu_helpers import to_f32_numpy
    from tests.test_gpu_grouped_prefix import GROUPS, grouped_batch
    for hq, hkv, d, dt in ((32, 8, 128, "bf16"), (16, 2, 64, "f16")):
        q, kc, vc, tables, lens, gs, gb = grouped_batch(GROUPS, hq, hkv, d, dt, seed=77, dev=dev)
        bt, cl, gs_d, gb_d = (torch.from_numpy(a).to(dev) for a in (tables, lens, gs, gb))
        scale = 1.0 / np.sqrt(d)
        out = pa.paged_attention_decode_grouped_prefix(q, kc, vc, bt, cl, gs_d, gb_d, scale)
        pa.check_status()
        ref = oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc),
                                        tables, lens, scale)
        assert_attention_close(out, ref, TORCH_DTYPES[dt])
    return 0


if __name__ == "__main__":
    sys.exit(main())
