"""The no-allocation decode entry point, for callers that cannot allocate
device memory (their host framework owns the whole device-memory budget), so
cannot provide the workspace the regular entry point takes.

It is called through the C ABI, twice in a row (the built-in scratch keeps the
previous call's contents, which must not matter), and each output must be
bit-identical to the regular entry point's on the same inputs and within the
attention tolerance of the oracle.  This file is collected last.
"""

import ctypes as C

import pytest
import torch

from tests.gpu_helpers import assert_attention_close, custom_batch, decode_inputs, oracle_decode

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice(gpu):
    import pagedattention_decode_attention_gb300 as pa
    from pagedattention_decode_attention_gb300 import capi
    lib = capi.lib()
    # multi-split sequences, so the scratch really holds partial results
    batch = custom_batch([5, 700, 2100, 5000, 33, 1], 32, 8, 128, "bf16", seed=71)
    q, kc, vc, bt, cl = decode_inputs(batch, gpu)
    ref = pa.paged_attention_decode(q, kc, vc, bt, cl, batch.scale)
    pa.check_status()
    want = oracle_decode(batch, q, kc, vc)
    assert_attention_close(ref, want, torch.bfloat16)
    stream = torch.cuda.current_stream(gpu).cuda_stream
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        rc = lib.pa_paged_attention_decode_noalloc(
            q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), cl.data_ptr(),
            batch.num_seqs, 32, 8, 128, batch.max_blocks, batch.num_blocks,
            C.c_float(batch.scale), capi.PA_BF16, out.data_ptr(), stream)
        assert rc == capi.PA_OK, lib.pa_last_error()
        torch.cuda.synchronize()
        pa.check_status()
        # same plan, same kernels, splits merged in a fixed order: bit-identical
        assert torch.equal(out, ref)
        assert_attention_close(out, want, torch.bfloat16)


def test_noalloc_rejects_shapes_beyond_its_scratch(gpu):
    from pagedattention_decode_attention_gb300 import capi
    lib = capi.lib()
    # 4096 sequences x 256 blocks each: far more partial results than the
    # built-in scratch holds.  Every pointer is NULL, so even without the size
    # guard the call would be refused on the host before any launch.
    rc = lib.pa_paged_attention_decode_noalloc(None, None, None, None, None, 4096, 32, 8, 128,
                                               4096, 100000, C.c_float(0.1), capi.PA_BF16, None,
                                               None)
    assert rc == capi.PA_ERR_INVALID_ARG
    assert b"built into the library" in lib.pa_last_error()
