"""Shared helpers for the GPU parity tests (inputs from the seeded generators,
expected values from ``oracle/`` only)."""

import numpy as np
import torch

import oracle.attention as oa
from pagedattention_decode_attention_gb300 import workloads as wl

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

# Tolerances (stated once, used by every attention parity test):
#   fp32 inputs: max |gpu - oracle| <= 1e-5
#   fp16 / bf16 inputs (fp32 accumulation): |gpu - oracle| <= 1e-2 + 2e-2 |oracle|
FP32_ATOL = 1e-5
LOWP_ATOL, LOWP_RTOL = 1e-2, 2e-2


def to_f32_numpy(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a (possibly 16-bit) tensor to float32 on the host."""
    return t.detach().float().cpu().numpy()


def assert_attention_close(gpu_out: torch.Tensor, ref: np.ndarray, dtype, rows=None):
    got = to_f32_numpy(gpu_out).astype(np.float64)
    if rows is not None:
        got, ref = got[rows], ref[rows]
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - ref)
    if dtype == torch.float32:
        worst = float(err.max()) if err.size else 0.0
        assert worst <= FP32_ATOL, f"max abs error {worst:.3e} > {FP32_ATOL}"
    else:
        bound = LOWP_ATOL + LOWP_RTOL * np.abs(ref)
        bad = err > bound
        assert not bad.any(), (
            f"{int(bad.sum())} of {err.size} elements outside tolerance; "
            f"worst excess {float((err - bound).max()):.3e}")


def decode_inputs(batch: wl.DecodeBatch, device, seed_offset=0):
    """Device tensors for one decode batch (N(0,1) values, seeded)."""
    dt = TORCH_DTYPES[batch.dtype]
    s = batch.seed + seed_offset
    q = wl.normal((batch.num_seqs, batch.num_q_heads, batch.head_dim), dt, s * 10 + 1, device)
    shape = (batch.num_blocks, batch.num_kv_heads, 16, batch.head_dim)
    kc = wl.normal(shape, dt, s * 10 + 2, device)
    vc = wl.normal(shape, dt, s * 10 + 3, device)
    bt = torch.from_numpy(batch.block_tables).to(device)
    cl = torch.from_numpy(batch.context_lens).to(device)
    return q, kc, vc, bt, cl


def oracle_decode(batch, q, kc, vc, seqs=None):
    """Oracle output (float64) from host copies of the generator's tensors."""
    return oa.paged_attention_decode(to_f32_numpy(q), to_f32_numpy(kc), to_f32_numpy(vc),
                                     batch.block_tables, batch.context_lens, batch.scale,
                                     seqs=seqs)


def custom_batch(lens, num_q_heads, num_kv_heads, head_dim, dtype, seed, slack_blocks=7,
                 max_blocks=None):
    gen = wl.rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    nb = int(wl.num_blocks_for(lens).sum()) + slack_blocks
    tables = wl.disjoint_tables(lens, nb, gen, max_blocks=max_blocks)
    return wl.DecodeBatch("custom", num_q_heads, num_kv_heads, head_dim, dtype, lens, tables, nb,
                          seed=seed)
