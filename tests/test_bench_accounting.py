"""The byte and flop counts the bench's rooflines divide by (CPU): each
matches a count made by hand on a small batch."""

import numpy as np

from pagedattention_decode_attention_gb300 import workloads as wl


def batch(lens, tables, hq=4, hkv=2, d=64, dtype="f16", extra=None):
    return wl.DecodeBatch("t", hq, hkv, d, dtype, np.array(lens, dtype=np.int32),
                          np.array(tables, dtype=np.int32), 64, extra=extra or {})


def test_algorithmic_bytes_by_hand():
    import bench
    b = batch([17, 3], [[5, 9], [7, -1]])        # 17 tokens in 2 blocks, 3 in 1
    got = bench.algorithmic_bytes(b)
    row = 2 * 64 * 2                              # one token's K and V row of one KV head, bytes
    assert got["tokens"] == 20
    assert got["kv"] == 20 * row * 2              # two KV heads
    qo = 2 * 2 * 4 * 64 * 2                       # q read + out written, 2 seqs x 4 heads
    tables = 3 * 4 + 2 * 4                        # 3 table entries, 2 lengths
    append = 2 * 2 * 2 * 2 * 64 * 2 + 2 * 8       # new K and V rows read + written, slots
    assert got["total"] == got["kv"] + qo + tables + append


def test_unique_bytes_count_a_shared_block_once():
    import bench
    # both sequences share physical block 5; the second also attends 4 tokens
    # of its own block 6; a block counts its attended tokens once
    b = batch([16, 20], [[5, -1], [5, 6]])
    per_token = 2 * 2 * 64 * 2                    # K and V, 2 KV heads, fp16
    assert bench.unique_kv_bytes(b) == (16 + 4) * per_token
    # a partial shared block counts the most tokens any sharer attends
    b = batch([10, 14], [[5], [5]])
    assert bench.unique_kv_bytes(b) == 14 * per_token


def test_prefill_flops_by_hand():
    import bench
    # a 3-token chunk on a 5-token context: positions 2, 3, 4 attend 3, 4, 5
    b = batch([5], [[1]], hq=8, d=128, extra={"query_lens": np.array([3])})
    assert bench.prefill_flops(b) == (3 + 4 + 5) * 4 * 128 * 8
    # a whole prompt (chunk = context) attends 1 + 2 + ... + n tokens
    b = batch([4], [[1]], hq=1, d=64, extra={"query_lens": np.array([4])})
    assert bench.prefill_flops(b) == (1 + 2 + 3 + 4) * 4 * 64


def test_cascade_launch_counts(monkeypatch):
    """The cascade lines' `gpu_launches`: the grouped decode is one plan and
    one attention launch per layer (its merges run inside that launch); the
    three phases are their plans and three launches per layer."""
    import bench
    monkeypatch.delenv("PA_CASCADE", raising=False)
    assert bench.cascade_launches_per_step(True, 8) == 1 + 8        # groups: grouped decode
    assert bench.cascade_launches_per_step(False, 32) == 2 + 3 * 32  # one prefix: phases
    monkeypatch.setenv("PA_CASCADE", "phases")
    assert bench.cascade_launches_per_step(True, 8) == 3 + 3 * 8
    monkeypatch.setenv("PA_CASCADE", "grouped")
    assert bench.cascade_launches_per_step(False, 32) == 1 + 32
