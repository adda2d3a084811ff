"""The batcher's ordered device operations, applied to host caches with the
oracle's copies, keep every running sequence's cache content exact through
prefix-cache hits, LRU eviction with recomputation, copy-on-write and swapping
to host memory and back (CPU only; the GPU test applies the same operations
with the device kernels)."""

import os

import pytest

from tests import batch_trace as bt


@pytest.fixture(scope="module", autouse=True)
def built():
    from pagedattention_decode_attention_gb300 import build, capi
    if not os.path.exists(capi.LIB_PATH):
        build.build()


def _run(seed, num_blocks, host_blocks, short_admissions=0):
    tiers = bt.HostTiers(num_blocks, host_blocks)
    checked = []

    def after(step, batcher, pool, rep):
        checked.append(bt.check_running_contents(batcher, pool, tiers))

    batcher, pool, stats = bt.run_trace(seed, num_blocks, host_blocks, 40, 3000, tiers.apply,
                                        after, short_admissions=short_admissions)
    assert batcher.idle, stats
    assert sum(checked) > 0
    return stats


@pytest.mark.parametrize("seed,num_blocks,host_blocks", [(11, 40, 12), (12, 56, 24)])
def test_trace_keeps_every_running_sequence_exact(seed, num_blocks, host_blocks):
    stats = _run(seed, num_blocks, host_blocks)
    # the trace really exercised what it is meant to
    assert stats["prefix_hit_tokens"] > 0, stats
    assert stats["evictions"] > 0, stats
    assert stats["swap_out"] > 0 and stats["swap_in"] > 0, stats
    assert stats["requeued"] > 0, stats
    assert stats["rekeyed_hits"] > 0, stats


def test_cut_short_admissions_leave_written_cached_blocks():
    """A prompt append that stops early still reports its slots: the blocks
    it filled were keyed into the prefix cache, and the request's next
    admission hits them."""
    stats = _run(11, 40, 12, short_admissions=6)
    assert stats["aborted_admissions"] == 6, stats


def test_dropping_a_cut_short_admissions_appends_is_caught(monkeypatch):
    """The content check is strong enough to see the mistake of dropping
    those appends (planted in the batcher's report, on the CPU)."""
    from pagedattention_decode_attention_gb300 import batching
    step = batching.ContinuousBatcher.step

    def dropping_step(self, next_token):
        rep = step(self, next_token)
        gone = {seq for _, seq in rep.aborted}
        rep.ops = [op for op in rep.ops
                   if not (op[0] == "append" and op[2] and op[2][0][0] in gone)]
        return rep

    monkeypatch.setattr(batching.ContinuousBatcher, "step", dropping_step)
    with pytest.raises(AssertionError, match="rows wrong"):
        _run(11, 40, 12, short_admissions=6)
