"""The continuous-batching driver on the native pool and on the pool model:
the same request stream must produce the same step reports (admissions with
prefix-cache hits, slots, copy-on-write pairs, preemptions by swapping,
resumptions, retirements) and the same final pool state.  CPU only."""

import os

import numpy as np
import pytest

from oracle.pool import BlockPool as ModelPool


@pytest.fixture(scope="module", autouse=True)
def built():
    from pagedattention_decode_attention_gb300 import build, capi
    if not os.path.exists(capi.LIB_PATH):
        build.build()


def _stream(seed, n_requests):
    """Requests sharing three system prompts, lognormal suffixes (median 30,
    clipped to [1, 200]) and U{5..80} new tokens; each carries how many
    requests arrive at the step it arrives in (0-3, at least one overall)."""
    gen = np.random.default_rng(seed)
    systems = [list(range(10_000 * (k + 1), 10_000 * (k + 1) + n)) for k, n in
               enumerate((48, 100, 200))]
    reqs = []
    for r in range(n_requests):
        sfx = int(np.clip(round(np.exp(gen.normal(np.log(30), 1.0))), 1, 200))
        prompt = systems[int(gen.integers(3))] + [int(x) for x in gen.integers(0, 50_000, sfx)]
        reqs.append((prompt, int(gen.integers(5, 81)), int(gen.integers(0, 4))))
    return reqs


def _drive(pool, reqs, steps):
    from pagedattention_decode_attention_gb300.batching import ContinuousBatcher
    b = ContinuousBatcher(pool, 16, max_running=48)
    reports, pending = [], list(reqs)
    arrivals = np.random.default_rng(len(reqs)).integers(0, 4, size=steps)
    tok = lambda r: (r.rid * 7919 + r.generated * 104729) % 50_000  # noqa: E731
    for step in range(steps):
        for _ in range(int(arrivals[step])):
            if pending:
                p, n, _ = pending.pop(0)
                b.submit(p, n)
        rep = b.step(tok)
        reports.append((rep.admitted, rep.slots, rep.cow_pairs, rep.swap_out, rep.swap_in,
                        rep.retired, rep.requeued))
        if not pending and b.idle:
            break
    return reports


def _pools(num_blocks, host_blocks, seed):
    from pagedattention_decode_attention_gb300 import BlockPool
    order = np.random.default_rng(seed).permutation(num_blocks)
    horder = np.random.default_rng(seed + 1).permutation(host_blocks)
    nat, mod = BlockPool(num_blocks, 16, order), ModelPool(num_blocks, 16, order)
    for p in (nat, mod):
        p.enable_prefix_cache()
        p.set_host_blocks(host_blocks, horder)
    return nat, mod


@pytest.mark.parametrize("seed,num_blocks,host_blocks", [(1, 160, 80), (2, 96, 40), (3, 400, 0)])
def test_batcher_native_equals_model(seed, num_blocks, host_blocks):
    reqs = _stream(seed, 70)
    nat, mod = _pools(num_blocks, host_blocks, seed)
    r_nat = _drive(nat, reqs, 2000)
    r_mod = _drive(mod, reqs, 2000)
    assert r_nat == r_mod
    st = nat.stats()
    assert st == mod.stats()
    assert st["live_seqs"] == 0 and st["used_blocks"] == 0      # everything retired
    assert st["prefix_hit_tokens"] > 0                          # shared system prompts hit


def test_batcher_under_pressure_preempts_and_evicts():
    reqs = _stream(4, 70)
    nat, mod = _pools(72, 48, 4)
    reports = _drive(nat, reqs, 4000)
    assert any(r[3] for r in reports) and any(r[4] for r in reports)   # swaps out and in
    assert nat.stats()["evictions"] > 0
    assert _drive(mod, reqs, 4000) == reports
