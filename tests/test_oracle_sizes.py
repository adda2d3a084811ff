"""Pins for the sizing / fragmentation oracle against the pages' printed numbers."""

from oracle import sizes
from tests.conftest import golden

GIB = 1 << 30
MIB = 1 << 20


def test_per_token_sizes():
    g = golden("kv_sizes.json")
    for key in ("mha_7b_per_token", "gqa_8b_per_token"):
        e = g[key]
        assert sizes.kv_cache_bytes(e["num_layers"], 1, e["num_kv_heads"], e["head_dim"],
                                    e["bytes_per_element"]) == e["bytes"], key


def test_request_and_batch_sizes():
    g = golden("kv_sizes.json")
    per7 = g["mha_7b_per_token"]
    f7 = lambda tokens, batch=1: sizes.kv_cache_bytes(32, tokens, 32, 128, 2, batch)
    assert f7(g["mha_7b_request_2048"]["tokens"]) == g["mha_7b_request_2048"]["bytes"]
    e = g["mha_7b_batch_10x2048"]
    assert f7(e["tokens"], e["batch"]) == e["bytes"]
    assert f7(g["mha_7b_prompt_4096"]["tokens"]) == g["mha_7b_prompt_4096"]["bytes"]
    assert per7["bytes"] == 512 * 1024

    f8 = lambda tokens: sizes.kv_cache_bytes(32, tokens, 8, 128, 2)
    assert f8(16) == g["gqa_8b_per_block"]["bytes"] == 2 * MIB
    e = g["gqa_8b_request_8k"]
    assert f8(e["tokens"]) == e["bytes"] == GIB
    assert sizes.blocks_for(e["tokens"]) == e["blocks"] == g["block_table_8k_entries"]["entries"]
    e = g["gqa_8b_context_128k"]
    assert f8(e["tokens"]) == e["bytes"] == 16 * GIB


def test_card_capacity_and_prefix_savings():
    g = golden("kv_sizes.json")
    e = g["gqa_8b_card_capacity"]
    per_block = sizes.kv_cache_bytes(32, 16, 8, 128, 2)
    assert e["free_bytes"] == 65 * GIB
    assert e["free_bytes"] // per_block == e["blocks"]
    assert e["blocks"] * 16 == e["tokens"]
    assert e["tokens"] // e["avg_request_tokens"] == e["requests"]
    e = g["gqa_8b_prefix_1k"]
    assert sizes.blocks_for(e["tokens"]) == e["blocks"]
    prefix = sizes.kv_cache_bytes(32, e["tokens"], 8, 128, 2)
    assert prefix == e["bytes"] == 128 * MIB
    assert e["sharers"] * prefix == e["saved_bytes_as_printed"]
    assert (e["sharers"] - 1) * prefix == e["saved_bytes_strict"]


def test_fragmentation_examples():
    g = golden("fragmentation.json")
    e = g["reserve_4096_use_512"]
    assert sizes.contiguous_waste_slots(e["reserved"], e["used"]) / e["reserved"] == e["waste_fraction"]
    for key in ("request_A", "request_B"):
        e = g[key]
        used = e["prompt"] + e["generated"] + e["future"]
        assert used == e["used"]
        assert sizes.contiguous_waste_slots(e["reserved"], used) == e["waste"]
        # paged: one 16-slot block each, the unfilled tail is the only waste
        assert sizes.blocks_for(used) == 1
        assert sizes.paged_waste_slots(used) == 16 - used
