"""KV-cache sizing and fragmentation accounting.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* OS-lab appendix, section 2.2: the KV cache of a batch is
  ``2 x num_layers x sequence_length x num_kv_heads x head_dim x
  bytes_per_element x batch_size`` (the 2 is keys plus values).
* OS-lab appendix, section 3.2 and "vLLM: treating the KV cache as virtual
  memory", section "跨域连接" (combinatorics): reserving the maximum length
  wastes ``L_max - L_i`` slots per request; paging wastes only the unfilled
  tail of the last block.
"""

from __future__ import annotations


def kv_cache_bytes(num_layers: int, seq_len: int, num_kv_heads: int, head_dim: int,
                   bytes_per_element: int, batch_size: int = 1) -> int:
    return 2 * num_layers * seq_len * num_kv_heads * head_dim * bytes_per_element * batch_size


def blocks_for(tokens: int, block_size: int = 16) -> int:
    """Physical blocks a request of ``tokens`` tokens holds under lazy allocation."""
    return -(-tokens // block_size)


def contiguous_waste_slots(reserved: int, used: int) -> int:
    """Slots reserved up front but never written (internal fragmentation)."""
    return reserved - used


def paged_waste_slots(used: int, block_size: int = 16) -> int:
    """Slots held but unwritten when only whole blocks are handed out."""
    return blocks_for(used, block_size) * block_size - used
