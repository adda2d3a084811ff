"""CPU oracle for the paged-KV decode path.

TEST INFRASTRUCTURE ONLY. This package is the slow, obviously-correct
restatement of what the pages define; it exists so the CUDA path can be
checked against it.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product package (``pagedattention_decode_attention_gb300``) never imports
it, and it never imports the product package: the two share no code.

Modules
-------
attention : gather-through-block-table + softmax attention in float64 (decode
            and causal chunked prefill),
            kv_append and block_copy as plain element copies.
pool      : a pure-Python model of the block pool (free list, refcounts,
            lazy allocation, fork, copy-on-write, prefix sharing, pinning).
sizes     : the KV-cache size formula and fragmentation accounting.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against facts other than itself (library routines, closed forms, the pages'
worked examples); none is "parity unpinned".
"""

from . import attention, pool, sizes  # noqa: F401

BLOCK_SIZE = 16
