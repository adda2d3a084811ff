"""GB300-native paged-KV decode attention.

Device entry points (hand-written sm_103a kernels behind the C ABI in
``include/pagedattn.h``):

* :func:`kv_append` -- write new tokens' K/V rows into their paged slots;
* :func:`paged_attention_decode` -- one decode step of attention over a block
  table, MHA and GQA (:func:`paged_attention_decode_plan` +
  :func:`paged_attention_decode_run` split it so one plan serves every layer;
  :func:`paged_attention_decode_append_run` also appends each sequence's new
  token in the same launch; :func:`paged_attention_decode_shared_prefix` reads
  a prefix shared by the whole batch once;
  :func:`paged_attention_decode_grouped_prefix` each group's own prefix once);
* :func:`paged_attention_prefill` -- chunked-prefill attention: each
  sequence's newest tokens attend causally over the paged cache
  (:func:`prefill_plan` + :func:`paged_attention_prefill_run` split it so one
  plan serves every layer);
* :func:`block_copy` -- copy-on-write block copies across all layers;
* :func:`block_swap` -- whole blocks between the device caches and
  page-locked host caches (preemption / offload), all layers in one launch;
* :class:`LayerCaches` -- every layer's caches checked once, for repeated
  copies and swaps at one C call each;

and the native host :class:`BlockPool` that produces tables, slots and copy
pairs.  The library is loaded on first use; if it has not been built the call
raises -- there is no fallback implementation.
"""

from .capi import PagedAttnError  # noqa: F401
from .capi import PA_SWAP_IN, PA_SWAP_OUT  # noqa: F401
from .ops import (LayerCaches, Prepared, alloc_prefill_workspace, alloc_workspace,  # noqa: F401
                  block_copy, block_swap, check_status, kv_append, paged_attention_decode,
                  paged_attention_decode_append_run, paged_attention_decode_shared_prefix,
                  paged_attention_decode_grouped_prefix, paged_attention_decode_grouped_prefix_run,
                  paged_attention_decode_shared_prefix_append_run,
                  paged_attention_decode_grouped_prefix_append_run,
                  grouped_prefix_plan, grouped_prefix_workspace_size,
                  paged_attention_decode_shared_prefix_run, shared_prefix_plan,
                  paged_attention_prefill, paged_attention_prefill_run, prefill_plan,
                  shared_prefix_workspace_size, prefill_workspace_size,
                  paged_attention_decode_plan, paged_attention_decode_run,
                  prepare_decode_append_run, prepare_decode_plan, prepare_decode_run,
                  paged_attention_decode_noalloc, prepare_kv_append, workspace_size)
from .pool import BlockPool  # noqa: F401

# the C entry points' own names for the calls above whose Python name is shorter
paged_attention_decode_workspace_size = workspace_size
paged_attention_decode_shared_prefix_workspace_size = shared_prefix_workspace_size
paged_attention_decode_shared_prefix_plan = shared_prefix_plan
paged_attention_decode_grouped_prefix_workspace_size = grouped_prefix_workspace_size
paged_attention_decode_grouped_prefix_plan = grouped_prefix_plan
paged_attention_prefill_workspace_size = prefill_workspace_size
paged_attention_prefill_plan = prefill_plan


def version() -> int:
    """The library's ABI version (``pa_version``)."""
    from . import capi
    return int(capi.lib().pa_version())

BLOCK_SIZE = 16
