"""Torch-facing binding of the device entry points.

Argument marshalling only: each function checks shapes / dtypes / devices of
the torch tensors, passes their raw pointers and the current CUDA stream to the
C ABI, and raises ``PagedAttnError`` on a non-zero status.  All computation
happens in the library's kernels.
"""

from __future__ import annotations

import ctypes as C

import torch

from . import capi

_DTYPES = {torch.float32: capi.PA_F32, torch.float16: capi.PA_F16, torch.bfloat16: capi.PA_BF16}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype} (float32, float16 or bfloat16)")
    return _DTYPES[t.dtype]


def _stream(device: torch.device, stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _cuda_contig(name: str, t: torch.Tensor, device: torch.device) -> None:
    _require(t.is_cuda and t.device == device, f"{name} must be on {device}")
    _require(t.is_contiguous(), f"{name} must be contiguous")


def workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   max_blocks_per_seq: int) -> int:
    out = C.c_size_t(0)
    capi.check(capi.lib().pa_paged_attention_decode_workspace_size(
        num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, C.byref(out)))
    return out.value


def alloc_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                    device) -> torch.Tensor:
    n = workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def kv_append(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              slot_mapping: torch.Tensor, stream=None) -> None:
    """Write ``k[i]`` / ``v[i]`` (``[T, Hkv, d]``) into slot ``slot_mapping[i]``
    of the paged caches (``[NB, Hkv, 16, d]``); negative slots are skipped."""
    dev = k_cache.device
    for name, t in (("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("slot_mapping", slot_mapping)):
        _cuda_contig(name, t, dev)
    _require(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    _require(k.dtype == v.dtype == k_cache.dtype == v_cache.dtype, "dtypes must match")
    _require(k_cache.dim() == 4 and k_cache.shape == v_cache.shape and k_cache.shape[2] == 16,
             "caches must be [num_blocks, num_kv_heads, 16, head_dim]")
    nb, hkv, _, d = k_cache.shape
    _require(k.shape == v.shape and k.dim() == 3 and tuple(k.shape[1:]) == (hkv, d),
             "k, v must be [num_tokens, num_kv_heads, head_dim]")
    _require(slot_mapping.shape == (k.shape[0],), "slot_mapping must be [num_tokens]")
    capi.check(capi.lib().pa_kv_append(
        k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        slot_mapping.data_ptr(), k.shape[0], hkv, d, nb, _dtype_code(k), _stream(dev, stream)))


def _decode_args(q, k_cache, v_cache, block_tables, context_lens):
    """Checks the decode operands (context_lens None: not passed) and returns
    (device, num_seqs, Hq, Hkv, d, num_blocks, max_blocks_per_seq)."""
    dev = q.device
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_tables", block_tables), ("context_lens", context_lens)):
        if t is not None:
            _cuda_contig(name, t, dev)
    _require(block_tables.dtype == torch.int32 and
             (context_lens is None or context_lens.dtype == torch.int32),
             "block_tables and context_lens must be int32")
    _require(q.dtype == k_cache.dtype == v_cache.dtype, "q and caches must share a dtype")
    _require(k_cache.dim() == 4 and k_cache.shape == v_cache.shape and k_cache.shape[2] == 16,
             "caches must be [num_blocks, num_kv_heads, 16, head_dim]")
    nb, hkv, _, d = k_cache.shape
    _require(q.dim() == 3 and q.shape[2] == d, "q must be [num_seqs, num_q_heads, head_dim]")
    b, hq, _ = q.shape
    _require(block_tables.dim() == 2 and block_tables.shape[0] == b,
             "block_tables must be [num_seqs, max_blocks_per_seq]")
    _require(context_lens is None or context_lens.shape == (b,), "context_lens must be [num_seqs]")
    return dev, b, hq, hkv, d, nb, block_tables.shape[1]


def paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """Decode attention of ``q`` (``[B, Hq, d]``) over paged ``k_cache`` /
    ``v_cache`` (``[NB, Hkv, 16, d]``) through ``block_tables`` (int32
    ``[B, max_blocks]``) for ``context_lens`` (int32 ``[B]``) tokens.  Plans
    and runs in one call."""
    return _decode(capi.lib().pa_paged_attention_decode, q, k_cache, v_cache, block_tables,
                   context_lens, scale, out, workspace, stream)


def paged_attention_decode_run(q, k_cache, v_cache, block_tables, context_lens, scale,
                               workspace: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    """Same as :func:`paged_attention_decode` on a workspace already planned by
    :func:`paged_attention_decode_plan` (one plan serves every layer of a step)."""
    return _decode(capi.lib().pa_paged_attention_decode_run, q, k_cache, v_cache, block_tables,
                   context_lens, scale, out, workspace, stream)


def _append_args(q, k_new, v_new, slot_mapping, hkv, d):
    dev, b = q.device, q.shape[0]
    for name, t in (("k_new", k_new), ("v_new", v_new), ("slot_mapping", slot_mapping)):
        _cuda_contig(name, t, dev)
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.shape == (b,),
             "slot_mapping must be int64 [num_seqs]")
    _require(k_new.dtype == v_new.dtype == q.dtype, "k_new / v_new must have q's dtype")
    _require(k_new.shape == v_new.shape == (b, hkv, d),
             "k_new, v_new must be [num_seqs, num_kv_heads, head_dim]")


def paged_attention_decode_append_run(q, k_new, v_new, slot_mapping, k_cache, v_cache,
                                      block_tables, context_lens, scale,
                                      workspace: torch.Tensor, out=None,
                                      stream=None) -> torch.Tensor:
    """:func:`kv_append` of one new token per sequence (row ``b`` of ``k_new`` /
    ``v_new`` to ``slot_mapping[b]``, the slot of the sequence's last token)
    followed by :func:`paged_attention_decode_run`, in one launch.  The
    workspace must hold a plan for these context lengths."""
    dev, b, hq, hkv, d, nb, mb = _decode_args(q, k_cache, v_cache, block_tables, context_lens)
    _append_args(q, k_new, v_new, slot_mapping, hkv, d)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, dev)
    _require(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    _cuda_contig("workspace", workspace, dev)
    capi.check(capi.lib().pa_paged_attention_decode_append_run(
        q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(),
        k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(),
        b, hq, hkv, d, mb, nb, float(scale), _dtype_code(q), out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(dev, stream)))
    return out


def _decode(fn, q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace, stream):
    dev, b, hq, hkv, d, nb, mb = _decode_args(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, dev)
    _require(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        workspace = alloc_workspace(b, hq, hkv, d, mb, dev)
    _cuda_contig("workspace", workspace, dev)
    capi.check(fn(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        context_lens.data_ptr(), b, hq, hkv, d, mb, nb, float(scale), _dtype_code(q),
        out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(dev, stream)))
    return out


def paged_attention_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale,
                                   out=None, stream=None) -> torch.Tensor:
    """:func:`paged_attention_decode` for callers that cannot allocate device
    memory: the library's built-in 128 MiB scratch replaces the workspace
    (calls on one device share it, so they must not overlap on the GPU)."""
    dev, b, hq, hkv, d, nb, mb = _decode_args(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, dev)
    _require(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    capi.check(capi.lib().pa_paged_attention_decode_noalloc(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        context_lens.data_ptr(), b, hq, hkv, d, mb, nb, float(scale), _dtype_code(q),
        out.data_ptr(), _stream(dev, stream)))
    return out


def paged_attention_decode_plan(context_lens: torch.Tensor, num_q_heads: int, num_kv_heads: int,
                                head_dim: int, max_blocks_per_seq: int, workspace: torch.Tensor,
                                stream=None) -> None:
    """Write the work list for these context lengths into ``workspace``."""
    dev = context_lens.device
    _cuda_contig("context_lens", context_lens, dev)
    _cuda_contig("workspace", workspace, dev)
    _require(context_lens.dtype == torch.int32 and context_lens.dim() == 1,
             "context_lens must be int32 [num_seqs]")
    capi.check(capi.lib().pa_paged_attention_decode_plan(
        context_lens.data_ptr(), context_lens.shape[0], num_q_heads, num_kv_heads, head_dim,
        max_blocks_per_seq, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(dev, stream)))


class Prepared:
    """A device entry point bound to fixed tensors.

    Validation and pointer marshalling happen once, in the ``prepare_*``
    function; each call re-issues only the C call with the stored arguments.
    Meant for per-layer loops that reuse the same buffers every decode step.
    The bound tensors are kept alive by this object.
    """

    def __init__(self, fn, args, keep):
        self._fn, self._args, self._keep = fn, args, keep

    def __call__(self) -> None:
        status = self._fn(*self._args)
        if status:
            capi.check(status)


def prepare_kv_append(k, v, k_cache, v_cache, slot_mapping, stream=None) -> Prepared:
    kv_append(k[:0], v[:0], k_cache, v_cache, slot_mapping[:0], stream)  # validates shapes
    nb, hkv, _, d = k_cache.shape
    args = (C.c_void_p(k.data_ptr()), C.c_void_p(v.data_ptr()), C.c_void_p(k_cache.data_ptr()),
            C.c_void_p(v_cache.data_ptr()), C.c_void_p(slot_mapping.data_ptr()), k.shape[0], hkv,
            d, nb, _dtype_code(k), C.c_void_p(_stream(k_cache.device, stream)))
    _require(slot_mapping.shape == (k.shape[0],), "slot_mapping must be [num_tokens]")
    return Prepared(capi.lib().pa_kv_append, args, (k, v, k_cache, v_cache, slot_mapping))


def prepare_decode_plan(context_lens, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                        workspace, stream=None) -> Prepared:
    dev = context_lens.device
    _cuda_contig("context_lens", context_lens, dev)
    _cuda_contig("workspace", workspace, dev)
    args = (C.c_void_p(context_lens.data_ptr()), context_lens.shape[0], num_q_heads, num_kv_heads,
            head_dim, max_blocks_per_seq, C.c_void_p(workspace.data_ptr()),
            C.c_size_t(workspace.numel() * workspace.element_size()), C.c_void_p(_stream(dev, stream)))
    return Prepared(capi.lib().pa_paged_attention_decode_plan, args, (context_lens, workspace))


def prepare_decode_run(q, k_cache, v_cache, block_tables, context_lens, scale, workspace, out,
                       stream=None) -> Prepared:
    dev, b, hq, hkv, d, nb, mb = _decode_args(q, k_cache, v_cache, block_tables, context_lens)
    _cuda_contig("out", out, dev)
    _cuda_contig("workspace", workspace, dev)
    _require(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    args = (C.c_void_p(q.data_ptr()), C.c_void_p(k_cache.data_ptr()), C.c_void_p(v_cache.data_ptr()),
            C.c_void_p(block_tables.data_ptr()), C.c_void_p(context_lens.data_ptr()), b, hq, hkv, d,
            mb, nb, C.c_float(scale), _dtype_code(q), C.c_void_p(out.data_ptr()),
            C.c_void_p(workspace.data_ptr()), C.c_size_t(workspace.numel() * workspace.element_size()),
            C.c_void_p(_stream(dev, stream)))
    return Prepared(capi.lib().pa_paged_attention_decode_run, args,
                    (q, k_cache, v_cache, block_tables, context_lens, workspace, out))


def prepare_decode_append_run(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                              context_lens, scale, workspace, out, stream=None) -> Prepared:
    dev, b, hq, hkv, d, nb, mb = _decode_args(q, k_cache, v_cache, block_tables, context_lens)
    _append_args(q, k_new, v_new, slot_mapping, hkv, d)
    _cuda_contig("out", out, dev)
    _cuda_contig("workspace", workspace, dev)
    _require(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    args = (C.c_void_p(q.data_ptr()), C.c_void_p(k_new.data_ptr()), C.c_void_p(v_new.data_ptr()),
            C.c_void_p(slot_mapping.data_ptr()), C.c_void_p(k_cache.data_ptr()),
            C.c_void_p(v_cache.data_ptr()), C.c_void_p(block_tables.data_ptr()),
            C.c_void_p(context_lens.data_ptr()), b, hq, hkv, d, mb, nb, C.c_float(scale),
            _dtype_code(q), C.c_void_p(out.data_ptr()), C.c_void_p(workspace.data_ptr()),
            C.c_size_t(workspace.numel() * workspace.element_size()),
            C.c_void_p(_stream(dev, stream)))
    return Prepared(capi.lib().pa_paged_attention_decode_append_run, args,
                    (q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, context_lens,
                     workspace, out))


def shared_prefix_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                 head_dim: int, max_blocks_per_seq: int) -> int:
    n = C.c_size_t(0)
    capi.check(capi.lib().pa_paged_attention_decode_shared_prefix_workspace_size(
        num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, C.byref(n)))
    return n.value


def shared_prefix_plan(context_lens: torch.Tensor, prefix_blocks: int, num_q_heads: int,
                       num_kv_heads: int, head_dim: int, max_blocks_per_seq: int, scale: float,
                       dtype: torch.dtype, workspace: torch.Tensor, stream=None) -> None:
    """The work lists of a shared-prefix (cascade) decode batch, into
    ``workspace``: one plan serves every
    :func:`paged_attention_decode_shared_prefix_run` over the same lengths."""
    dev = context_lens.device
    _cuda_contig("context_lens", context_lens, dev)
    _cuda_contig("workspace", workspace, dev)
    _require(context_lens.dtype == torch.int32, "context_lens must be int32")
    _require(dtype in _DTYPES, "dtype must be float32, float16 or bfloat16")
    capi.check(capi.lib().pa_paged_attention_decode_shared_prefix_plan(
        context_lens.data_ptr(), int(prefix_blocks), context_lens.shape[0], int(num_q_heads),
        int(num_kv_heads), int(head_dim), int(max_blocks_per_seq), float(scale), _DTYPES[dtype],
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(dev, stream)))


def paged_attention_decode_shared_prefix_run(q, k_cache, v_cache, block_tables, context_lens,
                                             prefix_blocks: int, scale: float, workspace,
                                             out=None, stream=None) -> torch.Tensor:
    """:func:`paged_attention_decode_shared_prefix` over a workspace that
    :func:`shared_prefix_plan` filled for the same lengths: the compute
    launches only."""
    return paged_attention_decode_shared_prefix(
        q, k_cache, v_cache, block_tables, context_lens, prefix_blocks, scale, out=out,
        workspace=workspace, stream=stream, _entry="pa_paged_attention_decode_shared_prefix_run")


def paged_attention_decode_shared_prefix(q, k_cache, v_cache, block_tables, context_lens,
                                         prefix_blocks: int, scale: float, out=None,
                                         workspace=None, stream=None,
                                         _entry="pa_paged_attention_decode_shared_prefix"
                                         ) -> torch.Tensor:
    """:func:`paged_attention_decode` for a batch whose tables all start with
    the same ``prefix_blocks`` blocks: the shared blocks are read once for all
    queries, each sequence's own blocks by the decode kernel, then the two
    parts are merged."""
    dev, b, hq, hkv, d, nb, mb = _decode_args(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, dev)
    _require(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        n = shared_prefix_workspace_size(b, hq, hkv, d, mb)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    _cuda_contig("workspace", workspace, dev)
    capi.check(getattr(capi.lib(), _entry)(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        context_lens.data_ptr(), int(prefix_blocks), b, hq, hkv, d, mb, nb, float(scale),
        _dtype_code(q), out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(dev, stream)))
    return out


def grouped_prefix_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                  head_dim: int, max_blocks_per_seq: int) -> int:
    n = C.c_size_t(0)
    capi.check(capi.lib().pa_paged_attention_decode_grouped_prefix_workspace_size(
        num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, C.byref(n)))
    return n.value


def _group_args(group_start, group_prefix_blocks, num_seqs, dev):
    for name, t in (("group_start", group_start), ("group_prefix_blocks", group_prefix_blocks)):
        _cuda_contig(name, t, dev)
        _require(t.dtype == torch.int32 and t.dim() == 1, f"{name} must be int32 [n]")
    g = group_prefix_blocks.shape[0]
    _require(group_start.shape[0] == g + 1, "group_start must have num_groups + 1 entries")
    _require(1 <= g <= num_seqs, "num_groups must be 1 .. num_seqs")
    return g


def grouped_prefix_plan(block_tables: torch.Tensor, context_lens: torch.Tensor,
                        group_start: torch.Tensor, group_prefix_blocks: torch.Tensor,
                        num_q_heads: int, num_kv_heads: int, head_dim: int, scale: float,
                        dtype: torch.dtype, workspace: torch.Tensor, stream=None) -> None:
    """Once per decode step: every sequence's table past its group's prefix
    and the work lists of a grouped shared-prefix (cascade) decode, into
    ``workspace``; one plan serves every
    :func:`paged_attention_decode_grouped_prefix_run` of the step."""
    dev = context_lens.device
    for name, t in (("block_tables", block_tables), ("context_lens", context_lens),
                    ("workspace", workspace)):
        _cuda_contig(name, t, dev)
    _require(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32,
             "block_tables and context_lens must be int32")
    _require(block_tables.dim() == 2 and block_tables.shape[0] == context_lens.shape[0],
             "block_tables must be [num_seqs, max_blocks_per_seq]")
    b = context_lens.shape[0]
    g = _group_args(group_start, group_prefix_blocks, b, dev)
    _require(dtype in _DTYPES, "dtype must be float32, float16 or bfloat16")
    capi.check(capi.lib().pa_paged_attention_decode_grouped_prefix_plan(
        block_tables.data_ptr(), context_lens.data_ptr(), group_start.data_ptr(),
        group_prefix_blocks.data_ptr(), g, b, int(num_q_heads), int(num_kv_heads), int(head_dim),
        block_tables.shape[1], float(scale), _DTYPES[dtype], workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(dev, stream)))


def paged_attention_decode_grouped_prefix_run(q, k_cache, v_cache, block_tables, group_start,
                                              group_prefix_blocks, scale: float, workspace,
                                              out=None, stream=None) -> torch.Tensor:
    """Per layer, over a workspace :func:`grouped_prefix_plan` filled: every
    group's prefix read once for its queries, each sequence's own blocks,
    then the merge."""
    dev, b, hq, hkv, d, nb, mb = _decode_args(q, k_cache, v_cache, block_tables, None)
    g = _group_args(group_start, group_prefix_blocks, b, dev)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, dev)
    _require(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    _cuda_contig("workspace", workspace, dev)
    capi.check(capi.lib().pa_paged_attention_decode_grouped_prefix_run(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        group_start.data_ptr(), group_prefix_blocks.data_ptr(), g, b, hq, hkv, d, mb, nb,
        float(scale), _dtype_code(q), out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(dev, stream)))
    return out


def paged_attention_decode_grouped_prefix(q, k_cache, v_cache, block_tables, context_lens,
                                          group_start, group_prefix_blocks, scale: float,
                                          out=None, workspace=None, stream=None) -> torch.Tensor:
    """:func:`paged_attention_decode` for a batch of groups of sequences, each
    group's tables starting with the same ``group_prefix_blocks[g]`` blocks
    (group g: sequences ``group_start[g] .. group_start[g + 1] - 1``): each
    group's shared blocks are read once for the group's queries."""
    dev, b, hq, hkv, d, nb, mb = _decode_args(q, k_cache, v_cache, block_tables, context_lens)
    g = _group_args(group_start, group_prefix_blocks, b, dev)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, dev)
    _require(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        n = grouped_prefix_workspace_size(b, hq, hkv, d, mb)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    _cuda_contig("workspace", workspace, dev)
    capi.check(capi.lib().pa_paged_attention_decode_grouped_prefix(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        context_lens.data_ptr(), group_start.data_ptr(), group_prefix_blocks.data_ptr(), g, b,
        hq, hkv, d, mb, nb, float(scale), _dtype_code(q), out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(dev, stream)))
    return out


def paged_attention_decode_shared_prefix_append_run(q, k_new, v_new, slot_mapping, k_cache,
                                                    v_cache, block_tables, context_lens,
                                                    prefix_blocks: int, scale: float, workspace,
                                                    out=None, stream=None) -> torch.Tensor:
    """:func:`paged_attention_decode_shared_prefix_run` with the step's new
    K/V rows (one per sequence, to ``slot_mapping[b]``, past the shared
    prefix) stored and attended in the same launches."""
    dev, b, hq, hkv, d, nb, mb = _decode_args(q, k_cache, v_cache, block_tables, context_lens)
    _append_args(q, k_new, v_new, slot_mapping, hkv, d)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, dev)
    _require(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    _cuda_contig("workspace", workspace, dev)
    capi.check(capi.lib().pa_paged_attention_decode_shared_prefix_append_run(
        q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(),
        k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(),
        int(prefix_blocks), b, hq, hkv, d, mb, nb, float(scale), _dtype_code(q), out.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(dev, stream)))
    return out


def paged_attention_decode_grouped_prefix_append_run(q, k_new, v_new, slot_mapping, k_cache,
                                                     v_cache, block_tables, group_start,
                                                     group_prefix_blocks, scale: float,
                                                     workspace, out=None,
                                                     stream=None) -> torch.Tensor:
    """:func:`paged_attention_decode_grouped_prefix_run` with the step's new
    K/V rows (one per sequence, to ``slot_mapping[b]``, past its group's
    prefix) stored and attended in the same launches."""
    dev, b, hq, hkv, d, nb, mb = _decode_args(q, k_cache, v_cache, block_tables, None)
    _append_args(q, k_new, v_new, slot_mapping, hkv, d)
    g = _group_args(group_start, group_prefix_blocks, b, dev)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, dev)
    _require(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    _cuda_contig("workspace", workspace, dev)
    capi.check(capi.lib().pa_paged_attention_decode_grouped_prefix_append_run(
        q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(),
        k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), group_start.data_ptr(),
        group_prefix_blocks.data_ptr(), g, b, hq, hkv, d, mb, nb, float(scale), _dtype_code(q),
        out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(dev, stream)))
    return out


def prefill_workspace_size(num_seqs: int, total_q: int, num_q_heads: int, num_kv_heads: int,
                           head_dim: int) -> int:
    n = C.c_size_t(0)
    capi.check(capi.lib().pa_paged_attention_prefill_workspace_size(
        num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, C.byref(n)))
    return n.value


def alloc_prefill_workspace(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim,
                            device) -> torch.Tensor:
    n = prefill_workspace_size(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def prefill_plan(context_lens: torch.Tensor, query_start: torch.Tensor, total_q: int,
                 num_q_heads: int, num_kv_heads: int, head_dim: int, max_blocks_per_seq: int,
                 scale: float, dtype: torch.dtype, workspace: torch.Tensor, stream=None) -> None:
    """The work list of a chunked-prefill batch, into ``workspace``: one plan
    serves every ``paged_attention_prefill_run`` over the same chunks."""
    dev = context_lens.device
    for name, t in (("context_lens", context_lens), ("query_start", query_start),
                    ("workspace", workspace)):
        _cuda_contig(name, t, dev)
    _require(context_lens.dtype == torch.int32 and query_start.dtype == torch.int32,
             "context_lens and query_start must be int32")
    b = context_lens.shape[0]
    _require(query_start.shape == (b + 1,), "query_start must be [num_seqs + 1]")
    _require(dtype in _DTYPES, "dtype must be float32, float16 or bfloat16")
    capi.check(capi.lib().pa_paged_attention_prefill_plan(
        context_lens.data_ptr(), query_start.data_ptr(), b, int(total_q), int(num_q_heads),
        int(num_kv_heads), int(head_dim), int(max_blocks_per_seq), float(scale),
        _DTYPES[dtype], workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(dev, stream)))


def paged_attention_prefill_run(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                block_tables: torch.Tensor, context_lens: torch.Tensor,
                                query_start: torch.Tensor, scale: float, workspace: torch.Tensor,
                                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """``paged_attention_prefill`` over a workspace that ``prefill_plan``
    filled for the same chunks: the attention kernel only."""
    return paged_attention_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start,
                                   scale, out=out, workspace=workspace, stream=stream,
                                   _entry="pa_paged_attention_prefill_run")


def paged_attention_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor,
                            query_start: torch.Tensor, scale: float,
                            out: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None, stream=None,
                            _entry: str = "pa_paged_attention_prefill") -> torch.Tensor:
    """Chunked-prefill attention: the query rows ``query_start[b] ..
    query_start[b+1]-1`` of ``q`` (``[total_q, Hq, d]``) are the newest tokens
    of sequence ``b`` (K/V already in the cache); each attends causally over
    the sequence's tokens up to itself."""
    dev = q.device
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_tables", block_tables), ("context_lens", context_lens),
                    ("query_start", query_start)):
        _cuda_contig(name, t, dev)
    _require(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
             and query_start.dtype == torch.int32,
             "block_tables, context_lens and query_start must be int32")
    _require(q.dtype == k_cache.dtype == v_cache.dtype, "q and caches must share a dtype")
    _require(k_cache.dim() == 4 and k_cache.shape == v_cache.shape and k_cache.shape[2] == 16,
             "caches must be [num_blocks, num_kv_heads, 16, head_dim]")
    nb, hkv, _, d = k_cache.shape
    _require(q.dim() == 3 and q.shape[2] == d, "q must be [total_q, num_q_heads, head_dim]")
    total_q, hq, _ = q.shape
    b = context_lens.shape[0]
    _require(block_tables.dim() == 2 and block_tables.shape[0] == b,
             "block_tables must be [num_seqs, max_blocks_per_seq]")
    _require(query_start.shape == (b + 1,), "query_start must be [num_seqs + 1]")
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, dev)
    _require(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    if workspace is None:
        workspace = alloc_prefill_workspace(b, total_q, hq, hkv, d, dev)
    _cuda_contig("workspace", workspace, dev)
    capi.check(getattr(capi.lib(), _entry)(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        context_lens.data_ptr(), query_start.data_ptr(), b, total_q, hq, hkv, d,
        block_tables.shape[1], nb, float(scale), _dtype_code(q), out.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(dev, stream)))
    return out


class LayerCaches:
    """Every layer's K and V cache (``[num_blocks, Hkv, 16, d]`` each), checked
    once, with the per-layer pointer arrays the multi-layer copies pass
    through the C ABI built once.  A copy-on-write step then costs one C call
    instead of a pass over every layer's tensors.

    ``host=False``: CUDA tensors on one device.  ``host=True``: contiguous
    page-locked CPU tensors (the swap tier).  The object holds references to
    the tensors; resizing or replacing their storage afterwards is not seen
    (build a new object)."""

    def __init__(self, k_caches, v_caches, host: bool = False):
        k, v = list(k_caches), list(v_caches)
        _require(len(k) == len(v) and len(k) > 0, "need one K and one V cache per layer")
        ref = k[0]
        _require(ref.dim() == 4 and ref.shape[2] == 16,
                 "caches must be [num_blocks, num_kv_heads, 16, head_dim]")
        self.device = None if host else ref.device
        for t in k + v:
            if host:
                _require(not t.is_cuda and t.is_pinned() and t.is_contiguous(),
                         "host caches must be contiguous page-locked CPU tensors")
            else:
                _cuda_contig("cache", t, self.device)
            _require(t.shape == ref.shape and t.dtype == ref.dtype,
                     "all layer caches must share shape and dtype")
        self.k, self.v, self.host = k, v, host
        self.num_layers = len(k)
        self.num_blocks, self.num_kv_heads, _, self.head_dim = ref.shape
        self.dtype = ref.dtype
        self._code = _dtype_code(ref)
        n = self.num_layers
        self._kp = (C.c_void_p * n)(*[t.data_ptr() for t in k])
        self._vp = (C.c_void_p * n)(*[t.data_ptr() for t in v])

    def _pairs(self, pairs: torch.Tensor, name: str) -> None:
        _require(pairs.is_cuda and pairs.device == self.device and pairs.is_contiguous(),
                 f"{name} must be contiguous on {self.device}")
        _require(pairs.dtype == torch.int64 and pairs.dim() == 2 and pairs.shape[1] == 2,
                 f"{name} must be int64 [n, 2]")

    def block_copy(self, src_dst_pairs: torch.Tensor, stream=None) -> None:
        """Copy whole blocks ``src -> dst`` (int64 ``[P, 2]`` on the device) in
        every layer, one launch."""
        _require(not self.host, "block_copy runs on device caches")
        self._pairs(src_dst_pairs, "src_dst_pairs")
        capi.check(capi.lib().pa_block_copy(
            self._kp, self._vp, self.num_layers, src_dst_pairs.data_ptr(),
            src_dst_pairs.shape[0], self.num_kv_heads, self.head_dim, self.num_blocks,
            self._code, _stream(self.device, stream)))

    def block_swap(self, host: "LayerCaches", pairs: torch.Tensor, direction: int,
                   stream=None) -> None:
        """Copy whole blocks between these device caches and the page-locked
        ``host`` caches, every layer in one launch: ``PA_SWAP_OUT`` copies
        device block ``pairs[i, 0]`` to host block ``pairs[i, 1]``,
        ``PA_SWAP_IN`` host ``pairs[i, 0]`` to device ``pairs[i, 1]`` (the
        pairs the pool's swap_out / swap_in return)."""
        _require(not self.host and host.host, "block_swap goes between device and host caches")
        _require(host.num_layers == self.num_layers and host.dtype == self.dtype
                 and (host.num_kv_heads, host.head_dim) == (self.num_kv_heads, self.head_dim),
                 "host caches must be [num_host_blocks, num_kv_heads, 16, head_dim] of the "
                 "device caches' dtype, one per layer")
        self._pairs(pairs, "pairs")
        capi.check(capi.lib().pa_block_swap(
            self._kp, self._vp, host._kp, host._vp, self.num_layers, pairs.data_ptr(),
            pairs.shape[0], int(direction), self.num_kv_heads, self.head_dim, self.num_blocks,
            host.num_blocks, self._code, _stream(self.device, stream)))


def block_swap(dev_k_caches, dev_v_caches, host_k_caches, host_v_caches,
               pairs: torch.Tensor, direction: int, stream=None) -> None:
    """:meth:`LayerCaches.block_swap` on caches given as per-layer lists
    (checked on every call)."""
    LayerCaches(dev_k_caches, dev_v_caches).block_swap(
        LayerCaches(host_k_caches, host_v_caches, host=True), pairs, direction, stream)


def block_copy(k_caches, v_caches, src_dst_pairs: torch.Tensor, stream=None) -> None:
    """:meth:`LayerCaches.block_copy` on caches given as per-layer lists
    (checked on every call)."""
    LayerCaches(k_caches, v_caches).block_copy(src_dst_pairs, stream)


def check_status(stream=None, device=None) -> None:
    """Synchronise the stream and raise if a kernel flagged an out-of-range
    index or a timed-out wait since the last check."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    capi.check(capi.lib().pa_check_status(_stream(dev, stream)))
