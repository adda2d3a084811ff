"""The C-ABI library loads, exports every symbol the public header declares, and
rejects bad arguments on the host before touching a GPU (CPU only)."""

import ctypes as C
import glob
import os
import re

import pytest

from tests.conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from pagedattention_decode_attention_gb300 import build, capi
    if not os.path.exists(capi.LIB_PATH):
        build.build()
    return capi.lib()


def declared_symbols():
    names = set()
    for header in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(header).read()
        names |= set(re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text))
    return names


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for required in ("pa_kv_append", "pa_paged_attention_decode", "pa_block_copy",
                     "pa_paged_attention_decode_workspace_size", "pa_pool_create",
                     "pa_pool_append_slot", "pa_pool_fork", "pa_pool_share_prefix",
                     "pa_pool_free_seq", "pa_pool_block_table", "pa_check_status"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in sorted(declared_symbols()) if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_declares_exactly_the_header(lib):
    from pagedattention_decode_attention_gb300 import capi
    assert set(capi.SIGNATURES) == declared_symbols()


def test_python_binding_carries_every_entry_point_name():
    """Each declared call has a Python function of the same name (without
    ``pa_``; pool calls as ``BlockPool`` methods).  Pool creation and
    destruction are the ``BlockPool`` constructor and finaliser; the error
    string travels inside ``PagedAttnError``."""
    import pagedattention_decode_attention_gb300 as pa
    missing = []
    for n in sorted(declared_symbols() - {"pa_pool_create", "pa_pool_destroy", "pa_last_error"}):
        if n.startswith("pa_pool_"):
            found = callable(getattr(pa.BlockPool, n[len("pa_pool_"):], None))
        else:
            found = callable(getattr(pa, n[len("pa_"):], None))
        if not found:
            missing.append(n)
    assert not missing, missing


def test_version(lib):
    import pagedattention_decode_attention_gb300 as pa
    assert lib.pa_version() >= 100 and pa.version() == lib.pa_version()


def test_workspace_size_is_host_only(lib):
    out = C.c_size_t(0)
    assert lib.pa_paged_attention_decode_workspace_size(128, 32, 8, 128, 512, C.byref(out)) == 0
    # header + units + arrivals + partial (lse, o) for 16 splits of 128 seqs
    assert out.value >= 128 * 16 * 32 * 128 * 4
    assert lib.pa_paged_attention_decode_workspace_size(1, 0, 1, 64, 1, C.byref(out)) == 1


@pytest.mark.parametrize("kwargs,status", [
    (dict(dtype=7), 2),                          # unknown dtype -> unsupported
    (dict(head_dim=96), 2),                      # head_dim not built
    (dict(num_q_heads=6, num_kv_heads=4), 1),    # ragged grouping
    (dict(num_q_heads=32, num_kv_heads=2), 2),   # 16 heads per KV head > 8 (16-bit path)
    (dict(workspace_bytes=16), 1),               # workspace too small
])
def test_decode_rejects_on_host(lib, kwargs, status):
    a = dict(q=256, k=256, v=256, bt=256, cl=256, num_seqs=2, num_q_heads=4, num_kv_heads=4,
             head_dim=64, max_blocks=4, num_blocks=8, scale=0.125, dtype=2, out=256,
             ws=256, workspace_bytes=1 << 20)
    a.update(kwargs)
    rc = lib.pa_paged_attention_decode(a["q"], a["k"], a["v"], a["bt"], a["cl"], a["num_seqs"],
                                       a["num_q_heads"], a["num_kv_heads"], a["head_dim"],
                                       a["max_blocks"], a["num_blocks"], a["scale"], a["dtype"],
                                       a["out"], a["ws"], a["workspace_bytes"], None)
    assert rc == status
    assert lib.pa_last_error()


def test_workspace_sizes_refuse_overflowing_shapes(lib):
    """Shapes whose workspace would wrap size_t arithmetic are refused, not
    reported as a small size."""
    out = C.c_size_t(0)
    big = (1 << 31) - 1
    assert lib.pa_paged_attention_decode_workspace_size(big, big, 1, 128, big, C.byref(out)) == 1
    assert b"workspace" in lib.pa_last_error()
    assert lib.pa_paged_attention_decode_shared_prefix_workspace_size(
        big, 1024, 1, 128, 1 << 20, C.byref(out)) == 1
    assert lib.pa_paged_attention_decode_grouped_prefix_workspace_size(
        big, 64, 8, 128, 1 << 20, C.byref(out)) == 1
    # the attention entry point refuses the same shapes before touching any pointer
    assert lib.pa_paged_attention_decode(256, 256, 256, 256, 256, big, 64, 8, 128, 1 << 20, 64,
                                         0.1, 2, 256, 256, 1 << 62, None) == 1


def test_one_shot_decode_checks_every_pointer_before_its_plan(lib):
    """A NULL query is refused on the host before the plan would be launched
    (on a machine without a GPU a launch attempt reports PA_ERR_CUDA
    instead), so a rejected call leaves the workspace untouched."""
    rc = lib.pa_paged_attention_decode(None, 256, 256, 256, 256, 2, 4, 4, 64, 4, 8, 0.125, 2,
                                       256, 256, 1 << 20, None)
    assert rc == 1 and b"NULL" in lib.pa_last_error()
    rc = lib.pa_paged_attention_decode(256, 256, 256 + 8, 256, 256, 2, 4, 4, 64, 4, 8, 0.125, 2,
                                       256, 256, 1 << 20, None)
    assert rc == 1 and b"aligned" in lib.pa_last_error()


def test_noalloc_refuses_shapes_beyond_its_scratch_on_host(lib):
    rc = lib.pa_paged_attention_decode_noalloc(None, None, None, None, None, 4096, 32, 8, 128,
                                               4096, 100000, C.c_float(0.1), 2, None, None)
    assert rc == 1 and b"built into the library" in lib.pa_last_error()
    big = (1 << 31) - 1
    rc = lib.pa_paged_attention_decode_noalloc(None, None, None, None, None, big, big, 8, 128,
                                               big, 100000, C.c_float(0.1), 2, None, None)
    assert rc == 1 and b"built-in scratch" in lib.pa_last_error()


def test_empty_batches_are_noops(lib):
    assert lib.pa_kv_append(None, None, None, None, None, 0, 8, 128, 16, 2, None) == 0
    assert lib.pa_block_copy(None, None, 1, None, 0, 8, 128, 16, 2, None) == 0
    assert lib.pa_paged_attention_decode(None, None, None, None, None, 0, 4, 4, 64, 4, 8,
                                         0.1, 1, None, None, 0, None) == 0


def test_copy_paths_reject_on_host(lib):
    # misaligned pointer, bad dtype, too many layers
    assert lib.pa_kv_append(8, 16, 16, 16, 16, 1, 8, 128, 16, 2, None) == 1
    assert lib.pa_kv_append(16, 16, 16, 16, 16, 1, 8, 128, 16, 5, None) == 2
    ptrs = (C.c_void_p * 1)(256)
    assert lib.pa_block_copy(ptrs, ptrs, 300, 256, 1, 8, 128, 16, 2, None) == 1


def _grouped(lib, **kw):
    a = dict(q=256, k=256, v=256, bt=256, cl=256, gs=256, gb=256, num_groups=2, num_seqs=4,
             num_q_heads=32, num_kv_heads=8, head_dim=128, max_blocks=8, num_blocks=64,
             scale=0.125, dtype=2, out=256, ws=256, workspace_bytes=1 << 30)
    a.update(kw)
    return lib.pa_paged_attention_decode_grouped_prefix(
        a["q"], a["k"], a["v"], a["bt"], a["cl"], a["gs"], a["gb"], a["num_groups"],
        a["num_seqs"], a["num_q_heads"], a["num_kv_heads"], a["head_dim"], a["max_blocks"],
        a["num_blocks"], a["scale"], a["dtype"], a["out"], a["ws"], a["workspace_bytes"], None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(num_groups=0), 1),              # no group
    (dict(num_groups=5), 1),              # more groups than sequences
    (dict(dtype=0), 2),                   # fp32 decodes exactly without the cascade
    (dict(workspace_bytes=4096), 1),      # workspace too small
    (dict(ws=264), 1),                    # workspace not 256-byte aligned
    (dict(gs=None), 1),                   # group arrays required
    (dict(bt=None), 1),                   # tables required by the plan
])
def test_grouped_prefix_rejects_on_host(lib, kwargs, status):
    assert _grouped(lib, **kwargs) == status
    assert lib.pa_last_error()


def test_grouped_prefix_workspace_covers_the_shared_layout(lib):
    g, s = C.c_size_t(0), C.c_size_t(0)
    assert lib.pa_paged_attention_decode_grouped_prefix_workspace_size(
        128, 32, 8, 128, 65, C.byref(g)) == 0
    assert lib.pa_paged_attention_decode_shared_prefix_workspace_size(
        128, 32, 8, 128, 65, C.byref(s)) == 0
    # plus each sequence's suffix table, suffix length and prefix block count
    assert g.value >= s.value + 128 * 65 * 4 + 2 * 128 * 4


def test_fused_cascade_runs_reject_on_host(lib):
    ptr = 256
    # new K/V rows and slots are required, and 16-byte aligned
    assert lib.pa_paged_attention_decode_shared_prefix_append_run(
        ptr, None, ptr, ptr, ptr, ptr, ptr, ptr, 4, 4, 32, 8, 128, 8, 64, 0.125, 2, ptr, ptr,
        1 << 30, None) == 1
    assert lib.pa_paged_attention_decode_grouped_prefix_append_run(
        ptr, ptr + 8, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 2, 4, 32, 8, 128, 8, 64, 0.125, 2, ptr,
        ptr, 1 << 30, None) == 1
    # a prefix longer than the table
    assert lib.pa_paged_attention_decode_shared_prefix_append_run(
        ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 9, 4, 32, 8, 128, 8, 64, 0.125, 2, ptr, ptr,
        1 << 30, None) == 1


def test_missing_library_fails_loudly(monkeypatch):
    """With the shared library absent every call raises: the pool, the
    version query and the attention entry point.  Nothing falls back to a
    host computation."""
    import torch

    import pagedattention_decode_attention_gb300 as pa
    from pagedattention_decode_attention_gb300 import capi
    monkeypatch.setattr(capi, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libpagedattn.so"))
    monkeypatch.setattr(capi, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        pa.BlockPool(4)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        pa.version()
    q = torch.zeros(1, 4, 64)
    kc = torch.zeros(2, 4, 16, 64)
    with pytest.raises(Exception):
        pa.paged_attention_decode(q, kc, kc.clone(), torch.zeros(1, 1, dtype=torch.int32),
                                  torch.ones(1, dtype=torch.int32), 0.125)
