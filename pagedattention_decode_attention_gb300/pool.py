"""Python handle on the native host block pool (``pa_pool_*`` in the C ABI)."""

from __future__ import annotations

import ctypes as C

import numpy as np

from . import capi


class BlockPool:
    """Free list + refcounts + lazy allocation + fork / copy-on-write + prefix
    sharing, implemented in C++; this class only marshals arguments."""

    def __init__(self, num_blocks: int, block_size: int = 16, initial_order=None):
        self._lib = capi.lib()
        handle = C.c_void_p()
        order = None
        if initial_order is not None:
            self._order = np.ascontiguousarray(initial_order, dtype=np.int32)
            order = self._order.ctypes.data_as(C.POINTER(C.c_int32))
        capi.check(self._lib.pa_pool_create(num_blocks, block_size, order, C.byref(handle)))
        self._h = handle
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if self._h:
            self._lib.pa_pool_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def new_seq(self) -> int:
        out = C.c_int()
        capi.check(self._lib.pa_pool_new_seq(self._h, C.byref(out)))
        return out.value

    def append_slot(self, seq: int):
        slot, src, dst = C.c_int64(), C.c_int64(), C.c_int64()
        capi.check(self._lib.pa_pool_append_slot(self._h, seq, C.byref(slot), C.byref(src),
                                                 C.byref(dst)))
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def append_slots(self, seqs):
        """One slot per sequence; returns (int64 slots [n], int64 pairs [p, 2])."""
        seqs = np.ascontiguousarray(seqs, dtype=np.int32)
        n = len(seqs)
        slots = np.empty(n, dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        npairs, done = C.c_int(), C.c_int()
        capi.check(self._lib.pa_pool_append_slots(
            self._h, seqs.ctypes.data_as(C.POINTER(C.c_int32)), n,
            slots.ctypes.data_as(C.POINTER(C.c_int64)), pairs.ctypes.data_as(C.POINTER(C.c_int64)),
            max(n, 1), C.byref(npairs), C.byref(done)))
        return slots, pairs[:npairs.value].copy()

    def fork(self, parent: int) -> int:
        out = C.c_int()
        capi.check(self._lib.pa_pool_fork(self._h, parent, C.byref(out)))
        return out.value

    def share_prefix(self, src_seq: int, dst_seq: int, num_tokens: int) -> None:
        capi.check(self._lib.pa_pool_share_prefix(self._h, src_seq, dst_seq, num_tokens))

    def pin(self, seq: int, num_tokens: int) -> None:
        capi.check(self._lib.pa_pool_pin(self._h, seq, num_tokens))

    def unpin(self, block: int) -> None:
        capi.check(self._lib.pa_pool_unpin(self._h, block))

    def free_seq(self, seq: int) -> None:
        capi.check(self._lib.pa_pool_free_seq(self._h, seq))

    def block_table(self, seq: int):
        n, ctx = C.c_int(), C.c_int()
        capi.check(self._lib.pa_pool_block_table(self._h, seq, None, 0, C.byref(n), C.byref(ctx)))
        buf = np.empty(max(n.value, 1), dtype=np.int32)
        capi.check(self._lib.pa_pool_block_table(self._h, seq,
                                                 buf.ctypes.data_as(C.POINTER(C.c_int32)),
                                                 n.value, C.byref(n), C.byref(ctx)))
        return buf[:n.value].tolist(), ctx.value

    def enable_prefix_cache(self, on: bool = True) -> None:
        """Key full blocks by content so later prompts reuse them (before the
        first sequence)."""
        capi.check(self._lib.pa_pool_enable_prefix_cache(self._h, int(bool(on))))

    def new_seq_with_prompt(self, tokens) -> tuple[int, int]:
        """New sequence for a prompt: returns ``(seq, hit_tokens)``; the first
        ``hit_tokens`` tokens are served by cached blocks, the caller appends
        the rest with :meth:`append_token`."""
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        seq, hit = C.c_int(), C.c_int()
        capi.check(self._lib.pa_pool_new_seq_with_prompt(
            self._h, toks.ctypes.data_as(C.POINTER(C.c_int32)), toks.shape[0], C.byref(seq),
            C.byref(hit)))
        return seq.value, hit.value

    def append_token(self, seq: int, token: int):
        """:meth:`append_slot` for a known token id (keys the block it fills)."""
        slot, src, dst = C.c_int64(), C.c_int64(), C.c_int64()
        capi.check(self._lib.pa_pool_append_token(self._h, seq, int(token), C.byref(slot),
                                                  C.byref(src), C.byref(dst)))
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def append_tokens(self, seqs, tokens):
        """:meth:`append_token` of ``tokens[i]`` to ``seqs[i]`` for every i, in
        order, in one call.  Stops where the pool runs out of blocks.  Returns
        (int64 slots of the appends made, int64 copy pairs [p, 2], number of
        appends made); other errors raise."""
        seqs = np.ascontiguousarray(seqs, dtype=np.int32)
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        if seqs.shape != toks.shape or seqs.ndim != 1:
            raise ValueError("seqs and tokens must be 1-D of one length")
        n = seqs.shape[0]
        slots = np.empty(max(n, 1), dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        npairs, done = C.c_int(), C.c_int()
        rc = self._lib.pa_pool_append_tokens(
            self._h, seqs.ctypes.data_as(C.POINTER(C.c_int32)),
            toks.ctypes.data_as(C.POINTER(C.c_int32)), n,
            slots.ctypes.data_as(C.POINTER(C.c_int64)), pairs.ctypes.data_as(C.POINTER(C.c_int64)),
            max(n, 1), C.byref(npairs), C.byref(done))
        if rc != capi.PA_ERR_NO_BLOCKS:
            capi.check(rc)
        return slots[:done.value], pairs[:npairs.value], done.value

    def set_host_blocks(self, num_host_blocks: int, initial_order=None) -> None:
        """Give the pool a host tier (swap space) of ``num_host_blocks`` blocks."""
        order = None
        if initial_order is not None:
            order = np.ascontiguousarray(initial_order, dtype=np.int32)
            if order.shape != (num_host_blocks,):
                raise ValueError("initial_order must have num_host_blocks entries")
        capi.check(self._lib.pa_pool_set_host_blocks(
            self._h, num_host_blocks,
            None if order is None else order.ctypes.data_as(C.POINTER(C.c_int32))))
        self._host_order = order

    def _swap(self, fn, seq: int) -> np.ndarray:
        table, _ = self.block_table(seq)
        buf = np.empty((max(len(table), 1), 2), dtype=np.int64)
        n = C.c_int()
        capi.check(fn(self._h, seq, buf.ctypes.data_as(C.POINTER(C.c_int64)), len(table),
                      C.byref(n)))
        return buf[:n.value]

    def swap_out(self, seq: int) -> np.ndarray:
        """Move ``seq`` to the host tier; returns int64 ``[n, 2]`` copy pairs
        (device block, host block) in logical order."""
        return self._swap(self._lib.pa_pool_swap_out, seq)

    def swap_in(self, seq: int) -> np.ndarray:
        """Bring ``seq`` back; returns int64 ``[n, 2]`` copy pairs (host block,
        device block) in logical order."""
        return self._swap(self._lib.pa_pool_swap_in, seq)

    def is_swapped(self, seq: int) -> bool:
        out = C.c_int()
        capi.check(self._lib.pa_pool_is_swapped(self._h, seq, C.byref(out)))
        return bool(out.value)

    def refcount(self, block: int) -> int:
        out = C.c_int()
        capi.check(self._lib.pa_pool_refcount(self._h, block, C.byref(out)))
        return out.value

    def stats(self) -> dict:
        st = capi.PoolStats()
        capi.check(self._lib.pa_pool_stats(self._h, C.byref(st)))
        return {name: getattr(st, name) for name, _ in capi.PoolStats._fields_}

    def tables(self, seqs, max_blocks: int) -> tuple[np.ndarray, np.ndarray]:
        """Block tables (int32 ``[n, max_blocks]``, -1 padded) and context
        lengths (int32 ``[n]``) of ``seqs``, ready to copy to the device."""
        tab = np.full((len(seqs), max_blocks), -1, dtype=np.int32)
        lens = np.zeros(len(seqs), dtype=np.int32)
        for i, s in enumerate(seqs):
            t, ctx = self.block_table(s)
            if len(t) > max_blocks:
                raise ValueError(f"sequence {s} holds {len(t)} blocks > max_blocks {max_blocks}")
            tab[i, :len(t)] = t
            lens[i] = ctx
        return tab, lens
