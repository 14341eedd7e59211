"""Python handle on the library's host-side block manager (``pkv_bm_*``).

The manager itself is C++ inside libpkv.so; this class marshals arguments and
turns its tables into the int32 tensors the attention calls take.  It runs
on the host only and needs no GPU.
"""

from __future__ import annotations

import ctypes

import numpy as np

from . import ops

BLOCK_SIZE = ops.BLOCK_SIZE


def _i32_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class BlockManager:
    """A pool of ``num_blocks`` 256-token blocks with reference counts and prefix reuse."""

    def __init__(self, num_blocks: int):
        self._lib = ops.load_library()
        self._h = self._lib.pkv_bm_create(int(num_blocks))
        if not self._h:
            raise ops.PkvError(-2, self._lib.pkv_last_error().decode())
        self.num_blocks = int(num_blocks)

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def _check(self, rc: int):
        if rc != 0:
            raise ops.PkvError(rc, self._lib.pkv_last_error().decode())

    @property
    def num_free_blocks(self) -> int:
        return int(self._lib.pkv_bm_num_free_blocks(self._h))

    def ref_count(self, block: int) -> int:
        return int(self._lib.pkv_bm_ref_count(self._h, int(block)))

    def allocate(self, seq_id: int, token_ids) -> int:
        """Blocks for a prompt; returns the number of leading tokens whose KV is already cached."""
        t = np.ascontiguousarray(token_ids, dtype=np.int32)
        cached = ctypes.c_int32(0)
        self._check(self._lib.pkv_bm_allocate(self._h, int(seq_id), _i32_ptr(t), t.size, ctypes.byref(cached)))
        return cached.value

    def append(self, seq_id: int, token_id: int) -> int:
        """One decode token; returns its cache slot."""
        slot = ctypes.c_int32(0)
        self._check(self._lib.pkv_bm_append(self._h, int(seq_id), int(token_id), ctypes.byref(slot)))
        return slot.value

    def free(self, seq_id: int):
        self._check(self._lib.pkv_bm_free(self._h, int(seq_id)))

    def seq_info(self, seq_id: int):
        """(num_tokens, num_blocks, num_cached_tokens) of a sequence."""
        n, b, c = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
        self._check(self._lib.pkv_bm_seq_info(self._h, int(seq_id), ctypes.byref(n), ctypes.byref(b),
                                              ctypes.byref(c)))
        return n.value, b.value, c.value

    def block_table(self, seq_ids, max_blocks: int | None = None) -> np.ndarray:
        """int32 [len(seq_ids), max_blocks], padded with -1."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        if max_blocks is None:
            max_blocks = max([self.seq_info(int(s))[1] for s in ids] + [1])
        out = np.empty((ids.size, int(max_blocks)), dtype=np.int32)
        self._check(self._lib.pkv_bm_block_table(self._h, ids.ctypes.data_as(ctypes.c_void_p), ids.size,
                                                 _i32_ptr(out), int(max_blocks)))
        return out

    def slot_mapping(self, seq_id: int, start: int, end: int) -> np.ndarray:
        """Cache rows of token positions [start, end) of one sequence."""
        out = np.empty(max(0, int(end) - int(start)), dtype=np.int32)
        self._check(self._lib.pkv_bm_slot_mapping(self._h, int(seq_id), int(start), int(end), _i32_ptr(out)))
        return out

    def prefill_batch(self, seq_ids):
        """The index arrays of one varlen prefill over the sequences' uncached tokens.

        Returns (slot_mapping, positions, cu_seqlens_q, cu_seqlens_k, block_table) as host int32 arrays:
        the query rows of sequence s are its tokens from its cached-prefix length on, and its keys are
        all its tokens (the chunk attends causally to prefix + chunk).
        """
        slots, pos, cu_q, cu_k = [], [], [0], [0]
        for s in seq_ids:
            n, _, cached = self.seq_info(int(s))
            slots.append(self.slot_mapping(int(s), cached, n))
            pos.append(np.arange(cached, n, dtype=np.int32))
            cu_q.append(cu_q[-1] + n - cached)
            cu_k.append(cu_k[-1] + n)
        return (np.concatenate(slots).astype(np.int32), np.concatenate(pos).astype(np.int32),
                np.asarray(cu_q, np.int32), np.asarray(cu_k, np.int32), self.block_table(seq_ids))
