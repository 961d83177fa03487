"""Python handle for the native refcounted block allocator (host only)."""

import ctypes

import numpy as np

from . import _lib


class OutOfBlocks(_lib.PagedKVError):
    pass


def _addr(a):
    """Address of a contiguous numpy array's data."""
    return a.ctypes.data


class BlockAllocator:
    """Fixed-size blocks, per-sequence block tables, refcounted sharing and
    copy-on-write; decides ids only (the caller owns every tensor)."""

    def __init__(self, num_blocks, block_size):
        self._lib = _lib.load()
        h = ctypes.c_void_p()
        self._check(self._lib.pkv_alloc_create(num_blocks, block_size, ctypes.byref(h)),
                    "pkv_alloc_create")
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def _check(self, st, what):
        if st == 4:
            raise OutOfBlocks(st, what)
        _lib.check(st, what)

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pkv_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def add_seq(self, seq_id, num_tokens):
        self._check(self._lib.pkv_alloc_add_seq(self._h, seq_id, num_tokens), "add_seq")

    def fork(self, parent, child):
        self._check(self._lib.pkv_alloc_fork(self._h, parent, child), "fork")

    def append_slot(self, seq_id):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        self._check(self._lib.pkv_alloc_append_slot(self._h, seq_id, ctypes.byref(slot),
                                                    ctypes.byref(src), ctypes.byref(dst)),
                    "append_slot")
        return slot.value, src.value, dst.value

    def append_slots(self, seq_ids):
        """Next slot of each sequence, in order; returns (slots [n], pairs [P, 2])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = len(ids)
        slots = np.empty(n, dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        count = ctypes.c_int(0)
        st = self._lib.pkv_alloc_append_slots(self._h, _addr(ids), n, _addr(slots), _addr(pairs),
                                              ctypes.byref(count))
        self._check(st, "append_slots")
        return slots, pairs[:count.value].copy()

    def free_seq(self, seq_id):
        self._check(self._lib.pkv_alloc_free_seq(self._h, seq_id), "free_seq")

    def block_table(self, seq_ids, max_blocks):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        out = np.empty((len(ids), max_blocks), dtype=np.int32)
        st = self._lib.pkv_alloc_block_table(self._h, _addr(ids), len(ids), _addr(out), max_blocks)
        self._check(st, "block_table")
        return out

    def seq_slots(self, seq_id, start, count):
        out = np.empty(count, dtype=np.int64)
        self._check(self._lib.pkv_alloc_seq_slots(self._h, seq_id, start, count, _addr(out)),
                    "seq_slots")
        return out

    def seq_info(self, seq_id):
        n, b = ctypes.c_int(), ctypes.c_int()
        self._check(self._lib.pkv_alloc_seq_info(self._h, seq_id, ctypes.byref(n),
                                                 ctypes.byref(b)), "seq_info")
        return n.value, b.value

    def refcount(self, block):
        r = ctypes.c_int()
        self._check(self._lib.pkv_alloc_refcount(self._h, block, ctypes.byref(r)), "refcount")
        return r.value

    def stats(self):
        s = _lib.AllocStats()
        self._check(self._lib.pkv_alloc_stats(self._h, ctypes.byref(s)), "stats")
        return {name: getattr(s, name) for name, _ in _lib.AllocStats._fields_}
