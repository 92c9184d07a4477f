"""Python handle on the native block manager (pa_bm_* of include/pa.h)."""
from __future__ import annotations

import ctypes

import numpy as np

from ._lib import check, lib


def inject_alloc_failure(k: int):
    """Test hook (pa_bm_inject_alloc_failure): the k-th host allocation point
    of the following block-manager calls fails as if host memory ran out
    (the call raises OutOfBlocks and changes nothing); k < 0 disarms."""
    lib().pa_bm_inject_alloc_failure(int(k))


class BlockManager:
    """Free list, refcounts, fork and copy-on-write over a pool of physical blocks.

    seed != 0 shuffles the initial free-list order (SplitMix64 Fisher-Yates),
    so that sequences land on scattered physical blocks.
    """

    def __init__(self, num_blocks: int, block_size: int, seed: int = 0):
        h = ctypes.c_void_p()
        check(lib().pa_bm_create(int(num_blocks), int(block_size), int(seed), ctypes.byref(h)))
        self._h = h
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq: int, n_tokens: int) -> np.ndarray:
        slots = np.empty(int(n_tokens), dtype=np.int64)
        check(lib().pa_bm_add_seq(self._h, int(seq), int(n_tokens),
                                  slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))))
        return slots

    def fork(self, parent: int, child: int):
        check(lib().pa_bm_fork(self._h, int(parent), int(child)))

    def append(self, seq: int):
        """-> (slot, cow_src, cow_dst); cow_* = -1 when no copy is needed."""
        s, a, b = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        check(lib().pa_bm_append(self._h, int(seq), ctypes.byref(s), ctypes.byref(a),
                                 ctypes.byref(b)))
        return s.value, a.value, b.value

    def append_n(self, seq: int, n: int):
        """-> (slots[n], cow pairs list)."""
        slots = np.empty(int(n), dtype=np.int64)
        a, b = ctypes.c_int64(), ctypes.c_int64()
        check(lib().pa_bm_append_n(self._h, int(seq), int(n),
                                   slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                   ctypes.byref(a), ctypes.byref(b)))
        return slots, ([(a.value, b.value)] if a.value >= 0 else [])

    def free_seq(self, seq: int):
        check(lib().pa_bm_free_seq(self._h, int(seq)))

    def block_table(self, seqs, max_blocks: int) -> np.ndarray:
        seqs = np.ascontiguousarray(seqs, dtype=np.int64)
        out = np.zeros((len(seqs), int(max_blocks)), dtype=np.int32)
        check(lib().pa_bm_block_table(self._h, seqs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                      len(seqs), out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                      int(max_blocks)))
        return out

    def seq_len(self, seq: int) -> int:
        v = ctypes.c_int64()
        check(lib().pa_bm_seq_len(self._h, int(seq), ctypes.byref(v)))
        return v.value

    def seq_blocks(self, seq: int) -> list:
        n = ctypes.c_int64()
        check(lib().pa_bm_seq_blocks(self._h, int(seq), None, 0, ctypes.byref(n)))
        out = np.zeros(max(n.value, 1), dtype=np.int32)
        check(lib().pa_bm_seq_blocks(self._h, int(seq),
                                     out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n.value,
                                     ctypes.byref(n)))
        return out[:n.value].tolist()

    def refcount(self, block: int) -> int:
        v = ctypes.c_int()
        check(lib().pa_bm_refcount(self._h, int(block), ctypes.byref(v)))
        return v.value

    def num_free(self) -> int:
        return int(lib().pa_bm_num_free(self._h))
