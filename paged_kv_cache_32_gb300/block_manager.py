"""Python binding of the host KV block manager (include/pa_block_manager.h).

Argument marshalling only: every operation runs in the C++ manager inside
libpa.so.  Typical decode step::

    bm = BlockManager(num_blocks, block_size)
    bm.allocate(seq, prompt_len)                 # or allocate_with_prefix(seq, tokens)
    slots, pairs = bm.append_slots(seqs)         # one new token per sequence
    tables, lens = bm.build_tables(seqs, width)  # metadata for pa_decode
    # pa_copy_blocks(pairs) -> pa_reshape_and_cache(slots) -> pa_decode(tables, lens)
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import lib as _lib

OK, ERR_INVALID_ARG, ERR_UNKNOWN_SEQ, ERR_NO_BLOCKS, ERR_SEQ_EXISTS = 0, -1, -2, -3, -4
_NAMES = {ERR_INVALID_ARG: "invalid argument", ERR_UNKNOWN_SEQ: "unknown sequence",
          ERR_NO_BLOCKS: "KV block pool exhausted", ERR_SEQ_EXISTS: "sequence already exists"}


class BlockManagerError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {_NAMES.get(status, 'error')} ({status})")
        self.status = status


_configured = False


def _L():
    global _configured
    L = _lib()
    if not _configured:
        vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        L.pa_bm_create.argtypes = [i32, i32, u64]
        L.pa_bm_create.restype = vp
        L.pa_bm_destroy.argtypes = [vp]
        L.pa_bm_destroy.restype = None
        L.pa_bm_num_free.argtypes = [vp]
        L.pa_bm_num_free.restype = i32
        L.pa_bm_ref_count.argtypes = [vp, i32]
        L.pa_bm_ref_count.restype = i32
        L.pa_bm_allocate.argtypes = [vp, i64, i32]
        L.pa_bm_allocate.restype = ctypes.c_int
        L.pa_bm_allocate_with_prefix.argtypes = [vp, i64, vp, i32, ctypes.POINTER(i32)]
        L.pa_bm_allocate_with_prefix.restype = ctypes.c_int
        L.pa_bm_append_slot.argtypes = [vp, i64, ctypes.POINTER(i64), ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.pa_bm_append_slot.restype = ctypes.c_int
        L.pa_bm_append_slots.argtypes = [vp, vp, i32, vp, vp, ctypes.POINTER(i32)]
        L.pa_bm_append_slots.restype = ctypes.c_int
        L.pa_bm_fork.argtypes = [vp, i64, i64]
        L.pa_bm_fork.restype = ctypes.c_int
        L.pa_bm_free.argtypes = [vp, i64]
        L.pa_bm_free.restype = ctypes.c_int
        L.pa_bm_seq_len.argtypes = [vp, i64]
        L.pa_bm_seq_len.restype = i32
        L.pa_bm_num_seq_blocks.argtypes = [vp, i64]
        L.pa_bm_num_seq_blocks.restype = i32
        L.pa_bm_max_seq_blocks.argtypes = [vp, vp, i32]
        L.pa_bm_max_seq_blocks.restype = i32
        L.pa_bm_build_tables.argtypes = [vp, vp, i32, i32, vp, vp]
        L.pa_bm_build_tables.restype = ctypes.c_int
        _configured = True
    return L


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, shuffle_seed: int = 0):
        self._h = _L().pa_bm_create(int(num_blocks), int(block_size), int(shuffle_seed))
        if not self._h:
            raise BlockManagerError(ERR_INVALID_ARG, "pa_bm_create")
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _L().pa_bm_destroy(h)
            self._h = None

    def _check(self, rc: int, where: str) -> None:
        if rc != OK:
            raise BlockManagerError(rc, where)

    def num_free(self) -> int:
        return _L().pa_bm_num_free(self._h)

    def ref_count(self, block: int) -> int:
        return _L().pa_bm_ref_count(self._h, int(block))

    def allocate(self, seq: int, num_tokens: int) -> None:
        self._check(_L().pa_bm_allocate(self._h, int(seq), int(num_tokens)), "allocate")

    def allocate_with_prefix(self, seq: int, tokens) -> int:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        hits = ctypes.c_int32(0)
        self._check(_L().pa_bm_allocate_with_prefix(self._h, int(seq), t.ctypes.data, len(t), ctypes.byref(hits)),
                    "allocate_with_prefix")
        return hits.value

    def append_slot(self, seq: int):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        self._check(_L().pa_bm_append_slot(self._h, int(seq), ctypes.byref(slot), ctypes.byref(src),
                                           ctypes.byref(dst)), "append_slot")
        return slot.value, src.value, dst.value

    def append_slots(self, seqs):
        s = np.ascontiguousarray(seqs, dtype=np.int64)
        slots = np.empty(len(s), np.int64)
        pairs = np.empty((max(len(s), 1), 2), np.int32)
        n = ctypes.c_int32(0)
        self._check(_L().pa_bm_append_slots(self._h, s.ctypes.data, len(s), slots.ctypes.data, pairs.ctypes.data,
                                            ctypes.byref(n)), "append_slots")
        return slots, pairs[:n.value].copy()

    def fork(self, parent: int, child: int) -> None:
        self._check(_L().pa_bm_fork(self._h, int(parent), int(child)), "fork")

    def free(self, seq: int) -> None:
        self._check(_L().pa_bm_free(self._h, int(seq)), "free")

    def seq_len(self, seq: int) -> int:
        r = _L().pa_bm_seq_len(self._h, int(seq))
        if r < 0:
            raise BlockManagerError(r, "seq_len")
        return r

    def num_seq_blocks(self, seq: int) -> int:
        r = _L().pa_bm_num_seq_blocks(self._h, int(seq))
        if r < 0:
            raise BlockManagerError(r, "num_seq_blocks")
        return r

    def build_tables(self, seqs, width: int | None = None):
        s = np.ascontiguousarray(seqs, dtype=np.int64)
        if width is None:
            width = _L().pa_bm_max_seq_blocks(self._h, s.ctypes.data, len(s))
            if width < 0:
                raise BlockManagerError(width, "max_seq_blocks")
            width = max(width, 1)
        tables = np.zeros((len(s), width), np.int32)
        lens = np.zeros(len(s), np.int32)
        self._check(_L().pa_bm_build_tables(self._h, s.ctypes.data, len(s), int(width), tables.ctypes.data,
                                            lens.ctypes.data), "build_tables")
        return tables, lens
