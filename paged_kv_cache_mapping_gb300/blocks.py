"""Host-side KV block manager (C ABI in include/pkv_blocks.h): a ctypes
wrapper that only marshals arguments; the manager itself is C++ in libpkv.so.

    bm = BlockManager(num_blocks, block_size)
    cached = bm.add_sequence(seq_id, prompt_token_ids)   # tokens already cached
    slots = bm.append(seq_id, token_ids)                 # their cache slots
    cu_q, seq_lens, tables, slots = bm.build_step(seq_ids, n_new, tokens, max_blocks)
    bm.free_sequence(seq_id)
"""
import ctypes

import numpy as np

from . import PkvError, load_library


class Stats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("free_blocks", ctypes.c_int32),
                ("cached_blocks", ctypes.c_int32), ("num_sequences", ctypes.c_int32),
                ("prefix_hit_blocks", ctypes.c_int64), ("evictions", ctypes.c_int64)]


def _lib():
    lib = load_library()
    if not getattr(lib, "_pkv_bm_ready", False):
        vp, i32, i64, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
        p32 = ctypes.POINTER(ctypes.c_int32)
        lib.pkv_bm_create.argtypes = [i32, i32, ctypes.POINTER(vp)]
        lib.pkv_bm_create.restype = st
        lib.pkv_bm_destroy.argtypes = [vp]
        lib.pkv_bm_destroy.restype = None
        lib.pkv_bm_add_sequence.argtypes = [vp, i64, p32, i32, p32]
        lib.pkv_bm_add_sequence.restype = st
        lib.pkv_bm_append.argtypes = [vp, i64, p32, i32, p32]
        lib.pkv_bm_append.restype = st
        lib.pkv_bm_free_sequence.argtypes = [vp, i64]
        lib.pkv_bm_free_sequence.restype = st
        lib.pkv_bm_block_table.argtypes = [vp, i64, p32, i32, p32, p32]
        lib.pkv_bm_block_table.restype = st
        lib.pkv_bm_build_step.argtypes = [vp, ctypes.POINTER(ctypes.c_int64), p32, p32, i32, i32, p32, p32, p32,
                                          p32]
        lib.pkv_bm_build_step.restype = st
        lib.pkv_bm_stats.argtypes = [vp, ctypes.POINTER(Stats)]
        lib.pkv_bm_stats.restype = st
        lib._pkv_bm_ready = True
    return lib


def _check(rc):
    if rc != 0:
        lib = load_library()
        raise PkvError(rc, f"{lib.pkv_status_string(rc).decode()}: {lib.pkv_last_error().decode()}")


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int):
        self._lib = _lib()
        self._h = ctypes.c_void_p()
        _check(self._lib.pkv_bm_create(int(num_blocks), int(block_size), ctypes.byref(self._h)))
        self.block_size = int(block_size)

    def close(self):
        if self._h:
            self._lib.pkv_bm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_sequence(self, seq_id: int, prompt) -> int:
        arr, ptr = _i32(prompt)
        out = ctypes.c_int32(0)
        _check(self._lib.pkv_bm_add_sequence(self._h, int(seq_id), ptr, arr.size, ctypes.byref(out)))
        return int(out.value)

    def append(self, seq_id: int, tokens) -> np.ndarray:
        arr, ptr = _i32(tokens)
        slots = np.empty(arr.size, np.int32)
        _check(self._lib.pkv_bm_append(self._h, int(seq_id), ptr, arr.size,
                                       slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return slots

    def free_sequence(self, seq_id: int):
        _check(self._lib.pkv_bm_free_sequence(self._h, int(seq_id)))

    def block_table(self, seq_id: int):
        nb, nt = ctypes.c_int32(0), ctypes.c_int32(0)
        _check(self._lib.pkv_bm_block_table(self._h, int(seq_id), None, 0, ctypes.byref(nb), ctypes.byref(nt)))
        table = np.empty(nb.value, np.int32)
        _check(self._lib.pkv_bm_block_table(self._h, int(seq_id), table.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                            nb.value, ctypes.byref(nb), ctypes.byref(nt)))
        return table, int(nt.value)

    def build_step(self, seq_ids, n_new, tokens, max_blocks: int):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        nn, nn_p = _i32(n_new)
        tk, tk_p = _i32(tokens)
        B = ids.size
        cu = np.empty(B + 1, np.int32)
        sl = np.empty(B, np.int32)
        bt = np.empty((B, max_blocks), np.int32)
        slots = np.empty(int(nn.sum()), np.int32)
        p = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        _check(self._lib.pkv_bm_build_step(self._h, ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), nn_p, tk_p,
                                           B, int(max_blocks), p(cu), p(sl), p(bt), p(slots)))
        return cu, sl, bt, slots

    def stats(self) -> dict:
        s = Stats()
        _check(self._lib.pkv_bm_stats(self._h, ctypes.byref(s)))
        return {k: getattr(s, k) for k, _ in Stats._fields_}
