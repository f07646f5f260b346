"""CPU oracle for paged KV cache attention (numpy wrapper over pkv_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by
the benchmark's CPU-baseline leg, never by the product path.  It shares no
code with the CUDA library.

Every array is a numpy array.  bf16 data travels as uint16 bit patterns and
e4m3 data as uint8 codes.  Formats: "f32", "bf16", "e4m3".

Functions and the passages they follow (see pkv_oracle.c for the full
statement of each definition):
  slot_mapping  -- nanoserve, "Architecture", step 2 "Prepare"; "How to design
                   an LLM serving system (a vLLM deep dive)", "PagedAttention".
  append        -- nanoserve, "Architecture", step 3 "Forward".
  attention     -- nanoserve, "Architecture", step 3, and its "Paged KV cache",
                   "Chunked prefill" and "Triton paged-attention decode
                   kernel" bullets; "PageServe", "What is implemented".
  e4m3_encode / e4m3_decode / bf16_decode -- "How Easy Is It to Start Serving
                   LLMs?", "What each setting does to performance" (FP8 KV).
  csr_to_block_tables -- "How Easy Is It to Start Serving LLMs?", "1.
                   Block-sparse KV memory" (pages as a CSR matrix); plain
                   Python loops, no C.
"""
import ctypes
import os

import numpy as np

from . import build_oracle

_FMT = {"f32": 0, "bf16": 1, "e4m3": 2}
_NP = {"f32": np.float32, "bf16": np.uint16, "e4m3": np.uint8}
_lib = None


def _load(path=None):
    global _lib
    if _lib is None or path is not None:
        path = path or build_oracle.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        lib.orc_bf16_decode_n.argtypes = [P, P, i64]
        lib.orc_e4m3_decode_n.argtypes = [P, P, i64]
        lib.orc_e4m3_encode_n.argtypes = [P, P, i64]
        lib.orc_slot_mapping.argtypes = [i32, P, P, P, i32, i32, P]
        lib.orc_slot_mapping.restype = ctypes.c_int
        lib.orc_append.argtypes = [P, P, ctypes.c_int, P, i64, i32, i32, P, P,
                                   ctypes.c_int, i32, i64, f32, f32]
        lib.orc_append.restype = ctypes.c_int
        lib.orc_attention.argtypes = [P, ctypes.c_int, P, P, P, i32, i32, P, P,
                                      ctypes.c_int, i32, i64, i32, i32, i32,
                                      f64, f64, f64, P, i32]
        lib.orc_attention.restype = ctypes.c_int
        lib.orc_attention_rows.argtypes = [P, ctypes.c_int, P, P, P, i32, i32, P,
                                           P, ctypes.c_int, i32, i64, i32, i32,
                                           i32, f64, f64, f64, i64, P, P, P, i32]
        lib.orc_attention_rows.restype = ctypes.c_int
        lib.orc_attention_v.argtypes = [P, ctypes.c_int, P, P, P, i32, i32, P, P,
                                        ctypes.c_int, i32, i64, i32, i32, i32,
                                        f64, f64, f64, f64, i64, P, i32]
        lib.orc_attention_v.restype = ctypes.c_int
        lib.orc_attention_rows_v.argtypes = [P, ctypes.c_int, P, P, P, i32, i32, P,
                                             P, ctypes.c_int, i32, i64, i32, i32,
                                             i32, f64, f64, f64, f64, i64, i64, P, P, P, i32]
        lib.orc_attention_rows_v.restype = ctypes.c_int
        _lib = lib
    return _lib


def use_library(path):
    """Test hook: route every call to another build of the oracle (the tests
    that plant a mistake in a copy of the oracle use it).  Returns the
    previously loaded library handle for restore_library()."""
    global _lib
    prev = _lib
    _load(path)
    return prev


def restore_library(prev):
    global _lib
    _lib = prev


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def fmt_of(a) -> str:
    for name, dt in _NP.items():
        if a.dtype == dt:
            return name
    raise TypeError(f"unsupported array dtype {a.dtype}")


# ---------------------------------------------------------------- formats
def bf16_decode(bits) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    _load().orc_bf16_decode_n(_ptr(bits), _ptr(out), bits.size)
    return out


def e4m3_decode(codes) -> np.ndarray:
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().orc_e4m3_decode_n(_ptr(codes), _ptr(out), codes.size)
    return out


def e4m3_encode(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().orc_e4m3_encode_n(_ptr(x), _ptr(out), x.size)
    return out


# ---------------------------------------------------------------- page lists
def csr_to_block_tables(kv_indptr, kv_indices, max_blocks):
    """Row i = the pages kv_indices[kv_indptr[i] .. kv_indptr[i+1]-1] in
    order, then -1; a row whose offsets decrease or leave [0, nnz], or that
    has more than max_blocks pages, is all -1 and flagged.
    Returns (tables [B, max_blocks] int32, bad [B] bool)."""
    indptr = [int(x) for x in kv_indptr]
    indices = [int(x) for x in kv_indices]
    B = len(indptr) - 1
    tables = np.full((B, max_blocks), -1, np.int32)
    bad = np.zeros(B, bool)
    for i in range(B):
        a, b = indptr[i], indptr[i + 1]
        if a < 0 or b < a or b > len(indices) or b - a > max_blocks:
            bad[i] = True
            continue
        for j in range(a, b):
            tables[i, j - a] = indices[j]
    return tables, bad


# ---------------------------------------------------------------- slots
def slot_mapping(cu_seqlens_q, seq_lens, block_tables, block_size) -> np.ndarray:
    cu = _c(cu_seqlens_q, np.int32)
    sl = _c(seq_lens, np.int32)
    bt = _c(block_tables, np.int32)
    B = sl.shape[0]
    out = np.empty(int(cu[B]), np.int64)
    rc = _load().orc_slot_mapping(B, _ptr(cu), _ptr(sl), _ptr(bt), bt.shape[1],
                                  int(block_size), _ptr(out))
    if rc:
        raise ValueError("slot_mapping: inconsistent lengths")
    return out


# ---------------------------------------------------------------- append
def append(k, v, slots, k_cache, v_cache, k_scale=1.0, v_scale=1.0) -> None:
    """Writes k[T,Hkv,D], v into the caches [NB, bs, Hkv, D] in place."""
    src = fmt_of(k)
    k = _c(k, k.dtype)
    v = _c(v, v.dtype)
    slots = _c(slots, np.int64)
    cfmt = fmt_of(k_cache)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    T, H, D = k.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    rc = _load().orc_append(_ptr(k), _ptr(v), _FMT[src], _ptr(slots), T, H, D,
                            _ptr(k_cache), _ptr(v_cache), _FMT[cfmt], bs, NB,
                            float(k_scale), float(v_scale))
    if rc:
        raise ValueError(f"append failed ({rc})")


# ---------------------------------------------------------------- attention
def attention(q, cu_seqlens_q, seq_lens, block_tables, k_cache, v_cache, scale,
              k_scale=1.0, v_scale=1.0, nthreads=1, rows=None, soft_cap=0.0,
              window_left=-1) -> np.ndarray:
    """fp64 attention.  q[T,Hq,D]; caches [NB,bs,Hkv,D].

    rows=None -> returns [T,Hq,D]; rows=(t[n], h[n]) -> returns [n, D].
    soft_cap > 0: each scaled score s becomes soft_cap * tanh(s / soft_cap);
    window_left >= 0: the query at position p sees keys p - window_left .. p.
    """
    variant = soft_cap > 0 or window_left >= 0
    qf = fmt_of(q)
    q = _c(q, q.dtype)
    cu = _c(cu_seqlens_q, np.int32)
    sl = _c(seq_lens, np.int32)
    bt = _c(block_tables, np.int32)
    cfmt = fmt_of(k_cache)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    T, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    assert D == D2
    B = sl.shape[0]
    lib = _load()
    if rows is None:
        out = np.zeros((T, Hq, D), np.float64)
        if variant:
            rc = lib.orc_attention_v(_ptr(q), _FMT[qf], _ptr(cu), _ptr(sl), _ptr(bt), B,
                                     bt.shape[1], _ptr(k_cache), _ptr(v_cache),
                                     _FMT[cfmt], bs, NB, Hq, Hkv, D, float(scale),
                                     float(k_scale), float(v_scale), float(soft_cap),
                                     int(window_left), _ptr(out), int(nthreads))
        else:
            rc = lib.orc_attention(_ptr(q), _FMT[qf], _ptr(cu), _ptr(sl), _ptr(bt), B,
                                   bt.shape[1], _ptr(k_cache), _ptr(v_cache),
                                   _FMT[cfmt], bs, NB, Hq, Hkv, D, float(scale),
                                   float(k_scale), float(v_scale), _ptr(out),
                                   int(nthreads))
    else:
        rt = _c(rows[0], np.int64)
        rh = _c(rows[1], np.int32)
        out = np.zeros((rt.shape[0], D), np.float64)
        if variant:
            rc = lib.orc_attention_rows_v(_ptr(q), _FMT[qf], _ptr(cu), _ptr(sl),
                                          _ptr(bt), B, bt.shape[1], _ptr(k_cache),
                                          _ptr(v_cache), _FMT[cfmt], bs, NB, Hq, Hkv,
                                          D, float(scale), float(k_scale),
                                          float(v_scale), float(soft_cap), int(window_left),
                                          rt.shape[0], _ptr(rt), _ptr(rh), _ptr(out),
                                          int(nthreads))
        else:
            rc = lib.orc_attention_rows(_ptr(q), _FMT[qf], _ptr(cu), _ptr(sl),
                                        _ptr(bt), B, bt.shape[1], _ptr(k_cache),
                                        _ptr(v_cache), _FMT[cfmt], bs, NB, Hq, Hkv,
                                        D, float(scale), float(k_scale),
                                        float(v_scale), rt.shape[0], _ptr(rt),
                                        _ptr(rh), _ptr(out), int(nthreads))
    if rc:
        raise ValueError(f"attention failed ({rc})")
    return out


def cpu_count() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------- one step
def run_step(wl, nthreads=1, rows=None, history_batch=1 << 22, soft_cap=0.0, window_left=-1):
    """Runs one step of a workload (see paged_kv_cache_mapping_gb300.workloads)
    on the oracle: history rows are appended first, then this step's rows are
    appended through their slots and every query row attends.

    Returns (out, k_cache, v_cache, step_slots)."""
    kc = np.zeros(wl.cache_shape(), wl.cache_np_dtype())
    vc = np.zeros(wl.cache_shape(), wl.cache_np_dtype())
    for s0, s1, cu, sl, k, v in wl.history_batches(history_batch):
        if k.shape[0]:
            slots = slot_mapping(cu, sl, wl.block_tables[s0:s1], wl.block_size)
            append(k, v, slots, kc, vc, wl.k_scale, wl.v_scale)
    slots = slot_mapping(wl.cu_seqlens_q, wl.seq_lens, wl.block_tables, wl.block_size)
    kn, vn = wl.new_rows()
    append(kn, vn, slots, kc, vc, wl.k_scale, wl.v_scale)
    out = attention(wl.q, wl.cu_seqlens_q, wl.seq_lens, wl.block_tables, kc, vc,
                    wl.scale, wl.k_scale, wl.v_scale, nthreads=nthreads, rows=rows,
                    soft_cap=soft_cap, window_left=window_left)
    return out, kc, vc, slots
