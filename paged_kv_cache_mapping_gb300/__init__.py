"""Paged KV cache append and attention for GB300 (sm_103a).

A thin ctypes binding over libpkv.so (C ABI in include/pkv.h).  The binding
only marshals arguments: every step -- slot computation, append, attention --
runs in the library's CUDA kernels.  PyTorch provides device memory and the
current stream.  There is no CPU fallback: if the library is missing or the
tensors are not on a CUDA device, the call raises.

Functions (same names as the C ABI):
  pkv_slot_mapping(cu_seqlens_q, seq_lens, block_tables, block_size, out=None)
  pkv_append(k, v, slot_mapping, k_cache, v_cache, k_scale=1.0, v_scale=1.0)
  pkv_attention_workspace_size(q, block_tables, k_cache)
  pkv_attention(q, cu_seqlens_q, seq_lens, block_tables, k_cache, v_cache,
                scale, out, k_scale=1.0, v_scale=1.0, max_q_len=0, workspace=None)
  pkv_attention_plan(q, cu_seqlens_q, seq_lens, block_tables, k_cache, workspace,
                     max_q_len=0, window_left=-1)
  pkv_attention_run(q, cu_seqlens_q, seq_lens, block_tables, k_cache, v_cache,
                    scale, out, workspace, k_scale=1.0, v_scale=1.0, max_q_len=0)
  pkv_attention_static_workspace(q, cu_seqlens_q, seq_lens, block_tables, k_cache,
                                 v_cache, scale, out, k_scale=1.0, v_scale=1.0, max_q_len=0)
  pkv_device_errors()
"""
import ctypes
import os

import torch

__all__ = ["PkvError", "pkv_slot_mapping", "pkv_csr_to_block_tables", "pkv_append", "pkv_attention", "pkv_attention_workspace_size",
           "pkv_attention_plan", "pkv_attention_run", "pkv_attention_static_workspace", "pkv_device_errors", "pkv_version", "library_path", "load_library",
           "EXPORTED", "STATIC_WORKSPACE_BYTES"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpkv.so")
EXPORTED = ("pkv_slot_mapping", "pkv_append", "pkv_attention_workspace_size", "pkv_attention", "pkv_attention_ex",
            "pkv_attention_plan", "pkv_attention_run",
            "pkv_attention_static_workspace", "pkv_device_errors", "pkv_status_string", "pkv_last_error",
            "pkv_version", "pkv_csr_to_block_tables", "pkv_bm_create", "pkv_bm_destroy", "pkv_bm_add_sequence", "pkv_bm_append",
            "pkv_bm_free_sequence", "pkv_bm_block_table", "pkv_bm_build_step", "pkv_bm_stats")
# PKV_STATIC_WORKSPACE_BYTES of include/pkv.h
STATIC_WORKSPACE_BYTES = 16 << 20

_DT = {torch.float32: 0, torch.bfloat16: 1, torch.float8_e4m3fn: 2, torch.int32: 3, torch.int64: 4}


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class _Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class _Variant(ctypes.Structure):
    _fields_ = [("logits_soft_cap", ctypes.c_float), ("window_left", ctypes.c_int32)]


_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Loads libpkv.so (built by ``python -m paged_kv_cache_mapping_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise PkvError(-1, f"{_LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_cache_mapping_gb300.build`")
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.POINTER(_Tensor)
        st = ctypes.c_int
        lib.pkv_slot_mapping.argtypes = [P, P, P, ctypes.c_int32, P, ctypes.c_void_p]
        lib.pkv_slot_mapping.restype = st
        lib.pkv_csr_to_block_tables.argtypes = [P, P, P, ctypes.c_void_p]
        lib.pkv_csr_to_block_tables.restype = st
        lib.pkv_append.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_void_p]
        lib.pkv_append.restype = st
        lib.pkv_attention_workspace_size.argtypes = [P, P, P, ctypes.POINTER(ctypes.c_size_t)]
        lib.pkv_attention_workspace_size.restype = st
        lib.pkv_attention.argtypes = [P, P, P, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_int32, P, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        lib.pkv_attention.restype = st
        lib.pkv_attention_ex.argtypes = [P, P, P, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                         ctypes.c_int32, P, ctypes.POINTER(_Variant), ctypes.c_void_p,
                                         ctypes.c_size_t, ctypes.c_void_p]
        lib.pkv_attention_ex.restype = st
        lib.pkv_attention_plan.argtypes = [P, P, P, P, P, ctypes.c_int32, ctypes.POINTER(_Variant), ctypes.c_void_p,
                                           ctypes.c_size_t, ctypes.c_void_p]
        lib.pkv_attention_plan.restype = st
        lib.pkv_attention_run.argtypes = [P, P, P, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                          ctypes.c_int32, P, ctypes.POINTER(_Variant), ctypes.c_void_p,
                                          ctypes.c_size_t, ctypes.c_void_p]
        lib.pkv_attention_run.restype = st
        lib.pkv_attention_static_workspace.argtypes = [P, P, P, P, P, P, ctypes.c_float, ctypes.c_float,
                                                       ctypes.c_float, ctypes.c_int32, P, ctypes.c_void_p]
        lib.pkv_attention_static_workspace.restype = st
        lib.pkv_device_errors.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
        lib.pkv_device_errors.restype = st
        lib.pkv_status_string.argtypes = [ctypes.c_int]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_last_error.argtypes = []
        lib.pkv_last_error.restype = ctypes.c_char_p
        lib.pkv_version.argtypes = []
        lib.pkv_version.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _tensor(t: torch.Tensor, name: str) -> _Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise PkvError(1, f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dim() > 4:
        raise PkvError(1, f"{name} has more than 4 dimensions")
    dt = _DT.get(t.dtype)
    if dt is None:
        raise PkvError(2, f"{name}: unsupported dtype {t.dtype}")
    d = _Tensor()
    d.data = t.data_ptr()
    d.dtype = dt
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(rc: int):
    if rc != 0:
        lib = load_library()
        raise PkvError(rc, f"{lib.pkv_status_string(rc).decode()}: {lib.pkv_last_error().decode()}")


def pkv_version() -> str:
    return load_library().pkv_version().decode()


def pkv_slot_mapping(cu_seqlens_q, seq_lens, block_tables, block_size: int, out=None, T: int = None):
    """Flat cache slot of every new row: [T] int32 (or the given out)."""
    lib = load_library()
    if out is None:
        if T is None:
            raise ValueError("give T (the host-side row count) or out")
        out = torch.empty(T, dtype=torch.int32, device=seq_lens.device)
    a, b, c, o = (_tensor(cu_seqlens_q, "cu_seqlens_q"), _tensor(seq_lens, "seq_lens"),
                  _tensor(block_tables, "block_tables"), _tensor(out, "slot_mapping"))
    _check(lib.pkv_slot_mapping(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), int(block_size),
                                ctypes.byref(o), _stream(seq_lens.device)))
    return out


def pkv_csr_to_block_tables(kv_indptr, kv_indices, block_tables):
    """Fills block_tables [B, max_blocks] int32 from the CSR page lists
    (kv_indptr [B+1], kv_indices [nnz], int32); returns block_tables."""
    lib = load_library()
    a, b, c = (_tensor(kv_indptr, "kv_indptr"), _tensor(kv_indices, "kv_indices"),
               _tensor(block_tables, "block_tables"))
    _check(lib.pkv_csr_to_block_tables(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), _stream(kv_indptr.device)))
    return block_tables


def pkv_append(k, v, slot_mapping, k_cache, v_cache, k_scale: float = 1.0, v_scale: float = 1.0):
    """Writes k, v [T, Hkv, D] into the caches [num_blocks, block_size, Hkv, D]."""
    lib = load_library()
    tk, tv, ts, tkc, tvc = (_tensor(k, "k"), _tensor(v, "v"), _tensor(slot_mapping, "slot_mapping"),
                            _tensor(k_cache, "k_cache"), _tensor(v_cache, "v_cache"))
    _check(lib.pkv_append(ctypes.byref(tk), ctypes.byref(tv), ctypes.byref(ts), ctypes.byref(tkc),
                          ctypes.byref(tvc), float(k_scale), float(v_scale), _stream(k.device)))


def pkv_attention_workspace_size(q, block_tables, k_cache) -> int:
    lib = load_library()
    tq, tb, tk = _tensor(q, "q"), _tensor(block_tables, "block_tables"), _tensor(k_cache, "k_cache")
    n = ctypes.c_size_t(0)
    _check(lib.pkv_attention_workspace_size(ctypes.byref(tq), ctypes.byref(tb), ctypes.byref(tk),
                                            ctypes.byref(n)))
    return int(n.value)


def pkv_attention(q, cu_seqlens_q, seq_lens, block_tables, k_cache, v_cache, scale: float, out,
                  k_scale: float = 1.0, v_scale: float = 1.0, max_q_len: int = 0, workspace=None,
                  soft_cap: float = 0.0, window_left: int = -1):
    """Causal GQA attention of q [T, Hq, D] over the paged caches into out.
    soft_cap > 0 or window_left >= 0 select the variants (pkv_attention_ex)."""
    lib = load_library()
    if workspace is None:
        workspace = torch.empty(pkv_attention_workspace_size(q, block_tables, k_cache), dtype=torch.uint8,
                                device=q.device)
    tq, tcu, tsl, tbt, tkc, tvc, to = (
        _tensor(q, "q"), _tensor(cu_seqlens_q, "cu_seqlens_q"), _tensor(seq_lens, "seq_lens"),
        _tensor(block_tables, "block_tables"), _tensor(k_cache, "k_cache"), _tensor(v_cache, "v_cache"),
        _tensor(out, "out"))
    ws = (ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(), _stream(q.device))
    if soft_cap > 0 or window_left >= 0:
        var = _Variant(float(soft_cap), int(window_left))
        _check(lib.pkv_attention_ex(ctypes.byref(tq), ctypes.byref(tcu), ctypes.byref(tsl), ctypes.byref(tbt),
                                    ctypes.byref(tkc), ctypes.byref(tvc), float(scale), float(k_scale),
                                    float(v_scale), int(max_q_len), ctypes.byref(to), ctypes.byref(var), *ws))
    else:
        _check(lib.pkv_attention(ctypes.byref(tq), ctypes.byref(tcu), ctypes.byref(tsl), ctypes.byref(tbt),
                                 ctypes.byref(tkc), ctypes.byref(tvc), float(scale), float(k_scale),
                                 float(v_scale), int(max_q_len), ctypes.byref(to), *ws))
    return out


def pkv_attention_plan(q, cu_seqlens_q, seq_lens, block_tables, k_cache, workspace, max_q_len: int = 0,
                       window_left: int = -1):
    """Writes the work lists of an attention call into workspace, from the
    device lengths; every later pkv_attention_run over the same lengths and
    shapes reuses them (one plan per model step, one run per layer)."""
    lib = load_library()
    tq, tcu, tsl, tbt, tkc = (_tensor(q, "q"), _tensor(cu_seqlens_q, "cu_seqlens_q"), _tensor(seq_lens, "seq_lens"),
                              _tensor(block_tables, "block_tables"), _tensor(k_cache, "k_cache"))
    var = _Variant(0.0, int(window_left))
    _check(lib.pkv_attention_plan(ctypes.byref(tq), ctypes.byref(tcu), ctypes.byref(tsl), ctypes.byref(tbt),
                                  ctypes.byref(tkc), int(max_q_len), ctypes.byref(var),
                                  ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(),
                                  _stream(q.device)))


def pkv_attention_run(q, cu_seqlens_q, seq_lens, block_tables, k_cache, v_cache, scale: float, out, workspace,
                      k_scale: float = 1.0, v_scale: float = 1.0, max_q_len: int = 0, soft_cap: float = 0.0,
                      window_left: int = -1):
    """Attention of one layer over the plan that pkv_attention_plan left in
    workspace (same lengths, shapes, max_q_len and window_left)."""
    lib = load_library()
    tq, tcu, tsl, tbt, tkc, tvc, to = (
        _tensor(q, "q"), _tensor(cu_seqlens_q, "cu_seqlens_q"), _tensor(seq_lens, "seq_lens"),
        _tensor(block_tables, "block_tables"), _tensor(k_cache, "k_cache"), _tensor(v_cache, "v_cache"),
        _tensor(out, "out"))
    var = _Variant(float(soft_cap), int(window_left))
    _check(lib.pkv_attention_run(ctypes.byref(tq), ctypes.byref(tcu), ctypes.byref(tsl), ctypes.byref(tbt),
                                 ctypes.byref(tkc), ctypes.byref(tvc), float(scale), float(k_scale), float(v_scale),
                                 int(max_q_len), ctypes.byref(to), ctypes.byref(var),
                                 ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(),
                                 _stream(q.device)))
    return out


def pkv_attention_static_workspace(q, cu_seqlens_q, seq_lens, block_tables, k_cache, v_cache, scale: float,
                                   out, k_scale: float = 1.0, v_scale: float = 1.0, max_q_len: int = 0):
    """pkv_attention with the library's fixed per-device scratch array as the
    workspace: allocates nothing.  Calls on one device must not overlap."""
    lib = load_library()
    tq, tcu, tsl, tbt, tkc, tvc, to = (
        _tensor(q, "q"), _tensor(cu_seqlens_q, "cu_seqlens_q"), _tensor(seq_lens, "seq_lens"),
        _tensor(block_tables, "block_tables"), _tensor(k_cache, "k_cache"), _tensor(v_cache, "v_cache"),
        _tensor(out, "out"))
    _check(lib.pkv_attention_static_workspace(ctypes.byref(tq), ctypes.byref(tcu), ctypes.byref(tsl),
                                              ctypes.byref(tbt), ctypes.byref(tkc), ctypes.byref(tvc),
                                              float(scale), float(k_scale), float(v_scale), int(max_q_len),
                                              ctypes.byref(to), _stream(q.device)))
    return out


def pkv_device_errors(device=None) -> int:
    """Synchronises the current stream and returns (and clears) the device
    error bits: 1 slot range, 2 block id range, 4 lengths, 8 wait timeout,
    16 a run without a matching plan."""
    lib = load_library()
    flags = ctypes.c_uint32(0)
    _check(lib.pkv_device_errors(_stream(device), ctypes.byref(flags)))
    return int(flags.value)
