"""The C ABI without a GPU: libpkv.so loads, exports every function that
include/pkv.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_mapping_gb300 as pkv
from paged_kv_cache_mapping_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.load_library()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    return re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)


def test_header_declares_the_binding_names():
    names = declared_functions()
    assert sorted(names) == sorted(pkv.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_no_other_symbol_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.library_path()], capture_output=True,
                         text=True).stdout
    syms = {l.split()[-1] for l in out.splitlines() if l.strip() and l.split()[-2] in "TtWw"}
    pkv_syms = {s for s in syms if s.startswith("pkv_")}
    assert pkv_syms == set(declared_functions())


def test_status_strings_and_version(lib):
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(3) == b"workspace too small"
    assert lib.pkv_status_string(99) == b"unknown status"
    assert re.match(rb"\d+\.\d+\.\d+", lib.pkv_version())


def _t(ptr, dtype, shape, stride=None):
    d = pkv._Tensor()
    d.data = ptr
    d.dtype = dtype
    d.ndim = len(shape)
    if stride is None:
        stride, acc = [], 1
        for n in reversed(shape):
            stride.insert(0, acc)
            acc *= n
    for i, (n, s) in enumerate(zip(shape, stride)):
        d.shape[i] = n
        d.stride[i] = s
    return d


F32, BF16, E4M3, I32, I64 = 0, 1, 2, 3, 4
FAKE = 0x10000  # never dereferenced: every case below fails validation first


def _attn(lib, q, cu, sl, bt, kc, vc, out, ws_bytes=1 << 30, max_q=0):
    r = lambda x: ctypes.byref(x)
    return lib.pkv_attention(r(q), r(cu), r(sl), r(bt), r(kc), r(vc), 0.1, 1.0, 1.0, max_q, r(out),
                             ctypes.c_void_p(FAKE), ws_bytes, None)


def good(T=4, Hq=32, Hkv=8, D=128, B=4, NB=100, bs=16, mb=8, qdt=BF16, kdt=BF16, odt=F32):
    return dict(q=_t(FAKE, qdt, [T, Hq, D]), cu=_t(FAKE, I32, [B + 1]), sl=_t(FAKE, I32, [B]),
                bt=_t(FAKE, I32, [B, mb]), kc=_t(FAKE, kdt, [NB, bs, Hkv, D]),
                vc=_t(FAKE, kdt, [NB, bs, Hkv, D]), out=_t(FAKE, odt, [T, Hq, D]))


@pytest.mark.parametrize("mutate,status", [
    (lambda a: a.update(q=_t(FAKE, BF16, [4, 30, 128])), 1),          # Hq not a multiple of Hkv
    (lambda a: a.update(out=_t(FAKE, F32, [4, 32, 64])), 1),          # out shape
    (lambda a: a.update(q=_t(FAKE, F32, [4, 32, 128])), 2),           # f32 q, bf16 cache
    (lambda a: a.update(kc=_t(FAKE, F32, [100, 16, 8, 128])), 1),     # k/v dtypes differ
    (lambda a: a.update(q=_t(FAKE, BF16, [4, 32, 96]), out=_t(FAKE, F32, [4, 32, 96]),
                        kc=_t(FAKE, BF16, [100, 16, 8, 96]), vc=_t(FAKE, BF16, [100, 16, 8, 96])), 2),
    (lambda a: a.update(bt=_t(FAKE, I64, [4, 8])), 1),                # table dtype
    (lambda a: a.update(cu=_t(FAKE, I32, [4])), 1),                   # cu length
    (lambda a: a.update(kc=_t(FAKE, BF16, [100, 16, 8, 128], [16384, 1024, 128, 2])), 1),  # strided cache
    (lambda a: a.update(q=_t(FAKE + 2, BF16, [4, 32, 128])), 1),      # misaligned q
    (lambda a: a.update(kc=_t(0, BF16, [100, 16, 8, 128])), 1),       # NULL cache
])
def test_attention_validation(lib, mutate, status):
    a = good()
    mutate(a)
    rc = _attn(lib, a["q"], a["cu"], a["sl"], a["bt"], a["kc"], a["vc"], a["out"])
    assert rc == status, lib.pkv_last_error()
    assert lib.pkv_last_error() != b""


def test_workspace_too_small_is_reported(lib):
    a = good()
    rc = _attn(lib, a["q"], a["cu"], a["sl"], a["bt"], a["kc"], a["vc"], a["out"], ws_bytes=100)
    assert rc == 3


def test_workspace_size_is_host_only(lib):
    a = good(B=64)
    n = ctypes.c_size_t(0)
    assert lib.pkv_attention_workspace_size(ctypes.byref(a["q"]), ctypes.byref(a["bt"]),
                                            ctypes.byref(a["kc"]), ctypes.byref(n)) == 0
    # block tables of 8 x 16 tokens: one split-KV chunk per sequence at most,
    # so at least one chunk output and log-sum-exp per (sequence, head)
    assert n.value >= 64 * 1 * 32 * (128 + 1) * 4
    c = good(B=64, mb=4096)  # 65536-token tables: 512 chunks of 128 tokens
    k = ctypes.c_size_t(0)
    lib.pkv_attention_workspace_size(ctypes.byref(c["q"]), ctypes.byref(c["bt"]), ctypes.byref(c["kc"]),
                                     ctypes.byref(k))
    assert k.value >= 64 * 128 * 32 * (128 + 1) * 4
    b = good(B=128)
    m = ctypes.c_size_t(0)
    lib.pkv_attention_workspace_size(ctypes.byref(b["q"]), ctypes.byref(b["bt"]), ctypes.byref(b["kc"]),
                                     ctypes.byref(m))
    assert m.value > n.value


def test_append_validation(lib):
    r = ctypes.byref
    k = _t(FAKE, BF16, [4, 8, 128])
    slots = _t(FAKE, I32, [4])
    kc = _t(FAKE, BF16, [100, 16, 8, 128])
    assert lib.pkv_append(r(k), r(k), r(_t(FAKE, I32, [5])), r(kc), r(kc), 1.0, 1.0, None) == 1
    assert lib.pkv_append(r(_t(FAKE, F32, [4, 8, 128])), r(_t(FAKE, F32, [4, 8, 128])), r(slots), r(kc),
                          r(kc), 1.0, 1.0, None) == 2
    k8 = _t(FAKE, E4M3, [100, 16, 8, 128])
    assert lib.pkv_append(r(k), r(k), r(slots), r(k8), r(k8), 0.0, 1.0, None) == 1  # zero scale
    assert lib.pkv_append(r(k), r(k), r(_t(FAKE, F32, [4])), r(kc), r(kc), 1.0, 1.0, None) == 1


def test_slot_mapping_validation(lib):
    r = ctypes.byref
    cu, sl, bt = _t(FAKE, I32, [5]), _t(FAKE, I32, [4]), _t(FAKE, I32, [4, 8])
    assert lib.pkv_slot_mapping(r(cu), r(sl), r(bt), 0, r(_t(FAKE, I32, [9])), None) == 1
    assert lib.pkv_slot_mapping(r(cu), r(sl), r(bt), 16, r(_t(FAKE, F32, [9])), None) == 1
    assert lib.pkv_slot_mapping(r(_t(FAKE, I32, [4])), r(sl), r(bt), 16, r(_t(FAKE, I32, [9])), None) == 1


def test_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(pkv.PkvError):
        pkv.pkv_slot_mapping(torch.zeros(5, dtype=torch.int32), torch.zeros(4, dtype=torch.int32),
                             torch.zeros(4, 4, dtype=torch.int32), 16, T=4)


def test_plan_and_run_validation(lib):
    """The split call checks its arguments on the host like pkv_attention:
    a short workspace, mismatched shapes and a variant the prefill kernel in
    use cannot take are refused before any launch."""
    r = ctypes.byref
    a = good()
    ws = ctypes.c_void_p(FAKE)
    args = (r(a["q"]), r(a["cu"]), r(a["sl"]), r(a["bt"]), r(a["kc"]))
    assert lib.pkv_attention_plan(*args, 0, None, ws, 100, None) == 3
    assert lib.pkv_attention_plan(r(a["q"]), r(_t(FAKE, I32, [4])), r(a["sl"]), r(a["bt"]), r(a["kc"]), 0, None,
                                  ws, 1 << 30, None) == 1
    assert lib.pkv_attention_run(*args, r(a["vc"]), 0.1, 1.0, 1.0, 0, r(a["out"]), None, ws, 100, None) == 3
    assert lib.pkv_attention_run(*args, r(a["vc"]), 0.1, 1.0, 1.0, 0, r(_t(FAKE, F32, [4, 32, 64])), None, ws,
                                 1 << 30, None) == 1
    assert lib.pkv_attention_run(*args, r(a["vc"]), 0.1, 1.0, 1.0, 0, None, None, ws, 1 << 30, None) == 1
    # a window with prefill rows on a block size that is not a multiple of 8
    # (the mma.sync prefill): unsupported, plan and run alike
    b = good(kdt=E4M3, bs=12)
    var = pkv._Variant(0.0, 64)
    assert lib.pkv_attention_plan(r(b["q"]), r(b["cu"]), r(b["sl"]), r(b["bt"]), r(b["kc"]), 8, r(var), ws,
                                  1 << 30, None) == 2
    assert lib.pkv_attention_run(r(b["q"]), r(b["cu"]), r(b["sl"]), r(b["bt"]), r(b["kc"]), r(b["vc"]), 0.1, 1.0,
                                 1.0, 8, r(b["out"]), r(var), ws, 1 << 30, None) == 2
