"""pkv_attention_static_workspace: the attention call that takes its scratch
from the library's fixed per-device array and allocates nothing.

The GPU test runs several calls in a row on different batches, so each call
starts from the array contents the previous one left, and compares every
result with pkv_attention on a caller-provided workspace.  This file is
named to be collected last, so the GPU test also runs after every other
test has used the device."""
import ctypes

import pytest
import torch

import paged_kv_cache_mapping_gb300 as pkv
from paged_kv_cache_mapping_gb300 import build as pkv_build
from paged_kv_cache_mapping_gb300 import workloads as W
from paged_kv_cache_mapping_gb300.harness import DeviceStep
from tests.gpu_util import TOL


def _desc(dtype, shape, ptr=0x10000):
    d = pkv._Tensor()
    d.data = ptr  # never dereferenced: the call is rejected on the host
    d.dtype = dtype
    d.ndim = len(shape)
    acc = 1
    for i in reversed(range(len(shape))):
        d.shape[i] = shape[i]
        d.stride[i] = acc
        acc *= shape[i]
    return d


def test_static_workspace_rejects_a_call_beyond_its_size():
    pkv_build.build()
    lib = pkv.load_library()
    BF16, I32, F32 = 1, 3, 0
    B, T, Hq, Hkv, D, mb, bs = 64, 64, 32, 8, 128, 256, 16  # 4096-token tables
    q, out = _desc(BF16, [T, Hq, D]), _desc(F32, [T, Hq, D])
    cu, sl, bt = _desc(I32, [B + 1]), _desc(I32, [B]), _desc(I32, [B, mb])
    kc, vc = _desc(BF16, [1000, bs, Hkv, D]), _desc(BF16, [1000, bs, Hkv, D])
    need = ctypes.c_size_t(0)
    assert lib.pkv_attention_workspace_size(ctypes.byref(q), ctypes.byref(bt), ctypes.byref(kc),
                                            ctypes.byref(need)) == 0
    assert need.value > pkv.STATIC_WORKSPACE_BYTES
    r = ctypes.byref
    rc = lib.pkv_attention_static_workspace(r(q), r(cu), r(sl), r(bt), r(kc), r(vc), 0.1, 1.0, 1.0, 1, r(out),
                                            None)
    assert rc == 3  # PKV_ERR_WORKSPACE_TOO_SMALL
    msg = lib.pkv_last_error().decode()
    assert str(need.value) in msg and str(pkv.STATIC_WORKSPACE_BYTES) in msg


def _decode_split():
    # 12 decode sequences up to 2600 tokens: several split-KV chunks each
    return W.qwen3_4b_decode(B=12, ctx=(1, 2600), block_size=16, num_blocks=0, seed=2102)


def _mixed():
    # decodes plus prefill chunks: the plan, prefill and decode kernels
    return W.mixed_prefill(n_decode=5, dec_ctx=(300, 1400), chunk=200, prefix=160, block_size=16,
                           num_blocks=1024, seed=2104)


def _fp8():
    return W.lognormal_fp8(B=20, median=700, sigma=1.0, cap=6000, seed=2106)


@pytest.mark.gpu
def test_static_workspace_matches_caller_workspace_over_consecutive_calls():
    pkv_build.build()
    steps = {name: DeviceStep(make()) for name, make in
             (("decode", _decode_split), ("mixed", _mixed), ("fp8", _fp8))}
    expected = {}
    for name, ds in steps.items():
        assert pkv.pkv_attention_workspace_size(ds.q, ds.bt, ds.caches[0][0]) <= pkv.STATIC_WORKSPACE_BYTES
        expected[name] = ds.step().clone()  # slots, append, attention with a caller workspace
    torch.cuda.synchronize()
    assert pkv.pkv_device_errors() == 0
    # consecutive calls on one stream; each finds the previous call's leftovers
    for name in ("decode", "mixed", "decode", "fp8", "fp8", "mixed"):
        ds, wl = steps[name], steps[name].wl
        kc, vc = ds.caches[0]
        out = torch.full_like(ds.out, float("nan"))
        pkv.pkv_attention_static_workspace(ds.q, ds.cu_q, ds.seq_lens, ds.bt, kc, vc, wl.scale, out,
                                           wl.k_scale, wl.v_scale, ds.max_q_len)
        torch.cuda.synchronize()
        assert pkv.pkv_device_errors() == 0, name
        # the same kernels on the same inputs with a plan that depends only on
        # the lengths: the results must be the same bits; the tolerance is
        # reported only to make a failure easier to read
        if not torch.equal(out, expected[name]):
            ref, got = expected[name].double(), out.double()
            err = (got - ref).abs().max().item()
            tol_abs, tol_rel = TOL[wl.kv]
            raise AssertionError(f"{name}: static-array result differs from the caller-workspace result "
                                 f"(max |diff| {err:.3e}; attention tolerance {tol_abs})")
