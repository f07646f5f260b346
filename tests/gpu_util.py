"""Shared pieces of the GPU parity tests: run a workload on the library and
on the oracle, and compare."""
import numpy as np
import torch

import oracle
from paged_kv_cache_mapping_gb300 import pkv_device_errors
from paged_kv_cache_mapping_gb300.harness import DeviceStep, cache_to_numpy
from tests.helpers import rel_l2

# Tolerances.  bf16 queries and caches, fp32 output, against the fp64 oracle:
# max |err| <= 2e-3 and relative L2 <= 1e-3, the accuracy bound of the
# attention path (bf16 inputs, fp32 accumulation and output).  fp8
# caches: max |err| <= 1e-2 against the oracle on the same dequantised
# values.  fp32 everything: the kernel accumulates in fp32 (unit roundoff
# 6e-8) over at most a few hundred terms per dot product and sum; the tiny
# fp32 workload measures about 1e-7 relative L2, so 1e-5 absolute and 1e-6
# relative L2 keep a margin of ten over the rounding.
TOL = {"bf16": (2e-3, 1e-3), "e4m3": (1e-2, 1e-2), "f32": (1e-5, 1e-6)}


def run_gpu(wl, out_dtype=torch.float32, **kw):
    ds = DeviceStep(wl, out_dtype=out_dtype, **kw)
    out = ds.step()
    torch.cuda.synchronize()
    flags = pkv_device_errors()
    assert flags == 0, f"device error flags 0x{flags:x}"
    return ds, out


def rows_of(wl):
    """(token, head) index arrays of every query row."""
    t = np.repeat(np.arange(wl.T), wl.Hq)
    h = np.tile(np.arange(wl.Hq), wl.T)
    return t, h


def check_attention(gpu_out, ref, kv, what=""):
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    tol_abs, tol_rel = TOL[kv]
    err = float(np.abs(g - ref).max()) if ref.size else 0.0
    rel = rel_l2(g, ref) if ref.size else 0.0
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    assert err <= tol_abs, f"{what}: max abs err {err:.3e} > {tol_abs}"
    assert rel <= tol_rel, f"{what}: rel L2 {rel:.3e} > {tol_rel}"
    return err, rel


def bf16_rne_of(x: torch.Tensor) -> torch.Tensor:
    """Round an fp32 tensor to bf16, nearest even (torch's own conversion)."""
    return x.to(torch.bfloat16)


def oracle_caches_equal(ds, okc, ovc, layer=0):
    kc, vc = ds.caches[layer]
    gk, gv = cache_to_numpy(kc), cache_to_numpy(vc)
    return np.array_equal(gk.view(np.uint8), okc.view(np.uint8)) and \
        np.array_equal(gv.view(np.uint8), ovc.view(np.uint8))
