"""The e4m3 append on the GPU against the oracle over the encoder's whole
range: every bf16 bit pattern (both signs of zero, subnormals, NaN, +-inf)
and fp32 values at and beside every rounding tie, at scales that push the
products into saturation and deep into the e4m3 subnormals, from bf16 and
from f32 source rows; then attention over caches in which a large share of
the codes saturated.

OCP e4m3 ("How Easy Is It to Start Serving LLMs?", "What each setting does to
performance", FP8 KV cache; the format's own definition): bias 7, largest
finite 448, no infinity, one NaN pattern per sign.  Codes are compared byte
for byte, except that where the input is NaN either NaN code (0x7F, 0xFF)
is accepted: the format leaves the sign of a converted NaN open.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_mapping_gb300 import pkv_append, pkv_device_errors
from paged_kv_cache_mapping_gb300 import workloads as W
from tests.gpu_util import check_attention, oracle_caches_equal, run_gpu

pytestmark = pytest.mark.gpu

NT = oracle.cpu_count()
HKV, D = 2, 128


def _is_nan_code(c):
    return (c & 0x7F) == 0x7F


def _append_both(k, v, scale_k, scale_v, src):
    """Appends rows k, v [T, HKV, D] (uint16 bf16 bits or float32) at slots
    0..T-1 of a one-token-per-block cache on the GPU and on the oracle;
    returns (gpu K, gpu V, oracle K, oracle V) codes as uint8 arrays."""
    T = k.shape[0]
    nb = T + 3
    okc = np.zeros((nb, 1, HKV, D), np.uint8)
    ovc = np.zeros_like(okc)
    slots = np.arange(T, dtype=np.int64)
    oracle.append(k, v, slots, okc, ovc, scale_k, scale_v)
    dev = torch.device("cuda")
    if src == "bf16":
        kt = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).to(dev)
        vt = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        kt, vt = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)
    gkc = torch.full((nb, 1, HKV, D), 0x55, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
    gvc = torch.full((nb, 1, HKV, D), 0x55, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
    pkv_append(kt, vt, torch.from_numpy(slots.astype(np.int32)).to(dev), gkc, gvc, scale_k, scale_v)
    torch.cuda.synchronize()
    assert pkv_device_errors() == 0
    gk = gkc.view(torch.uint8).cpu().numpy()
    gv = gvc.view(torch.uint8).cpu().numpy()
    # slots past the rows are canaries: untouched
    assert (gk[T:] == 0x55).all() and (gv[T:] == 0x55).all()
    return gk[:T], gv[:T], okc[:T], ovc[:T]


def _assert_codes(g, o, x_nan, what):
    g, o = g.reshape(-1), o.reshape(-1)
    x_nan = x_nan.reshape(-1)
    assert _is_nan_code(o[x_nan]).all(), f"{what}: oracle gave a non-NaN code for NaN"
    assert _is_nan_code(g[x_nan]).all(), f"{what}: GPU gave a non-NaN code for NaN"
    fin = ~x_nan
    bad = np.nonzero(g[fin] != o[fin])[0]
    assert bad.size == 0, (f"{what}: {bad.size} codes differ, first at {np.nonzero(fin)[0][bad[0]]}: "
                           f"gpu 0x{g[fin][bad[0]]:02x} oracle 0x{o[fin][bad[0]]:02x}")


def _all_bf16_rows(perm_seed):
    """Every bf16 bit pattern once, laid out as rows [256, HKV, D]; V holds a
    seeded permutation of the same patterns."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    k = bits.reshape(-1, HKV, D)
    v = np.random.default_rng(perm_seed).permutation(bits).reshape(-1, HKV, D)
    return np.ascontiguousarray(k), np.ascontiguousarray(v)


def _bf16_nan(b):
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


# scales: exact (1), one that saturates everything above 1 (1/448), a
# dense-subnormal one (1000: |x| / 1000 < 2^-6 for |x| < 15.6), an inexact
# product (3.7), and the harness's usual kind, max |x| / 448 for |x| <= 4
SCALES = [1.0, 1.0 / 448.0, 1000.0, 3.7, 4.0 / 448.0]


@pytest.mark.parametrize("scale", SCALES)
def test_every_bf16_pattern_encodes_like_the_oracle(scale):
    k, v = _all_bf16_rows(7)
    gk, gv, ok, ov = _append_both(k, v, scale, scale * 0.5, "bf16")
    _assert_codes(gk, ok, _bf16_nan(k), f"K scale {scale}")
    _assert_codes(gv, ov, _bf16_nan(v), f"V scale {scale * 0.5}")
    # the cases this range is meant to reach really occur
    codes = ok.reshape(-1)[~_bf16_nan(k).reshape(-1)]
    assert (codes & 0x7F == 0x7E).any()  # +-448 (saturated or exact)
    if scale == 1000.0:
        assert ((codes & 0x78) == 0).mean() > 0.3  # dense subnormals and zeros


def _tie_values():
    """fp32 values at every midpoint between adjacent e4m3 magnitudes (and
    the midpoint between 448 and the next binade step), with the fp32
    neighbours on either side, both signs; plus zeros, infinities and NaN."""
    mags = np.array([oracle.e4m3_decode(np.array([c], np.uint8))[0] for c in range(0x7F)], np.float64)
    mids = (mags[:-1] + mags[1:]) / 2
    mids = np.concatenate([mids, [480.0, 464.0]])  # beyond the largest finite
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)  # every midpoint is an fp32 value
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(0))
    vals = np.concatenate([m32, up, dn])
    vals = np.concatenate([vals, -vals, np.array([0.0, -0.0, np.inf, -np.inf, np.nan, -np.nan,
                                                   np.float32(1e-30), np.float32(-1e-45)], np.float32)])
    return vals.astype(np.float32)


@pytest.mark.parametrize("scale", [1.0, 0.5, 3.7, 1000.0])
def test_f32_source_ties_and_specials(scale):
    vals = _tie_values()
    rng = np.random.default_rng(11)
    # pad to whole rows with random fp32 bit patterns (finite and not)
    per_row = HKV * D
    n_pad = (-vals.size) % per_row + 4 * per_row
    rand = rng.integers(0, 1 << 32, size=n_pad, dtype=np.uint64).astype(np.uint32).view(np.float32)
    k = np.concatenate([vals, rand]).reshape(-1, HKV, D)
    v = np.ascontiguousarray(k[::-1])
    gk, gv, ok, ov = _append_both(np.ascontiguousarray(k), v, scale, scale, "f32")
    _assert_codes(gk, ok, np.isnan(k), f"f32 K scale {scale}")
    _assert_codes(gv, ov, np.isnan(v), f"f32 V scale {scale}")


def test_f32_source_matches_bf16_source_on_bf16_values():
    """An f32 row holding bf16 values encodes to the same codes as the bf16
    row (the product is the same fp32 multiply)."""
    k, v = _all_bf16_rows(9)
    kf = W.bf16_bits_to_f32(k)
    vf = W.bf16_bits_to_f32(v)
    for scale in (1.0, 1.0 / 448.0, 1000.0):
        gk, gv, _, _ = _append_both(k, v, scale, scale, "bf16")
        fk, fv, _, _ = _append_both(np.ascontiguousarray(kf), np.ascontiguousarray(vf), scale, scale, "f32")
        nan_k, nan_v = _bf16_nan(k), _bf16_nan(v)
        assert np.array_equal(gk.reshape(-1)[~nan_k.reshape(-1)], fk.reshape(-1)[~nan_k.reshape(-1)])
        assert np.array_equal(gv.reshape(-1)[~nan_v.reshape(-1)], fv.reshape(-1)[~nan_v.reshape(-1)])


@pytest.mark.parametrize("shrink", [8.0, 64.0])
def test_attention_over_saturated_caches(shrink):
    """Scales well below max|X| / 448: a large share of the K and V codes
    saturate at +-448.  The caches must still equal the oracle's byte for
    byte, and attention must match the oracle run on the same codes."""
    wl = W.lognormal_fp8(B=10, median=600, sigma=0.8, cap=3000, seed=2207)
    wl.k_scale = float(np.float32(wl.k_scale / shrink))
    wl.v_scale = float(np.float32(wl.v_scale / shrink))
    ref, okc, ovc, _ = oracle.run_step(wl, nthreads=NT)
    sat = ((okc & 0x7F) == 0x7E).mean()
    assert sat > (0.2 if shrink == 8.0 else 0.6), sat
    ds, out = run_gpu(wl)
    assert oracle_caches_equal(ds, okc, ovc)
    check_attention(out, ref, "e4m3", f"saturated fp8 (scales / {shrink})")
