"""Logits soft cap and sliding window (pkv_attention_ex) against the oracle
with the same variant: decode rows (bf16 and e4m3, split across chunks, the
window cutting into the first chunk) and tensor-core prefill rows (bf16 and
e4m3 caches)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_mapping_gb300 import PkvError
from paged_kv_cache_mapping_gb300 import workloads as W
from tests.gpu_util import TOL, check_attention, run_gpu

pytestmark = pytest.mark.gpu

NT = oracle.cpu_count()


def _decode():
    return W.qwen3_4b_decode(B=12, ctx=(1, 2600), block_size=16, num_blocks=0, seed=2401)


def _fp8():
    return W.lognormal_fp8(B=20, median=700, sigma=1.0, cap=6000, seed=2402)


def _mixed():
    return W.mixed_prefill(n_decode=5, dec_ctx=(300, 1400), chunk=200, prefix=160, block_size=16,
                           num_blocks=1024, seed=2403)


def _mixed_fp8():
    return W.mixed_prefill(n_decode=5, dec_ctx=(300, 1400), chunk=200, prefix=160, block_size=16,
                           num_blocks=1024, seed=2406, kv="e4m3")


def _fp8_pf_d64():
    return W.build("fp8 pf", Hq=16, Hkv=4, D=64, block_size=8, seq_lens=[300, 77, 1, 900],
                   q_lens=[120, 77, 1, 1], src="bf16", kv="e4m3", seed=2405, pool_slack=0.1)


def _g16():
    return W.build("g16", Hq=64, Hkv=4, D=128, block_size=32, seq_lens=[1, 90, 700, 1500],
                   q_lens=[1, 1, 130, 1], src="bf16", kv="bf16", seed=2404, pool_slack=0.1)


def _g32_decode():
    # one KV head for 32 query heads: decode rows too wide for the decode
    # kernel's head columns take the tensor-core prefill
    return W.build("g32", Hq=32, Hkv=1, D=128, block_size=16, seq_lens=[1, 90, 700, 1500],
                   q_lens=[1, 1, 1, 1], src="bf16", kv="bf16", seed=2407, pool_slack=0.1)


@pytest.mark.parametrize("make,cap,window", [
    (_decode, 0.0, 300), (_decode, 20.0, -1), (_decode, 5.0, 1000), (_decode, 0.0, 0),
    (_fp8, 30.0, 500), (_fp8, 0.0, 129),
    (_mixed, 15.0, 200), (_mixed, 0.0, 64), (_mixed, 3.0, -1),
    (_g16, 0.0, 100), (_g32_decode, 10.0, 300),
    (_mixed_fp8, 15.0, 200), (_mixed_fp8, 0.0, 64), (_fp8_pf_d64, 10.0, -1)],
    ids=["dec-w300", "dec-cap20", "dec-cap5-w1000", "dec-w0", "fp8-cap30-w500", "fp8-w129",
         "mixed-cap15-w200", "mixed-w64", "mixed-cap3", "g16-w100", "g32-dec-cap10-w300",
         "mixed-fp8-cap15-w200", "mixed-fp8-w64", "fp8-pf-d64-cap10"])
def test_variant_matches_oracle(make, cap, window):
    wl = make()
    ref = oracle.run_step(wl, nthreads=NT, soft_cap=cap, window_left=window)[0]
    _, out = run_gpu(wl, soft_cap=cap, window_left=window)
    check_attention(out, ref, wl.kv, f"cap {cap} window {window}")


def test_variants_off_equal_plain_bitwise():
    wl = _mixed()
    _, a = run_gpu(wl)
    _, b = run_gpu(wl, soft_cap=0.0, window_left=10 ** 7)
    assert torch.equal(a, b)


def test_variants_outside_the_built_paths_are_refused():
    with pytest.raises(PkvError) as e:
        run_gpu(W.tiny(), window_left=3)  # fp32
    assert e.value.status == 2
    # prefill rows on a block size that is not a multiple of 8 (the mma.sync kernel)
    bs4_prefill = W.build("bs4 pf", Hq=16, Hkv=4, D=64, block_size=4, seq_lens=[300, 77], q_lens=[120, 77],
                          src="bf16", kv="e4m3", seed=2405, pool_slack=0.1)
    with pytest.raises(PkvError) as e:
        run_gpu(bs4_prefill, soft_cap=10.0)
    assert e.value.status == 2
    # a query group wider than a tensor-core tile (G 256) also takes the mma.sync kernel
    g256 = W.build("g256", Hq=256, Hkv=1, D=64, block_size=16, seq_lens=[300, 77], q_lens=[1, 1],
                   src="bf16", kv="bf16", seed=2408, pool_slack=0.1)
    with pytest.raises(PkvError) as e:
        run_gpu(g256, window_left=50)
    assert e.value.status == 2
