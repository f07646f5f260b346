"""Full-size workloads, in the launch configuration the benchmark times,
against the oracle.

Slots and the whole caches are compared bit for bit (the oracle replays the
full-size append); attention is compared on a seeded sample of (token, head)
rows that the oracle computes one by one, always including the first and
last rows of the shortest and the longest sequence and, for prefill chunks,
their first and last query tokens.  Outputs across the page layouts are
compared bitwise on the whole tensor."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_mapping_gb300 import pkv_device_errors
from paged_kv_cache_mapping_gb300 import workloads as W
from paged_kv_cache_mapping_gb300.harness import DeviceStep, cache_to_numpy
from tests.gpu_util import TOL
from tests.helpers import rel_l2

pytestmark = pytest.mark.gpu

NT = oracle.cpu_count()
N_SAMPLE = 160


def sample_rows(wl, seed):
    g = np.random.default_rng(seed)
    cu = wl.cu_seqlens_q
    live = [s for s in range(wl.B) if wl.q_lens[s] > 0]
    lens = wl.seq_lens
    picks = set()
    for s in (min(live, key=lambda s: lens[s]), max(live, key=lambda s: lens[s])):
        for t in (int(cu[s]), int(cu[s + 1]) - 1):
            for h in (0, wl.Hq - 1):
                picks.add((t, h))
    for s in live:  # both ends of every prefill chunk
        if wl.q_lens[s] > 1:
            for t in (int(cu[s]), int(cu[s]) + 1, int(cu[s + 1]) - 1):
                picks.add((t, int(g.integers(wl.Hq))))
    while len(picks) < N_SAMPLE:
        picks.add((int(g.integers(wl.T)), int(g.integers(wl.Hq))))
    t, h = zip(*sorted(picks))
    return np.array(t, np.int64), np.array(h, np.int32)


def bench_step(wl, out_dtype):
    """The benchmark's configuration: 4 layer caches, max_q_len from the batch."""
    ds = DeviceStep(wl, out_dtype=out_dtype, layers=4, max_q_len=int(wl.q_lens.max()))
    out = ds.step(layer=1).clone()
    torch.cuda.synchronize()
    assert pkv_device_errors() == 0
    return ds, out


FULL = {
    "qwen3_4b_decode_b64": lambda: W.qwen3_4b_decode(),
    "mixed_prefill": lambda: W.mixed_prefill(),
    "mixed_prefill_fp8": lambda: W.mixed_prefill(kv="e4m3"),
    "long_fp8_b8": lambda: W.long_fp8(),
    "lognormal_fp8_b256": lambda: W.lognormal_fp8(),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_against_oracle(name):
    wl = FULL[name]()
    t, h = sample_rows(wl, seed=7000 + len(name))
    ref, okc, ovc, oslots = oracle.run_step(wl, nthreads=NT, rows=(t, h))
    ds, out_bf16 = bench_step(wl, torch.bfloat16)
    # slots and caches, bit for bit (layer 1 received the same appends as layer 0)
    assert np.array_equal(ds.slots.cpu().numpy().astype(np.int64), oslots.astype(np.int64))
    kc, vc = ds.caches[1]
    assert np.array_equal(cache_to_numpy(kc).view(np.uint8), okc.view(np.uint8)), "k cache differs"
    assert np.array_equal(cache_to_numpy(vc).view(np.uint8), ovc.view(np.uint8)), "v cache differs"
    # f32 output on the same caches; bf16 output is its round-to-nearest-even
    out_f32 = torch.empty(ds.out.shape, dtype=torch.float32, device=ds.out.device)
    ds.attention_only(layer=1, out=out_f32)
    torch.cuda.synchronize()
    assert torch.equal(out_f32.to(torch.bfloat16), out_bf16), "bf16 output is not the rounded f32 output"
    got = out_f32[torch.from_numpy(t).cuda(), torch.from_numpy(h.astype(np.int64)).cuda()]
    got = got.cpu().numpy().astype(np.float64)
    tol_abs, tol_rel = TOL[wl.kv]
    err = float(np.abs(got - ref).max())
    rel = rel_l2(got, ref)
    assert np.isfinite(got).all()
    assert err <= tol_abs and rel <= tol_rel, f"{name}: max |err| {err:.3e}, rel L2 {rel:.3e}"


def test_layout_sweep_full_size_bitwise_and_sampled():
    outs = {}
    ref = None
    for bs in (1, 16, 64):
        for contiguous in (False, True):
            wl = W.layout_sweep(bs, contiguous)
            ds = DeviceStep(wl, out_dtype=torch.float32, layers=1, max_q_len=1)
            o = ds.step().cpu()
            assert pkv_device_errors() == 0
            outs[(bs, contiguous)] = o
            if ref is None:  # the logical K/V are the same in every layout
                t, h = sample_rows(wl, seed=7100)
                ref = oracle.run_step(wl, nthreads=NT, rows=(t, h))[0]
                got = o[torch.from_numpy(t), torch.from_numpy(h.astype(np.int64))].numpy().astype(np.float64)
                tol_abs, tol_rel = TOL["bf16"]
                assert float(np.abs(got - ref).max()) <= tol_abs and rel_l2(got, ref) <= tol_rel
            del ds
            torch.cuda.empty_cache()
    first = outs[(1, False)]
    for key, o in outs.items():
        assert torch.equal(o, first), f"layout {key} differs from bs 1 scattered"
