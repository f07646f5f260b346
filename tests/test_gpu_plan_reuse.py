"""One plan per model step, one run per layer ("How Easy Is It to Start
Serving LLMs?", "3. Load balancing: keep every SM busy": the plan is made
once from the lengths, kept in a fixed GPU buffer and reused by every
layer).  Each run over a reused plan must give the bits pkv_attention (plan
+ run) gives on the same inputs; a run on a workspace planned for other
shapes must do nothing and say so."""
import numpy as np
import pytest
import torch

from paged_kv_cache_mapping_gb300 import (pkv_append, pkv_attention, pkv_attention_plan, pkv_attention_run,
                                          pkv_device_errors, pkv_slot_mapping)
from paged_kv_cache_mapping_gb300 import workloads as W
from paged_kv_cache_mapping_gb300.harness import DeviceStep

pytestmark = pytest.mark.gpu

LAYERS = 5


def _decode():
    return W.qwen3_4b_decode(B=12, ctx=(1, 2600), block_size=16, num_blocks=0, seed=2401)


def _mixed_tc():
    return W.mixed_prefill(n_decode=5, dec_ctx=(300, 1400), chunk=200, prefix=160, block_size=16,
                           num_blocks=1024, seed=2402)


def _mixed_bs8():  # block size 8: the tensor-core prefill with boxes of 8 slots
    return W.build("mixed bs8", Hq=32, Hkv=8, D=128, block_size=8, seq_lens=[700, 130, 1, 300],
                   q_lens=[1, 130, 1, 45], src="bf16", kv="bf16", seed=2403, pool_slack=0.1)


def _mixed_bs4():  # block size 4: the mma.sync prefill kernel
    return W.build("mixed bs4", Hq=32, Hkv=8, D=128, block_size=4, seq_lens=[700, 130, 1, 300],
                   q_lens=[1, 130, 1, 45], src="bf16", kv="bf16", seed=2407, pool_slack=0.1)


def _mixed_fp8():  # e4m3 caches: the tensor-core prefill on f16-converted tiles
    return W.mixed_prefill(n_decode=5, dec_ctx=(300, 1400), chunk=200, prefix=160, block_size=16,
                           num_blocks=1024, seed=2408, kv="e4m3")


def _fp8():
    return W.lognormal_fp8(B=24, median=700, sigma=1.0, cap=6000, seed=2404)


CASES = {"decode": (_decode, {}), "mixed_tc": (_mixed_tc, {}), "mixed_bs8": (_mixed_bs8, {}),
         "mixed_mma": (_mixed_bs4, {}), "fp8": (_fp8, {}), "mixed_fp8": (_mixed_fp8, {}),
         "decode_window": (_decode, {"window_left": 300}),
         "mixed_tc_window": (_mixed_tc, {"window_left": 100}),
         "mixed_fp8_window": (_mixed_fp8, {"window_left": 100})}


def _layer_inputs(ds, layers, seed):
    """Per layer: new K/V rows and a query that differ from layer to layer."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    out = []
    for _ in range(layers):
        def rnd(t):
            return torch.randn(t.shape, generator=g).to(t.dtype).to(t.device)
        out.append((rnd(ds.q), rnd(ds.k_new), rnd(ds.v_new)))
    return out


@pytest.mark.parametrize("name", list(CASES))
def test_runs_over_one_plan_equal_the_full_call(name):
    make, kw = CASES[name]
    wl = make()
    ds = DeviceStep(wl, layers=LAYERS, **kw)
    ref_ws = torch.empty_like(ds.ws)
    inputs = _layer_inputs(ds, LAYERS, 77)
    # the soft cap may change from layer to layer (not on the mma.sync prefill path)
    caps = [0.0] * LAYERS if name == "mixed_mma" else [0.0, 30.0, 0.0, 5.0, 0.0]
    # the per-step part once, then append + run per layer
    pkv_slot_mapping(ds.cu_q, ds.seq_lens, ds.bt, wl.block_size, out=ds.slots)
    ds.plan()
    runs = []
    for layer, (q, k, v) in enumerate(inputs):
        kc, vc = ds.caches[layer]
        pkv_append(k, v, ds.slots, kc, vc, wl.k_scale, wl.v_scale)
        o = torch.full_like(ds.out, float("nan"))
        pkv_attention_run(q, ds.cu_q, ds.seq_lens, ds.bt, kc, vc, wl.scale, o, ds.ws, wl.k_scale, wl.v_scale,
                          ds.max_q_len, soft_cap=caps[layer], window_left=ds.window_left)
        runs.append(o)
    torch.cuda.synchronize()
    assert pkv_device_errors() == 0
    # the same layers through the full call, each on its own
    for layer, (q, k, v) in enumerate(inputs):
        kc, vc = ds.caches[layer]
        o = torch.full_like(ds.out, float("nan"))
        pkv_attention(q, ds.cu_q, ds.seq_lens, ds.bt, kc, vc, wl.scale, o, wl.k_scale, wl.v_scale, ds.max_q_len,
                      ref_ws, soft_cap=caps[layer], window_left=ds.window_left)
        torch.cuda.synchronize()
        assert torch.isfinite(o).all()
        assert torch.equal(runs[layer], o), f"{name}: layer {layer} differs from pkv_attention"
    assert pkv_device_errors() == 0


def test_a_run_without_a_matching_plan_does_nothing_and_is_recorded():
    a = DeviceStep(_decode())
    b = DeviceStep(W.qwen3_4b_decode(B=5, ctx=(1, 2600), block_size=16, num_blocks=0, seed=2405))
    # a's workspace is large enough for b's shapes; plan a, then run b on it
    assert a.ws.numel() >= b.ws.numel()
    a.step()
    a.plan()
    torch.cuda.synchronize()
    assert pkv_device_errors() == 0
    o = torch.full_like(b.out, float("nan"))
    kc, vc = b.caches[0]
    pkv_attention_run(b.q, b.cu_q, b.seq_lens, b.bt, kc, vc, b.wl.scale, o, a.ws, max_q_len=1)
    assert pkv_device_errors() == 16
    assert torch.isnan(o).all()
    # the mixed kernels check too: a decode plan run as a prefill batch
    m = DeviceStep(_mixed_tc())
    expected = m.step().clone()  # the step's rows appended, then the full call
    ws = torch.empty(max(m.ws.numel(), a.ws.numel()), dtype=torch.uint8, device="cuda")
    pkv_attention_plan(a.q, a.cu_q, a.seq_lens, a.bt, a.caches[0][0], ws, max_q_len=1)
    o = torch.full_like(m.out, float("nan"))
    pkv_attention_run(m.q, m.cu_q, m.seq_lens, m.bt, *m.caches[0], m.wl.scale, o, ws, max_q_len=m.max_q_len)
    assert pkv_device_errors() == 16
    assert torch.isnan(o).all()
    # a fresh plan makes the workspace usable again
    pkv_attention_plan(m.q, m.cu_q, m.seq_lens, m.bt, m.caches[0][0], ws, max_q_len=m.max_q_len)
    pkv_attention_run(m.q, m.cu_q, m.seq_lens, m.bt, *m.caches[0], m.wl.scale, o, ws, max_q_len=m.max_q_len)
    torch.cuda.synchronize()
    assert pkv_device_errors() == 0
    assert torch.equal(o, expected)


def test_plan_and_layer_runs_replay_from_a_cuda_graph():
    ds = DeviceStep(_mixed_tc(), layers=3, out_dtype=torch.bfloat16)
    outs = [torch.empty_like(ds.out) for _ in range(3)]

    def model_step():
        ds.model_step_start()
        for layer in range(3):
            ds.layer_step(layer, outs[layer])

    model_step()
    eager = [o.clone() for o in outs]
    torch.cuda.synchronize()
    assert pkv_device_errors() == 0
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        model_step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        model_step()
    for _ in range(3):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for o, e in zip(outs, eager):
            assert torch.equal(o, e)
    assert pkv_device_errors() == 0


def test_many_runs_keep_the_plan():
    """Forty runs in a row over one plan (more than a model's layers): the
    counters each run resets stay consistent."""
    ds = DeviceStep(_decode(), layers=2)
    ds.step(1)
    first = ds.step(0).clone()
    ds.plan()
    for i in range(40):
        ds.run(i % 2)
    torch.cuda.synchronize()
    assert pkv_device_errors() == 0
    assert torch.equal(ds.out, first)
    assert np.isfinite(ds.out.float().cpu().numpy()).all()
