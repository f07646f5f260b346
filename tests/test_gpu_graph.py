"""A whole step (slot mapping, append, attention) captured into a CUDA graph
and replayed gives the same bits as the step run eagerly: every launch of the
path, including the programmatic-dependent-launch edges and the tensor-core
prefill's tensor maps, survives capture.  The first, eager call on a device
does the one-time set-up (symbol addresses, shared-memory limits) outside the
capture."""
import pytest
import torch

from paged_kv_cache_mapping_gb300 import pkv_device_errors
from paged_kv_cache_mapping_gb300 import workloads as W
from paged_kv_cache_mapping_gb300.harness import DeviceStep

pytestmark = pytest.mark.gpu


def _decode():
    return W.qwen3_4b_decode(B=12, ctx=(1, 2600), block_size=16, num_blocks=0, seed=2201)


def _mixed():
    return W.mixed_prefill(n_decode=5, dec_ctx=(300, 1400), chunk=200, prefix=160, block_size=16,
                           num_blocks=1024, seed=2202)


def _fp8():
    return W.lognormal_fp8(B=24, median=700, sigma=1.0, cap=6000, seed=2203)


@pytest.mark.parametrize("make", [_decode, _mixed, _fp8], ids=["decode", "mixed", "fp8"])
def test_graph_replay_matches_eager(make):
    ds = DeviceStep(make(), out_dtype=torch.bfloat16)
    eager = ds.step().clone()
    torch.cuda.synchronize()
    assert pkv_device_errors() == 0
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # one more eager step on the capture stream
        ds.step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ds.step()
    for _ in range(3):
        ds.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(ds.out, eager)
    assert pkv_device_errors() == 0
