"""The device plan at and past its one-warp-per-sequence limit (512
sequences): batches of 512, 513 and 700 sequences, most of them decoding
(split into several chunks, so merges run) and a few prefilling, against the
oracle row by row; and the same rows give the same bits whatever batch they
sit in, so the two ways of writing the work lists agree."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_mapping_gb300 import workloads as W
from tests.gpu_util import check_attention, run_gpu

pytestmark = pytest.mark.gpu

NT = oracle.cpu_count()


def batch(B, seed):
    g = np.random.default_rng(seed)
    lens = g.integers(1, 400, size=B).astype(np.int32)
    q = np.ones(B, np.int32)
    for i in (3, B // 2, B - 1):  # a few prefill rows
        q[i] = int(min(lens[i], 20))
    return W.build(f"plan B{B}", Hq=8, Hkv=2, D=64, block_size=16, seq_lens=lens, q_lens=q,
                   src="bf16", kv="bf16", seed=seed, pool_slack=0.1)


@pytest.mark.parametrize("B", [512, 513, 700])
def test_plan_limits_against_the_oracle(B):
    wl = batch(B, 3000 + B)
    ref = oracle.run_step(wl, nthreads=NT)[0]
    _, out = run_gpu(wl)
    check_attention(out, ref, "bf16", f"B{B}")


def test_rows_do_not_depend_on_the_plan_path():
    """The first 300 sequences of a 700-sequence batch (per-thread lists)
    and the same 300 alone (per-warp lists) give bitwise equal rows."""
    big = batch(700, 3700)
    n = 300
    _, out_big = run_gpu(big)
    out_big = out_big.clone()
    _, out_small = run_gpu(big.select(list(range(n))))
    t = int(np.sum(big.q_lens[:n]))
    assert torch.equal(out_big[:t], out_small)
