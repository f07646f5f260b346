"""Multi-step serving loop driven by the host block manager: requests with
shared system prompts arrive, prefill in chunks, decode, finish and free
their blocks; a small pool forces cached blocks to be evicted and reused.
Each step's slots and block tables come from the manager (and must equal the
GPU slot computation), the kernels append and attend, and every output row
is compared with the oracle run on each sequence's logical K/V.

A token's K/V are drawn from a generator seeded with the chained hash of the
tokens up to and including it, so two sequences with the same prefix have the
same K/V there -- the property that makes sharing cached blocks correct."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_mapping_gb300 import (PkvError, pkv_append, pkv_attention, pkv_device_errors,
                                          pkv_slot_mapping)
from paged_kv_cache_mapping_gb300.blocks import BlockManager
from paged_kv_cache_mapping_gb300.workloads import bf16_bits, bf16_bits_to_f32
from tests.gpu_util import TOL
from tests.helpers import rel_l2

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS, NB = 8, 2, 64, 16, 40
MASK = (1 << 64) - 1


def kv_of(tokens):
    """bf16 K and V bits [n, HKV, D] for a token sequence (content-chained)."""
    k = np.empty((len(tokens), HKV, D), np.uint16)
    v = np.empty_like(k)
    c = 1469598103934665603
    for i, t in enumerate(tokens):
        c = ((c ^ (int(t) + 0x9E3779B97F4A7C15)) * 1099511628211) & MASK
        g = np.random.default_rng(c)
        x = g.standard_normal((2, HKV, D), dtype=np.float32)
        k[i], v[i] = bf16_bits(x[0]), bf16_bits(x[1])
    return k, v


def test_block_manager_drives_the_kernels_through_churn():
    dev = torch.device("cuda")
    rng = np.random.default_rng(77)
    bm = BlockManager(NB, BS)
    kc = torch.zeros((NB, BS, HKV, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    systems = [rng.integers(0, 5000, 40), rng.integers(0, 5000, 40)]
    live = {}  # sid -> dict(tokens, done, prompt_len, gen, max_gen)
    next_id = 0
    scale = D ** -0.5
    max_blocks = 16
    rows_checked = 0
    for step in range(14):
        # admit up to two requests
        for _ in range(int(rng.integers(0, 3))):
            prompt = np.concatenate([systems[int(rng.integers(2))], rng.integers(0, 5000, int(rng.integers(5, 60)))])
            cached = bm.add_sequence(next_id, prompt)
            live[next_id] = dict(tokens=list(prompt), done=cached, prompt_len=len(prompt), gen=0,
                                 max_gen=int(rng.integers(2, 6)))
            next_id += 1
        if not live:
            continue
        # this step's tokens: a prefill chunk of at most 48 or one decode token
        while True:
            ids, n_new, toks = [], [], []
            for sid, s in live.items():
                if s["done"] < s["prompt_len"]:
                    n = min(48, s["prompt_len"] - s["done"])
                    new = s["tokens"][s["done"]:s["done"] + n]
                else:
                    new = [int(rng.integers(0, 5000))]
                ids.append(sid)
                n_new.append(len(new))
                toks += list(new)
            try:
                cu, sl, bt, slots = bm.build_step(ids, n_new, np.array(toks, np.int32), max_blocks)
                break
            except PkvError as e:  # pool full: the newest request gives its blocks back
                assert e.status == 6
                newest = max(live)
                bm.free_sequence(newest)
                del live[newest]
                if not live:
                    break
        if not live:
            continue
        for sid, n in zip(ids, n_new):  # record what was appended
            s = live[sid]
            if s["done"] < s["prompt_len"]:
                s["done"] += n
            else:
                s["tokens"].append(int(toks[int(cu[ids.index(sid)])]))
                s["done"] += 1
                s["gen"] += 1
        T = int(cu[-1])
        # this step's new K/V rows, from each sequence's logical content
        k_new = np.empty((T, HKV, D), np.uint16)
        v_new = np.empty_like(k_new)
        logical = {}
        for b, sid in enumerate(ids):
            kk, vv = kv_of(live[sid]["tokens"][:int(sl[b])])
            logical[sid] = (kk, vv)
            k_new[cu[b]:cu[b + 1]] = kk[int(sl[b]) - n_new[b]:]
            v_new[cu[b]:cu[b + 1]] = vv[int(sl[b]) - n_new[b]:]
        to_dev = lambda a, dt=torch.int32: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
        cu_t, sl_t, bt_t, slots_t = to_dev(cu), to_dev(sl), to_dev(bt), to_dev(slots)
        assert torch.equal(pkv_slot_mapping(cu_t, sl_t, bt_t, BS, T=T), slots_t)
        k_t = torch.from_numpy(k_new.view(np.int16)).to(dev).view(torch.bfloat16)
        v_t = torch.from_numpy(v_new.view(np.int16)).to(dev).view(torch.bfloat16)
        pkv_append(k_t, v_t, slots_t, kc, vc)
        q = bf16_bits(rng.standard_normal((T, HQ, D), dtype=np.float32))
        q_t = torch.from_numpy(q.view(np.int16)).to(dev).view(torch.bfloat16)
        out = torch.empty((T, HQ, D), dtype=torch.float32, device=dev)
        pkv_attention(q_t, cu_t, sl_t, bt_t, kc, vc, scale, out, max_q_len=int(max(n_new)))
        torch.cuda.synchronize()
        assert pkv_device_errors() == 0
        # oracle on contiguous logical caches (one block run per sequence)
        nb = [-(-int(n) // BS) for n in sl]
        okc = np.zeros((sum(nb), BS, HKV, D), np.uint16)
        ovc = np.zeros_like(okc)
        obt = np.full((len(ids), max(nb)), -1, np.int32)
        base = 0
        for b, sid in enumerate(ids):
            kk, vv = logical[sid]
            n = int(sl[b])
            okc.reshape(-1, HKV, D)[base * BS:base * BS + n] = kk
            ovc.reshape(-1, HKV, D)[base * BS:base * BS + n] = vv
            obt[b, :nb[b]] = np.arange(base, base + nb[b])
            base += nb[b]
        ref = oracle.attention(q, cu, sl, obt, okc, ovc, scale, nthreads=oracle.cpu_count())
        got = out.cpu().numpy().astype(np.float64)
        tol_abs, tol_rel = TOL["bf16"]
        err = float(np.abs(got - ref).max())
        assert err <= tol_abs and rel_l2(got, ref) <= tol_rel, f"step {step}: max |err| {err:.3e}"
        rows_checked += T
        # finish
        for sid in [sid for sid, s in live.items() if s["gen"] >= s["max_gen"]]:
            bm.free_sequence(sid)
            del live[sid]
    st = bm.stats()
    assert rows_checked > 300
    assert st["prefix_hit_blocks"] > 0, st
    assert st["evictions"] > 0, st
