"""CUDA path (through the C ABI) against the CPU oracle, element by element,
on seeded inputs small enough for the oracle, spanning several tiles,
split-KV chunks and ragged tails."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_mapping_gb300 import (PkvError, pkv_attention, pkv_csr_to_block_tables, pkv_device_errors,
                                          pkv_slot_mapping)
from paged_kv_cache_mapping_gb300 import workloads as W
from paged_kv_cache_mapping_gb300.harness import DeviceStep, cache_to_numpy
from tests.gpu_util import bf16_rne_of, check_attention, oracle_caches_equal, run_gpu

pytestmark = pytest.mark.gpu

NT = oracle.cpu_count()


def small_decode(seed=2002, B=12, ctx=(1, 2600), bs=16):
    return W.qwen3_4b_decode(B=B, ctx=ctx, block_size=bs, num_blocks=0, seed=seed)


def small_mixed(seed=2004):
    return W.mixed_prefill(n_decode=5, dec_ctx=(300, 1400), chunk=200, prefix=160, block_size=16,
                           num_blocks=1024, seed=seed)


def small_fp8(seed=2005):
    return W.long_fp8(B=3, ctx=(5000, 21000), seed=seed)


def small_lognormal(seed=2006):
    return W.lognormal_fp8(B=24, median=700, sigma=1.0, cap=6000, seed=seed)


CASES = {
    "tiny_fp32": W.tiny,
    "decode_bf16": small_decode,
    "decode_bf16_bs1": lambda: small_decode(seed=2012, B=5, ctx=(1, 1300), bs=1),
    "decode_bf16_bs7": lambda: small_decode(seed=2013, B=5, ctx=(1, 1300), bs=7),
    "mixed_bf16": small_mixed,
    "long_fp8": small_fp8,
    "lognormal_fp8": small_lognormal,
}


@pytest.fixture(scope="module")
def computed():
    cache = {}

    def get(name):
        if name not in cache:
            wl = CASES[name]()
            ref, okc, ovc, oslots = oracle.run_step(wl, nthreads=NT)
            ds, out = run_gpu(wl)
            cache[name] = (wl, ref, okc, ovc, oslots, ds, out.clone())
        return cache[name]
    return get


@pytest.mark.parametrize("name", list(CASES))
def test_slot_mapping_bitexact(computed, name):
    wl, ref, okc, ovc, oslots, ds, out = computed(name)
    assert np.array_equal(ds.slots.cpu().numpy().astype(np.int64), oslots)
    s64 = torch.empty(wl.T, dtype=torch.int64, device="cuda")
    pkv_slot_mapping(ds.cu_q, ds.seq_lens, ds.bt, wl.block_size, out=s64)
    assert np.array_equal(s64.cpu().numpy(), oslots)
    assert pkv_device_errors() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_append_caches_bitexact(computed, name):
    wl, ref, okc, ovc, oslots, ds, out = computed(name)
    assert oracle_caches_equal(ds, okc, ovc), "cache bytes differ from the oracle's"


@pytest.mark.parametrize("name", list(CASES))
def test_attention_matches_oracle(computed, name):
    wl, ref, okc, ovc, oslots, ds, out = computed(name)
    check_attention(out, ref, wl.kv, name)


@pytest.mark.parametrize("name", ["decode_bf16", "mixed_bf16", "long_fp8", "tiny_fp32"])
def test_bf16_output_is_rounded_f32_output(computed, name):
    wl, ref, okc, ovc, oslots, ds, out = computed(name)
    ob = torch.empty(out.shape, dtype=torch.bfloat16, device="cuda")
    ds.attention_only(out=ob)
    torch.cuda.synchronize()
    assert torch.equal(ob.view(torch.int16), bf16_rne_of(out).view(torch.int16))
    # bf16 output against the oracle: |err| <= tol + 2^-8 |ref|
    g = ob.float().cpu().numpy()
    tol = {"bf16": 2e-3, "e4m3": 1e-2, "f32": 1e-5}[wl.kv]
    assert (np.abs(g - ref) <= tol + 2.0 ** -8 * np.abs(ref)).all()


def test_decode_multi_chunk_covered(computed):
    wl = computed("decode_bf16")[0]
    assert (wl.seq_lens > 512).sum() >= 3 and (wl.seq_lens % 64 != 0).all()
    wl = computed("long_fp8")[0]
    assert (wl.seq_lens > 4096).all()


def test_repeat_is_deterministic(computed):
    wl, ref, okc, ovc, oslots, ds, out = computed("decode_bf16")
    o2 = ds.step().clone()
    torch.cuda.synchronize()
    assert torch.equal(o2, out)


def test_layout_invariance_bitwise():
    """Block size 1, 16, 64 with scattered and contiguous tables: identical
    bits (all tiling is in logical tokens)."""
    outs = []
    ref = None
    for bs in (1, 16, 64):
        for contiguous in (False, True):
            wl = W.layout_sweep(bs, contiguous, B=4, ctx=777, seed=2003)
            ds, out = run_gpu(wl)
            outs.append(out.clone())
            if ref is None:
                ref = oracle.run_step(wl, nthreads=NT)[0]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    check_attention(outs[0], ref, "bf16", "layout")


def test_batch_composition_invariance_bitwise():
    both = W.build("pair", Hq=32, Hkv=8, D=128, block_size=16, seq_lens=[700, 5000, 33],
                   q_lens=[1, 1, 5], src="bf16", kv="bf16", seed=2007, pool_slack=0.2)
    _, o_all = run_gpu(both)
    o_all = o_all.clone()
    for sel, rows in (([0], slice(0, 1)), ([2], slice(2, 7)), ([2, 1, 0], None)):
        sub = both.select(sel)
        _, o = run_gpu(sub)
        if rows is not None:
            assert torch.equal(o, o_all[rows])
        else:
            assert torch.equal(o[0:5], o_all[2:7])
            assert torch.equal(o[5:6], o_all[1:2])
            assert torch.equal(o[6:7], o_all[0:1])


@pytest.mark.parametrize("Hq,Hkv,D,kv", [(8, 8, 128, "bf16"), (16, 2, 64, "bf16"), (32, 2, 128, "bf16"),
                                         (12, 4, 64, "bf16"), (32, 16, 128, "bf16"), (32, 16, 128, "e4m3"),
                                         (48, 16, 64, "e4m3"), (12, 3, 64, "e4m3"), (8, 1, 64, "e4m3"),
                                         (20, 5, 128, "e4m3")])
def test_head_shapes(Hq, Hkv, D, kv):
    """G = 1, 8, 16 (the latter through the tile path), 3; D = 64; 16 KV
    heads, where a decode item covers 8 of them, so a token pair's rows are
    not one contiguous run and go as two copies; and e4m3 items of 3, 1 and 5
    KV heads (at D = 64 the two rows of a pair then sit 64 bytes off a
    128-byte multiple apart and the MMA rows keep their unrotated order)."""
    wl = W.build("heads", Hq=Hq, Hkv=Hkv, D=D, block_size=16, seq_lens=[1, 90, 600, 1500],
                 q_lens=[1, 1, 3, 1], src="bf16", kv=kv, seed=2008, pool_slack=0.1)
    ref = oracle.run_step(wl, nthreads=NT)[0]
    _, out = run_gpu(wl)
    check_attention(out, ref, kv, f"Hq{Hq} Hkv{Hkv} D{D} {kv}")


@pytest.mark.parametrize("Hq,Hkv,D,kv,bs,q_lens", [
    (32, 1, 128, "bf16", 16, [1, 1, 1, 1, 1]),     # G 32, decode rows only: tensor-core prefill, 4 tokens a tile
    (32, 1, 128, "bf16", 16, [1, 1, 3, 1, 130]),
    (128, 1, 64, "bf16", 16, [1, 1, 3, 1, 130]),   # G 128: one token a tile
    (40, 2, 64, "e4m3", 16, [1, 1, 3, 1, 130]),    # G 20: 6 tokens, 120 of 128 rows
    (96, 1, 64, "e4m3", 8, [1, 1, 3, 1, 130]),     # G 96: one token, 96 rows, boxes of 8 slots
    (256, 1, 64, "bf16", 16, [1, 1, 3, 1, 130]),   # G 256: beyond a tile, the mma.sync prefill
    (20, 4, 128, "bf16", 16, [1, 1, 1, 1, 1]),     # G 5 and 7: decode kernel, head columns 5-7 idle
    (28, 4, 128, "e4m3", 16, [1, 1, 1, 1, 1]),
])
def test_wide_query_groups(Hq, Hkv, D, kv, bs, q_lens):
    """Query groups wider than the decode kernel's eight head columns (the
    rows of a sequence are its tokens times the group, as for a prefill
    chunk), up to and past the 128 rows of a tensor-core tile, and groups
    that fill only part of the decode kernel's columns."""
    wl = W.build("wide groups", Hq=Hq, Hkv=Hkv, D=D, block_size=bs, seq_lens=[1, 90, 600, 1500, 300],
                 q_lens=q_lens, src="bf16", kv=kv, seed=2015, pool_slack=0.1)
    ref, okc, ovc, _ = oracle.run_step(wl, nthreads=NT)
    ds, out = run_gpu(wl)
    assert oracle_caches_equal(ds, okc, ovc)
    check_attention(out, ref, kv, f"Hq{Hq} Hkv{Hkv} D{D} {kv} bs{bs} q{q_lens}")
    out16 = torch.empty(out.shape, dtype=torch.bfloat16, device=out.device)
    ds.attention_only(out=out16)
    torch.cuda.synchronize()
    assert torch.equal(out16, bf16_rne_of(out))
    assert pkv_device_errors() == 0


# Prefill through the tensor-core (tcgen05) kernel: bf16 caches with block
# sizes that are multiples of 16.  Chunks with and without a cached prefix,
# token counts that are not multiples of a tile, a decode in the same batch.
@pytest.mark.parametrize("Hq,Hkv,D,bs", [(32, 8, 128, 16), (32, 8, 64, 32), (8, 8, 128, 64), (64, 8, 128, 16),
                                         (48, 3, 64, 16), (12, 4, 128, 48)])
def test_tensor_core_prefill_shapes(Hq, Hkv, D, bs):
    wl = W.build("tc prefill", Hq=Hq, Hkv=Hkv, D=D, block_size=bs, seq_lens=[700, 130, 1, 300, 64],
                 q_lens=[129, 130, 1, 45, 64], src="bf16", kv="bf16", seed=2010, pool_slack=0.1)
    ref = oracle.run_step(wl, nthreads=NT)[0]
    ds, out = run_gpu(wl)
    check_attention(out, ref, "bf16", f"tc prefill Hq{Hq} Hkv{Hkv} D{D} bs{bs}")
    out16 = torch.empty(out.shape, dtype=torch.bfloat16, device=out.device)
    ds.attention_only(out=out16)
    torch.cuda.synchronize()
    assert torch.equal(out16, bf16_rne_of(out))


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_tensor_core_prefill_layout_invariance_bitwise(kv):
    """Block sizes 8 and 24 take boxes of 8 slots, the others boxes of 16:
    the tiles and their arithmetic are the same in every layout."""
    outs = []
    for bs in (8, 16, 24, 32, 64):
        for contiguous in (False, True):
            wl = W.build("tc layout", Hq=32, Hkv=8, D=128, block_size=bs, seq_lens=[900, 333, 1],
                         q_lens=[300, 333, 1], src="bf16", kv=kv, seed=2011, contiguous=contiguous,
                         pool_slack=0.2)
            outs.append(run_gpu(wl)[1].cpu())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


# Prefill rows on e4m3 caches and on block sizes that are 8 mod 16 go
# through the tensor-core kernel too (codes converted to f16 in shared
# memory, boxes of 8 slots); block sizes that are not multiples of 8 keep the
# mma.sync kernel.  G 4, 4, 3, 8, 4, 3, 4, 4.
@pytest.mark.parametrize("kv,Hq,Hkv,D,bs", [("e4m3", 32, 8, 128, 16), ("e4m3", 16, 4, 64, 8),
                                            ("e4m3", 12, 4, 128, 24), ("e4m3", 64, 8, 64, 32),
                                            ("bf16", 32, 8, 128, 8), ("bf16", 12, 4, 64, 24),
                                            ("bf16", 32, 8, 128, 4), ("e4m3", 16, 4, 128, 12)])
def test_prefill_cache_formats_and_block_sizes(kv, Hq, Hkv, D, bs):
    wl = W.build("pf formats", Hq=Hq, Hkv=Hkv, D=D, block_size=bs, seq_lens=[700, 130, 1, 300, 64],
                 q_lens=[129, 130, 1, 45, 64], src="bf16", kv=kv, seed=2014, pool_slack=0.1)
    ref, okc, ovc, _ = oracle.run_step(wl, nthreads=NT)
    ds, out = run_gpu(wl)
    assert oracle_caches_equal(ds, okc, ovc)
    check_attention(out, ref, kv, f"prefill {kv} Hq{Hq} Hkv{Hkv} D{D} bs{bs}")
    out16 = torch.empty(out.shape, dtype=torch.bfloat16, device=out.device)
    ds.attention_only(out=out16)
    torch.cuda.synchronize()
    assert torch.equal(out16, bf16_rne_of(out))


def test_fp8_d64_and_prefill():
    wl = W.build("fp8 mixed", Hq=16, Hkv=4, D=64, block_size=8, seq_lens=[1, 2000, 300, 77],
                 q_lens=[1, 1, 120, 77], src="bf16", kv="e4m3", seed=2009, pool_slack=0.1)
    ref, okc, ovc, _ = oracle.run_step(wl, nthreads=NT)
    ds, out = run_gpu(wl)
    assert oracle_caches_equal(ds, okc, ovc)
    check_attention(out, ref, "e4m3", "fp8 D64 mixed")


def test_edge_lengths_and_empty_rows():
    """N = 1, q_s = 0 sequences, a sequence filling its table exactly, a
    prefill chunk that is the whole sequence."""
    wl = W.build("edges", Hq=32, Hkv=8, D=128, block_size=16, seq_lens=[1, 50, 64, 64, 30],
                 q_lens=[1, 0, 64, 1, 0], src="bf16", kv="bf16", seed=2010, max_blocks=4)
    ref = oracle.run_step(wl, nthreads=NT)[0]
    _, out = run_gpu(wl)
    check_attention(out, ref, "bf16", "edges")


def test_pure_decode_hint_matches_unknown_hint():
    wl = small_decode(seed=2011, B=6)
    ds = DeviceStep(wl, max_q_len=1)
    a = ds.step().clone()
    b = torch.empty_like(a)
    pkv_attention(ds.q, ds.cu_q, ds.seq_lens, ds.bt, *ds.caches[0], wl.scale, b, max_q_len=0,
                  workspace=ds.ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_empty_batch():
    wl = W.tiny()
    ds = DeviceStep(wl)
    q = ds.q[:0]
    out = torch.empty_like(q)
    cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    sl = torch.zeros(0, dtype=torch.int32, device="cuda")
    bt = ds.bt[:0]
    pkv_attention(q, cu, sl, bt, *ds.caches[0], wl.scale, out, workspace=ds.ws)
    torch.cuda.synchronize()


def test_out_of_range_block_id_is_recorded_not_faulted():
    """A block id outside the pool inside a sequence's visible range: the
    kernels skip it and record bit 2; nothing is read out of bounds."""
    wl = small_decode(seed=2014, B=4, ctx=(100, 700))
    ds = DeviceStep(wl, max_q_len=1)
    torch.cuda.synchronize()
    assert pkv_device_errors() == 0
    bad = ds.bt.clone()
    bad[1, 2] = wl.num_blocks + 5
    bad[2, 0] = -3
    out = torch.empty_like(ds.out)
    pkv_attention(ds.q, ds.cu_q, ds.seq_lens, bad, *ds.caches[0], wl.scale, out, max_q_len=1,
                  workspace=ds.ws)
    assert pkv_device_errors() & 2
    slots = torch.empty(wl.T, dtype=torch.int32, device="cuda")
    pkv_slot_mapping(ds.cu_q, ds.seq_lens, bad, wl.block_size, out=slots)
    torch.cuda.synchronize()
    pkv_device_errors()


def test_inconsistent_lengths_are_recorded():
    wl = small_decode(seed=2015, B=3, ctx=(10, 40))
    ds = DeviceStep(wl, max_q_len=1)
    torch.cuda.synchronize()
    bad_lens = ds.seq_lens.clone()
    bad_lens[0] = wl.max_blocks * wl.block_size + 1  # beyond the block table
    out = torch.zeros_like(ds.out)
    pkv_attention(ds.q, ds.cu_q, bad_lens, ds.bt, *ds.caches[0], wl.scale, out, max_q_len=1,
                  workspace=ds.ws)
    assert pkv_device_errors() & 4


def test_host_validation_errors():
    wl = W.tiny()
    ds = DeviceStep(wl)
    with pytest.raises(PkvError) as e:
        pkv_attention(ds.q, ds.cu_q, ds.seq_lens, ds.bt, *ds.caches[0], wl.scale,
                      torch.empty(1, device="cuda"))
    assert e.value.status == 1
    with pytest.raises(PkvError) as e:
        pkv_attention(ds.q.bfloat16(), ds.cu_q, ds.seq_lens, ds.bt, *ds.caches[0], wl.scale, ds.out)
    assert e.value.status == 2
    # the f32 path needs no workspace; a bf16 call with a short one is refused
    wl2 = small_decode(seed=2016, B=2, ctx=(10, 20))
    ds2 = DeviceStep(wl2)
    with pytest.raises(PkvError) as e:
        pkv_attention(ds2.q, ds2.cu_q, ds2.seq_lens, ds2.bt, *ds2.caches[0], wl2.scale, ds2.out,
                      workspace=ds2.ws[:16])
    assert e.value.status == 3


def test_cpu_tensors_fail_loudly():
    wl = W.tiny()
    with pytest.raises(PkvError):
        pkv_slot_mapping(torch.zeros(5, dtype=torch.int32), torch.zeros(4, dtype=torch.int32),
                         torch.zeros(4, 4, dtype=torch.int32), 16, T=4)


def test_csr_page_lists_give_the_same_tables_and_attention():
    wl = W.qwen3_4b_decode(B=12, ctx=(1, 2600), block_size=16, num_blocks=0, seed=2302)
    nb = -(-wl.seq_lens.astype(np.int64) // wl.block_size)
    indptr = np.concatenate([[0], np.cumsum(nb)]).astype(np.int32)
    indices = np.concatenate([wl.block_tables[i, :nb[i]] for i in range(wl.B)]).astype(np.int32)
    max_blocks = wl.block_tables.shape[1]
    ref, bad = oracle.csr_to_block_tables(indptr, indices, max_blocks)
    assert not bad.any()
    dev = torch.device("cuda")
    bt = torch.full((wl.B, max_blocks), 12345, dtype=torch.int32, device=dev)
    pkv_csr_to_block_tables(torch.from_numpy(indptr).to(dev), torch.from_numpy(indices).to(dev), bt)
    torch.cuda.synchronize()
    assert pkv_device_errors() == 0
    assert np.array_equal(bt.cpu().numpy(), ref)
    ds, out = run_gpu(wl)
    ds.bt.copy_(bt)
    out2 = ds.attention_only(out=torch.empty_like(out))
    torch.cuda.synchronize()
    assert torch.equal(out2, out)
    # bad rows: filled with -1 and recorded, never faulted
    bad_ptr = torch.tensor([0, 3, 2, 9], dtype=torch.int32, device=dev)
    bt2 = torch.zeros((3, 4), dtype=torch.int32, device=dev)
    pkv_csr_to_block_tables(bad_ptr, torch.arange(6, dtype=torch.int32, device=dev), bt2)
    torch.cuda.synchronize()
    assert pkv_device_errors() & 4
    ref2, bad2 = oracle.csr_to_block_tables([0, 3, 2, 9], list(range(6)), 4)
    assert bad2.tolist() == [False, True, True] and np.array_equal(bt2.cpu().numpy(), ref2)
