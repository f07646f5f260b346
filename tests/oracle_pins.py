"""Pins of the CPU oracle to things other than itself.

Each pin_* function raises AssertionError when the oracle (module ``orc``)
disagrees with the pages or with the mathematics:
  * brute force on tiny inputs (high-precision mpmath, no max subtraction),
  * a library routine (torch scaled_dot_product_attention in float64 on the
    gathered contiguous K/V; torch's bf16 and float8_e4m3fn conversions),
  * closed forms (one key, zero query, constant values, two keys),
  * the OCP e4m3 values in tests/golden/e4m3_ocp_spec.txt,
  * the invariants the pages state (block size, paged = contiguous = full
    recompute, shared prefix, neighbour independence, batch composition).
The same functions run against copies of the oracle with a planted mistake
(test_oracle_pins.py) to show that each such mistake fails at least one pin.
"""
import math
import os

import mpmath
import numpy as np
import torch

from paged_kv_cache_mapping_gb300 import workloads as W
from tests.helpers import (bf16_to_f64, e4m3_to_f64, flat_rows, page_walk_slots,
                           random_tables, values)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------ value formats
def pin_bf16_decode(orc):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = orc.bf16_decode(bits)
    ref = bf16_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _golden_e4m3():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_ocp_spec.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                code, val = line.split()[:2]
                rows.append((int(code, 16), float(val)))
    return rows


def pin_e4m3_decode(orc):
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_decode(codes)
    ref = e4m3_to_f64(codes)  # torch float8_e4m3fn
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    for code, val in _golden_e4m3():
        g = orc.e4m3_decode(np.array([code], np.uint8))[0]
        if math.isnan(val):
            assert math.isnan(g), hex(code)
        else:
            assert g == val and math.copysign(1, g) == math.copysign(1, val), hex(code)
    pos = got[:0x7F]
    assert np.all(np.diff(pos) > 0)            # strictly increasing magnitudes
    assert np.array_equal(got[0x80:0xFF], -pos)  # sign bit mirrors


def _nearest_e4m3(prod):
    """Nearest search over the 127 non-negative finite codes (decoded by
    torch): for every fp32 value, the code of the same sign whose value is
    nearest, ties to the code with an even mantissa, magnitudes beyond the
    largest code (infinity included) to the largest code, NaN to NaN.
    Nearness is decided exactly, by comparing 2|x| with the sum of the two
    neighbouring code values."""
    codes = np.arange(0x7F, dtype=np.uint8)           # +0 .. 448
    mags = e4m3_to_f64(codes)
    a = np.abs(prod.astype(np.float64))
    sign = np.where(np.signbit(prod), 0x80, 0).astype(np.uint8)
    hi = np.clip(np.searchsorted(mags, a, side="left"), 0, mags.size - 1)
    lo = np.clip(hi - 1, 0, mags.size - 1)
    exact = mags[hi] == a
    twice, both = 2.0 * a, mags[lo] + mags[hi]
    pick = np.where(twice < both, lo, np.where(twice > both, hi,
                    np.where(codes[lo] % 2 == 0, lo, hi)))
    pick = np.where(exact, hi, pick)
    pick = np.where(a >= mags[-1], mags.size - 1, pick)
    out = codes[pick] | sign
    nan = np.isnan(prod)
    out[nan] = 0x7F | sign[nan]
    return out


def pin_e4m3_encode(orc):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = W.bf16_bits_to_f32(bits)
    for scale in (1.0, 0.5, 3.0, 1.0 / 64, 0.0138, 7.25, 1e-3):
        inv = np.float32(1.0) / np.float32(scale)
        with np.errstate(over="ignore", invalid="ignore"):
            prod = (x * inv).astype(np.float32)  # one fp32 multiply
        got = orc.e4m3_encode(prod)
        ref = _nearest_e4m3(prod)
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, (scale, prod[bad[:4]], got[bad[:4]], ref[bad[:4]])
        # library cross-check inside the finite range
        ok = np.abs(prod) < 448
        tq = torch.from_numpy(prod[ok]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(tq, got[ok]), scale


# ------------------------------------------------------------ slots
def pin_slot_mapping(orc):
    g = np.random.default_rng(11)
    for bs in (1, 3, 7, 16, 32):
        B = 5
        n = g.integers(1, 90, size=B)
        ql = np.minimum(g.integers(0, 9, size=B), n)
        tab = random_tables(g, n, bs, num_blocks=int(sum(-(-n // bs))) + 7,
                            width=int(max(-(-n // bs))) + 2)
        cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
        got = orc.slot_mapping(cu, n.astype(np.int32), tab, bs)
        ref = np.concatenate([page_walk_slots(tab[s], int(n[s]), bs)[n[s] - ql[s]:]
                              for s in range(B)])
        assert np.array_equal(got, ref), bs


# ------------------------------------------------------------ page lists
def pin_csr_tables(orc):
    # two requests sharing their prompt's pages 7 and 2, stored once
    tab, bad = orc.csr_to_block_tables([0, 3, 7], [7, 2, 5, 7, 2, 9, 4], 5)
    assert tab.tolist() == [[7, 2, 5, -1, -1], [7, 2, 9, 4, -1]] and not bad.any()
    # round trip: tables -> CSR (one row per request, pages in order) -> tables
    g = np.random.default_rng(12)
    n = g.integers(0, 9, size=6)
    tables = np.full((6, 10), -1, np.int32)
    indptr, indices = [0], []
    for i, k in enumerate(n):
        pages = g.integers(0, 50, size=k)
        tables[i, :k] = pages
        indices += list(pages)
        indptr.append(len(indices))
    got, bad = orc.csr_to_block_tables(indptr, indices, 10)
    assert np.array_equal(got, tables) and not bad.any()
    # bad rows: decreasing offsets, too many pages, offsets past nnz
    got, bad = orc.csr_to_block_tables([0, 2, 1, 5, 9], [1, 2, 3, 4, 5], 3)
    assert bad.tolist() == [False, True, True, True]
    assert got[0].tolist() == [1, 2, -1] and (got[1:] == -1).all()


# ------------------------------------------------------------ append
def pin_append(orc):
    g = np.random.default_rng(12)
    T, H, D, NB, bs = 37, 3, 16, 20, 7
    for src, kv in (("f32", "f32"), ("bf16", "bf16"), ("bf16", "e4m3"), ("f32", "e4m3")):
        if src == "f32":
            k = g.standard_normal((T, H, D), dtype=np.float32) * 3
            v = g.standard_normal((T, H, D), dtype=np.float32) * 3
        else:
            k = W.bf16_bits(g.standard_normal((T, H, D), dtype=np.float32) * 3)
            v = W.bf16_bits(g.standard_normal((T, H, D), dtype=np.float32) * 3)
        dt = {"f32": np.float32, "bf16": np.uint16, "e4m3": np.uint8}[kv]
        canary_k = g.integers(0, 1 << 8, size=(NB, bs, H, D * np.dtype(dt).itemsize),
                              dtype=np.uint8).view(dt)
        canary_v = canary_k[::-1].copy()
        kc, vc = canary_k.copy(), canary_v.copy()
        slots = g.choice(NB * bs, size=T, replace=False).astype(np.int64)
        slots[::5] = -1  # padding rows are skipped
        ks, vs = 0.0217, 0.0371
        orc.append(k, v, slots, kc, vc, ks, vs)
        w = slots >= 0
        if kv == "e4m3":
            kx = values(k, src).astype(np.float32) * (np.float32(1) / np.float32(ks))
            vx = values(v, src).astype(np.float32) * (np.float32(1) / np.float32(vs))
            kexp = _nearest_e4m3(kx.astype(np.float32).ravel()).reshape(k.shape)
            vexp = _nearest_e4m3(vx.astype(np.float32).ravel()).reshape(v.shape)
        else:
            kexp, vexp = k, v
        assert np.array_equal(flat_rows(kc, slots[w]).view(np.uint8),
                              np.ascontiguousarray(kexp[w]).view(np.uint8)), (src, kv)
        assert np.array_equal(flat_rows(vc, slots[w]).view(np.uint8),
                              np.ascontiguousarray(vexp[w]).view(np.uint8)), (src, kv)
        untouched = np.setdiff1d(np.arange(NB * bs), slots[w])
        assert np.array_equal(flat_rows(kc, untouched).view(np.uint8),
                              flat_rows(canary_k, untouched).view(np.uint8))
        assert np.array_equal(flat_rows(vc, untouched).view(np.uint8),
                              flat_rows(canary_v, untouched).view(np.uint8))


# ------------------------------------------------------------ attention
def _random_problem(g, *, B, Hq, Hkv, D, bs, kv, src, max_n=12, max_q=3, scale=None):
    n = g.integers(1, max_n + 1, size=B).astype(np.int32)
    ql = np.minimum(g.integers(0, max_q + 1, size=B), n).astype(np.int32)
    ql[0] = max(ql[0], 1)
    NB = int(sum(-(-n // bs))) + 5
    tab = random_tables(g, n, bs, NB, width=int(max(-(-n // bs))) + 1)
    if kv == "e4m3":
        codes = g.integers(0, 256, size=(NB, bs, Hkv, D), dtype=np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN patterns
        kc = codes
        vc = g.permutation(codes.ravel()).reshape(codes.shape)
    elif kv == "bf16":
        kc = W.bf16_bits(g.standard_normal((NB, bs, Hkv, D), dtype=np.float32))
        vc = W.bf16_bits(g.standard_normal((NB, bs, Hkv, D), dtype=np.float32))
    else:
        kc = g.standard_normal((NB, bs, Hkv, D), dtype=np.float32)
        vc = g.standard_normal((NB, bs, Hkv, D), dtype=np.float32)
    T = int(ql.sum())
    q = g.standard_normal((T, Hq, D), dtype=np.float32) * 1.5
    if src == "bf16":
        q = W.bf16_bits(q)
    cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    if scale is None:
        scale = float(np.float32(1 / math.sqrt(D)))
    return dict(q=q, cu=cu, n=n, tab=tab, kc=kc, vc=vc, scale=scale, bs=bs,
                Hq=Hq, Hkv=Hkv, kv=kv, src=src, ks=0.0123 if kv == "e4m3" else 1.0,
                vs=0.0311 if kv == "e4m3" else 1.0)


def _run(orc, P):
    return orc.attention(P["q"], P["cu"], P["n"], P["tab"], P["kc"], P["vc"], P["scale"],
                         P["ks"], P["vs"])


def _gathered(P, s):
    """Logical K and V of sequence s (fp64), gathered by walking its pages."""
    slots = page_walk_slots(P["tab"][s], int(P["n"][s]), P["bs"])
    K = values(flat_rows(P["kc"], slots), P["kv"], P["ks"])
    V = values(flat_rows(P["vc"], slots), P["kv"], P["vs"])
    return K, V


def pin_attention_bruteforce(orc):
    """mpmath at 40 digits, softmax without max subtraction, tiny inputs."""
    g = np.random.default_rng(13)
    mpmath.mp.dps = 40
    for kv, src in (("f32", "f32"), ("bf16", "bf16"), ("e4m3", "bf16")):
        P = _random_problem(g, B=3, Hq=4, Hkv=2, D=6, bs=3, kv=kv, src=src, max_n=8)
        out = _run(orc, P)
        Q = values(P["q"], src)
        G = P["Hq"] // P["Hkv"]
        for s in range(3):
            K, V = _gathered(P, s)
            N = int(P["n"][s])
            q_s = int(P["cu"][s + 1] - P["cu"][s])
            for i in range(q_s):
                t = int(P["cu"][s]) + i
                pos = N - q_s + i
                for h in range(P["Hq"]):
                    kh = h // G
                    w = []
                    for j in range(pos + 1):
                        sc = mpmath.mpf(P["scale"]) * mpmath.fsum(
                            mpmath.mpf(float(Q[t, h, d])) * mpmath.mpf(float(K[j, kh, d]))
                            for d in range(Q.shape[2]))
                        w.append(mpmath.exp(sc))
                    den = mpmath.fsum(w)
                    for d in range(Q.shape[2]):
                        num = mpmath.fsum(w[j] * mpmath.mpf(float(V[j, kh, d]))
                                          for j in range(pos + 1))
                        ref = float(num / den)
                        assert abs(out[t, h, d] - ref) <= 1e-12 * max(1.0, abs(ref)), \
                            (kv, s, i, h, d, out[t, h, d], ref)


def _sdpa_reference(P):
    """torch SDPA in float64 on each sequence's gathered contiguous K/V, the
    KV heads repeated to the query heads, causal mask offset by N - q_s."""
    Q = torch.from_numpy(values(P["q"], P["src"]))
    G = P["Hq"] // P["Hkv"]
    out = torch.zeros_like(Q)
    for s in range(len(P["n"])):
        a, b = int(P["cu"][s]), int(P["cu"][s + 1])
        if b == a:
            continue
        K, V = _gathered(P, s)
        K = torch.from_numpy(K).repeat_interleave(G, dim=1).transpose(0, 1)
        V = torch.from_numpy(V).repeat_interleave(G, dim=1).transpose(0, 1)
        q = Q[a:b].transpose(0, 1)
        N, qs = int(P["n"][s]), b - a
        mask = torch.arange(N)[None, :] <= (N - qs + torch.arange(qs))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(
            q, K, V, attn_mask=mask, scale=P["scale"])
        out[a:b] = o.transpose(0, 1)
    return out.numpy()


def pin_attention_sdpa(orc):
    g = np.random.default_rng(14)
    cases = [dict(B=4, Hq=8, Hkv=2, D=32, bs=7, kv="bf16", src="bf16", max_n=120, max_q=9),
             dict(B=3, Hq=6, Hkv=3, D=16, bs=1, kv="f32", src="f32", max_n=40, max_q=40),
             dict(B=3, Hq=4, Hkv=4, D=24, bs=16, kv="e4m3", src="bf16", max_n=70, max_q=5),
             dict(B=2, Hq=8, Hkv=1, D=8, bs=5, kv="bf16", src="bf16", max_n=30, max_q=30)]
    for c in cases:
        P = _random_problem(g, **c)
        out = _run(orc, P)
        ref = _sdpa_reference(P)
        err = np.abs(out - ref).max()
        assert err <= 1e-12 * max(1.0, np.abs(ref).max()), (c, err)


def pin_closed_forms(orc):
    g = np.random.default_rng(15)
    base = dict(B=3, Hq=4, Hkv=2, D=8, bs=3, kv="f32", src="f32", max_n=10, max_q=2)
    # one key: o = v_0 exactly
    P = _random_problem(g, **base)
    P["n"][:] = 1
    P["cu"] = np.array([0, 1, 2, 3], np.int32)
    P["q"] = P["q"][:1].repeat(3, axis=0)
    out = _run(orc, P)
    G = P["Hq"] // P["Hkv"]
    for s in range(3):
        K, V = _gathered(P, s)
        for h in range(P["Hq"]):
            assert np.array_equal(out[s, h], V[0, h // G]), "N=1"
    # zero query or zero scale: o = mean of the visible values
    for zero in ("q", "scale"):
        P = _random_problem(g, **base)
        if zero == "q":
            P["q"][:] = 0
        else:
            P["scale"] = 0.0
        out = _run(orc, P)
        for s in range(3):
            K, V = _gathered(P, s)
            N, a, b = int(P["n"][s]), int(P["cu"][s]), int(P["cu"][s + 1])
            for i in range(b - a):
                pos = N - (b - a) + i
                for h in range(P["Hq"]):
                    ref = V[:pos + 1, h // G].mean(axis=0)
                    assert np.allclose(out[a + i, h], ref, rtol=1e-14, atol=1e-15), zero
    # every value row equal to c: o = c
    P = _random_problem(g, **base)
    c = g.standard_normal(8).astype(np.float32)
    P["vc"][:] = c
    out = _run(orc, P)
    T = int(P["cu"][-1])
    assert np.allclose(out[:T], np.broadcast_to(c.astype(np.float64), out[:T].shape),
                       rtol=1e-14, atol=0)
    # every key equal: o = mean of the visible values
    P = _random_problem(g, **base)
    P["kc"][:] = g.standard_normal(8).astype(np.float32)
    out = _run(orc, P)
    for s in range(3):
        K, V = _gathered(P, s)
        N, a, b = int(P["n"][s]), int(P["cu"][s]), int(P["cu"][s + 1])
        for i in range(b - a):
            pos = N - (b - a) + i
            for h in range(P["Hq"]):
                assert np.allclose(out[a + i, h], V[:pos + 1, h // G].mean(axis=0),
                                   rtol=1e-13, atol=1e-15), "equal keys"
    # two keys along one axis: the weight of key 1 is the logistic of the
    # score difference scale * q0 * (k1 - k0)
    # (also with logits far beyond exp's range: the softmax is shift
    # invariant, so the result must stay finite and exact)
    for k0, k1, sc in ((0.5, -1.25, 0.75), (-1.25, 0.5, 300.0)):
        P = _random_problem(g, B=1, Hq=1, Hkv=1, D=4, bs=1, kv="f32", src="f32", max_n=2)
        P["n"][:] = 2
        P["tab"] = random_tables(g, [2], 1, P["kc"].shape[0])
        P["cu"] = np.array([0, 1], np.int32)
        P["q"] = np.array([[[2.0, 0, 0, 0]]], np.float32)
        P["scale"] = sc
        slots = page_walk_slots(P["tab"][0], 2, 1)
        P["kc"].reshape(-1, 1, 4)[slots[0], 0] = [k0, 9, 9, 9]
        P["kc"].reshape(-1, 1, 4)[slots[1], 0] = [k1, -7, 3, 1]
        K, V = _gathered(P, 0)
        out = _run(orc, P)
        z = sc * 2.0 * (k1 - k0)
        w1 = 1.0 / (1.0 + math.exp(-z)) if z > -700 else 0.0
        ref = (1 - w1) * V[0, 0] + w1 * V[1, 0]
        assert np.allclose(out[0, 0], ref, rtol=1e-14, atol=1e-15), ("two keys", sc)


# ------------------------------------------------------------ invariants
def _oracle_step(orc, wl):
    return orc.run_step(wl)[0]


def pin_invariant_block_size_and_layout(orc):
    outs = []
    for bs in (1, 3, 7, 16, 32):
        for contiguous in (False, True):
            wl = W.build("inv", Hq=4, Hkv=2, D=16, block_size=bs,
                         seq_lens=[1, 19, 40, 7], q_lens=[1, 3, 1, 7], src="bf16",
                         kv="bf16", seed=21, contiguous=contiguous, pool_slack=0.5)
            outs.append(_oracle_step(orc, wl))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def pin_invariant_full_recompute(orc):
    """One-shot causal prefill of a sequence equals appending its tokens one
    by one and decoding each (incremental paged decode)."""
    full = W.build("full", Hq=4, Hkv=2, D=16, block_size=5, seq_lens=[23], q_lens=[23],
                   src="bf16", kv="bf16", seed=22)
    o_full = _oracle_step(orc, full)
    kc = np.zeros(full.cache_shape(), np.uint16)
    vc = np.zeros_like(kc)
    for p in range(23):
        cu = np.array([0, 1], np.int32)
        sl = np.array([p + 1], np.int32)
        slots = orc.slot_mapping(cu, sl, full.block_tables, full.block_size)
        orc.append(full.k_tokens[p:p + 1], full.v_tokens[p:p + 1], slots, kc, vc)
        o = orc.attention(full.q[p:p + 1], cu, sl, full.block_tables, kc, vc, full.scale)
        assert np.array_equal(o[0], o_full[p]), p


def pin_invariant_shared_prefix(orc):
    kw = dict(n_decode=3, dec_ctx=(40, 60), chunk=12, prefix=32, block_size=8,
              num_blocks=64, seed=23)
    shared = W.mixed_prefill(**kw)
    # unshared: the same logical data with every sequence owning its blocks
    un = W.build("unshared", Hq=32, Hkv=8, D=128, block_size=8,
                 seq_lens=shared.seq_lens, q_lens=shared.q_lens, src="bf16", kv="bf16",
                 seed=23, num_blocks=64)
    un.k_tokens[:] = shared.k_tokens
    un.v_tokens[:] = shared.v_tokens
    un.q[:] = shared.q
    assert (shared.block_tables[0, :4] == shared.block_tables[3, :4]).all()
    assert not np.isin(un.block_tables[0, :4], un.block_tables[3, :4]).any()
    assert np.array_equal(_oracle_step(orc, shared), _oracle_step(orc, un))


def pin_invariant_batch(orc):
    """Neighbour independence and batch composition: a short sequence alone,
    batched with a long one, or batched in another order gives the same rows."""
    kw = dict(Hq=4, Hkv=2, D=16, block_size=4, src="bf16", kv="bf16", seed=24)
    both = W.build("both", seq_lens=[9, 300], q_lens=[2, 1], num_blocks=90, **kw)
    alone = both.select([0])
    swapped = both.select([1, 0])
    o_both = _oracle_step(orc, both)
    o_alone = _oracle_step(orc, alone)
    o_sw = _oracle_step(orc, swapped)
    assert np.array_equal(o_both[:2], o_alone)
    assert np.array_equal(o_both[:2], o_sw[1:3])
    assert np.array_equal(o_both[2:], o_sw[:1])


# ------------------------------------------------------------ variants
def _run_v(orc, P, soft_cap=0.0, window_left=-1):
    return orc.attention(P["q"], P["cu"], P["n"], P["tab"], P["kc"], P["vc"], P["scale"],
                         P["ks"], P["vs"], soft_cap=soft_cap, window_left=window_left)


def pin_variants_reduce_and_window_closed_form(orc):
    g = np.random.default_rng(15)
    P = _random_problem(g, B=4, Hq=4, Hkv=2, D=16, bs=5, kv="bf16", src="bf16", max_n=40, max_q=6)
    plain = _run(orc, P)
    # a window wider than any sequence and a cap of +inf-like size change nothing
    assert np.array_equal(_run_v(orc, P, window_left=10 ** 6), plain)
    assert np.abs(_run_v(orc, P, soft_cap=1e12) - plain).max() <= 1e-12
    # window 0: each query sees only its own key, so the output is its V row
    out = _run_v(orc, P, window_left=0)
    G = P["Hq"] // P["Hkv"]
    for s in range(len(P["n"])):
        K, V = _gathered(P, s)
        N, a, b = int(P["n"][s]), int(P["cu"][s]), int(P["cu"][s + 1])
        for i in range(b - a):
            for h in range(P["Hq"]):
                assert np.array_equal(out[a + i, h], V[N - (b - a) + i, h // G])


def pin_window_sdpa(orc):
    """torch SDPA in float64 with a banded causal mask on the gathered K/V."""
    g = np.random.default_rng(16)
    for W_left in (1, 3, 17):
        P = _random_problem(g, B=4, Hq=6, Hkv=2, D=16, bs=7, kv="bf16", src="bf16", max_n=60, max_q=12)
        out = _run_v(orc, P, window_left=W_left)
        Q = torch.from_numpy(values(P["q"], P["src"]))
        G = P["Hq"] // P["Hkv"]
        for s in range(len(P["n"])):
            a, b = int(P["cu"][s]), int(P["cu"][s + 1])
            if b == a:
                continue
            K, V = _gathered(P, s)
            K = torch.from_numpy(K).repeat_interleave(G, dim=1).transpose(0, 1)
            V = torch.from_numpy(V).repeat_interleave(G, dim=1).transpose(0, 1)
            N, qs = int(P["n"][s]), b - a
            pos = (N - qs + torch.arange(qs))[:, None]
            j = torch.arange(N)[None, :]
            mask = (j <= pos) & (j >= pos - W_left)
            o = torch.nn.functional.scaled_dot_product_attention(Q[a:b].transpose(0, 1), K, V,
                                                                 attn_mask=mask, scale=P["scale"])
            ref = o.transpose(0, 1).numpy()
            assert np.abs(out[a:b] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max()), (W_left, s)


def pin_soft_cap_bruteforce(orc):
    """mpmath at 40 digits: cap * tanh(scale q.k / cap), softmax without max subtraction."""
    g = np.random.default_rng(17)
    mpmath.mp.dps = 40
    for cap, W_left in ((2.0, -1), (0.7, 2)):
        P = _random_problem(g, B=3, Hq=4, Hkv=2, D=6, bs=3, kv="bf16", src="bf16", max_n=8, scale=1.3)
        out = _run_v(orc, P, soft_cap=cap, window_left=W_left)
        Q = values(P["q"], P["src"])
        G = P["Hq"] // P["Hkv"]
        for s in range(3):
            K, V = _gathered(P, s)
            N, a, b = int(P["n"][s]), int(P["cu"][s]), int(P["cu"][s + 1])
            for i in range(b - a):
                pos = N - (b - a) + i
                lo = 0 if W_left < 0 else max(0, pos - W_left)
                for h in range(P["Hq"]):
                    kh = h // G
                    w = []
                    for j in range(lo, pos + 1):
                        dot = mpmath.fsum(mpmath.mpf(float(Q[a + i, h, d])) * mpmath.mpf(float(K[j, kh, d]))
                                          for d in range(Q.shape[2]))
                        sc = mpmath.mpf(cap) * mpmath.tanh(mpmath.mpf(P["scale"]) * dot / mpmath.mpf(cap))
                        w.append(mpmath.exp(sc))
                    den = mpmath.fsum(w)
                    for d in range(Q.shape[2]):
                        num = mpmath.fsum(w[j - lo] * mpmath.mpf(float(V[j, kh, d])) for j in range(lo, pos + 1))
                        ref = float(num / den)
                        assert abs(out[a + i, h, d] - ref) <= 1e-12 * max(1.0, abs(ref)), (cap, W_left, s, i, h, d)


ALL_PINS = [pin_bf16_decode, pin_e4m3_decode, pin_e4m3_encode, pin_slot_mapping, pin_csr_tables,
            pin_append, pin_attention_bruteforce, pin_attention_sdpa, pin_closed_forms,
            pin_invariant_block_size_and_layout, pin_invariant_full_recompute,
            pin_invariant_shared_prefix, pin_invariant_batch, pin_variants_reduce_and_window_closed_form,
            pin_window_sdpa, pin_soft_cap_bruteforce]
