"""Seeded synthetic inputs shaped like the pages' workloads.

This module draws random numbers and lays out block tables; it holds none of
the method's arithmetic (no slot computation, no append, no attention).  The
tests, the benchmark and the smoke check feed the same arrays to the CUDA
library and to the CPU oracle.

Recipe (every workload):
  * numpy ``Generator(PCG64([seed, stream, s]))``; ``seed`` is fixed per
    workload preset, ``stream`` 1 = K, 2 = V, 3 = Q, 4 = lengths, 5 = pool
    permutation, and ``s`` the sequence index where there is one.
  * Values: i.i.d. standard normal drawn in float32
    (``standard_normal(dtype=float32)``); bf16 workloads round each draw to
    bf16 (round to nearest, ties to even) and keep the bit pattern (uint16).
  * Block tables: sequence s owns ceil(N_s / block_size) blocks taken in turn
    from a seeded permutation of the pool ("scattered") or from the identity
    order ("contiguous"); entries past a sequence's last block are -1.
    Shared prefix blocks are listed by every sharer and stored once
    (nanoserve, "Prefix caching"; "How Easy Is It to Start Serving LLMs?",
    "1. Block-sparse KV memory": requests sharing a prompt list the same
    page ids).
  * seq_lens counts this step's new tokens; the last q_s tokens of every
    sequence are this step's new rows, the rest is history that a setup step
    writes into the cache before the timed step.
  * fp8 workloads: per-tensor scales max|K| / 448 and max|V| / 448 over the
    generated tokens, rounded to fp32.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

E4M3_MAX = 448.0


def rng(seed: int, stream: int, index: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream, index]))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (input prep)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal(g: np.random.Generator, shape, fmt: str) -> np.ndarray:
    x = g.standard_normal(shape, dtype=np.float32)
    return bf16_bits(x) if fmt == "bf16" else x


@dataclass
class Workload:
    """One synthetic step of paged attention."""

    name: str
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    src: str                 # format of q, k, v rows: "f32" | "bf16"
    kv: str                  # cache format: "f32" | "bf16" | "e4m3"
    seq_lens: np.ndarray     # int32 [B], N_s including this step's rows
    q_lens: np.ndarray       # int32 [B], new rows (queries) this step
    write_start: np.ndarray  # int32 [B], first position this sequence writes
    block_tables: np.ndarray  # int32 [B, max_blocks], -1 padded
    cu_seqlens_k: np.ndarray  # int64 [B+1], offsets of each sequence in k/v_tokens
    k_tokens: np.ndarray     # [sum N_s, Hkv, D] logical K of every position
    v_tokens: np.ndarray
    q: np.ndarray            # [T, Hq, D]
    scale: float
    k_scale: float = 1.0
    v_scale: float = 1.0
    seed: int = 0
    meta: dict = field(default_factory=dict)

    # ---- shapes
    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.q_lens.sum())

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    def cache_shape(self):
        return (self.num_blocks, self.block_size, self.Hkv, self.D)

    def cache_np_dtype(self):
        return {"f32": np.float32, "bf16": np.uint16, "e4m3": np.uint8}[self.kv]

    # ---- this step's new rows
    def new_rows(self):
        ks, vs = [], []
        for s in range(self.B):
            a = int(self.cu_seqlens_k[s] + self.seq_lens[s] - self.q_lens[s])
            b = int(self.cu_seqlens_k[s] + self.seq_lens[s])
            ks.append(self.k_tokens[a:b])
            vs.append(self.v_tokens[a:b])
        return np.concatenate(ks), np.concatenate(vs)

    # ---- history written before the step, in batches of whole sequences
    def history_batches(self, max_tokens: int = 1 << 22):
        """Yields (s0, s1, cu_seqlens, seq_lens_hist, k, v): the rows of
        positions [write_start_s, N_s - q_s) of sequences s0..s1-1, packed,
        with seq_lens_hist = N_s - q_s (so that they are the "new" rows of a
        setup step that ends where this step's rows begin)."""
        hist_end = (self.seq_lens - self.q_lens).astype(np.int32)
        n_rows = np.maximum(hist_end - self.write_start, 0).astype(np.int64)
        s0 = 0
        while s0 < self.B:
            s1, tot = s0, 0
            while s1 < self.B and (s1 == s0 or tot + n_rows[s1] <= max_tokens):
                tot += int(n_rows[s1])
                s1 += 1
            cu = np.concatenate([[0], np.cumsum(n_rows[s0:s1])]).astype(np.int32)
            ks, vs = [], []
            for s in range(s0, s1):
                a = int(self.cu_seqlens_k[s] + self.write_start[s])
                b = int(self.cu_seqlens_k[s] + hist_end[s])
                ks.append(self.k_tokens[a:b])
                vs.append(self.v_tokens[a:b])
            yield s0, s1, cu, hist_end[s0:s1].copy(), np.concatenate(ks), np.concatenate(vs)
            s0 = s1

    def select(self, seqs) -> "Workload":
        """Sub-workload of the given sequences (same pool and values).  A
        sharer whose prefix owner is not selected writes the shared blocks
        itself (the values are the same)."""
        seqs = [int(s) for s in seqs]
        owners = self.meta.get("owner", np.arange(self.B))
        ws = self.write_start.copy()
        for s in seqs:
            if owners[s] != s and owners[s] not in seqs:
                ws[s] = 0
        parts_k, parts_v, cuk = [], [], [0]
        for s in seqs:
            a, b = int(self.cu_seqlens_k[s]), int(self.cu_seqlens_k[s + 1])
            parts_k.append(self.k_tokens[a:b])
            parts_v.append(self.v_tokens[a:b])
            cuk.append(cuk[-1] + b - a)
        cq = self.cu_seqlens_q
        q = np.concatenate([self.q[cq[s]:cq[s + 1]] for s in seqs])
        new_owner = np.array([seqs.index(owners[s]) if owners[s] in seqs else i
                              for i, s in enumerate(seqs)], np.int64)
        return Workload(
            name=self.name + "[sel]", Hq=self.Hq, Hkv=self.Hkv, D=self.D,
            block_size=self.block_size, num_blocks=self.num_blocks, src=self.src,
            kv=self.kv, seq_lens=self.seq_lens[seqs].copy(),
            q_lens=self.q_lens[seqs].copy(), write_start=ws[seqs].copy(),
            block_tables=self.block_tables[seqs].copy(),
            cu_seqlens_k=np.array(cuk, np.int64), k_tokens=np.concatenate(parts_k),
            v_tokens=np.concatenate(parts_v), q=q, scale=self.scale,
            k_scale=self.k_scale, v_scale=self.v_scale, seed=self.seed,
            meta={"owner": new_owner, "selected_from": seqs})

    # ---- accounting used by the benchmark (bytes a pass must move)
    def kv_bytes_read(self) -> int:
        """K and V rows every query row set must read once per KV head: the
        keys visible to the sequence's last query, N_s rows."""
        eb = {"f32": 4, "bf16": 2, "e4m3": 1}[self.kv]
        return int(self.seq_lens[self.q_lens > 0].astype(np.int64).sum()) * self.Hkv * self.D * eb * 2


def build(name: str, *, Hq: int, Hkv: int, D: int, block_size: int,
          seq_lens, q_lens, src: str = "bf16", kv: str = "bf16", seed: int = 0,
          num_blocks: int | None = None, contiguous: bool = False,
          max_blocks: int | None = None, shared=(), threads: int = 8,
          pool_slack: float = 0.0) -> Workload:
    """General builder.

    shared: iterable of (owner, sharers, n_prefix_tokens); n_prefix_tokens is
    a multiple of block_size; the owner's first blocks are also the sharers'
    first blocks and the sharers' logical K/V there are the owner's.
    """
    seq_lens = np.asarray(seq_lens, np.int32)
    q_lens = np.asarray(q_lens, np.int32)
    B = seq_lens.shape[0]
    bs = block_size
    nblk = -(-seq_lens.astype(np.int64) // bs)
    owner = np.arange(B)
    share_blocks = np.zeros(B, np.int64)
    for own, sharers, n_pre in shared:
        assert n_pre % bs == 0
        for sh in sharers:
            owner[sh] = own
            share_blocks[sh] = n_pre // bs
            assert seq_lens[sh] >= n_pre and seq_lens[own] - q_lens[own] >= n_pre
    needed = int((nblk - share_blocks).sum())
    if num_blocks is None:
        num_blocks = needed + int(math.ceil(needed * pool_slack))
    assert needed <= num_blocks, (needed, num_blocks)
    if max_blocks is None:
        max_blocks = int(nblk.max()) if B else 1
    pool = (np.arange(num_blocks, dtype=np.int64) if contiguous
            else rng(seed, 5).permutation(num_blocks))
    tables = np.full((B, max_blocks), -1, np.int32)
    order = sorted(range(B), key=lambda s: (owner[s] != s, s))  # owners first
    cursor = 0
    for s in order:
        k0 = int(share_blocks[s])
        if k0:
            tables[s, :k0] = tables[owner[s], :k0]
        n_own = int(nblk[s]) - k0
        tables[s, k0:k0 + n_own] = pool[cursor:cursor + n_own]
        cursor += n_own
    write_start = (share_blocks * bs).astype(np.int32)

    cuk = np.concatenate([[0], np.cumsum(seq_lens.astype(np.int64))])
    tot = int(cuk[-1])
    dt = np.uint16 if src == "bf16" else np.float32
    k_tokens = np.empty((tot, Hkv, D), dt)
    v_tokens = np.empty((tot, Hkv, D), dt)

    def fill(s):
        a, n = int(cuk[s]), int(seq_lens[s])
        ws = int(write_start[s])
        if n > ws:
            k_tokens[a + ws:a + n] = _normal(rng(seed, 1, s), (n - ws, Hkv, D), src)
            v_tokens[a + ws:a + n] = _normal(rng(seed, 2, s), (n - ws, Hkv, D), src)

    with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        list(ex.map(fill, range(B)))
    for s in range(B):  # shared positions copy the owner's logical rows
        ws = int(write_start[s])
        if ws:
            o = int(cuk[owner[s]])
            k_tokens[cuk[s]:cuk[s] + ws] = k_tokens[o:o + ws]
            v_tokens[cuk[s]:cuk[s] + ws] = v_tokens[o:o + ws]
    T = int(q_lens.sum())
    q = _normal(rng(seed, 3), (T, Hq, D), src)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    k_scale = v_scale = 1.0
    if kv == "e4m3":
        def absmax(a):
            x = bf16_bits_to_f32(a) if src == "bf16" else a
            return float(np.abs(x).max()) if x.size else 1.0
        k_scale = float(np.float32(absmax(k_tokens) / E4M3_MAX))
        v_scale = float(np.float32(absmax(v_tokens) / E4M3_MAX))
    return Workload(name=name, Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                    num_blocks=int(num_blocks), src=src, kv=kv, seq_lens=seq_lens,
                    q_lens=q_lens, write_start=write_start, block_tables=tables,
                    cu_seqlens_k=cuk, k_tokens=k_tokens, v_tokens=v_tokens, q=q,
                    scale=scale, k_scale=k_scale, v_scale=v_scale, seed=seed,
                    meta={"owner": owner})


# ---------------------------------------------------------------- presets
# The five workloads the pages' measurements are shaped like.  Qwen3-4B
# attention has 32 query heads, 8 KV heads and head dimension 128 ("How Easy
# Is It to Start Serving LLMs?", "Four phases, nine scripts", Phase 4).

def tiny(seed: int = 1001) -> Workload:
    """Four decoding sequences with 5, 17, 33 and 64 keys (the new token
    included), fp32, Hq 4, Hkv 2, D 64, block size 16, a pool of 64 blocks."""
    return build("tiny decode fp32 (N=5,17,33,64; Hq4 Hkv2 D64 bs16)", Hq=4, Hkv=2,
                 D=64, block_size=16, seq_lens=[5, 17, 33, 64], q_lens=[1] * 4,
                 src="f32", kv="f32", seed=seed, num_blocks=64)


def qwen3_4b_decode(B: int = 64, ctx=(512, 4096), block_size: int = 16,
                    num_blocks: int = 20000, seed: int = 1002) -> Workload:
    """Decode step at Qwen3-4B heads: B sequences with contexts uniform in
    ctx (inclusive), one new token each, bf16, block size 16, blocks drawn
    from a shuffled pool."""
    lens = rng(seed, 4).integers(ctx[0], ctx[1] + 1, size=B).astype(np.int32)
    mb = -(-ctx[1] // block_size)
    nb = max(num_blocks, int((-(-lens.astype(np.int64) // block_size)).sum()))
    return build(f"Qwen3-4B decode B{B} ctx U[{ctx[0]},{ctx[1]}] bs{block_size} bf16",
                 Hq=32, Hkv=8, D=128, block_size=block_size, seq_lens=lens,
                 q_lens=np.ones(B, np.int32), src="bf16", kv="bf16", seed=seed,
                 num_blocks=nb, max_blocks=mb)


def layout_sweep(block_size: int, contiguous: bool, B: int = 32, ctx: int = 2048,
                 seed: int = 1003) -> Workload:
    """B sequences of ctx keys at Qwen3-4B heads; the pool holds exactly the
    needed blocks.  The logical K/V and Q do not depend on the layout."""
    lens = np.full(B, ctx, np.int32)
    lay = "contiguous" if contiguous else "scattered"
    return build(f"layout B{B} ctx{ctx} bs{block_size} {lay}", Hq=32, Hkv=8, D=128,
                 block_size=block_size, seq_lens=lens, q_lens=np.ones(B, np.int32),
                 src="bf16", kv="bf16", seed=seed, contiguous=contiguous)


def mixed_prefill(n_decode: int = 16, dec_ctx=(1024, 8192), chunk: int = 512,
                  prefix: int = 1024, block_size: int = 16, num_blocks: int = 8192,
                  seed: int = 1004, kv: str = "bf16") -> Workload:
    """Chunked-prefill step: n_decode decodes, then chunk A (chunk new tokens
    after a cached prefix whose blocks decodes 0 and 1 share) and chunk B
    (chunk tokens, no prior context), packed decodes first.  kv: the cache
    format ("bf16", or "e4m3" with per-tensor scales)."""
    dec = rng(seed, 4).integers(dec_ctx[0], dec_ctx[1] + 1, size=n_decode)
    lens = np.concatenate([dec, [prefix + chunk, chunk]]).astype(np.int32)
    ql = np.concatenate([np.ones(n_decode), [chunk, chunk]]).astype(np.int32)
    a = n_decode
    sharers = [s for s in (0, 1) if s < n_decode]
    mb = -(-max(dec_ctx[1], prefix + chunk) // block_size)
    return build(f"mixed prefill {n_decode} decodes + 2x{chunk} chunks {kv}",
                 Hq=32, Hkv=8, D=128, block_size=block_size, seq_lens=lens,
                 q_lens=ql, src="bf16", kv=kv, seed=seed,
                 num_blocks=num_blocks, max_blocks=mb,
                 shared=[(a, sharers, prefix)] if sharers and prefix else ())


def long_fp8(B: int = 8, ctx=(32768, 131072), seed: int = 1005) -> Workload:
    """Long-context decode with an fp8 e4m3 cache: B sequences with contexts
    uniform in ctx, bf16 queries, per-tensor K and V scales."""
    lens = rng(seed, 4).integers(ctx[0], ctx[1] + 1, size=B).astype(np.int32)
    return build(f"long fp8 B{B} ctx U[{ctx[0]},{ctx[1]}] e4m3", Hq=32, Hkv=8,
                 D=128, block_size=16, seq_lens=lens, q_lens=np.ones(B, np.int32),
                 src="bf16", kv="e4m3", seed=seed, max_blocks=-(-ctx[1] // 16),
                 pool_slack=0.05)


def lognormal_fp8(B: int = 256, median: int = 2048, sigma: float = 1.0,
                  cap: int = 16384, seed: int = 1006) -> Workload:
    """Decode with log-normal contexts (median 2048, sigma 1, clamped to
    [1, cap]) and an fp8 e4m3 cache."""
    g = rng(seed, 4)
    lens = np.clip(np.rint(np.exp(g.normal(math.log(median), sigma, size=B))), 1,
                   cap).astype(np.int32)
    return build(f"lognormal fp8 B{B} median{median} cap{cap} e4m3", Hq=32, Hkv=8,
                 D=128, block_size=16, seq_lens=lens, q_lens=np.ones(B, np.int32),
                 src="bf16", kv="e4m3", seed=seed, max_blocks=-(-cap // 16),
                 pool_slack=0.05)
