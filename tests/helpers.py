"""Test-side helpers that restate the layout in a second, independent way.

They never call the oracle or the CUDA library: they derive slots by walking
a sequence's pages token by token (the way a block manager fills them) and
read rows through the flat [num_blocks * block_size] view of a cache.
"""
import numpy as np
import torch


def page_walk_slots(table_row, n_tokens, block_size):
    """Slots of positions 0..n_tokens-1 of one sequence, found by filling its
    pages in order: a page takes block_size tokens, then the next listed
    page starts at offset 0."""
    slots = np.empty(n_tokens, np.int64)
    page, off = 0, 0
    for p in range(n_tokens):
        slots[p] = int(table_row[page]) * block_size + off
        off += 1
        if off == block_size:
            page, off = page + 1, 0
    return slots


def flat_rows(cache, slots):
    """Rows [len(slots), H, D] of a cache [NB, bs, H, D] at the given flat slots."""
    nb, bs = cache.shape[:2]
    return cache.reshape(nb * bs, *cache.shape[2:])[slots]


def bf16_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def e4m3_to_f64(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def values(arr, fmt, scale=1.0):
    if fmt == "f32":
        return arr.astype(np.float64)
    if fmt == "bf16":
        return bf16_to_f64(arr)
    return e4m3_to_f64(arr) * scale


def random_tables(rng, seq_lens, block_size, num_blocks, width=None, contiguous=False):
    nblk = [-(-int(n) // block_size) for n in seq_lens]
    width = width or max(nblk + [1])
    pool = np.arange(num_blocks) if contiguous else rng.permutation(num_blocks)
    assert sum(nblk) <= num_blocks
    tab = np.full((len(seq_lens), width), -1, np.int32)
    c = 0
    for s, n in enumerate(nblk):
        tab[s, :n] = pool[c:c + n]
        c += n
    return tab


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (den if den > 0 else 1.0))
