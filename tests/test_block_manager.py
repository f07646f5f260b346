"""Host block manager (include/pkv_blocks.h) against its definition: slots
follow block tables, blocks are taken only at block boundaries, full blocks
are shared only between sequences whose token prefixes match, reference
counts free blocks exactly when no table holds them, cached free blocks are
evicted in release order, and a request that does not fit changes nothing."""
import numpy as np
import pytest

from paged_kv_cache_mapping_gb300 import PkvError
from paged_kv_cache_mapping_gb300 import build as pkv_build
from paged_kv_cache_mapping_gb300.blocks import BlockManager

BS = 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkv_build.build()


def slots_of(table, start, n, bs=BS):
    p = np.arange(start, start + n)
    return table[p // bs] * bs + p % bs


def test_slots_follow_the_table_and_blocks_come_at_boundaries():
    bm = BlockManager(64, BS)
    assert bm.add_sequence(1, np.arange(5)) == 0
    s = bm.append(1, np.arange(5))
    table, n = bm.block_table(1)
    assert n == 5 and table.size == 1
    assert np.array_equal(s, slots_of(table, 0, 5))
    s2 = bm.append(1, np.arange(11))  # fills block 0 exactly
    table, n = bm.block_table(1)
    assert n == 16 and table.size == 1 and np.array_equal(s2, slots_of(table, 5, 11))
    bm.append(1, [7])  # crosses the boundary
    table, n = bm.block_table(1)
    assert n == 17 and table.size == 2
    assert bm.stats()["free_blocks"] == 62


def test_prefix_sharing_leaves_the_last_prompt_token_to_compute():
    bm = BlockManager(64, BS)
    prompt = np.arange(100, 140)  # 2 full blocks + 8
    assert bm.add_sequence(1, prompt) == 0
    bm.append(1, prompt)
    assert bm.add_sequence(2, prompt) == 32
    t1, _ = bm.block_table(1)
    t2, n2 = bm.block_table(2)
    assert n2 == 32 and np.array_equal(t2, t1[:2])
    bm.append(2, prompt[32:])
    t2, n2 = bm.block_table(2)
    assert n2 == 40 and t2[2] != t1[2]
    # a prompt of exactly two blocks keeps its last token to compute: one block cached
    assert bm.add_sequence(3, prompt[:32]) == 16
    st = bm.stats()
    assert st["prefix_hit_blocks"] == 3 and st["num_sequences"] == 3


def test_an_edit_in_the_first_block_shares_nothing():
    bm = BlockManager(64, BS)
    prompt = np.arange(200, 260)
    bm.add_sequence(1, prompt)
    bm.append(1, prompt)
    edited = prompt.copy()
    edited[3] += 1
    assert bm.add_sequence(2, edited) == 0
    edited2 = prompt.copy()
    edited2[20] += 1  # second block differs: only the first is shared
    assert bm.add_sequence(3, edited2) == 16


def test_cached_blocks_survive_release_and_are_evicted_in_release_order():
    bm = BlockManager(8, BS)
    prompt = np.arange(300, 340)
    bm.add_sequence(1, prompt)
    bm.append(1, prompt)  # 3 blocks, 2 full and cached
    bm.free_sequence(1)
    st = bm.stats()
    assert st["free_blocks"] == 8 and st["cached_blocks"] == 2
    assert bm.add_sequence(2, prompt) == 32  # hits the released blocks
    bm.free_sequence(2)
    # fill the pool with something else: blocks never cached and the
    # released partial blocks go first, the cached prefix (released last) after
    bm.add_sequence(3, np.arange(5))
    bm.append(3, np.arange(16 * 6))  # 6 blocks
    st = bm.stats()  # cached: the prompt's 2 released blocks + sequence 3's 6 full ones
    assert st["evictions"] == 0 and st["cached_blocks"] == 8 and st["free_blocks"] == 2
    bm.append(3, np.arange(32))  # 2 more: the prompt's cached blocks are evicted
    st = bm.stats()
    assert st["free_blocks"] == 0 and st["evictions"] == 2 and st["cached_blocks"] == 8
    bm.free_sequence(3)
    assert bm.add_sequence(5, prompt) == 0


def test_a_request_that_does_not_fit_changes_nothing():
    bm = BlockManager(4, BS)
    bm.add_sequence(1, np.arange(10))
    bm.append(1, np.arange(10))
    before = bm.stats()
    with pytest.raises(PkvError) as ei:
        bm.append(1, np.arange(16 * 4))
    assert ei.value.status == 6
    assert bm.stats() == before
    t, n = bm.block_table(1)
    assert n == 10 and t.size == 1
    bm.add_sequence(2, np.arange(3))
    with pytest.raises(PkvError):
        bm.build_step([1, 2], [16, 40], np.zeros(56, np.int32), 8)
    assert bm.stats()["free_blocks"] == 3 and bm.block_table(2)[1] == 0


def test_build_step_packs_the_kernels_inputs():
    bm = BlockManager(64, BS)
    for sid, n in ((7, 20), (9, 3)):
        bm.add_sequence(sid, np.arange(n))
    cu, sl, bt, slots = bm.build_step([7, 9], [20, 3], np.arange(23), max_blocks=4)
    assert cu.tolist() == [0, 20, 23] and sl.tolist() == [20, 3]
    t7, _ = bm.block_table(7)
    t9, _ = bm.block_table(9)
    assert bt[0, :2].tolist() == t7.tolist() and bt[0, 2:].tolist() == [-1, -1]
    assert bt[1, 0] == t9[0] and (bt[1, 1:] == -1).all()
    assert np.array_equal(slots[:20], slots_of(t7, 0, 20)) and np.array_equal(slots[20:], slots_of(t9, 0, 3))
    with pytest.raises(PkvError):
        bm.build_step([7, 7], [1, 1], np.arange(2), max_blocks=4)  # one sequence twice


def test_random_churn_keeps_the_invariants():
    rng = np.random.default_rng(5)
    nb = 40
    bm = BlockManager(nb, BS)
    prefixes = [rng.integers(0, 1000, 48) for _ in range(3)]
    live = {}  # seq id -> token ids so far
    next_id = 0
    for step in range(400):
        op = rng.random()
        if op < 0.3 or not live:
            prompt = np.concatenate([prefixes[rng.integers(3)][:rng.integers(0, 49)],
                                     rng.integers(0, 1000, rng.integers(1, 30))])
            cached = bm.add_sequence(next_id, prompt)
            assert cached % BS == 0 and cached <= len(prompt) - 1
            try:
                bm.append(next_id, prompt[cached:])
                live[next_id] = list(prompt)
            except PkvError as e:
                assert e.status == 6
                bm.free_sequence(next_id)
            next_id += 1
        elif op < 0.75:
            sid = int(rng.choice(list(live)))
            new = rng.integers(0, 1000, rng.integers(1, 20))
            try:
                bm.append(sid, new)
                live[sid] += list(new)
            except PkvError as e:
                assert e.status == 6
        else:
            sid = int(rng.choice(list(live)))
            bm.free_sequence(sid)
            del live[sid]
        # invariants
        owners = {}
        for sid, toks in live.items():
            table, n = bm.block_table(sid)
            assert n == len(toks) and table.size == -(-n // BS)
            for i, b in enumerate(table):
                owners.setdefault(int(b), []).append((sid, i))
        for b, who in owners.items():
            if len(who) > 1:  # a shared block: full, same index, same token prefix
                (s0, i0) = who[0]
                for s1, i1 in who[1:]:
                    assert i1 == i0
                    end = (i0 + 1) * BS
                    assert len(live[s0]) >= end and len(live[s1]) >= end
                    assert live[s0][:end] == live[s1][:end]
        st = bm.stats()
        assert st["free_blocks"] == nb - len(owners)
        assert st["num_sequences"] == len(live)
