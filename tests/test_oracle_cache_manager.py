"""Pins of the plain-Python KV-cache page manager model (oracle side).

Checked against what holds for any correct paged cache, independently of the
model's own bookkeeping:
  * a byte-level pool simulation: every reported slot is written with a tag
    naming (sequence, token), every reported copy is carried out; reading a
    sequence back through its block table must give exactly its history
    (inherited prefix, then its own tokens);
  * conservation: free blocks + referenced blocks = pool size, and each
    block's count equals the number of tables that hold it;
  * hand-worked small cases of the stated policy (stack order, copy-on-write,
    last-in-first-out preemption);
  * failure atomicity: a refused request leaves every observable unchanged.
"""
import copy

import numpy as np
import pytest

from oracle.kv_cache_manager import (ERR_INVALID_ARG, ERR_OUT_OF_BLOCKS, OK,
                                     KVCacheManagerModel)


class PoolSim:
    """Token tags in a [num_blocks * P] array, written only through slots."""

    def __init__(self, n, P):
        self.P = P
        self.cell = np.full(n * P, -1, np.int64)
        self.hist = {}

    def apply(self, m, seq_ids, counts, slots, copies):
        for a, b in copies:                 # copies come before the new writes
            self.cell[b * self.P:(b + 1) * self.P] = self.cell[a * self.P:(a + 1) * self.P]
        k = 0
        for s, c in zip(seq_ids, counts):
            for _ in range(c):
                tag = s * 1_000_000 + len(self.hist[s])
                self.cell[slots[k]] = tag
                self.hist[s].append(tag)
                k += 1
        assert k == len(slots)

    def check(self, m):
        ids = sorted(m.seqs)
        tab, lens = m.block_tables(ids)
        for r, s in enumerate(ids):
            L = int(lens[r])
            got = [int(self.cell[tab[r, i // m.P] * m.P + i % m.P]) for i in range(L)]
            assert got == self.hist[s], f"sequence {s} reads back wrong tokens"
            assert all(tab[r, j] == -1 for j in range(-(-L // m.P), m.M))


def conservation(m):
    held = {}
    for pages, _, _ in m.seqs.values():
        for b in pages:
            held[b] = held.get(b, 0) + 1
    assert len(m.free) + len(held) == m.N
    assert len(set(m.free)) == len(m.free) and not (set(m.free) & set(held))
    for b in range(m.N):
        assert m.ref[b] == held.get(b, 0)


def snapshot(m):
    return copy.deepcopy((m.free, m.ref, m.seqs, m.admitted))


def test_hand_worked_append_fork_and_copy_on_write():
    m = KVCacheManagerModel(num_blocks=4, block_size=2, max_blocks_per_seq=3)
    assert m.add(0) == OK
    st, slots, cp = m.append([0], [3])
    assert st == OK and slots.tolist() == [0, 1, 2] and cp.shape == (0, 2)
    assert m.pages(0) == [0, 1] and m.num_free() == 2
    # child shares the first 3 tokens: pages 0 and 1 (page 1 half full)
    assert m.fork(0, 1, 3) == OK and m.pages(1) == [0, 1] and m.ref[:2] == [2, 2]
    # the child writes into the shared half page: copy it to block 2 first
    st, slots, cp = m.append([1], [1])
    assert st == OK and cp.tolist() == [[1, 2]] and slots.tolist() == [2 * 2 + 1]
    assert m.pages(1) == [0, 2] and m.ref[1] == 1 and m.ref[2] == 1
    # the parent now owns page 1 alone: writes in place, no copy
    st, slots, cp = m.append([0], [1])
    assert st == OK and cp.shape == (0, 2) and slots.tolist() == [1 * 2 + 1]
    # the parent's next token needs a new page: block 3, the last free one
    st, slots, cp = m.append([0], [1])
    assert st == OK and slots.tolist() == [3 * 2 + 0] and m.num_free() == 0
    # release pushes pages last first; shared page 0 stays with the child
    assert m.release(0) == OK
    assert m.free == [3, 1] and m.ref[0] == 1
    st, slots, _ = m.append([1], [1])            # pops block 1 (top of the stack)
    assert st == OK and slots.tolist() == [1 * 2]


def test_page_aligned_fork_needs_no_copy():
    m = KVCacheManagerModel(8, 4, 4)
    m.add(7)
    m.append([7], [8])
    m.fork(7, 8, 8)
    st, slots, cp = m.append([8, 7], [1, 1])
    assert st == OK and cp.shape == (0, 2)
    assert slots.tolist() == [2 * 4, 3 * 4]      # fresh pages, child first (call order)


def test_two_sharers_append_in_one_call():
    # both sharers of a partial page append in the same call: the first one
    # copies, the second then owns the original alone and writes in place
    m = KVCacheManagerModel(6, 4, 3)
    m.add(0)
    m.append([0], [5])                           # pages 0, 1 (1 token in page 1)
    m.fork(0, 1, 5)
    assert m.blocks_needed([1, 0], [1, 1]) == 1
    st, slots, cp = m.append([1, 0], [1, 1])
    assert st == OK and cp.tolist() == [[1, 2]]
    assert slots.tolist() == [2 * 4 + 1, 1 * 4 + 1]


def test_out_of_blocks_is_atomic():
    m = KVCacheManagerModel(3, 2, 8)
    m.add(0)
    m.add(1)
    m.append([0], [3])
    before = snapshot(m)
    st, slots, cp = m.append([1, 0], [2, 2])     # needs 2 blocks, 1 free
    assert st == ERR_OUT_OF_BLOCKS and len(slots) == 0 and len(cp) == 0
    assert snapshot(m) == before


def test_invalid_requests_are_refused_without_change():
    m = KVCacheManagerModel(4, 2, 2)
    m.add(0)
    before = snapshot(m)
    assert m.append([0, 0], [1, 1])[0] == ERR_INVALID_ARG      # duplicate
    assert m.append([5], [1])[0] == ERR_INVALID_ARG            # unknown
    assert m.append([0], [5])[0] == ERR_INVALID_ARG            # beyond the table
    assert m.fork(0, 1, 1) == ERR_INVALID_ARG                  # beyond its length
    assert m.add(0) == ERR_INVALID_ARG
    assert m.release(3) == ERR_INVALID_ARG
    assert snapshot(m) == before


def test_lifo_preemption_order_and_protection():
    m = KVCacheManagerModel(6, 2, 4)
    for s in (10, 11, 12):
        m.add(s)
    m.append([10, 11, 12], [4, 2, 2])            # 2 + 1 + 1 pages; 2 free
    st, victims = m.preempt_for(4, protected=[12])
    assert st == OK and victims == [11, 10] and m.num_free() == 5
    assert sorted(m.seqs) == [12]
    # one victim at a time when fewer blocks are needed
    m2 = KVCacheManagerModel(6, 2, 4)
    for s in (10, 11, 12):
        m2.add(s)
    m2.append([10, 11, 12], [4, 2, 2])
    st, victims = m2.preempt_for(3, protected=[12])
    assert st == OK and victims == [11] and m2.num_free() == 3
    st, victims = m2.preempt_for(5, protected=[12])
    assert st == OK and victims == [10] and m2.num_free() == 5
    before = snapshot(m2)
    st, victims = m2.preempt_for(6, protected=[12])             # impossible
    assert st == ERR_OUT_OF_BLOCKS and victims == [] and snapshot(m2) == before


def test_preemption_counts_shared_pages_once():
    m = KVCacheManagerModel(5, 2, 4)
    m.add(0)
    m.append([0], [4])                           # pages 0, 1
    m.fork(0, 1, 4)                              # shares both
    m.append([1], [2])                           # + page 2
    assert m.num_free() == 2
    st, victims = m.preempt_for(3)               # the child frees only page 2
    assert st == OK and victims == [1] and m.num_free() == 3
    conservation(m)


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_read_back_and_conserve(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.choice([1, 2, 4, 16]))
    m = KVCacheManagerModel(int(rng.integers(8, 64)), P, int(rng.integers(4, 24)))
    sim = PoolSim(m.N, P)
    next_id = 0
    for _ in range(300):
        op = rng.random()
        live = sorted(m.seqs)
        if op < 0.15 or not live:
            assert m.add(next_id) == OK
            sim.hist[next_id] = []
            next_id += 1
        elif op < 0.3:
            parent = int(rng.choice(live))
            n = int(rng.integers(0, m.length(parent) + 1))
            assert m.fork(parent, next_id, n) == OK
            sim.hist[next_id] = list(sim.hist[parent][:n])
            next_id += 1
        elif op < 0.42:
            s = int(rng.choice(live))
            assert m.release(s) == OK
            del sim.hist[s]
        elif op < 0.5:
            st, victims = m.preempt_for(int(rng.integers(0, m.N + 2)))
            for v in victims:
                del sim.hist[v]
            assert st in (OK, ERR_OUT_OF_BLOCKS)
        else:
            k = int(rng.integers(1, min(6, len(live)) + 1))
            ids = [int(x) for x in rng.choice(live, k, replace=False)]
            counts = [int(x) for x in rng.integers(0, 2 * P + 2, k)]
            before = snapshot(m)
            need = m.blocks_needed(ids, counts)
            st, slots, cp = m.append(ids, counts)
            if st == OK:
                assert len(before[0]) - len(m.free) == need
                sim.apply(m, ids, counts, slots, cp)
            else:
                assert snapshot(m) == before
                assert st == (ERR_INVALID_ARG if need < 0 else ERR_OUT_OF_BLOCKS)
        conservation(m)
        sim.check(m)


def test_oracle_copy_blocks_duplicates_whole_blocks_only():
    # the device copy-on-write's oracle: destination blocks become exact
    # copies of their sources in both pools (every kv head, every slot);
    # no other block changes
    import oracle
    rng = np.random.default_rng(9)
    kp = rng.integers(0, 1 << 16, (7, 3, 4, 8)).astype(np.uint16)
    vp = rng.integers(0, 1 << 16, (7, 3, 4, 8)).astype(np.uint16)
    k0, v0 = kp.copy(), vp.copy()
    oracle.copy_blocks(kp, vp, np.array([[1, 5], [3, 6]], np.int32))
    assert np.array_equal(kp[5], k0[1]) and np.array_equal(vp[5], v0[1])
    assert np.array_equal(kp[6], k0[3]) and np.array_equal(vp[6], v0[3])
    for b in (0, 1, 2, 3, 4):
        assert np.array_equal(kp[b], k0[b]) and np.array_equal(vp[b], v0[b])
    oracle.copy_blocks(kp, vp, np.zeros((0, 2), np.int32))    # no pairs: no change
    assert np.array_equal(kp[6], k0[3])
