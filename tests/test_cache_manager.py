"""The native host page manager (pkv_cache_* through the C ABI) against the
plain-Python oracle model: identical statuses, slot mappings, copy-on-write
pairs, preemption victims, block tables and lengths, step by step, on random
operation sequences and on the hand-worked cases.  Host code only: runs
without a GPU."""
import numpy as np
import pytest

import paged_kv_attention_31_gb300 as pkv
from oracle.kv_cache_manager import KVCacheManagerModel


def _same_state(nat, ref):
    assert nat.num_free() == ref.num_free()
    assert nat.num_seqs() == len(ref.seqs)
    ids = sorted(ref.seqs)
    t1, l1 = nat.block_tables(ids)
    t2, l2 = ref.block_tables(ids)
    assert np.array_equal(t1, t2) and np.array_equal(l1, l2)
    for s in ids:
        assert nat.length(s) == ref.length(s)


def _both(N, P, M):
    return pkv.KVCacheManager(N, P, M), KVCacheManagerModel(N, P, M)


def test_status_codes_agree():
    assert pkv.PKV_ERR_OUT_OF_BLOCKS == 7
    assert "blocks" in pkv.status_string(7)


def test_hand_worked_case_matches():
    nat, ref = _both(4, 2, 3)
    for m in (nat, ref):
        assert m.add(0) == 0
    for ids, cnt in (([0], [3]),):
        a, b = nat.append(ids, cnt), ref.append(ids, cnt)
        assert a[0] == b[0] and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert nat.fork(0, 1, 3) == ref.fork(0, 1, 3) == 0
    for ids, cnt in (([1], [1]), ([0], [1]), ([0], [1]), ([0], [1]), ([1], [5])):
        a, b = nat.append(ids, cnt), ref.append(ids, cnt)
        assert a[0] == b[0] and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
        _same_state(nat, ref)


def test_create_rejects_bad_sizes():
    for args in ((0, 16, 4), (4, 0, 4), (4, 16, 0), (-1, 16, 4)):
        with pytest.raises(pkv.PkvError):
            pkv.KVCacheManager(*args)


def test_block_tables_of_unknown_sequence_is_an_error():
    nat = pkv.KVCacheManager(8, 4, 2)
    nat.add(3)
    with pytest.raises(pkv.PkvError):
        nat.block_tables([3, 4])


@pytest.mark.parametrize("seed", range(12))
def test_random_operations_match_oracle(seed):
    rng = np.random.default_rng(1000 + seed)
    P = int(rng.choice([1, 2, 4, 16, 32, 64]))
    N = int(rng.integers(4, 96))
    M = int(rng.integers(2, 40))
    nat, ref = _both(N, P, M)
    next_id = int(rng.integers(0, 1 << 40))          # large ids: int64 end to end
    for _ in range(400):
        live = sorted(ref.seqs)
        op = rng.random()
        if op < 0.12 or not live:
            assert nat.add(next_id) == ref.add(next_id)
            next_id += int(rng.integers(1, 5))
        elif op < 0.25:
            parent = int(rng.choice(live))
            n = int(rng.integers(-1, ref.length(parent) + 2))   # includes invalid
            assert nat.fork(parent, next_id, n) == ref.fork(parent, next_id, n)
            next_id += 1
        elif op < 0.35:
            s = int(rng.choice(live)) if rng.random() < 0.9 else -5
            assert nat.release(s) == ref.release(s)
        elif op < 0.45:
            need = int(rng.integers(0, N + 3))
            prot = [int(x) for x in rng.choice(live, min(len(live), int(rng.integers(0, 3))),
                                               replace=False)]
            a, b = nat.preempt_for(need, prot), ref.preempt_for(need, prot)
            assert a == (b[0], b[1])
        else:
            k = int(rng.integers(1, min(8, len(live)) + 1))
            ids = [int(x) for x in rng.choice(live, k, replace=False)]
            if rng.random() < 0.05:
                ids.append(ids[0])                                   # duplicate
            counts = [int(x) for x in rng.integers(0, 2 * P + 3, len(ids))]
            assert nat.blocks_needed(ids, counts) == ref.blocks_needed(ids, counts)
            a, b = nat.append(ids, counts), ref.append(ids, counts)
            assert a[0] == b[0]
            assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
        _same_state(nat, ref)
