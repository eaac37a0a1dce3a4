"""Host block allocator: free-list and reference-count invariants (CPU only)."""
import threading

import numpy as np
import pytest

import kv_cache_attention_rope_gb300 as kv


def test_create_rejects_bad_sizes():
    with pytest.raises(kv.KvattnError):
        kv.BlockAllocator(0)
    with pytest.raises(kv.KvattnError):
        kv.BlockAllocator(2**31)


def test_all_or_nothing_and_failure_count():
    a = kv.BlockAllocator(10)
    ids = a.alloc(7)
    assert sorted(ids) == list(range(7)) or len(set(ids)) == 7
    assert a.num_free == 3
    with pytest.raises(kv.KvattnError) as e:
        a.alloc(4)
    assert e.value.name == "KVATTN_ERR_OUT_OF_BLOCKS"
    assert a.num_free == 3 and a.num_failures == 1
    more = a.alloc(3)
    assert a.num_free == 0
    assert set(ids) | set(more) == set(range(10))


def test_freed_blocks_are_reused_lifo():
    a = kv.BlockAllocator(100)
    ids = a.alloc(10)
    a.free(ids[3:5])
    again = a.alloc(2)
    assert set(again) == set(ids[3:5])


def test_double_free_and_bad_ids_change_nothing():
    a = kv.BlockAllocator(8)
    ids = a.alloc(4)
    a.free([ids[0]])
    with pytest.raises(kv.KvattnError):
        a.free([ids[0]])                     # double free
    with pytest.raises(kv.KvattnError):
        a.free([ids[1], ids[1]])             # one reference, two frees
    with pytest.raises(kv.KvattnError):
        a.free([ids[2], 99])                 # out of range: ids[2] must stay allocated
    assert a.refcount(ids[2]) == 1
    assert a.num_free == 5
    assert a.refcount(-1) == -1 and a.refcount(8) == -1


def test_shared_blocks_return_on_last_reference():
    a = kv.BlockAllocator(4)
    ids = a.alloc(2)
    a.share(ids)
    assert a.refcount(ids[0]) == 2
    a.free(ids)
    assert a.num_free == 2 and a.refcount(ids[0]) == 1
    a.free([ids[0], ids[1]])
    assert a.num_free == 4 and a.refcount(ids[0]) == 0
    with pytest.raises(kv.KvattnError):
        a.share([ids[0]])                    # not allocated


def test_random_sequence_against_a_set_model():
    rng = np.random.default_rng(0)
    n = 500
    a = kv.BlockAllocator(n)
    refs = {}
    for _ in range(3000):
        op = rng.integers(0, 3)
        if op == 0:
            k = int(rng.integers(0, 20))
            free_now = n - len(refs)
            if k > free_now:
                with pytest.raises(kv.KvattnError):
                    a.alloc(k)
            else:
                for i in a.alloc(k):
                    assert int(i) not in refs
                    refs[int(i)] = 1
        elif op == 1 and refs:
            pick = rng.choice(list(refs), size=min(len(refs), int(rng.integers(1, 8))), replace=False)
            a.free(pick)
            for i in pick:
                refs[int(i)] -= 1
                if refs[int(i)] == 0:
                    del refs[int(i)]
        elif op == 2 and refs:
            pick = rng.choice(list(refs), size=1)
            a.share(pick)
            refs[int(pick[0])] += 1
        assert a.num_free == n - len(refs)
    for i, r in refs.items():
        assert a.refcount(i) == r


def test_threads_never_hand_out_a_block_twice():
    a = kv.BlockAllocator(4000)
    got = [[] for _ in range(8)]

    def worker(k):
        for _ in range(200):
            ids = a.alloc(2)
            got[k].extend(ids.tolist())
            if len(got[k]) > 100:
                a.free(got[k][:50])
                del got[k][:50]

    th = [threading.Thread(target=worker, args=(k,)) for k in range(8)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    held = [i for g in got for i in g]
    assert len(held) == len(set(held))
    assert a.num_free == 4000 - len(held)


def test_table_grow_and_release():
    a = kv.BlockAllocator(20)
    row = np.full(8, -1, dtype=np.int32)
    a.grow(row, 16, 0, 1)          # first token: one block
    assert (row[:1] >= 0).all() and (row[1:] == -1).all()
    a.grow(row, 16, 1, 16)         # still one block
    assert (row[1:] == -1).all()
    a.grow(row, 16, 16, 17)        # token 17 opens block 2
    assert row[1] >= 0 and row[2] == -1
    a.grow(row, 16, 17, 128)       # 8 blocks in total
    assert (row >= 0).all() and len(set(row.tolist())) == 8
    with pytest.raises(kv.KvattnError):
        a.grow(row, 16, 128, 129)  # row too narrow
    assert a.num_free == 12
    a.release(row, 16, 128)
    assert (row == -1).all() and a.num_free == 20


def test_table_grow_is_all_or_nothing():
    a = kv.BlockAllocator(3)
    row = np.full(8, -1, dtype=np.int32)
    with pytest.raises(kv.KvattnError):
        a.grow(row, 16, 0, 64)     # needs 4 blocks, 3 exist
    assert (row == -1).all() and a.num_free == 3 and a.num_failures == 1


def test_claim_adopts_an_existing_table():
    a = kv.BlockAllocator(10)
    a.claim([7, 2, 5])
    assert a.num_free == 7 and a.refcount(7) == 1
    with pytest.raises(kv.KvattnError):
        a.claim([1, 2])          # 2 is taken: nothing changes
    assert a.refcount(1) == 0
    with pytest.raises(kv.KvattnError):
        a.claim([3, 3])          # repeated
    with pytest.raises(kv.KvattnError):
        a.claim([10])            # out of range
    got = set(a.alloc(7).tolist())
    assert got == {0, 1, 3, 4, 6, 8, 9}
    a.free([2])
    assert a.alloc(1).tolist() == [2]
