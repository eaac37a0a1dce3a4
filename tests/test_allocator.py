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


def test_fork_shares_the_prefix_blocks():
    a = kv.BlockAllocator(16)
    BS = 16
    parent = np.full(4, -1, dtype=np.int32)
    a.grow(parent, BS, 0, 37)                  # 3 blocks, the last one partial
    child = np.full(4, -1, dtype=np.int32)
    a.fork(parent, child, BS, 37)
    assert list(child[:3]) == list(parent[:3]) and child[3] == -1
    assert [a.refcount(b) for b in parent[:3]] == [2, 2, 2]
    assert a.num_free == 13
    # a fork of a block that is not allocated changes nothing
    bad = np.array([parent[0], 15, -1, -1], dtype=np.int32)
    with pytest.raises(kv.KvattnError):
        a.fork(bad, np.full(4, -1, dtype=np.int32), BS, 20)
    assert a.refcount(parent[0]) == 2
    with pytest.raises(kv.KvattnError):
        a.fork(parent, child, BS, 5 * BS)      # wider than the row


def test_prepare_append_copies_a_shared_partial_block_once():
    a = kv.BlockAllocator(16)
    BS = 16
    parent = np.full(4, -1, dtype=np.int32)
    a.grow(parent, BS, 0, 37)
    child = np.full(4, -1, dtype=np.int32)
    a.fork(parent, child, BS, 37)
    shared_last = int(parent[2])
    # the child appends at position 37, inside the shared block 2: copy on write
    cow = a.prepare_append(child, BS, 37, 38)
    assert cow is not None and cow[0] == shared_last and cow[1] != shared_last
    assert child[2] == cow[1] and a.refcount(cow[1]) == 1 and a.refcount(shared_last) == 1
    assert list(child[:2]) == list(parent[:2])  # full blocks stay shared
    # the parent now holds the old block alone: its append writes in place
    assert a.prepare_append(parent, BS, 37, 38) is None and parent[2] == shared_last
    # appends that start a block, or append nothing, never copy
    assert a.prepare_append(child, BS, 38, 48) is None
    assert a.prepare_append(child, BS, 48, 50) is None and child[3] >= 0
    assert a.prepare_append(child, BS, 50, 50) is None
    # releasing both sequences returns every block
    a.release(child, BS, 50)
    a.release(parent, BS, 38)
    assert a.num_free == 16


def test_prepare_append_is_all_or_nothing():
    a = kv.BlockAllocator(4)
    BS = 16
    parent = np.full(4, -1, dtype=np.int32)
    a.grow(parent, BS, 0, 20)                  # 2 blocks
    child = np.full(4, -1, dtype=np.int32)
    a.fork(parent, child, BS, 20)
    before = child.copy()
    # copy (1 block) + 2 new blocks > 2 free: nothing changes
    with pytest.raises(kv.KvattnError) as e:
        a.prepare_append(child, BS, 20, 60)
    assert e.value.name == "KVATTN_ERR_OUT_OF_BLOCKS"
    assert np.array_equal(child, before) and a.num_free == 2 and a.num_failures == 1
    assert a.refcount(parent[1]) == 2
    # copy + 1 new block fits
    assert a.prepare_append(child, BS, 20, 40) is not None and a.num_free == 0
    # a partial block that is not allocated is an error
    row = np.array([-1, -1, -1, -1], dtype=np.int32)
    with pytest.raises(kv.KvattnError):
        a.prepare_append(row, BS, 5, 6)
    with pytest.raises(kv.KvattnError):
        a.prepare_append(child, BS, 40, 39)    # shrinking


def test_random_sequences_with_forks_against_a_model():
    """Sequences that grow, fork (shared prefix) and get released, driven
    through fork / prepare_append / release, checked against a plain model of
    which block holds which token of which sequence: a token is never written
    into a block another live sequence still reads, and every count matches."""
    rng = np.random.default_rng(3)
    BS, W, n = 16, 12, 160
    a = kv.BlockAllocator(n)
    seqs = {}            # id -> (table row, length)
    next_id = 0

    def refs_model():
        c = {}
        for sid, (row, L) in seqs.items():
            for b in row[: (L + BS - 1) // BS]:
                c[int(b)] = c.get(int(b), 0) + 1
        return c

    for _ in range(1500):
        op = rng.integers(0, 4)
        if op == 0 or not seqs:                       # new sequence
            row = np.full(W, -1, dtype=np.int32)
            L = int(rng.integers(1, 60))
            try:
                a.grow(row, BS, 0, L)
            except kv.KvattnError:
                continue
            seqs[next_id] = (row, L)
            next_id += 1
        elif op == 1:                                 # fork a prefix of a live sequence
            sid = int(rng.choice(list(seqs)))
            row, L = seqs[sid]
            P = int(rng.integers(1, L + 1))
            child = np.full(W, -1, dtype=np.int32)
            a.fork(row, child, BS, P)
            seqs[next_id] = (child, P)
            next_id += 1
        elif op == 2:                                 # append to a sequence
            sid = int(rng.choice(list(seqs)))
            row, L = seqs[sid]
            new = min(W * BS, L + int(rng.integers(1, 40)))
            if new == L:
                continue
            before = row.copy()
            shared_partial = L % BS != 0 and refs_model().get(int(row[(L - 1) // BS]), 0) > 1
            try:
                cow = a.prepare_append(row, BS, L, new)
            except kv.KvattnError:
                assert np.array_equal(row, before)    # all or nothing
                continue
            assert (cow is not None) == shared_partial
            if cow is not None:
                assert cow[0] == before[(L - 1) // BS] and row[(L - 1) // BS] == cow[1]
            # every block this append writes into is held by this sequence alone
            seqs[sid] = (row, new)
            held = refs_model()
            for blk in row[L // BS: (new + BS - 1) // BS]:
                assert held[int(blk)] == 1
        else:                                         # release a sequence
            sid = int(rng.choice(list(seqs)))
            row, L = seqs.pop(sid)
            a.release(row, BS, L)
        model = refs_model()
        assert a.num_free == n - len(model)
        for b, r in model.items():
            assert a.refcount(b) == r
    for sid, (row, L) in list(seqs.items()):
        a.release(row, BS, L)
    assert a.num_free == n
