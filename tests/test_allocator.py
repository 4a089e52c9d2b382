"""The product allocator (C ABI, host only) against the oracle's free-list model,
block id for block id."""
import random

import numpy as np
import pytest

from oracle.free_list import FreeListModel, OutOfBlocks as ModelOOM, DoubleFree as ModelDF


@pytest.mark.parametrize("seed", [0, 7, 12345, 2**64 - 1])
def test_hand_out_order_matches_model(pkv, seed):
    n = 4096
    a = pkv.pf_alloc_create(n, seed)
    model = FreeListModel(n, seed)
    got = pkv.pf_alloc_blocks(a, n)
    assert got.tolist() == model.alloc(n)
    assert pkv.pf_alloc_free_count(a) == 0


def test_exhaustion_and_all_or_nothing(pkv):
    a = pkv.pf_alloc_create(10, 3)
    first = pkv.pf_alloc_blocks(a, 8)
    with pytest.raises(pkv.OutOfBlocks):
        pkv.pf_alloc_blocks(a, 3)
    assert pkv.pf_alloc_free_count(a) == 2
    rest = pkv.pf_alloc_blocks(a, 2)
    assert sorted(first.tolist() + rest.tolist()) == list(range(10))
    with pytest.raises(pkv.OutOfBlocks):
        pkv.pf_alloc_blocks(a, 1)


def test_double_free_changes_nothing(pkv):
    a = pkv.pf_alloc_create(8, 0)
    ids = pkv.pf_alloc_blocks(a, 4)
    with pytest.raises(pkv.DoubleFree):
        pkv.pf_free_blocks(a, [ids[0], ids[1], ids[0]])
    assert pkv.pf_alloc_free_count(a) == 4
    with pytest.raises(pkv.DoubleFree):
        pkv.pf_free_blocks(a, [7])            # never allocated
    with pytest.raises(pkv.DoubleFree):
        pkv.pf_free_blocks(a, [-1])
    pkv.pf_free_blocks(a, ids)
    assert pkv.pf_alloc_free_count(a) == 8
    with pytest.raises(pkv.DoubleFree):
        pkv.pf_free_blocks(a, ids[:1])


def test_lifo_reuse_matches_model(pkv):
    a = pkv.pf_alloc_create(64, 9)
    m = FreeListModel(64, 9)
    rng = random.Random(1)
    live = []
    for _ in range(2000):
        if live and rng.random() < 0.45:
            k = rng.randrange(len(live))
            ids = live.pop(k)
            pkv.pf_free_blocks(a, ids)
            m.free(ids)
        else:
            n = rng.randint(0, 6)
            try:
                want = m.alloc(n)
            except ModelOOM:
                with pytest.raises(pkv.OutOfBlocks):
                    pkv.pf_alloc_blocks(a, n)
                continue
            got = pkv.pf_alloc_blocks(a, n).tolist()
            assert got == want
            live.append(got)
        assert pkv.pf_alloc_free_count(a) == m.free_count()


def test_demand_paging_churn_matches_model_no_leaks(pkv):
    # PageForge "Allocator stress test": 500 alloc/free cycles of 16 sequences.
    B, N, MAXB = 16, 512, 32
    a = pkv.pf_alloc_create(N, 5)
    m = FreeListModel(N, 5)
    rng = random.Random(2)
    for _ in range(500):
        seqs = []
        for _ in range(16):
            L = rng.randint(1, MAXB * B)
            row = np.zeros(MAXB, dtype=np.int32)
            mrow = [0] * MAXB
            cur = 0
            while cur < L:
                new = min(L, cur + rng.randint(1, 48))
                pkv.pf_seq_reserve(a, B, row, cur, new)
                m.seq_reserve(mrow, B, cur, new)
                cur = new
            assert row.tolist() == mrow
            seqs.append((row, mrow, L))
        for row, mrow, L in seqs:
            pkv.pf_seq_release(a, B, row, L)
            m.seq_release(mrow, B, L)
        assert pkv.pf_alloc_free_count(a) == N == m.free_count()


def test_seq_reserve_rejects_short_row_and_is_atomic_on_oom(pkv):
    a = pkv.pf_alloc_create(4, 0)
    row = np.zeros(3, dtype=np.int32)
    with pytest.raises(pkv.PagedKVError):
        pkv.pf_seq_reserve(a, 16, row, 0, 49)      # needs 4 blocks, row holds 3
    pkv.pf_seq_reserve(a, 16, row, 0, 33)          # 3 blocks
    assert row.tolist() == [0, 1, 2]
    other = np.zeros(4, dtype=np.int32)
    with pytest.raises(pkv.OutOfBlocks):
        pkv.pf_seq_reserve(a, 16, other, 0, 40)    # needs 3, 1 free
    assert other.tolist() == [0, 0, 0, 0] and pkv.pf_alloc_free_count(a) == 1
    with pytest.raises(pkv.PagedKVError):
        pkv.pf_seq_reserve(a, 16, row, 33, 20)     # shrinking is not a reserve


def test_shared_blocks_and_copy_on_write_match_model(pkv):
    """Forks, copy-on-write and frees of shared blocks: the product and the
    model hand out the same ids and keep the same reference counts, and fail
    on the same steps (PagedAttention blog, "Copy-on-Write for Parallel
    Sampling")."""
    B, N, MAXB = 16, 96, 12
    a = pkv.pf_alloc_create(N, 5)
    m = FreeListModel(N, 5)
    rng = random.Random(3)
    seqs = []   # (product row, model row, length)
    for step in range(3000):
        r = rng.random()
        if r < 0.25 or not seqs:                 # new sequence
            L = rng.randrange(1, MAXB * B)
            row = np.zeros(MAXB, dtype=np.int32)
            mrow = [0] * MAXB
            try:
                m.seq_reserve(mrow, B, 0, L)
                ok = True
            except ModelOOM:
                ok = False
            if ok:
                pkv.pf_seq_reserve(a, B, row, 0, L)
                seqs.append((row, mrow, L))
            else:
                with pytest.raises(pkv.OutOfBlocks):
                    pkv.pf_seq_reserve(a, B, row, 0, L)
        elif r < 0.45:                            # fork a prefix
            row, mrow, L = seqs[rng.randrange(len(seqs))]
            Lc = rng.randrange(1, L + 1)
            child = np.zeros(MAXB, dtype=np.int32)
            pkv.pf_seq_fork(a, B, row, Lc, child)
            mchild = m.seq_fork(mrow, B, Lc) + [0] * (MAXB - -(-Lc // B))
            seqs.append((child, mchild, Lc))
        elif r < 0.7:                             # write into a block: copy-on-write first
            row, mrow, L = seqs[rng.randrange(len(seqs))]
            j = rng.randrange(-(-L // B))
            try:
                want = m.cow(mrow, j)
                ok = True
            except ModelOOM:
                ok = False
            if ok:
                got = pkv.pf_alloc_cow(a, row, j)
                assert got == want
            else:
                before = row.copy()
                with pytest.raises(pkv.OutOfBlocks):
                    pkv.pf_alloc_cow(a, row, j)
                assert np.array_equal(row, before)
        else:                                     # a sequence finishes
            row, mrow, L = seqs.pop(rng.randrange(len(seqs)))
            pkv.pf_seq_release(a, B, row, L)
            m.seq_release(mrow, B, L)
        assert pkv.pf_alloc_free_count(a) == m.free_count()
        if step % 97 == 0:
            assert [pkv.pf_alloc_refcount(a, b) for b in range(N)] == [m.refcount(b) for b in range(N)]
        for row, mrow, L in seqs[-3:]:
            assert row.tolist() == mrow
    # a block listed more often than it is referenced: error, no change
    for row, mrow, L in seqs:
        pkv.pf_seq_release(a, B, row, L)
        m.seq_release(mrow, B, L)
    assert pkv.pf_alloc_free_count(a) == N == m.free_count()
    ids = pkv.pf_alloc_blocks(a, 2)
    pkv.pf_alloc_share(a, ids[:1])
    with pytest.raises(pkv.DoubleFree):
        pkv.pf_free_blocks(a, [ids[0], ids[0], ids[0]])
    assert pkv.pf_alloc_refcount(a, ids[0]) == 2
    with pytest.raises(pkv.PagedKVError):
        pkv.pf_alloc_share(a, [N - 1 if N - 1 not in ids else 0])   # a free block
    assert pkv.pf_alloc_refcount(a, -1) == -1
