"""Pins of the plain-Python free-list model (oracle/free_list.py)."""
import pytest

from conftest import read_golden
from oracle.free_list import (DoubleFree, FreeListModel, OutOfBlocks, SplitMix64,
                              hand_out_order)


def test_splitmix64_known_answers():
    for row in read_golden("splitmix64.txt"):
        rng = SplitMix64(int(row[1], 0))
        assert [rng.next() for _ in range(3)] == [int(x, 0) for x in row[2:5]]


def test_unshuffled_stack_hands_out_block_zero_first():
    # "Why Naive KV-Caches Waste >60% VRAM", "Implementation Walkthrough": the
    # stack starts as reversed(range(n)) and pop() returns block 0 first.
    a = FreeListModel(5)
    assert [a.alloc(1)[0] for _ in range(5)] == [0, 1, 2, 3, 4]
    with pytest.raises(OutOfBlocks):
        a.alloc(1)


def test_shuffled_order_is_a_permutation_and_seeded():
    o1 = hand_out_order(4096, 7)
    assert sorted(o1) == list(range(4096))
    assert o1 == hand_out_order(4096, 7)
    assert o1 != hand_out_order(4096, 8)
    assert o1 != list(range(4096))
    # Fisher-Yates with an unbiased draw: position of block 0 is uniform
    counts = [0] * 4
    for seed in range(1, 4001):
        counts[hand_out_order(4, seed).index(0)] += 1
    assert all(900 < c < 1100 for c in counts)


def test_lifo_reuse_and_double_free():
    a = FreeListModel(8)
    x = a.alloc(3)
    a.free([x[1]])
    assert a.alloc(1) == [x[1]]          # last freed comes back first
    with pytest.raises(DoubleFree):
        a.free([x[0], x[0]])
    assert a.free_count() == 5           # failed free changed nothing
    a.free(x)
    with pytest.raises(DoubleFree):
        a.free([x[0]])
    with pytest.raises(DoubleFree):
        a.free([99])


def test_all_or_nothing():
    a = FreeListModel(4)
    a.alloc(3)
    with pytest.raises(OutOfBlocks):
        a.alloc(2)
    assert a.free_count() == 1
    assert len(a.alloc(1)) == 1


def test_churn_500_cycles_16_sequences_no_leaks():
    # PageForge, "Allocator stress test": 500 alloc/free cycles of 16 sequences,
    # 0 leaks, 0 out-of-memory errors.
    import random
    rng = random.Random(5)
    a = FreeListModel(512, shuffle_seed=3)
    for _ in range(500):
        tables = []
        for _ in range(16):
            L = rng.randint(1, 512)
            row = [0] * 32
            cur = 0
            while cur < L:                       # demand paging, a few tokens at a time
                new = min(L, cur + rng.randint(1, 40))
                a.seq_reserve(row, 16, cur, new)
                cur = new
            tables.append((row, L))
        assert a.free_count() == 512 - sum(-(-L // 16) for _, L in tables)
        for row, L in tables:
            a.seq_release(row, 16, L)
        assert a.free_count() == 512
    assert not any(a.owned)


def test_second_batch_gets_first_batch_pages_back():
    # PageForge, "Does the pool actually come back to zero?": batch 2 claims the
    # exact physical pages batch 1 returned.
    a = FreeListModel(512, shuffle_seed=11)
    first = [a.alloc(4) for _ in range(8)]
    for ids in first:
        a.free(ids)
    second = [a.alloc(4) for _ in range(8)]
    assert sorted(sum(first, [])) == sorted(sum(second, []))
    assert a.free_count() == 512 - 32


def test_demand_paging_appends_only_when_last_block_is_full():
    # PagedAttention blog, "Architecture": append into the last block while it
    # has room, otherwise allocate a new block and extend the table.
    a = FreeListModel(10)
    row = [-1] * 4
    a.seq_reserve(row, 16, 0, 1)
    assert row == [0, -1, -1, -1]
    a.seq_reserve(row, 16, 1, 16)
    assert row == [0, -1, -1, -1] and a.free_count() == 9
    a.seq_reserve(row, 16, 16, 17)
    assert row == [0, 1, -1, -1]
    a.seq_reserve(row, 16, 17, 64)
    assert row == [0, 1, 2, 3]
    with pytest.raises(ValueError):
        a.seq_reserve(row, 16, 64, 65)


def _cow_golden():
    g = {}
    for row in read_golden("copy_on_write.txt"):
        g.setdefault(row[0], []).append(row[1:])
    return g


def test_copy_on_write_example_tables():
    """The three sequences of the copy-on-write example, built by forking the
    prefix: the model reproduces the printed tables id for id, counts three
    references on each shared block, and a write into a shared block changes
    only the writer's table."""
    g = _cow_golden()
    B = int(g["block_size"][0][0])
    prefix = int(g["prefix_tokens"][0][0])
    want = {row[0]: [int(x) for x in row[1:]] for row in g["table"]}
    shared = [int(x) for x in g["shared"][0]]
    a = FreeListModel(16)
    a.free(a.alloc(16))                      # every block free again ...
    a.alloc(16)
    a.free([0, 9, 5, 2, 13, 7])              # ... so the stack hands out 7, 13, 2, 5, 9, then 0
    tab_a = a.alloc(prefix // B)             # the prompt's blocks
    tab_a += a.alloc(1)                      # A's first own block
    tab_b = a.seq_fork(tab_a, B, prefix) + a.alloc(1)
    tab_c = a.seq_fork(tab_a, B, prefix) + a.alloc(1)
    assert {"A": tab_a, "B": tab_b, "C": tab_c} == want
    assert [a.refcount(b) for b in shared] == [3, 3]
    assert [a.refcount(t[-1]) for t in (tab_a, tab_b, tab_c)] == [1, 1, 1]
    # B writes into block 13: a new block for B only
    before_a, before_c = list(tab_a), list(tab_c)
    old, new = a.cow(tab_b, 1)
    assert old == 13 and tab_b == [7, new, 5] and new == 0
    assert tab_a == before_a and tab_c == before_c
    assert a.refcount(13) == 2 and a.refcount(new) == 1
    # a private block needs no copy
    assert a.cow(tab_b, 2) is None and tab_b[2] == 5


def test_beam_search_prefix_saving():
    """Beam width 4 over a 1024-token prefix: the prefix is stored once, so
    3 of its 4 copies are eliminated."""
    g = _cow_golden()
    B = int(g["block_size"][0][0])
    width = int(g["beam_width"][0][0])
    tokens = int(g["beam_prefix_tokens"][0][0])
    n = tokens // B
    a = FreeListModel(4 * n)
    root = a.alloc(n)
    beams = [root] + [a.seq_fork(root, B, tokens) for _ in range(width - 1)]
    used = 4 * n - a.free_count()
    assert used == n
    assert (width * n - used) // n == int(g["copies_eliminated"][0][0])
    assert all(a.refcount(b) == width for b in root)
    # the prefix returns to the pool only with its last beam
    for i, t in enumerate(beams):
        a.free(t)
        assert a.free_count() == (4 * n if i == width - 1 else 3 * n)


def test_shared_frees_and_double_free():
    a = FreeListModel(8)
    x = a.alloc(2)
    a.share(x)
    a.share([x[0]])
    assert [a.refcount(b) for b in x] == [3, 2]
    # listing a block more often than it is referenced: error, no change
    with pytest.raises(DoubleFree):
        a.free([x[1], x[1], x[1]])
    assert [a.refcount(b) for b in x] == [3, 2] and a.free_count() == 6
    # a block returns to the stack when its last reference goes, in list order
    a.free([x[1], x[0], x[1], x[0]])
    assert a.refcount(x[0]) == 1 and a.stack[-1] == x[1]
    a.free([x[0]])
    assert a.stack[-2:] == [x[1], x[0]] and a.free_count() == 8
    with pytest.raises(ValueError):
        a.share([x[0]])                      # free blocks cannot be shared


def test_cow_without_free_blocks_changes_nothing():
    a = FreeListModel(3)
    x = a.alloc(3)
    a.share([x[0]])
    row = [x[0]]
    with pytest.raises(OutOfBlocks):
        a.cow(row, 0)
    assert row == [x[0]] and a.refcount(x[0]) == 2 and a.free_count() == 0
