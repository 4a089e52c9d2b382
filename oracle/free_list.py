"""Plain-Python model of the host free-list block allocator.

TEST INFRASTRUCTURE ONLY: the tests compare the product allocator's block ids
with this model, id for id.  The product never imports this module.

What it models
--------------
* A LIFO stack of free physical block ids; ``alloc`` pops, ``free`` pushes
  ("Why Naive KV-Caches Waste >60% VRAM", "Implementation Walkthrough": the
  allocator is a stack initialised to ``reversed(range(num_blocks))`` so block
  0 is handed out first, ``allocate`` pops and raises when the stack is empty,
  ``free`` appends).  O(1) per block (PageForge, "Five techniques", 02).
* ``alloc(n)`` is all-or-nothing and a failed call changes nothing; freeing a
  block that is not allocated is an error and also changes nothing (PageFault
  README, "Test": exhaustion, double free, all-or-nothing).
* Demand paging: a sequence that grows from ``cur_len`` to ``new_len`` tokens
  gets ``ceil(new_len/B) - ceil(cur_len/B)`` new blocks appended to its table
  row; tokens go into the last block while it has room (PagedAttention blog,
  "Architecture").
* Shared blocks (PagedAttention blog, "Copy-on-Write for Parallel
  Sampling"): a reference count per block tracks the sequences whose tables
  point at it.  ``alloc`` gives a block one reference, ``share`` (a fork:
  the child's table points at the parent's blocks) adds one, and ``free``
  drops one per listed id; a block goes back on the stack when its last
  reference goes, in list order.  Before a write into a block that other
  sequences still reference, ``cow`` gives the writer a fresh block (the
  caller copies the contents), moves one reference from the old block to it
  and patches only the writer's table entry -- fork()'s copy-on-write.
  Listing a block more times than it has references is a double free.
* A "shuffled" pool (what a pool looks like after churn, PageFault README,
  "Four stages") permutes the initial hand-out order with a Fisher-Yates
  shuffle driven by SplitMix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014: state += 0x9E3779B97F4A7C15,
  then the two xor-shift-multiply mixing rounds).  Seed 0 means no shuffle.
  Draws in [0, n) reject the low ``2**64 mod n`` values so they are unbiased.
"""

MASK64 = (1 << 64) - 1


class SplitMix64:
    def __init__(self, seed):
        self.state = seed & MASK64

    def next(self):
        self.state = (self.state + 0x9E3779B97F4A7C15) & MASK64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        return z ^ (z >> 31)

    def below(self, n):
        """Uniform integer in [0, n) by rejection of the biased low range."""
        threshold = ((1 << 64) - n) % n
        while True:
            r = self.next()
            if r >= threshold:
                return r % n


def hand_out_order(n_blocks, shuffle_seed):
    """Order in which a fresh allocator hands out its blocks."""
    order = list(range(n_blocks))
    if shuffle_seed:
        rng = SplitMix64(shuffle_seed)
        for i in range(n_blocks - 1, 0, -1):
            j = rng.below(i + 1)
            order[i], order[j] = order[j], order[i]
    return order


class OutOfBlocks(Exception):
    pass


class DoubleFree(Exception):
    pass


class FreeListModel:
    def __init__(self, n_blocks, shuffle_seed=0):
        self.n_blocks = n_blocks
        self.stack = list(reversed(hand_out_order(n_blocks, shuffle_seed)))
        self.refs = [0] * n_blocks      # references per block; 0 = free

    @property
    def owned(self):
        return [r > 0 for r in self.refs]

    def free_count(self):
        return len(self.stack)

    def refcount(self, b):
        return self.refs[b]

    def alloc(self, n):
        if n < 0:
            raise ValueError("negative block count")
        if n > len(self.stack):
            raise OutOfBlocks(f"need {n} blocks, {len(self.stack)} free")
        ids = [self.stack.pop() for _ in range(n)]
        for b in ids:
            self.refs[b] = 1
        return ids

    def free(self, ids):
        listed = {}
        for b in ids:
            listed[b] = listed.get(b, 0) + 1
            if not (0 <= b < self.n_blocks) or listed[b] > self.refs[b]:
                raise DoubleFree(f"block {b} is not allocated (or listed more often than it is referenced)")
        for b in ids:
            self.refs[b] -= 1
            if self.refs[b] == 0:
                self.stack.append(b)

    def share(self, ids):
        for b in ids:
            if not (0 <= b < self.n_blocks) or self.refs[b] == 0:
                raise ValueError(f"block {b} is not allocated")
        for b in ids:
            self.refs[b] += 1

    def cow(self, table_row, j):
        """Make table_row[j] private before a write into it.  Returns None when
        the block has no other reference, else (old block, new block); the
        caller copies the old block's contents into the new one."""
        b = table_row[j]
        if not (0 <= b < self.n_blocks) or self.refs[b] == 0:
            raise ValueError(f"block {b} is not allocated")
        if self.refs[b] == 1:
            return None
        if not self.stack:
            raise OutOfBlocks("need 1 block, 0 free")
        d = self.stack.pop()
        self.refs[d] = 1
        self.refs[b] -= 1
        table_row[j] = d
        return b, d

    def seq_fork(self, parent_row, block_size, length):
        """A child sequence that shares the parent's first `length` tokens."""
        n = -(-length // block_size)
        child = list(parent_row[:n])
        self.share(child)
        return child

    def seq_reserve(self, table_row, block_size, cur_len, new_len):
        """Grow a sequence's table row from cur_len to new_len tokens."""
        have = -(-cur_len // block_size)
        need = -(-new_len // block_size)
        if need > len(table_row):
            raise ValueError("table row too short")
        if need > have:
            table_row[have:need] = self.alloc(need - have)
        return table_row

    def seq_release(self, table_row, block_size, length):
        n = -(-length // block_size)
        self.free(list(table_row[:n]))
