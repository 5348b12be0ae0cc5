"""Block bookkeeping of the pages, as plain Python (test infrastructure only).

The hot path never runs this: it decides which blocks a sequence uses and
which copy-on-write copies a step needs, and the tests compare the copies the
GPU makes with it.  Three pieces, each following one page:

- ``BlockPool``: the FIFO free queue with reference counts of
  "分页 KV Cache" (ai-infra handbook), paged.py ``BlockPool``: allocate pops
  from the head and sets ref 1, returns None when short; free decrements and
  appends a block to the tail when its count reaches 0.
- ``CountingPool``: the pool of "KV cache：容量推导、分页与回收",
  kv_cache.py ``Pool``: fresh ids from a counter, retain / release, a block
  disappears at ref 0, and it may carry token labels as its content.
- ``Sequence``: that page's ``Sequence``: ``fork`` retains every block;
  ``append`` opens a new block when the length is a multiple of the block
  size, otherwise copies a shared tail (ref > 1) into a fresh block and
  releases the old one, then writes the token.

Both pools expose the same four calls, so ``Sequence`` runs on either.
"""
from collections import deque
import math


class BlockPool:
    """FIFO free queue + reference counts."""

    def __init__(self, num_blocks: int):
        self.num_blocks = num_blocks
        self.ref_cnt = [0] * num_blocks
        self.free_queue = deque(range(num_blocks))

    def num_free(self) -> int:
        return len(self.free_queue)

    def allocate(self, n: int):
        if n > len(self.free_queue):
            return None
        out = []
        for _ in range(n):
            b = self.free_queue.popleft()
            self.ref_cnt[b] = 1
            out.append(b)
        return out

    def free(self, blocks) -> None:
        for b in blocks:
            self.ref_cnt[b] -= 1
            if self.ref_cnt[b] == 0:
                self.free_queue.append(b)

    # the Sequence interface
    def new_block(self, content=()):
        got = self.allocate(1)
        if got is None:
            raise MemoryError("block pool exhausted")
        return got[0]

    def retain(self, b: int) -> None:
        self.ref_cnt[b] += 1

    def release(self, b: int) -> None:
        self.free([b])

    def refs(self, b: int) -> int:
        return self.ref_cnt[b]

    def content(self, b: int):
        return None


class CountingPool:
    """Counter-issued ids, refcounts, optional per-block token content."""

    def __init__(self, block_size: int = 4):
        if block_size <= 0:
            raise ValueError("block_size must be positive")
        self.block_size = block_size
        self.next_id = 0
        self.data = {}
        self.ref = {}

    def new_block(self, content=()):
        b = self.next_id
        self.next_id += 1
        self.data[b] = list(content)
        self.ref[b] = 1
        return b

    def retain(self, b: int) -> None:
        self.ref[b] += 1

    def release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            del self.ref[b]
            del self.data[b]

    def refs(self, b: int) -> int:
        return self.ref[b]

    def content(self, b: int):
        return self.data[b]


class Sequence:
    """A sequence's block list and length over a pool; records its CoW copies."""

    def __init__(self, pool, block_size: int, blocks=None, length: int = 0):
        self.pool = pool
        self.block_size = block_size
        self.blocks = list(blocks or [])
        self.length = length

    def append(self, token=None):
        """Add one token.  Returns ("new", b), ("cow", old, new) or ("in_place", b)."""
        offset = self.length % self.block_size
        if offset == 0:
            b = self.pool.new_block()
            self.blocks.append(b)
            event = ("new", b)
        elif self.pool.refs(self.blocks[-1]) > 1:
            old = self.blocks[-1]
            old_content = self.pool.content(old)
            new = self.pool.new_block(old_content if old_content is not None else ())
            self.blocks[-1] = new
            self.pool.release(old)
            event = ("cow", old, new)
        else:
            event = ("in_place", self.blocks[-1])
        content = self.pool.content(self.blocks[-1])
        if content is not None:
            content.append(token)
        self.length += 1
        return event

    def fork(self):
        for b in self.blocks:
            self.pool.retain(b)
        return Sequence(self.pool, self.block_size, list(self.blocks), self.length)

    def tokens(self):
        out = []
        for b in self.blocks:
            out.extend(self.pool.content(b))
        return out

    def close(self) -> None:
        for b in self.blocks:
            self.pool.release(b)
        self.blocks, self.length = [], 0


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """ceil(T / block_size): the blocks a T-token sequence occupies."""
    return math.ceil(num_tokens / block_size)


def round_robin_tables(seq_lens, block_size: int, num_blocks: int):
    """Give each request one block at a time, in turn, until each holds its
    context (the interleaved layout of the handbook's verification script)."""
    pool = BlockPool(num_blocks)
    tables = [[] for _ in seq_lens]
    while any(len(t) * block_size < s for t, s in zip(tables, seq_lens)):
        for t, s in zip(tables, seq_lens):
            if len(t) * block_size < s:
                t += pool.allocate(1)
    return tables


def parallel_sampling_blocks(prompt_len: int, gen_len: int, n: int, block_size: int):
    """Physical blocks held after n samples of one prompt each generate gen_len
    tokens, with and without sharing.  Sharing: the prompt's sequence is the
    first sample and n - 1 forks share its blocks; every sample then appends
    its tokens one by one under the copy-on-write rule.  Returns
    (unshared, shared)."""
    unshared = n * blocks_needed(prompt_len + gen_len, block_size)
    pool = CountingPool(block_size)
    first = Sequence(pool, block_size)
    for _ in range(prompt_len):
        first.append()
    samples = [first] + [first.fork() for _ in range(n - 1)]
    for _ in range(gen_len):
        for s in samples:
            s.append()
    return unshared, len(pool.ref)


def cow_step(groups, block_size: int, pool):
    """One decode step for parallel-sampling groups: every sample appends one
    token.  `groups` is a list of lists of Sequence.  Returns the (src, dst)
    block pairs the step must copy, in the order the appends happen."""
    pairs = []
    for g in groups:
        for s in g:
            ev = s.append()
            if ev[0] == "cow":
                pairs.append((ev[1], ev[2]))
    return pairs
