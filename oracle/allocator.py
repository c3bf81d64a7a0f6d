"""Block allocator model written from the pages.  Test infrastructure only.

[P1] "3.3 页面级显存管理", 3.3.2 (dynamic page allocation; batch allocation at
     prefill, one more page whenever the token count exceeds
     num_blocks * block_size; the BlockAllocator sketch with refcounts and
     share_blocks), 3.3.4 (one global pool, O(1) alloc and free)
[P2] "vLLM三大核心技术分页内存与共享解码", "Copy-on-Write共享解码的显存优化原理"
     (refcount per physical block; write in place at refcount 1, else copy
     to a new block, repoint the table, decrement the old block; a block
     returns to the free pool when its count drops to 0) and
     "三项技术的协同效应与性能增益分析" (O(1) alloc/free from a free list)
[P3] "3.1 PagedAttention的核心原理", 3.1.2 (block table + refcounts),
     3.1.5 (CoW steps 1-4)
[P4] notes on the vLLM paper, "Memory Sharing与写时复制" (the refcount lives
     in the physical block's metadata)

Readings where the pages disagree or are silent:
  * order of the free list: a stack; the block freed last is handed out
    first and a fresh pool hands out the highest id first (the pool list
    popped from its end, as in [P1]'s sketches).  policy="fifo" (take from
    the front, return to the back) exists only to replay [P2]'s demo.
  * a block is freed when its count reaches exactly 0; releasing a block
    whose count is already 0 is an error.
  * allocation is all-or-nothing: on shortage nothing is taken.
"""
from __future__ import annotations


class OutOfBlocks(MemoryError):
    pass


class BlockAllocatorModel:
    def __init__(self, num_blocks: int, initial_free=None, policy: str = "lifo"):
        assert policy in ("lifo", "fifo")
        self.num_blocks = int(num_blocks)
        self.policy = policy
        if initial_free is None:
            self.free = list(range(self.num_blocks))
            self.rc = {}
        else:
            self.free = [int(b) for b in initial_free]
            fs = set(self.free)
            assert len(fs) == len(self.free), "duplicate id in free list"
            assert all(0 <= b < self.num_blocks for b in fs)
            # every block not on the free list is held once
            self.rc = {b: 1 for b in range(self.num_blocks) if b not in fs}

    # -- pool ----------------------------------------------------------
    def _take(self) -> int:
        return self.free.pop() if self.policy == "lifo" else self.free.pop(0)

    def alloc(self, n: int) -> list:
        """n blocks, refcount 1 each; all-or-nothing."""
        if n < 0:
            raise ValueError(n)
        if len(self.free) < n:
            raise OutOfBlocks(f"need {n}, free {len(self.free)}")
        out = []
        for _ in range(n):
            b = self._take()
            self.rc[b] = 1
            out.append(b)
        return out

    def incref(self, ids) -> None:
        """Share: one more holder for each block ([P1] share_blocks)."""
        for b in ids:
            if self.rc.get(int(b), 0) <= 0:
                raise ValueError(f"incref of free block {b}")
        for b in ids:
            self.rc[int(b)] += 1

    def decref(self, ids) -> int:
        """Release one hold on each block; a block at 0 goes back to the pool."""
        for b in ids:
            if not (0 <= int(b) < self.num_blocks):
                raise ValueError(f"bad id {b}")
        freed = 0
        for b in ids:
            b = int(b)
            if self.rc.get(b, 0) <= 0:
                raise ValueError(f"decref of free block {b}")
            self.rc[b] -= 1
            if self.rc[b] == 0:
                del self.rc[b]
                self.free.append(b)
                freed += 1
        return freed

    def cow(self, b: int):
        """Copy-on-write before a write into block b.

        Returns (block to write, needs_copy).  At refcount 1 the block is
        written in place; otherwise a new block is taken, the old one loses
        one holder, and the caller copies old -> new and repoints its table.
        """
        b = int(b)
        if self.rc.get(b, 0) <= 0:
            raise ValueError(f"cow of free block {b}")
        if self.rc[b] == 1:
            return b, False
        (new,) = self.alloc(1)
        self.rc[b] -= 1
        return new, True

    def refcount(self, b: int) -> int:
        return self.rc.get(int(b), 0)

    @property
    def num_free(self) -> int:
        return len(self.free)

    @property
    def num_shared(self) -> int:
        return sum(1 for c in self.rc.values() if c > 1)

    # -- one sequence's share of a decode step -------------------------
    def append(self, table: list, ctx_before: int, n_new: int, block_size: int) -> list:
        """Make room for tokens [ctx_before, ctx_before + n_new) of a sequence.

        Blocks of `table` that these tokens land in and that other
        sequences also hold are copied first (copy-on-write, in logical
        order); then as many new blocks are appended as the token count now
        needs ([P1] 3.3.2: a new page once the count exceeds
        num_blocks * block_size; a prefill takes them in one batch).
        All-or-nothing.  Returns the (src, dst) copies the caller must do.
        """
        if n_new <= 0:
            return []
        ctx_after = ctx_before + n_new
        first = ctx_before // block_size
        last = (ctx_after - 1) // block_size
        shared = [lb for lb in range(first, min(last + 1, len(table)))
                  if self.refcount(table[lb]) > 1]
        need_new = max(0, -(-ctx_after // block_size) - len(table))
        if self.num_free < need_new + len(shared):
            raise OutOfBlocks(f"need {need_new + len(shared)}, free {self.num_free}")
        pairs = []
        for lb in shared:
            new, copied = self.cow(table[lb])
            assert copied
            pairs.append((table[lb], new))
            table[lb] = new
        table.extend(self.alloc(need_new))
        return pairs


def fork_tables(alloc: BlockAllocatorModel, tables: list, parents) -> list:
    """Every sequence b continues from sequence parents[b]: it takes a new
    hold on each of the parent's blocks ([P1] 3.3.2 share_blocks; beam search
    and parallel sampling in [P4] "Memory Sharing与写时复制"), then the old
    tables are released.  Taking the new holds first keeps blocks that
    survive the fork from passing through refcount 0."""
    new = [list(tables[int(p)]) for p in parents]
    for t in new:
        alloc.incref(t)
    for t in tables:
        alloc.decref(t)
    return new
