"""Oracle model of the host block manager (TEST INFRASTRUCTURE ONLY).

A deliberately plain Python restatement of the bookkeeping the pages
describe, used to pin the product's C++ allocator op-for-op. It shares no
code with it.

Sources:
  * "PagedAttention: virtual memory for the KV cache" digest, section
    "调度器机制简述" (scheduler sketch): a free list of block ids,
    ``allocate_block`` that reports exhaustion (-1), ``ceil(len / B)`` blocks
    for a new request, a new block when the last one is full, and
    ``handle_write_with_cow``: if the written block's ref count is > 1,
    allocate a new block, copy, point this request's table at it, and drop
    one reference from the old block. Section "具体实例演示" gives the worked
    example this model is pinned to.
  * "01 · PagedAttention 与 KV cache 块管理", §3 and §4.3: blocks carry a
    ref count; freeing walks a request's blocks in reverse and returns a block
    to the free queue when its count reaches 0; uncached blocks go to the head
    of the queue (LIFO reuse); allocation takes from the head.
  * "PagedAttention原理（下）", §4.3: the COW steps (P shared with refcount 2,
    allocate Q, copy P into Q, retarget the writer's table, refcount(P) - 1),
    and the rule that COW is decided by refcount > 1, not by block identity.
  * "第4章 PagedAttention：虚拟内存的启示", §4.4.3: slot = table[pos // B] * B
    + pos % B; §4.7.3: a block in the free queue never has a live reference.

Readings where the pages leave a choice open (each also listed in the
design notes): allocation is all-or-nothing per call; the initial free-list
order is given by the caller (an explicit list reproduces the worked
example, a seeded permutation gives "random non-repeating physical ids");
freed blocks go to the head of the list.
"""
from __future__ import annotations


class OutOfBlocks(Exception):
    """The free list cannot satisfy the request (the pages' -1 / None)."""


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int, order=None):
        self.num_blocks = num_blocks
        self.block_size = block_size
        if order is None:
            order = list(range(num_blocks))
        order = [int(b) for b in order]
        assert sorted(order) == list(range(num_blocks)), "order must list every block once"
        self.free = list(order)          # head of the queue = index 0
        self.ref = [0] * num_blocks
        self.tables = {}                 # seq id -> list of physical block ids
        self.lens = {}                   # seq id -> number of cached tokens
        self._next_id = 0

    # -- free list ---------------------------------------------------------
    def _pop(self) -> int:
        if not self.free:
            raise OutOfBlocks()
        b = self.free.pop(0)
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        assert self.ref[b] >= 0
        if self.ref[b] == 0:
            self.free.insert(0, b)

    def num_free(self) -> int:
        return len(self.free)

    # -- sequences ---------------------------------------------------------
    def add_seq(self, num_tokens: int) -> int:
        need = -(-num_tokens // self.block_size)
        if need > len(self.free):
            raise OutOfBlocks()
        sid = self._next_id
        self._next_id += 1
        self.tables[sid] = [self._pop() for _ in range(need)]
        self.lens[sid] = num_tokens
        return sid

    def fork(self, parent: int) -> int:
        sid = self._next_id
        self._next_id += 1
        self.tables[sid] = list(self.tables[parent])
        for b in self.tables[sid]:
            self.ref[b] += 1
        self.lens[sid] = self.lens[parent]
        return sid

    def append_token(self, sid: int):
        """Returns (slot, cow_pair or None) for the token at position len."""
        table = self.tables[sid]
        pos = self.lens[sid]
        cow = None
        if pos % self.block_size == 0:
            table.append(self._pop())
        else:
            last = table[-1]
            if self.ref[last] > 1:
                fresh = self._pop()
                cow = (last, fresh)
                table[-1] = fresh
                self.ref[last] -= 1
        self.lens[sid] = pos + 1
        slot = table[pos // self.block_size] * self.block_size + pos % self.block_size
        return slot, cow

    def free_seq(self, sid: int) -> None:
        for b in reversed(self.tables.pop(sid)):
            self._release(b)
        del self.lens[sid]

    def table(self, sid: int):
        return list(self.tables[sid])

    def seq_len(self, sid: int) -> int:
        return self.lens[sid]

    # -- invariant the pages state (§4.7.3 of the vLLM book chapter) -------
    def check_invariants(self) -> None:
        in_free = set(self.free)
        assert len(in_free) == len(self.free)
        for b in range(self.num_blocks):
            assert (self.ref[b] == 0) == (b in in_free)
        counted = [0] * self.num_blocks
        for t in self.tables.values():
            for b in t:
                counted[b] += 1
        assert counted == self.ref
