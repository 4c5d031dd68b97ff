"""Prefix-cache block pool model (TEST INFRASTRUCTURE ONLY).

A plain restatement of the prefix-caching bookkeeping described on
"01 · PagedAttention 与 KV cache 块管理" (§4.2 free queue, §4.3 block pool,
§4.4 chained hashes, §4.5 allocation, §5 details), used by the tests to
check the product's C++ implementation op for op. Only tests/ import it.

Rules (each from the page, readings marked):
  * Block 0 is the null block: never on the free queue, never handed out
    (§5).
  * Free queue, head first = evicted first. Initially blocks 1..N-1 in
    ascending order (reading: the page fixes no initial order).
  * Chained hash of a full block: SHA-256 over the parent block's hash and
    the block's token ids (§4.4). Reading: the root parent is 32 zero bytes,
    token ids are serialised as little-endian int32, no extra keys.
  * A new sequence's prompt is matched from its first block; the first miss
    ends the match, and the match may cover at most num_tokens - 1 tokens
    (the last token is always recomputed) (§4.4, §4.5).
  * Hit = touch: ref count + 1, and a block with count 0 leaves the free
    queue from wherever it is (§4.3).
  * Allocation pops the free queue's head; a popped block loses its cached
    hash then (lazy eviction) (§4.3, §5). All-or-nothing: if the free queue
    cannot supply the blocks a prompt needs, nothing changes (reading of
    "return None when there are not enough free blocks", §4.5).
  * A block becomes cached when it is full: its hash is set and recorded
    (reading: a prompt's full blocks are recorded at allocation, since this
    step writes their K/V before anything reads them; a decode block when
    its last slot is reserved). If another block already holds that hash,
    the first one stays the lookup target.
  * With caching off for a request (cache=False) it neither matches nor
    records, at admission or when decode fills a block: every block is
    popped fresh and stays unhashed (the plain allocation of §4.3 without
    the hash steps of §4.4).
  * Free: the sequence's blocks in reverse table order, count - 1; a block
    reaching 0 goes to the queue head if it has no hash (LIFO reuse) and to
    the tail if it has one (FIFO, so cached blocks live longest) (§4.3).
"""
from __future__ import annotations

import hashlib
import struct

NONE_HASH = bytes(32)


class OutOfBlocks(RuntimeError):
    pass


def block_hash(parent: bytes, tokens) -> bytes:
    """SHA-256 of the parent hash followed by the token ids (little-endian int32)."""
    return hashlib.sha256(parent + b"".join(struct.pack("<i", int(t)) for t in tokens)).digest()


def chain_hashes(tokens, block_size: int) -> list:
    """Hashes of every full block of a token sequence, each chained on the previous."""
    out, parent = [], NONE_HASH
    for b in range(len(tokens) // block_size):
        parent = block_hash(parent, tokens[b * block_size:(b + 1) * block_size])
        out.append(parent)
    return out


class PrefixCacheModel:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks < 2 or block_size <= 0:
            raise ValueError("need at least the null block and one more")
        self.num_blocks, self.block_size = num_blocks, block_size
        self.free = list(range(1, num_blocks))       # head first
        self.ref = [0] * num_blocks
        self.hash = [None] * num_blocks
        self.cached = {}                             # hash -> [blocks], first is the lookup target
        self.seqs = {}
        self.next_id = 0

    # -- internals
    def _evict(self, b):
        h = self.hash[b]
        if h is not None:
            lst = self.cached[h]
            lst.remove(b)
            if not lst:
                del self.cached[h]
            self.hash[b] = None

    def _pop(self):
        b = self.free.pop(0)
        self._evict(b)
        self.ref[b] = 1
        return b

    def _record(self, b, h):
        self.hash[b] = h
        self.cached.setdefault(h, []).append(b)

    # -- operations
    def add_seq(self, tokens, cache=True):
        """Returns (seq_id, tokens found in the cache)."""
        tokens = [int(t) for t in tokens]
        B, n = self.block_size, len(tokens)
        hashes = chain_hashes(tokens, B) if cache else []
        hits = []
        for i, h in enumerate(hashes):
            if (i + 1) * B > n - 1 or h not in self.cached:
                break
            hits.append(self.cached[h][0])
        need = -(-n // B) - len(hits)
        available = len(self.free) - sum(1 for b in hits if self.ref[b] == 0)
        if need > available:
            raise OutOfBlocks(f"need {need}, {available} free")
        for b in hits:
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1
        table = list(hits)
        for i in range(len(hits), -(-n // B)):
            b = self._pop()
            table.append(b)
            if i < len(hashes):
                self._record(b, hashes[i])
        sid = self.next_id
        self.next_id += 1
        self.seqs[sid] = {"table": table, "tokens": tokens, "hashes": hashes, "cache": cache}
        return sid, len(hits) * B

    def append_token(self, sid, token):
        """Reserve the slot of the sequence's next token; returns the slot."""
        s = self.seqs[sid]
        B = self.block_size
        pos = len(s["tokens"])
        if pos % B == 0:
            if not self.free:
                raise OutOfBlocks("no free block")
            s["table"].append(self._pop())
        s["tokens"].append(int(token))
        if (pos + 1) % B == 0 and s["cache"]:
            parent = s["hashes"][-1] if s["hashes"] else NONE_HASH
            h = block_hash(parent, s["tokens"][pos + 1 - B:pos + 1])
            s["hashes"].append(h)
            self._record(s["table"][pos // B], h)
        return s["table"][pos // B] * B + pos % B

    def free_seq(self, sid):
        s = self.seqs.pop(sid)
        for b in reversed(s["table"]):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                if self.hash[b] is None:
                    self.free.insert(0, b)
                else:
                    self.free.append(b)

    def table(self, sid):
        return list(self.seqs[sid]["table"])

    def seq_len(self, sid):
        return len(self.seqs[sid]["tokens"])

    def check_invariants(self):
        assert 0 not in self.free and self.ref[0] == 0
        assert len(set(self.free)) == len(self.free)
        for b in range(1, self.num_blocks):
            assert (self.ref[b] == 0) == (b in self.free), b
        counts = [0] * self.num_blocks
        for s in self.seqs.values():
            for b in s["table"]:
                counts[b] += 1
        assert counts == self.ref
        for h, lst in self.cached.items():
            for b in lst:
                assert self.hash[b] == h
