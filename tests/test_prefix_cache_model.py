"""Pins for the prefix-cache model (oracle/prefix_cache.py) against what
"01 · PagedAttention 与 KV cache 块管理" fixes: chained SHA-256 hashes, a
match that ends at the first miss and never covers the last prompt token,
touch out of the middle of the free queue, LIFO reuse of unhashed blocks and
FIFO (tail) return of cached ones with the chain's tail first, lazy
eviction, the null block."""
import hashlib
import struct

import pytest

from oracle.prefix_cache import NONE_HASH, OutOfBlocks, PrefixCacheModel, block_hash, chain_hashes

B = 16


def _toks(seed, n):
    return [(seed * 7919 + 31 * i) % 50021 for i in range(n)]


def test_block_hash_is_sha256_of_parent_and_int32_tokens():
    t = [1, 2, 3, -4]
    ref = hashlib.sha256(NONE_HASH + struct.pack("<4i", *t)).digest()
    assert block_hash(NONE_HASH, t) == ref
    assert NONE_HASH == bytes(32)


def test_hashes_are_chained():
    """Block i's hash covers blocks 0..i: changing a token of block 0 changes
    every later hash; equal blocks after different prefixes hash differently."""
    a = _toks(1, 64)
    b = list(a)
    b[3] += 1
    ha, hb = chain_hashes(a, B), chain_hashes(b, B)
    assert len(ha) == 4 and all(x != y for x, y in zip(ha, hb))
    c = _toks(2, 16) + a[16:64]
    assert chain_hashes(c, B)[1] != ha[1]
    assert chain_hashes(a[:40], B) == ha[:2]


def test_match_covers_at_most_all_but_the_last_token():
    m = PrefixCacheModel(64, B)
    p = _toks(3, 64)
    s0, hit0 = m.add_seq(p)
    assert hit0 == 0
    s1, hit1 = m.add_seq(p)          # 4 full blocks cached, but the last token must be recomputed
    assert hit1 == 48
    assert m.table(s1)[:3] == m.table(s0)[:3] and m.table(s1)[3] != m.table(s0)[3]
    s2, hit2 = m.add_seq(p + [7])    # 65 tokens: all 4 full blocks may hit
    assert hit2 == 64 and m.table(s2)[:4] == m.table(s0)[:4]
    m.check_invariants()


def test_first_miss_ends_the_match():
    m = PrefixCacheModel(64, B)
    p = _toks(4, 80)
    m.add_seq(p)
    q = list(p)
    q[20] += 1                       # block 1 differs
    _, hit = m.add_seq(q)
    assert hit == 16                 # block 0 only; blocks 2.. are different hashes (chained)
    m.check_invariants()


def test_free_returns_unhashed_to_head_and_cached_to_tail_chain_tail_first():
    m = PrefixCacheModel(12, B)
    s, _ = m.add_seq(_toks(5, 40))   # blocks 1, 2 (full, cached), 3 (partial)
    assert m.table(s) == [1, 2, 3]
    assert m.free == list(range(4, 12))
    m.free_seq(s)
    assert m.free[0] == 3                        # unhashed: LIFO at the head
    assert m.free[-2:] == [2, 1]                 # cached: tail, the chain's tail first
    assert 0 not in m.free
    m.check_invariants()


def test_touch_takes_a_cached_free_block_out_of_the_middle_and_eviction_is_lazy():
    m = PrefixCacheModel(8, B)
    p = _toks(6, 33)                             # blocks 1, 2 full + 3 partial
    s, _ = m.add_seq(p)
    m.free_seq(s)                                # queue: 3, 4, 5, 6, 7, 2, 1
    assert m.free == [3, 4, 5, 6, 7, 2, 1]
    s2, hit = m.add_seq(p)                       # both full blocks hit while still free
    assert hit == 32 and m.table(s2)[:2] == [1, 2]
    assert m.free == [4, 5, 6, 7]                # 3 reused for the partial block
    m.free_seq(s2)                               # queue: 3, 4, 5, 6, 7, 2, 1
    # six new blocks pop up to block 2 (the chain's tail goes first): its hash
    # is evicted on reuse, block 1 keeps its own
    hog, _ = m.add_seq(_toks(99, 16 * 6))
    assert m.table(hog) == [3, 4, 5, 6, 7, 2]
    m.free_seq(hog)
    _, hit = m.add_seq(p)
    assert hit == 16
    m.check_invariants()


def test_null_block_is_never_handed_out_and_allocation_is_all_or_nothing():
    m = PrefixCacheModel(5, B)                   # 4 usable blocks
    s, _ = m.add_seq(_toks(7, 50))               # 4 blocks
    assert 0 not in m.table(s) and m.free == []
    before = (list(m.free), list(m.ref))
    with pytest.raises(OutOfBlocks):
        m.add_seq(_toks(8, 1))
    assert (m.free, m.ref) == before
    for t in range(14):                          # positions 50..63 fit the last block
        m.append_token(s, t)
    with pytest.raises(OutOfBlocks):
        m.append_token(s, 1)                     # position 64 needs a fifth block
    m.check_invariants()


def test_decode_blocks_become_cached_when_full():
    m = PrefixCacheModel(16, B)
    p = _toks(9, 30)
    s, _ = m.add_seq(p)
    toks = list(p)
    for t in (5, 6):                             # the second block fills at token 32
        slot = m.append_token(s, t)
        toks.append(t)
        assert slot == m.table(s)[(len(toks) - 1) // B] * B + (len(toks) - 1) % B
    assert m.hash[m.table(s)[1]] == chain_hashes(toks, B)[1]
    _, hit = m.add_seq(toks + [1])
    assert hit == 32
    m.check_invariants()


def test_caching_off_is_plain_allocation():
    """With caching off a request neither matches nor records: the same
    prompt twice gets fresh blocks, none carries a hash, and freeing returns
    them all to the head (LIFO), exactly the plain pool of section 4.3."""
    m = PrefixCacheModel(16, B)
    p = _toks(11, 40)
    s0, hit0 = m.add_seq(p, cache=False)
    s1, hit1 = m.add_seq(p, cache=False)
    assert (hit0, hit1) == (0, 0)
    assert m.table(s0) == [1, 2, 3] and m.table(s1) == [4, 5, 6]
    assert all(h is None for h in m.hash) and m.cached == {}
    for t in range(8):                            # block 3 fills at token 48: still unhashed
        m.append_token(s0, t)
    assert m.hash[3] is None
    m.free_seq(s0)
    assert m.free[:3] == [1, 2, 3]
    _, hit = m.add_seq(p)                         # a caching request finds nothing either
    assert hit == 0
    m.check_invariants()
