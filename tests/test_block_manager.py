"""Pins for the oracle's block-manager model against the pages' printed
examples and stated invariants (CPU only)."""
import json
import os

import numpy as np
import pytest

from oracle.block_manager import BlockManagerModel, OutOfBlocks
from paged_kv_cache_120_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _toy():
    g = _golden("worked_example.json")
    m = BlockManagerModel(g["num_blocks"], g["block_size"], order=workloads.toy_free_order())
    ids = {r: m.add_seq(g["requests"][r]["tokens"]) for r in ("A", "B", "C")}
    return g, m, ids


def test_worked_example_tables_and_counts():
    """Digest "具体实例演示": tables [3,7], [0,5,9], [4]; 96 slots, 84 tokens, 12 padded, 58 free."""
    g, m, ids = _toy()
    for r, sid in ids.items():
        assert m.table(sid) == g["requests"][r]["table"]
    slots = sum(len(m.table(s)) for s in ids.values()) * g["block_size"]
    tokens = sum(m.seq_len(s) for s in ids.values())
    assert (slots, tokens, slots - tokens) == (g["slots_used"], g["tokens_stored"], g["padded_slots"])
    assert m.num_free() == g["free_blocks_after"]
    assert 3 * 2048 == g["contiguous_reserved_slots"]
    m.check_invariants()


def test_worked_example_decode_step_slots_and_growth():
    """One new token each -> slots 121/159/76; B growing past 48 tokens -> [0,5,9,11]."""
    g, m, ids = _toy()
    slots = [m.append_token(ids[r]) for r in ("A", "B", "C")]
    assert slots == [(121, None), (159, None), (76, None)]
    b = ids["B"]
    seen = {}
    while m.seq_len(b) < 48 + workloads.TOY_GROWTH_TOKENS:
        slot, cow = m.append_token(b)
        assert cow is None
        seen[m.seq_len(b)] = m.table(b)
    assert seen[49] == g["b_table_after_growth"] == seen[64]
    assert seen[65] == [0, 5, 9, 11, 12] == seen[68]
    m.check_invariants()


def test_block_size_tradeoff_for_a_47_token_request():
    """Digest "注意力内核为何能正常工作": B=4 -> 12 lookups / 1 wasted; 16 -> 3 / 1; 64 -> 1 / 17."""
    g = _golden("block_size_tradeoff.json")
    for case in g["cases"]:
        m = BlockManagerModel(64, case["block_size"])
        sid = m.add_seq(g["tokens"])
        n = len(m.table(sid))
        assert n == case["lookups"]
        assert n * case["block_size"] - g["tokens"] == case["wasted_slots"]


def test_internal_fragmentation_example():
    """vLLM book §4.1.2: a 100-token request at 64-token granularity takes 128 slots, 28 wasted."""
    g = _golden("sizing.json")["internal_fragmentation"]
    m = BlockManagerModel(8, g["granularity"])
    sid = m.add_seq(g["tokens"])
    slots = len(m.table(sid)) * g["granularity"]
    assert (slots, slots - g["tokens"]) == (g["slots"], g["wasted"])


def test_parallel_sampling_shares_the_prompt_blocks():
    """vLLM book §4.7.1: a 48-token prompt, n=3: 9 blocks unshared, 3 blocks shared."""
    g = _golden("sizing.json")["parallel_sampling"]
    unshared = BlockManagerModel(32, g["block_size"])
    for _ in range(g["samples"]):
        unshared.add_seq(g["prompt_tokens"])
    assert 32 - unshared.num_free() == g["blocks_unshared"]
    shared = BlockManagerModel(32, g["block_size"])
    p = shared.add_seq(g["prompt_tokens"])
    for _ in range(g["samples"] - 1):
        shared.fork(p)
    assert 32 - shared.num_free() == g["blocks_shared"]
    assert all(shared.ref[b] == 3 for b in shared.table(p))


def test_cow_steps_of_the_lecture():
    """Lecture §4.3: A and B share P (ref 2); A writes -> new Q, copy P->Q, A's table -> Q, ref(P) = 1."""
    m = BlockManagerModel(8, 16)
    a = m.add_seq(20)                     # blocks [0, 1], last block half full
    b = m.fork(a)
    p = m.table(a)[-1]
    assert m.ref[p] == 2
    slot, cow = m.append_token(a)
    q = m.table(a)[-1]
    assert cow == (p, q) and q != p
    assert m.table(b)[-1] == p            # the other sharer still sees P
    assert m.ref[p] == 1 and m.ref[q] == 1
    assert slot == q * 16 + 20 % 16
    slot_b, cow_b = m.append_token(b)     # B is now the only owner: write in place
    assert cow_b is None and slot_b == p * 16 + 4
    m.check_invariants()


def test_cow_is_decided_by_refcount_not_by_block_identity():
    """Lecture §4.3 pitfall: a single owner never copies."""
    m = BlockManagerModel(4, 16)
    a = m.add_seq(3)
    for _ in range(10):
        _, cow = m.append_token(a)
        assert cow is None


def test_exhaustion_reports_and_leaves_state_unchanged():
    """Digest scheduler sketch: allocate_block returns -1 when the free list is empty."""
    m = BlockManagerModel(3, 16)
    a = m.add_seq(40)                     # 3 blocks
    before = (m.table(a), m.num_free(), list(m.ref))
    with pytest.raises(OutOfBlocks):
        m.add_seq(1)
    with pytest.raises(OutOfBlocks):
        for _ in range(9):
            m.append_token(a)             # 41..48 fit, 49 needs a 4th block
    assert m.seq_len(a) == 48
    assert m.num_free() == 0
    assert before[1] == 0
    m.check_invariants()


def test_free_returns_blocks_head_first_in_reverse_table_order():
    """Free walks the table in reverse; a block whose count reaches 0 goes to the head."""
    m = BlockManagerModel(6, 16)
    a = m.add_seq(40)                     # blocks 0, 1, 2
    m.free_seq(a)
    assert m.free[:3] == [0, 1, 2]
    b = m.add_seq(1)
    assert m.table(b) == [0]
    m.check_invariants()


def test_random_operations_keep_the_free_list_invariant():
    """vLLM book §4.7.3: a block with live references is never in the free queue."""
    rng = np.random.default_rng(13)
    m = BlockManagerModel(64, 16, order=rng.permutation(64))
    live = []
    for _ in range(2000):
        op = rng.integers(0, 4)
        try:
            if op == 0 or not live:
                live.append(m.add_seq(int(rng.integers(0, 60))))
            elif op == 1:
                live.append(m.fork(live[rng.integers(len(live))]))
            elif op == 2:
                m.append_token(live[rng.integers(len(live))])
            else:
                m.free_seq(live.pop(rng.integers(len(live))))
        except OutOfBlocks:
            pass
        m.check_invariants()
