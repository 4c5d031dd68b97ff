"""CPU checks of the product's prefix-cache block pool (pa_pcache_*) against
the oracle model, operation for operation: hits, block tables, slots,
reference counts, every block's hash and the free queue's exact order."""
import numpy as np
import pytest

from oracle.prefix_cache import OutOfBlocks, PrefixCacheModel, chain_hashes
from paged_kv_cache_120_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def _same(pc, m, live):
    assert pc.free_queue() == m.free
    assert pc.num_free() == len(m.free)
    for b in range(m.num_blocks):
        assert pc.ref_count(b) == m.ref[b], b
        assert pc.block_hash(b) == m.hash[b], b
    for sid in live:
        assert pc.table(sid) == m.table(sid)
        assert pc.seq_len(sid) == m.seq_len(sid)


def test_hashes_match_hashlib_chain(lib):
    pc = binding.PrefixCache(16, 4)
    toks = list(range(1000, 1014))
    sid, hit = pc.add_seq(toks)
    assert hit == 0
    want = chain_hashes(toks, 4)
    assert [pc.block_hash(b) for b in pc.table(sid)[:3]] == want
    assert pc.block_hash(pc.table(sid)[3]) is None      # partial block: no hash


def test_null_block_and_bad_arguments(lib):
    with pytest.raises(binding.PAError):
        binding.PrefixCache(1, 16)
    pc = binding.PrefixCache(4, 16)
    assert 0 not in pc.free_queue() and pc.num_free() == 3
    with pytest.raises(binding.PAError) as e:
        pc.add_seq(list(range(100)))                    # 7 blocks > 3
    assert e.value.code == binding.PA_ERR_OUT_OF_BLOCKS
    assert pc.free_queue() == [1, 2, 3]
    with pytest.raises(binding.PAError) as e:
        pc.free_seq(123)
    assert e.value.code == binding.PA_ERR_NOT_FOUND


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_model(lib, seed):
    """Prompts drawn from a few shared system prefixes plus random tails and
    random full-prompt repeats; random appends and frees. Every operation's
    result and the whole pool state must match the model."""
    rng = np.random.default_rng(seed)
    B = int(rng.choice([4, 16]))
    nb = int(rng.integers(24, 80))
    pc, m = binding.PrefixCache(nb, B), PrefixCacheModel(nb, B)
    prefixes = [list(rng.integers(0, 1000, size=int(rng.integers(1, 6 * B)))) for _ in range(3)]
    history = []
    live = []
    for _ in range(300):
        op = rng.random()
        if op < 0.4 or not live:
            if history and rng.random() < 0.3:
                toks = list(history[int(rng.integers(len(history)))])
            else:
                toks = list(prefixes[int(rng.integers(3))]) + list(rng.integers(0, 1000, size=int(rng.integers(0, 3 * B))))
            if not toks:
                toks = [1]
            try:
                want = m.add_seq(toks)
            except OutOfBlocks:
                with pytest.raises(binding.PAError) as e:
                    pc.add_seq(toks)
                assert e.value.code == binding.PA_ERR_OUT_OF_BLOCKS
            else:
                got = pc.add_seq(toks)
                assert got == want
                live.append(got[0])
                history.append(toks)
        elif op < 0.8:
            sid = live[int(rng.integers(len(live)))]
            tok = int(rng.integers(0, 1000))
            try:
                want = m.append_token(sid, tok)
            except OutOfBlocks:
                with pytest.raises(binding.PAError) as e:
                    pc.append_token(sid, tok)
                assert e.value.code == binding.PA_ERR_OUT_OF_BLOCKS
            else:
                assert pc.append_token(sid, tok) == want
        else:
            sid = live.pop(int(rng.integers(len(live))))
            m.free_seq(sid)
            pc.free_seq(sid)
        m.check_invariants()
        _same(pc, m, live)
    for sid in live:
        L = m.seq_len(sid)
        assert pc.slots(sid, 0, L).tolist() == [m.table(sid)[p // B] * B + p % B for p in range(L)]
