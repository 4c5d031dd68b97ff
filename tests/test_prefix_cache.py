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


def _model_admit(m, prompts, cache):
    """The model's reading of one admission wave: add_seq in order, stopping at
    the first request the pool cannot supply."""
    got = []
    for p in prompts:
        try:
            got.append(m.add_seq(p, cache=cache))
        except OutOfBlocks:
            break
    return got


@pytest.mark.parametrize("seed,cache", [(s, c) for s in range(4) for c in (True, False)])
def test_admit_waves_match_the_model(lib, seed, cache):
    """Waves of requests sharing a system prompt go through pa_pcache_admit and
    pa_pcache_free_seqs; each wave's ids, hits, lengths, cu_seqlens_q, slots
    and tables, and the pool after it, match the model; some waves run the
    pool dry part-way."""
    rng = np.random.default_rng(50 + seed)
    B = 16 if seed % 2 else 4
    nb = int(rng.integers(40, 90))
    pc, m = binding.PrefixCache(nb, B), PrefixCacheModel(nb, B)
    system = list(rng.integers(0, 500, size=int(rng.integers(B, 5 * B))))
    maxb = 12 if B == 16 else 40
    live = []
    for wave in range(25):
        n = int(rng.integers(1, 7))
        prompts = [system[:int(rng.integers(1, len(system) + 1))] + list(rng.integers(0, 500, size=int(
            rng.integers(0, 3 * B)))) for _ in range(n)]
        prompts = [p if p else [7] for p in prompts]
        prompts = [p[:maxb * B] for p in prompts]
        flat = np.array([t for p in prompts for t in p], np.int32)
        cu = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
        want = _model_admit(m, prompts, cache)
        count, out = pc.admit(flat, cu, maxb, flags=0 if cache else binding.PA_PCACHE_NO_CACHE)
        assert count == len(want)
        assert out["seq_ids"][:count].tolist() == [w[0] for w in want]
        assert out["num_cached"][:count].tolist() == [w[1] for w in want]
        assert out["seq_lens"][:count].tolist() == [len(p) for p in prompts[:count]]
        q = [0]
        for r in range(count):
            sid, hit = want[r]
            L = len(prompts[r])
            tab = m.table(sid)
            assert out["block_tables"][r].tolist() == tab + [-1] * (maxb - len(tab))
            assert out["slot_mapping"][q[-1]:q[-1] + L - hit].tolist() == \
                [tab[p // B] * B + p % B for p in range(hit, L)]
            q.append(q[-1] + L - hit)
        assert out["cu_seqlens_q"][:count + 1].tolist() == q
        live += [w[0] for w in want]
        if not cache:
            assert all(h == 0 for _, h in want)
        # decode a token or two, then free a random subset in one call
        for sid in live[-3:]:
            tok = int(rng.integers(0, 500))
            try:
                s_want = m.append_token(sid, tok)
            except OutOfBlocks:
                continue
            assert pc.append_token(sid, tok) == s_want
        k = int(rng.integers(0, len(live) + 1))
        idx = rng.permutation(len(live))[:k]
        gone = [live[i] for i in idx]
        for sid in gone:
            m.free_seq(sid)
        pc.free_seqs(np.array(gone, np.int32))
        live = [s for s in live if s not in gone]
        m.check_invariants()
        _same(pc, m, live)


def test_admit_and_free_seqs_argument_errors(lib):
    pc = binding.PrefixCache(32, 16)
    toks = np.arange(40, dtype=np.int32)
    with pytest.raises(binding.PAError) as e:                      # a request with no tokens
        pc.admit(toks, np.array([0, 20, 20, 40], np.int64), 4)
    assert e.value.code == binding.PA_ERR_INVALID_ARG
    with pytest.raises(binding.PAError) as e:                      # 3 blocks > max_blocks_per_seq 2
        pc.admit(toks, np.array([0, 40], np.int64), 2)
    assert e.value.code == binding.PA_ERR_INVALID_ARG
    with pytest.raises(binding.PAError) as e:                      # unknown flag
        pc.admit(toks, np.array([0, 40], np.int64), 4, flags=6)
    assert e.value.code == binding.PA_ERR_INVALID_ARG
    assert pc.num_free() == 31                                     # nothing admitted by any of them
    count, out = pc.admit(toks, np.array([0, 17, 40], np.int64), 4)
    assert count == 2
    with pytest.raises(binding.PAError) as e:                      # listed twice: nothing freed
        pc.free_seqs(np.array([out["seq_ids"][0]] * 2, np.int32))
    assert e.value.code == binding.PA_ERR_INVALID_ARG
    with pytest.raises(binding.PAError) as e:
        pc.free_seqs(np.array([out["seq_ids"][0], 99], np.int32))
    assert e.value.code == binding.PA_ERR_NOT_FOUND
    assert pc.num_free() == 31 - 4
    pc.free_seqs(out["seq_ids"][:2].copy())
    assert pc.num_free() == 31


def test_admit_stops_at_the_first_request_that_does_not_fit(lib):
    """A 12-block pool (11 usable): a wave of 3 requests needing 4, 5 and 4 new
    blocks admits the first two; the third and everything after it are
    untouched, and the same wave's remainder fits once the first two leave."""
    B, nb = 16, 12
    pc, m = binding.PrefixCache(nb, B), PrefixCacheModel(nb, B)
    prompts = [list(range(1, 64)), list(range(100, 180)), list(range(200, 260)), [5, 6]]
    flat = np.array([t for p in prompts for t in p], np.int32)
    cu = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
    want = _model_admit(m, prompts, True)
    assert len(want) == 2
    count, out = pc.admit(flat, cu, 8)
    assert count == 2 and out["seq_ids"][:2].tolist() == [w[0] for w in want]
    assert out["cu_seqlens_q"][:3].tolist() == [0, 63, 143]
    _same(pc, m, [w[0] for w in want])
    for sid, _ in want:
        m.free_seq(sid)
    pc.free_seqs(out["seq_ids"][:2].copy())
    rest = prompts[2:]
    want2 = _model_admit(m, rest, True)
    flat2 = np.array([t for p in rest for t in p], np.int32)
    cu2 = np.concatenate([[0], np.cumsum([len(p) for p in rest])]).astype(np.int64)
    count2, out2 = pc.admit(flat2, cu2, 8)
    assert count2 == len(want2) == 2
    assert out2["seq_ids"].tolist() == [w[0] for w in want2]
    _same(pc, m, [w[0] for w in want2])


def test_admit_into_host_tensors_and_their_checks(lib):
    """admit and free_seqs take CPU tensors (int32, contiguous) as well as
    numpy arrays, addressed in place: a wrong dtype, a strided view or a
    too-small buffer is an argument error and admits nothing."""
    import torch
    pc = binding.PrefixCache(32, 16)
    toks = torch.arange(40, dtype=torch.int32)
    cu = np.array([0, 17, 40], np.int64)
    out = {k: torch.full((64,), -7, dtype=torch.int32) for k in binding.PrefixCache._ADMIT_OUT}
    count, got = pc.admit(toks, cu, 4, 0, out)
    assert count == 2 and got is out
    want_count, want = binding.PrefixCache(32, 16).admit(toks.numpy(), cu, 4)
    assert want_count == 2
    for k in ("seq_ids", "num_cached", "cu_seqlens_q", "seq_lens"):
        n = len(want[k])
        assert out[k][:n].tolist() == want[k].tolist(), k
    assert out["slot_mapping"][:40].tolist() == want["slot_mapping"].tolist()
    assert out["block_tables"][:8].tolist() == want["block_tables"].ravel().tolist()
    pc.free_seqs(out["seq_ids"][:2].clone())
    free = pc.num_free()
    bad = [dict(out, seq_ids=torch.zeros(64, dtype=torch.int64)),          # dtype
           dict(out, slot_mapping=torch.zeros(128, dtype=torch.int32)[::2]),  # strided
           dict(out, slot_mapping=torch.zeros(39, dtype=torch.int32))]       # too small for 40 tokens
    for o in bad:
        with pytest.raises(binding.PAError) as e:
            pc.admit(toks, cu, 4, 0, o)
        assert e.value.code == binding.PA_ERR_INVALID_ARG
    with pytest.raises(binding.PAError):
        pc.admit(toks.to(torch.int64), cu, 4, 0, out)
    with pytest.raises(binding.PAError):
        pc.free_seqs(out["seq_ids"][:2].to(torch.int64))
    assert pc.num_free() == free
