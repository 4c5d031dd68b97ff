"""The prefix cache feeding the device kernels: requests that share a system
prompt reuse its cached blocks (their K/V written once, by the first
request), write and prefill only their uncached tokens, then decode over
tables that share blocks. Every output against the oracle run on the same
tables and the same writes; after eviction a prompt is recomputed."""
import math

import numpy as np
import pytest

import oracle
from oracle.prefix_cache import PrefixCacheModel
from paged_kv_cache_120_gb300 import binding, build, workloads

from harness import TOL, max_abs_err, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.lib()
    assert binding.pa_get_device_error() == 0
    return torch.device("cuda:0")


@pytest.mark.parametrize("dtype,Hq,Hkv", [(workloads.F16, 8, 8), (workloads.BF16, 32, 8)])
def test_shared_system_prompt_prefill_then_decode(dev, dtype, Hq, Hkv):
    import torch
    B, D, nb = 16, 128, 200
    rng = np.random.default_rng(3 + Hq)
    system = list(rng.integers(0, 32000, size=200))          # 12 full blocks + 8 tokens
    prompts = [system + list(rng.integers(0, 32000, size=int(n))) for n in (37, 5, 90, 16, 1)]
    pc, m = binding.PrefixCache(nb, B), PrefixCacheModel(nb, B)
    pool = workloads.normal_values((2, nb, B, Hkv, D), dtype, 40, dev)
    pool_bits = u16(pool).copy()
    scale = 1 / math.sqrt(D)
    ids, hits = [], []
    for r, p in enumerate(prompts):
        sid, hit = pc.add_seq(p)
        assert (sid, hit) == m.add_seq(p)
        assert hit == (0 if r == 0 else 192)                 # 12 full system blocks after the first
        ids.append(sid)
        hits.append(hit)
        # this request's K/V for its uncached positions, then prefill of those queries
        n_new = len(p) - hit
        slots = pc.slots(sid, hit, n_new)
        k = workloads.normal_values((n_new, Hkv, D), dtype, 100 + r, dev)
        v = workloads.normal_values((n_new, Hkv, D), dtype, 200 + r, dev)
        q = workloads.normal_values((n_new, Hq, D), dtype, 300 + r, dev)
        binding.pa_reshape_and_cache(k, v, pool, torch.from_numpy(slots).to(dev))
        assert oracle.reshape_and_cache(u16(k), u16(v), pool_bits, slots, nb, B, Hkv, D) == n_new
        bt = pc.block_tables([sid], -(-len(p) // B))
        out = torch.empty_like(q)
        binding.pa_prefill(out, q, pool, torch.from_numpy(bt).to(dev),
                           torch.tensor([0, n_new], dtype=torch.int32, device=dev),
                           torch.tensor([len(p)], dtype=torch.int32, device=dev), scale, n_new)
        torch.cuda.synchronize()
        want = oracle.prefill(u16(q), pool_bits, bt, np.array([0, n_new], np.int32),
                              np.array([len(p)], np.int32), scale, Hq, Hkv, D, nb, B, dtype)
        assert max_abs_err(oracle.decode_elems(u16(out), dtype), want) <= TOL[dtype]
        assert np.array_equal(u16(pool), pool_bits)
    # the system prompt's blocks are shared by every table
    tabs = pc.block_tables(ids, 20)
    assert all((tabs[i, :12] == tabs[0, :12]).all() for i in range(len(ids)))
    assert pc.ref_count(int(tabs[0, 0])) == len(ids)
    # decode steps over the shared tables
    for step_i in range(3):
        toks = rng.integers(0, 32000, size=len(ids))
        slots = np.array([pc.append_token(sid, int(t)) for sid, t in zip(ids, toks)], np.int32)
        assert slots.tolist() == [m.append_token(sid, int(t)) for sid, t in zip(ids, toks)]
        k = workloads.normal_values((len(ids), Hkv, D), dtype, 400 + step_i, dev)
        v = workloads.normal_values((len(ids), Hkv, D), dtype, 500 + step_i, dev)
        q = workloads.normal_values((len(ids), Hq, D), dtype, 600 + step_i, dev)
        binding.pa_reshape_and_cache(k, v, pool, torch.from_numpy(slots).to(dev))
        assert oracle.reshape_and_cache(u16(k), u16(v), pool_bits, slots, nb, B, Hkv, D) == len(ids)
        lens = np.array([pc.seq_len(sid) for sid in ids], np.int32)
        bt = pc.block_tables(ids, int(-(-lens.max() // B)))
        out = torch.empty_like(q)
        ws = binding.decode_workspace(q, pool)
        binding.pa_decode(out, q, pool, torch.from_numpy(bt).to(dev), torch.from_numpy(lens).to(dev), scale, ws,
                          flags=binding.PA_DECODE_SHARED_BLOCKS)
        torch.cuda.synchronize()
        want = oracle.decode(u16(q), pool_bits, bt, lens, scale, Hq, Hkv, D, nb, B, dtype)
        assert max_abs_err(oracle.decode_elems(u16(out), dtype), want) <= TOL[dtype]
    assert binding.pa_get_device_error() == 0


def test_evicted_prompt_is_recomputed(dev):
    """Free every request, then push enough other prompts through the pool to
    reuse the system prompt's blocks: the next request with that prompt hits
    nothing and its recomputed outputs still match the oracle."""
    import torch
    B, D, nb, H = 16, 128, 40, 4
    rng = np.random.default_rng(8)
    system = list(rng.integers(0, 32000, size=100))
    pc = binding.PrefixCache(nb, B)
    pool = workloads.normal_values((2, nb, B, H, D), workloads.F16, 41, dev)
    s0, hit = pc.add_seq(system + [1, 2, 3])
    assert hit == 0
    pc.free_seq(s0)
    s1, hit = pc.add_seq(system + [4])
    assert hit == 96
    pc.free_seq(s1)
    hog, _ = pc.add_seq(list(rng.integers(0, 32000, size=(nb - 1) * B)))   # the whole pool
    pc.free_seq(hog)
    s2, hit = pc.add_seq(system + [5, 6])
    assert hit == 0
    p_len = len(system) + 2
    slots = pc.slots(s2, 0, p_len)
    k = workloads.normal_values((p_len, H, D), workloads.F16, 42, dev)
    v = workloads.normal_values((p_len, H, D), workloads.F16, 43, dev)
    q = workloads.normal_values((p_len, H, D), workloads.F16, 44, dev)
    pool_bits = u16(pool).copy()
    binding.pa_reshape_and_cache(k, v, pool, torch.from_numpy(slots).to(dev))
    oracle.reshape_and_cache(u16(k), u16(v), pool_bits, slots, nb, B, H, D)
    bt = pc.block_tables([s2], -(-p_len // B))
    out = torch.empty_like(q)
    cu = torch.tensor([0, p_len], dtype=torch.int32, device=dev)
    sl = torch.tensor([p_len], dtype=torch.int32, device=dev)
    binding.pa_prefill(out, q, pool, torch.from_numpy(bt).to(dev), cu, sl, 1 / math.sqrt(D), p_len)
    torch.cuda.synchronize()
    want = oracle.prefill(u16(q), pool_bits, bt, np.array([0, p_len], np.int32), np.array([p_len], np.int32),
                          1 / math.sqrt(D), H, H, D, nb, B, workloads.F16)
    assert max_abs_err(oracle.decode_elems(u16(out), workloads.F16), want) <= TOL[workloads.F16]
    assert binding.pa_get_device_error() == 0


@pytest.mark.parametrize("dtype,Hq,Hkv", [(workloads.F16, 8, 8), (workloads.BF16, 16, 8)])
def test_admitted_wave_one_packed_prefill(dev, dtype, Hq, Hkv):
    """Two waves through pa_pcache_admit: the second hits the first's system
    prompt. Each wave's uncached tokens are written with one
    pa_reshape_and_cache and attended with one pa_prefill over the packed
    queries (cu_seqlens_q from the admission); outputs against the oracle on
    the same tables, the pool bit-exact against the oracle's writes, and the
    cached block hashes against the model's SHA-256 chain."""
    import torch
    B, D, nb = 16, 128, 160
    rng = np.random.default_rng(21 + Hq)
    system = list(rng.integers(0, 32000, size=150))
    pc, m = binding.PrefixCache(nb, B), PrefixCacheModel(nb, B)
    pool = workloads.normal_values((2, nb, B, Hkv, D), dtype, 60, dev)
    pool_bits = u16(pool).copy()
    scale = 1 / math.sqrt(D)
    maxb = 16
    for wave in range(2):
        prompts = [system + list(rng.integers(0, 32000, size=int(n))) for n in rng.integers(1, 90, size=5)]
        flat = np.array([t for p in prompts for t in p], np.int32)
        cu_t = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
        count, out = pc.admit(flat, cu_t, maxb)
        assert count == len(prompts)
        want_ids = [m.add_seq(p) for p in prompts]
        assert [(int(a), int(b)) for a, b in zip(out["seq_ids"], out["num_cached"])] == want_ids
        if wave == 1:
            assert all(h == 144 for _, h in want_ids)      # 9 full system blocks
        cu_q = out["cu_seqlens_q"]
        n = int(cu_q[-1])
        k = workloads.normal_values((n, Hkv, D), dtype, 700 + wave, dev)
        v = workloads.normal_values((n, Hkv, D), dtype, 710 + wave, dev)
        q = workloads.normal_values((n, Hq, D), dtype, 720 + wave, dev)
        slots = out["slot_mapping"][:n]
        binding.pa_reshape_and_cache(k, v, pool, torch.from_numpy(slots).to(dev))
        assert oracle.reshape_and_cache(u16(k), u16(v), pool_bits, slots, nb, B, Hkv, D) == n
        o = torch.empty_like(q)
        binding.pa_prefill(o, q, pool, torch.from_numpy(out["block_tables"]).to(dev),
                           torch.from_numpy(cu_q).to(dev), torch.from_numpy(out["seq_lens"]).to(dev), scale,
                           int(np.diff(cu_q).max()))
        torch.cuda.synchronize()
        want = oracle.prefill(u16(q), pool_bits, out["block_tables"], cu_q, out["seq_lens"], scale, Hq, Hkv, D,
                              nb, B, dtype)
        assert max_abs_err(oracle.decode_elems(u16(o), dtype), want) <= TOL[dtype]
        assert np.array_equal(u16(pool), pool_bits)
        for b in range(nb):
            assert pc.block_hash(b) == m.hash[b]
        pc.free_seqs(out["seq_ids"].copy())
        for sid, _ in want_ids:
            m.free_seq(sid)
    assert binding.pa_get_device_error() == 0
