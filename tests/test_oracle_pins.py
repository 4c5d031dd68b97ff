"""Pins for the oracle: it is checked against what the pages print and what
the mathematics fixes, never against itself or the CUDA path.

Each test names the fact it pins. Together they are chosen so that a
plausible slip anywhere in the oracle (a decoder bias, a swapped K/V index,
a transposed pool dimension, a dropped scale, a wrong GQA mapping, a wrong
merge sign) fails at least one of them; tests/test_oracle_mutants.py plants
such slips in a copy of the oracle and checks exactly that.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- decoders

def test_f16_decoder_matches_numpy_for_every_pattern():
    """IEEE binary16 decoding == numpy's float16 (a library routine), all 65536 patterns."""
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode_elems(bits, oracle.F16)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.f16_to_double(0x3C00) == 1.0
    assert oracle.f16_to_double(0x0001) == 2.0 ** -24


def test_bf16_decoder_matches_float32_upper_half_for_every_pattern():
    """bfloat16 is the upper half of a binary32: decode == (bits << 16) viewed as float32."""
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode_elems(bits, oracle.BF16)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen to quiet NaNs
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.bf16_to_double(0x3F80) == 1.0


# ------------------------------------------------------------ slot mapping

def test_slot_formula_printed_example():
    """vLLM book §4.4.3: table [7,3,12,25], length 50 -> the new token's slot is 402."""
    g = _golden("slot_mapping_example.json")
    assert oracle.slot(g["table"], g["block_size"], g["new_token_position"]) == g["expected_slot"]


def test_slot_formula_worked_example_new_tokens():
    """Worked example tables [3,7],[0,5,9],[4] at lengths 25/47/12: the next token's slots."""
    g = _golden("worked_example.json")
    got = [oracle.slot(g["requests"][r]["table"], g["block_size"], g["requests"][r]["tokens"])
           for r in ("A", "B", "C")]
    assert got == [7 * 16 + 9, 9 * 16 + 15, 4 * 16 + 12] == [121, 159, 76]


def test_slot_formula_every_position_covers_table_once():
    """Brute force: positions 0..nB-1 hit every slot of the table's blocks exactly once, in order."""
    table = [5, 1, 7]
    B = 16
    slots = [oracle.slot(table, B, p) for p in range(len(table) * B)]
    expected = [b * B + o for b in table for o in range(B)]
    assert slots == expected


# --------------------------------------------------------- write and copy

def _pool(nb, bs, h, d, rng):
    return rng.integers(0, 65536, size=(2, nb, bs, h, d), dtype=np.uint16)


def test_reshape_and_cache_matches_numpy_scatter():
    """kv[0][slot // B][slot % B] = key[t], kv[1][...] = value[t]; negative slots skipped."""
    rng = np.random.default_rng(0)
    nb, bs, h, d, t = 6, 16, 3, 8, 7
    pool = _pool(nb, bs, h, d, rng)
    key = rng.integers(0, 65536, size=(t, h, d), dtype=np.uint16)
    val = rng.integers(0, 65536, size=(t, h, d), dtype=np.uint16)
    slots = np.array([0, 17, 95, -1, 40, 63, -5], dtype=np.int32)
    ref = pool.copy()
    flat = ref.reshape(2, nb * bs, h, d)
    for i, s in enumerate(slots):
        if s >= 0:
            flat[0, s] = key[i]
            flat[1, s] = val[i]
    got = pool.copy()
    n = oracle.reshape_and_cache(key, val, got, slots, nb, bs, h, d)
    assert n == 5
    assert np.array_equal(got, ref)


def test_reshape_and_cache_rejects_slot_beyond_pool():
    rng = np.random.default_rng(1)
    pool = _pool(2, 16, 1, 8, rng)
    key = np.zeros((1, 1, 8), dtype=np.uint16)
    assert oracle.reshape_and_cache(key, key, pool, [32], 2, 16, 1, 8) == -1


def test_copy_blocks_matches_numpy_block_assignment():
    """COW copy: whole block (all slots, K and V, all heads) of src -> dst, every layer."""
    rng = np.random.default_rng(2)
    nb, bs, h, d = 8, 16, 2, 8
    pools = [_pool(nb, bs, h, d, rng) for _ in range(3)]
    pairs = [(1, 4), (6, 2), (0, 7)]
    refs = [p.copy() for p in pools]
    for r in refs:
        for s, t in pairs:
            r[:, t] = r[:, s]
    assert oracle.copy_blocks(pools, pairs, nb, bs, h, d) == 0
    for p, r in zip(pools, refs):
        assert np.array_equal(p, r)


# ------------------------------------------------------------- attention

def _f16(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def test_single_token_returns_its_value_row_exactly():
    """Closed form: softmax over one token is 1, so o = v_0 bit for bit."""
    rng = np.random.default_rng(3)
    q = _f16(rng.standard_normal(64))
    k = _f16(rng.standard_normal((1, 64)))
    v = _f16(rng.standard_normal((1, 64)))
    out = oracle.attention_contiguous(q, k, v, 0.125, oracle.F16)
    assert np.array_equal(out, v.view(np.float16)[0].astype(np.float64))


def test_empty_sequence_gives_zero_row():
    q = _f16(np.ones(64))
    k = np.zeros((0, 64), dtype=np.uint16)
    out = oracle.attention_contiguous(q, k, k, 0.125, oracle.F16)
    assert np.array_equal(out, np.zeros(64))


def test_equal_scores_give_the_mean_of_values():
    """q = 0 makes every score equal, so o is the arithmetic mean of the V rows."""
    rng = np.random.default_rng(4)
    L, D = 37, 64
    q = _f16(np.zeros(D))
    k = _f16(rng.standard_normal((L, D)))
    v = _f16(rng.standard_normal((L, D)))
    out = oracle.attention_contiguous(q, k, v, 0.125, oracle.F16)
    mean = v.view(np.float16).astype(np.float64).mean(axis=0)
    assert np.allclose(out, mean, rtol=0, atol=1e-14)


def test_two_tokens_closed_form_with_scale():
    """Scores 2*scale and 0: o = sigma(2s) v0 + sigma(-2s) v1, sigma via tanh."""
    D, scale = 64, 0.3
    q = np.zeros(D); q[0] = 1.0
    k = np.zeros((2, D)); k[0, 0] = 2.0
    v = np.zeros((2, D)); v[0, :] = 1.5; v[1, :] = -0.25; v[1, 5] = 3.0
    out = oracle.attention_contiguous(_f16(q), _f16(k), _f16(v), scale, oracle.F16)
    sig = lambda z: 0.5 * (1.0 + math.tanh(0.5 * z))
    expect = sig(2 * scale) * v[0] + sig(-2 * scale) * v[1]
    assert np.allclose(out, expect, rtol=0, atol=1e-14)


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_attention_matches_scipy_softmax_brute_force(dtype):
    """Random tiny cases against scipy.special.softmax and numpy matmul (library routines)."""
    rng = np.random.default_rng(5 + dtype)
    for L, D in [(1, 64), (5, 64), (16, 128), (33, 128)]:
        raw_q, raw_k, raw_v = rng.standard_normal(D), rng.standard_normal((L, D)), rng.standard_normal((L, D))
        if dtype == oracle.F16:
            q, k, v = _f16(raw_q), _f16(raw_k), _f16(raw_v)
            val = lambda a: a.view(np.float16).astype(np.float64)
        else:
            tob = lambda a: (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)
            q, k, v = tob(raw_q), tob(raw_k), tob(raw_v)
            val = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        scale = 1.0 / math.sqrt(D)
        w = scipy.special.softmax(scale * (val(k) @ val(q)))
        expect = w @ val(v)
        got = oracle.attention_contiguous(q, k, v, scale, dtype)
        assert np.allclose(got, expect, rtol=0, atol=1e-13)


@pytest.mark.parametrize("part_len", [1, 3, 16, 50, 1000])
def test_online_merge_equals_two_pass(part_len):
    """vLLM book §4.6: the (m, s, O) recurrence reaches the two-pass softmax result."""
    rng = np.random.default_rng(6)
    L, D = 211, 64
    q = _f16(rng.standard_normal(D) * 2)
    k = _f16(rng.standard_normal((L, D)))
    v = _f16(rng.standard_normal((L, D)))
    two = oracle.attention_contiguous(q, k, v, 0.125, oracle.F16)
    online = oracle.attention_online(q, k, v, 0.125, oracle.F16, part_len)
    assert np.allclose(online, two, rtol=0, atol=1e-13)


# --------------------------------------------------------------- paged decode

def _paged_case(rng, lens, B, Hq, Hkv, D, nb, dtype=oracle.F16):
    max_blk = max(1, max(-(-L // B) for L in lens))
    perm = rng.permutation(nb)
    bt = np.full((len(lens), max_blk), -1, dtype=np.int32)
    i = 0
    for s, L in enumerate(lens):
        n = -(-L // B)
        bt[s, :n] = perm[i:i + n]
        i += n
    pool = _f16(rng.standard_normal((2, nb, B, Hkv, D)))
    q = _f16(rng.standard_normal((len(lens), Hq, D)))
    return q, pool, bt, np.array(lens, dtype=np.int32)


def _gather(pool, bt_row, L, B, h):
    """Independent numpy gather: token i lives at pool[c, bt[i // B], i % B, h]."""
    idx_b = np.array([bt_row[i // B] for i in range(L)], dtype=np.int64)
    idx_o = np.arange(L) % B
    return pool[0, idx_b, idx_o, h], pool[1, idx_b, idx_o, h]


def test_paged_decode_equals_contiguous_attention_on_gathered_kv():
    """Digest "常见误解": paging changes where K/V live, not the result."""
    rng = np.random.default_rng(7)
    lens, B, Hq, Hkv, D, nb = [1, 15, 16, 17, 47, 90], 16, 4, 2, 64, 40
    q, pool, bt, sl = _paged_case(rng, lens, B, Hq, Hkv, D, nb)
    out = oracle.decode(q, pool, bt, sl, 0.125, Hq, Hkv, D, nb, B, oracle.F16)
    for s, L in enumerate(lens):
        for hq in range(Hq):
            k, v = _gather(pool, bt[s], L, B, hq // (Hq // Hkv))
            val = lambda a: a.view(np.float16).astype(np.float64)
            w = scipy.special.softmax(0.125 * (val(k) @ val(q[s, hq])))
            assert np.allclose(out[s, hq], w @ val(v), rtol=0, atol=1e-13)


def test_gqa_maps_contiguous_query_groups_to_one_kv_head():
    """Each kv head h has V = const c_h; q heads h*G..h*G+G-1 must return exactly c_h."""
    rng = np.random.default_rng(8)
    lens, B, Hq, Hkv, D, nb = [20, 33], 16, 6, 3, 64, 12
    q, pool, bt, sl = _paged_case(rng, lens, B, Hq, Hkv, D, nb)
    consts = [0.5, -2.0, 3.25]
    for h, c in enumerate(consts):
        pool[1, :, :, h, :] = _f16(np.full((nb, B, D), c))
    out = oracle.decode(q, pool, bt, sl, 0.125, Hq, Hkv, D, nb, B, oracle.F16)
    for hq in range(Hq):
        assert np.allclose(out[:, hq, :], consts[hq // 2], rtol=0, atol=1e-14)


def test_decode_invariant_under_physical_block_permutation():
    """Moving blocks to other physical ids (and rewriting tables) leaves outputs bit-identical."""
    rng = np.random.default_rng(9)
    lens, B, Hq, Hkv, D, nb = [5, 16, 31, 64, 70], 16, 8, 2, 64, 30
    q, pool, bt, sl = _paged_case(rng, lens, B, Hq, Hkv, D, nb)
    ref = oracle.decode(q, pool, bt, sl, 0.125, Hq, Hkv, D, nb, B, oracle.F16)
    sigma = rng.permutation(nb)            # block b moves to sigma[b]
    pool2 = np.empty_like(pool)
    pool2[:, sigma] = pool
    bt2 = np.where(bt >= 0, sigma[np.maximum(bt, 0)], -1).astype(np.int32)
    got = oracle.decode(q, pool2, bt2, sl, 0.125, Hq, Hkv, D, nb, B, oracle.F16)
    assert np.array_equal(got, ref)


def test_decode_ignores_padding_slots_of_the_last_block():
    """Only the L valid tokens are read: poisoning the unused slots (NaN) changes nothing."""
    rng = np.random.default_rng(10)
    lens, B, Hq, Hkv, D, nb = [3, 18, 40], 16, 2, 2, 64, 10
    q, pool, bt, sl = _paged_case(rng, lens, B, Hq, Hkv, D, nb)
    ref = oracle.decode(q, pool, bt, sl, 0.125, Hq, Hkv, D, nb, B, oracle.F16)
    poisoned = pool.copy()
    for s, L in enumerate(lens):
        last = bt[s, (L - 1) // B]
        poisoned[:, last, L % B if L % B else B:, :, :] = 0x7E00   # fp16 NaN
    got = oracle.decode(q, poisoned, bt, sl, 0.125, Hq, Hkv, D, nb, B, oracle.F16)
    assert np.array_equal(got, ref)


def test_decode_sampled_equals_full_batch():
    rng = np.random.default_rng(11)
    lens, B, Hq, Hkv, D, nb = [9, 50, 17], 16, 4, 1, 64, 12
    q, pool, bt, sl = _paged_case(rng, lens, B, Hq, Hkv, D, nb)
    full = oracle.decode(q, pool, bt, sl, 0.125, Hq, Hkv, D, nb, B, oracle.F16)
    seqs, heads = np.array([2, 0, 1]), np.array([3, 1, 0])
    got = oracle.decode_sampled(seqs, heads, q, pool, bt, sl, 0.125, Hq, Hkv, D, nb, B, oracle.F16)
    assert np.array_equal(got, full[seqs, heads])


def test_zero_length_sequence_gives_zero_rows():
    rng = np.random.default_rng(12)
    q, pool, bt, sl = _paged_case(rng, [4, 20], 16, 2, 2, 64, 6)
    sl = np.array([0, 20], dtype=np.int32)
    out = oracle.decode(q, pool, bt, sl, 0.125, 2, 2, 64, 6, 16, oracle.F16)
    assert np.array_equal(out[0], np.zeros((2, 64)))


# --------------------------------------------------------------- sizing

def test_sizing_numbers_printed_by_the_pages():
    """vLLM book §4.1.1 / §4.3.1: 819,200 B per token; 320 KB per block per layer; 12.5 MB complete block."""
    g = _golden("sizing.json")["llama2_13b"]
    shape_one_block = (2, 1, g["block_size"], g["num_kv_heads"], g["head_size"])
    per_token = 2 * g["num_layers"] * g["num_kv_heads"] * g["head_size"] * g["dtype_bytes"]
    assert per_token == g["kv_bytes_per_token"]
    assert int(np.prod(shape_one_block)) * g["dtype_bytes"] == g["block_bytes_per_layer"]
    assert g["num_layers"] * g["block_bytes_per_layer"] == g["complete_block_bytes"]
