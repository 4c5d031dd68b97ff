"""Pins for the oracle's causal chunked prefill (the varlen read path).

What fixes it: a chunk of q_len query tokens is the last q_len tokens of
the sequence's cached context, so query i (position p = seq_len - q_len + i)
sees tokens 0..p. With q_len = 1 it is the pinned decode; every row is a
softmax over an explicitly gathered prefix (checked against SciPy's softmax
on tiny cases); tokens after p cannot change row i; and the placement of
blocks cannot change anything.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle


def _f16(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def _case(rng, ctx, qlens, B=16, Hq=4, Hkv=2, D=16, spare=3):
    """Sequences with total lengths ctx[s], the last qlens[s] of them queried."""
    nblk = [-(-L // B) for L in ctx]
    nb = sum(nblk) + spare
    perm = rng.permutation(nb)
    maxb = max(1, max(nblk))
    bt = np.full((len(ctx), maxb), -1, np.int32)
    k = 0
    for s, n in enumerate(nblk):
        bt[s, :n] = perm[k:k + n]
        k += n
    pool = _f16(rng.normal(0, 1, (2, nb, B, Hkv, D)))
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = _f16(rng.normal(0, 1, (int(cu[-1]), Hq, D)))
    return dict(pool=pool, bt=bt, cu=cu, sl=np.array(ctx, np.int32), q=q, nb=nb, B=B, Hq=Hq,
                Hkv=Hkv, D=D, scale=1 / math.sqrt(D))


def _run(c, pool=None, bt=None):
    return oracle.prefill(c["q"], c["pool"] if pool is None else pool,
                          c["bt"] if bt is None else bt, c["cu"], c["sl"], c["scale"], c["Hq"],
                          c["Hkv"], c["D"], c["nb"], c["B"], oracle.F16)


def test_single_query_chunks_are_the_pinned_decode():
    rng = np.random.default_rng(1)
    c = _case(rng, [5, 40, 16, 1], [1, 1, 1, 1])
    got = _run(c)
    ref = oracle.decode(c["q"], c["pool"], c["bt"], c["sl"], c["scale"], c["Hq"], c["Hkv"],
                        c["D"], c["nb"], c["B"], oracle.F16)
    assert np.array_equal(got, ref)


def test_rows_match_scipy_softmax_over_the_causal_prefix():
    """Brute force: gather K/V of positions 0..p through the table by hand and
    apply scipy.special.softmax; GQA head map hq // (Hq / Hkv)."""
    rng = np.random.default_rng(2)
    c = _case(rng, [7, 35, 20], [3, 35, 6])
    got = _run(c)
    vals = c["pool"].view(np.float16).astype(np.float64)
    q = c["q"].view(np.float16).astype(np.float64)
    G = c["Hq"] // c["Hkv"]
    for s in range(3):
        L, ql = int(c["sl"][s]), int(c["cu"][s + 1] - c["cu"][s])
        for i in range(ql):
            p = L - ql + i
            for hq in range(c["Hq"]):
                h = hq // G
                K = np.stack([vals[0, c["bt"][s, t // c["B"]], t % c["B"], h] for t in range(p + 1)])
                V = np.stack([vals[1, c["bt"][s, t // c["B"]], t % c["B"], h] for t in range(p + 1)])
                w = scipy.special.softmax(c["scale"] * (K @ q[c["cu"][s] + i, hq]))
                assert np.allclose(got[c["cu"][s] + i, hq], w @ V, rtol=1e-12, atol=1e-13)


def test_tokens_after_a_query_do_not_change_its_row():
    """Causality: overwrite every cached token after position p of query 0 of
    sequence 1 with other values; that row is unchanged, later rows change."""
    rng = np.random.default_rng(3)
    c = _case(rng, [30, 50], [4, 10])
    before = _run(c)
    s, L, ql = 1, 50, 10
    p0 = L - ql
    pool2 = c["pool"].copy()
    for t in range(p0 + 1, L):
        pool2[:, c["bt"][s, t // c["B"]], t % c["B"]] = _f16(rng.normal(0, 3, (2, c["Hkv"], c["D"])))
    after = _run(c, pool=pool2)
    row0 = c["cu"][s]
    assert np.array_equal(after[row0], before[row0])
    assert not np.allclose(after[row0 + 1:row0 + ql], before[row0 + 1:row0 + ql])
    assert np.array_equal(after[:c["cu"][1]], before[:c["cu"][1]])


def test_last_query_sees_the_whole_sequence_and_first_sees_one_less_per_step():
    rng = np.random.default_rng(4)
    c = _case(rng, [33, 64, 17], [5, 64, 2])
    got = _run(c)
    full = oracle.decode(c["q"][c["cu"][1:] - 1], c["pool"], c["bt"], c["sl"], c["scale"], c["Hq"],
                         c["Hkv"], c["D"], c["nb"], c["B"], oracle.F16)
    assert np.array_equal(got[c["cu"][1:] - 1], full)
    # query i of a chunk of q_len is the decode over seq_len - q_len + i + 1 tokens
    shorter = oracle.decode(c["q"][c["cu"][:-1]], c["pool"], c["bt"],
                            c["sl"] - (c["cu"][1:] - c["cu"][:-1]) + 1, c["scale"], c["Hq"],
                            c["Hkv"], c["D"], c["nb"], c["B"], oracle.F16)
    assert np.array_equal(got[c["cu"][:-1]], shorter)


def test_prefill_invariant_under_block_permutation():
    rng = np.random.default_rng(5)
    c = _case(rng, [40, 70], [12, 70], spare=10)
    got = _run(c)
    sigma = rng.permutation(c["nb"])
    pool2 = np.empty_like(c["pool"])
    pool2[:, sigma] = c["pool"]
    bt2 = np.where(c["bt"] >= 0, sigma[np.maximum(c["bt"], 0)], -1).astype(np.int32)
    assert np.array_equal(_run(c, pool=pool2, bt=bt2), got)


def test_empty_chunks_write_nothing():
    rng = np.random.default_rng(6)
    c = _case(rng, [10, 20, 5], [0, 3, 0])
    got = _run(c)
    assert got.shape == (3, c["Hq"], c["D"])
    ref = oracle.decode(c["q"][[0, 1, 2]], c["pool"], c["bt"][[1, 1, 1]],
                        np.array([18, 19, 20], np.int32), c["scale"], c["Hq"], c["Hkv"], c["D"],
                        c["nb"], c["B"], oracle.F16)
    assert np.array_equal(got, ref)


# ----------------------------------------------------------- FP8 cache

def _fp8_case(rng, ctx, qlens, B=16, Hq=4, Hkv=2, D=16, spare=3):
    c = _case(rng, ctx, qlens, B, Hq, Hkv, D, spare)
    codes = rng.integers(0, 254, c["pool"].shape).astype(np.uint8)
    c["codes"] = np.where(codes >= 0x7F, codes + 1, codes).astype(np.uint8)  # every finite code
    return c


def test_fp8_single_query_chunks_are_the_pinned_fp8_decode():
    rng = np.random.default_rng(11)
    c = _fp8_case(rng, [5, 40, 16, 1], [1, 1, 1, 1])
    got = oracle.prefill_fp8(c["q"], c["codes"], c["bt"], c["cu"], c["sl"], c["scale"], c["Hq"], c["Hkv"],
                             c["D"], c["nb"], c["B"], oracle.F16, 0.02, 0.05)
    ref = oracle.decode_fp8(c["q"], c["codes"], c["bt"], c["sl"], c["scale"], c["Hq"], c["Hkv"], c["D"],
                            c["nb"], c["B"], oracle.F16, 0.02, 0.05)
    assert np.array_equal(got, ref)


def test_fp8_prefill_equals_16bit_prefill_on_the_dequantized_pool():
    """Power-of-two scales (different for K and V) make every dequantised
    value an fp16 value: the FP8 prefill must equal the pinned 16-bit prefill
    on a pool holding those values, row for row, bit for bit."""
    rng = np.random.default_rng(12)
    c = _fp8_case(rng, [7, 35, 20, 64], [3, 35, 6, 17])
    ks, vs = 0.25, 2.0
    vals = np.vectorize(oracle.e4m3_to_double)(c["codes"])
    vals[0] *= ks
    vals[1] *= vs
    pool16 = vals.astype(np.float16)
    assert np.array_equal(pool16.astype(np.float64), vals)
    got = oracle.prefill_fp8(c["q"], c["codes"], c["bt"], c["cu"], c["sl"], c["scale"], c["Hq"], c["Hkv"],
                             c["D"], c["nb"], c["B"], oracle.F16, ks, vs)
    ref = _run(c, pool=pool16.view(np.uint16))
    assert np.array_equal(got, ref)
