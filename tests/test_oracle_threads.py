"""The oracle's row-parallel batch functions give the same bits on one thread
and on all of them.

Each output row (one sequence or query row, one q-head) is computed by the
same single-threaded code whatever the thread count, so threading may change
only the time. These tests check that on every batch-level function, with
ragged lengths, GQA, an empty sequence and a prefill batch whose chunks
differ in length (including an empty chunk).
"""
import os

import numpy as np
import pytest

import oracle

B, HQ, HKV, D = 16, 8, 2, 64


def _batch(seed, lens):
    rng = np.random.default_rng(seed)
    nblk = [-(-L // B) for L in lens]
    nb = sum(nblk) + 3
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((len(lens), max(1, max(nblk))), -1, np.int32)
    i = 0
    for s, n in enumerate(nblk):
        bt[s, :n] = perm[i:i + n]
        i += n
    pool = rng.standard_normal((2, nb, B, HKV, D)).astype(np.float16).view(np.uint16)
    fp8 = rng.integers(0, 256, size=(2, nb, B, HKV, D), dtype=np.uint8)
    fp8[(fp8 & 0x7F) == 0x7F] = 0x10      # no NaN codes: finite outputs compare exactly
    q = rng.standard_normal((len(lens), HQ, D)).astype(np.float16).view(np.uint16)
    return nb, bt, np.array(lens, np.int32), pool, fp8, q


@pytest.fixture
def restore_threads():
    n = oracle.threads()
    yield
    oracle.set_threads(n)


def _both(fn):
    oracle.set_threads(1)
    one = fn()
    oracle.set_threads(max(4, os.cpu_count() or 1))
    many = fn()
    return one, many


def test_threaded_decode_is_bit_identical(restore_threads):
    lens = [1, 37, 0, 200, 16, 95, 3, 64]
    nb, bt, sl, pool, fp8, q = _batch(3, lens)
    scale = D ** -0.5
    one, many = _both(lambda: oracle.decode(q, pool, bt, sl, scale, HQ, HKV, D, nb, B, oracle.F16))
    assert np.array_equal(one, many)
    one, many = _both(lambda: oracle.decode_fp8(q, fp8, bt, sl, scale, HQ, HKV, D, nb, B, oracle.F16,
                                                0.03, 0.02))
    assert np.array_equal(one, many)
    seqs = np.array([0, 3, 3, 5, 7, 1], np.int32)
    heads = np.array([0, 7, 2, 5, 1, 3], np.int32)
    one, many = _both(lambda: oracle.decode_sampled(seqs, heads, q, pool, bt, sl, scale, HQ, HKV, D,
                                                    nb, B, oracle.F16))
    assert np.array_equal(one, many)
    full = oracle.decode(q, pool, bt, sl, scale, HQ, HKV, D, nb, B, oracle.F16)
    assert np.array_equal(many, full[seqs, heads])
    one, many = _both(lambda: oracle.decode_fp8_sampled(seqs, heads, q, fp8, bt, sl, scale, HQ, HKV,
                                                        D, nb, B, oracle.F16, 0.03, 0.02))
    assert np.array_equal(one, many)


def test_threaded_prefill_is_bit_identical(restore_threads):
    lens = [40, 70, 33, 90]
    chunks = [5, 0, 33, 17]
    nb, bt, sl, pool, fp8, _ = _batch(4, lens)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    rng = np.random.default_rng(9)
    q = rng.standard_normal((int(cu[-1]), HQ, D)).astype(np.float16).view(np.uint16)
    scale = D ** -0.5
    one, many = _both(lambda: oracle.prefill(q, pool, bt, cu, sl, scale, HQ, HKV, D, nb, B, oracle.F16))
    assert np.array_equal(one, many)
    # each prefill row is the decode definition over its causal prefix
    s, i = 3, 4
    row = int(cu[s]) + i
    vis = np.array([int(sl[s]) - chunks[s] + i + 1], np.int32)
    want = oracle.decode(q[row:row + 1], pool, bt[s:s + 1], vis, scale, HQ, HKV, D, nb, B, oracle.F16)
    assert np.array_equal(many[row], want[0])
    one, many = _both(lambda: oracle.prefill_fp8(q, fp8, bt, cu, sl, scale, HQ, HKV, D, nb, B, oracle.F16,
                                                 0.03, 0.02))
    assert np.array_equal(one, many)
