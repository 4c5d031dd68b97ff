"""Pins for the oracle's FP8 (E4M3) cache functions.

The E4M3 format is fixed by the OCP 8-bit floating point specification
(1 sign bit, 4 exponent bits with bias 7, 3 fraction bits, no infinities,
S.1111.111 = NaN, largest finite 448). PyTorch's ``float8_e4m3fn`` is an
independent implementation of it, so it serves as the library routine the
decoder and the rounding are checked against; closed forms and invariants
cover what PyTorch does differently (it does not saturate).

The decode pin reduces the FP8 path to the already-pinned 16-bit path: with
power-of-two scales every dequantised value is exact in fp16, so decoding the
byte pool must give exactly what the 16-bit decode gives on a pool holding
those values.
"""
import math

import numpy as np
import pytest
import torch

import oracle

E4M3 = torch.float8_e4m3fn


def _torch_codes(x):
    """E4M3 codes of fp32 values as PyTorch rounds them (nearest, ties to even)."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(E4M3).view(torch.uint8).numpy()


def _torch_values(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(E4M3).to(torch.float64).numpy()


# ----------------------------------------------------------------- decoder

def test_e4m3_decoder_matches_torch_for_every_code():
    """Every one of the 256 codes decodes to PyTorch's float8_e4m3fn value."""
    got = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    ref = _torch_values(np.arange(256))
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decoder_closed_forms():
    """Values the format's definition fixes: 1.0, 2.0, the extremes, signed zero."""
    assert oracle.e4m3_to_double(0x38) == 1.0           # exponent 7 = bias, fraction 0
    assert oracle.e4m3_to_double(0x40) == 2.0
    assert oracle.e4m3_to_double(0x7E) == 448.0         # 2^8 * 1.75
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6     # smallest normal
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9     # smallest subnormal
    assert oracle.e4m3_to_double(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_to_double(0xB8) == -1.0
    z = oracle.e4m3_to_double(0x80)
    assert z == 0.0 and math.copysign(1.0, z) == -1.0


# ----------------------------------------------------------------- encoder

def test_e4m3_encoder_round_trips_every_finite_code():
    """Rounding an exactly representable value returns its own code."""
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_from_float(oracle.e4m3_to_double(c)) == c, hex(c)


def test_e4m3_encoder_matches_torch_on_random_and_tie_values():
    """Nearest-even rounding == PyTorch's conversion, including every midpoint
    between adjacent codes (the ties) and the subnormal range."""
    rng = np.random.default_rng(7)
    finite = [oracle.e4m3_to_double(c) for c in range(0x7F)]  # 0 .. 448, ascending
    mids = [(a + b) / 2 for a, b in zip(finite[:-1], finite[1:])]
    xs = np.concatenate([
        np.array(mids), -np.array(mids),
        rng.uniform(-460, 460, 4000), rng.normal(0, 1, 4000), rng.uniform(-0.02, 0.02, 2000),
        np.array([464.0, -464.0, 2.0 ** -10, -(2.0 ** -10), 2.0 ** -11]),
    ]).astype(np.float32)
    got = np.array([oracle.e4m3_from_float(float(x)) for x in xs], dtype=np.uint8)
    assert np.array_equal(got, _torch_codes(xs))


def test_e4m3_encoder_ties_go_to_the_even_code():
    assert oracle.e4m3_from_float(1.0625) == 0x38   # between 1.0 (0x38) and 1.125 (0x39)
    assert oracle.e4m3_from_float(1.1875) == 0x3A   # between 1.125 (0x39) and 1.25 (0x3A)
    assert oracle.e4m3_from_float(2.0 ** -10) == 0x00
    assert oracle.e4m3_from_float(3 * 2.0 ** -10) == 0x02


def test_e4m3_encoder_saturates_and_keeps_nan():
    """Beyond the largest finite value the cache stores +-448 (a reading: the
    saturating conversion; PyTorch's cast gives NaN there instead)."""
    for x in (448.0, 449.0, 464.0, 480.0, 1e6, float("inf")):
        assert oracle.e4m3_from_float(x) == 0x7E
        assert oracle.e4m3_from_float(-x) == 0xFE
    assert oracle.e4m3_from_float(float("nan")) == 0x7F


# ---------------------------------------------------------------- quantise

@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_quantize_is_fp32_division_then_rounding(dtype):
    """code = e4m3(fp32(x) / fp32(scale)), checked against PyTorch doing the
    same division and cast (within the range where PyTorch does not give NaN)."""
    rng = np.random.default_rng(11)
    x = rng.normal(0, 3, 3000).astype(np.float32)
    tdt = torch.float16 if dtype == oracle.F16 else torch.bfloat16
    xt = torch.from_numpy(x).to(tdt)
    bits = xt.view(torch.int16).numpy().view(np.uint16)
    for scale in (1.0, 0.0371, 0.5, 3.3):
        q = (xt.float() / torch.tensor(scale, dtype=torch.float32))
        ok = q.abs() < 464
        ref = q.to(E4M3).view(torch.uint8).numpy()
        got = np.array([oracle.quantize_e4m3(int(b), dtype, scale) for b in bits], dtype=np.uint8)
        assert ok.float().mean() > 0.9
        assert np.array_equal(got[ok.numpy()], ref[ok.numpy()])
        assert np.all(np.isin(got[~ok.numpy()], [0x7E, 0xFE]))


# ------------------------------------------------------------- write path

def test_reshape_and_cache_fp8_places_quantized_rows_by_slot():
    """Token t's K/V rows land at pool[0/1][slot // B][slot % B] as codes of
    row / scale; negative slots are skipped and nothing else changes."""
    rng = np.random.default_rng(3)
    nb, B, H, D = 6, 16, 2, 8
    T = 5
    key = rng.normal(0, 2, (T, H, D)).astype(np.float16)
    val = rng.normal(0, 2, (T, H, D)).astype(np.float16)
    slots = np.array([17, -1, 0, 95, 40], dtype=np.int32)
    pool = rng.integers(0, 256, (2, nb, B, H, D), dtype=np.uint8)
    before = pool.copy()
    ks, vs = 0.25, 0.0625
    n = oracle.reshape_and_cache_fp8(key, val, pool, slots, nb, B, H, D, oracle.F16, ks, vs)
    assert n == 4
    expect = before.copy()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        expect[0, s // B, s % B] = _torch_codes(key[t].astype(np.float32) / np.float32(ks))
        expect[1, s // B, s % B] = _torch_codes(val[t].astype(np.float32) / np.float32(vs))
    assert np.array_equal(pool, expect)


def test_reshape_and_cache_fp8_rejects_slot_beyond_pool():
    pool = np.zeros((2, 2, 16, 1, 8), dtype=np.uint8)
    key = np.ones((1, 1, 8), dtype=np.float16)
    assert oracle.reshape_and_cache_fp8(key, key, pool, np.array([32], np.int32), 2, 16, 1, 8,
                                        oracle.F16, 1.0, 1.0) == -1


# -------------------------------------------------------------- read path

def _random_codes(rng, shape):
    """Codes of every finite E4M3 value (no NaN codes)."""
    c = rng.integers(0, 254, shape).astype(np.uint8)
    return np.where(c >= 0x7F, c + 1, c).astype(np.uint8)  # skip 0x7F; 0xFF is never drawn


@pytest.mark.parametrize("dtype,Hq,Hkv,D", [(oracle.F16, 4, 4, 16), (oracle.BF16, 8, 2, 32),
                                            (oracle.F16, 6, 1, 16)])
def test_fp8_decode_equals_16bit_decode_on_dequantized_pool(dtype, Hq, Hkv, D):
    """With power-of-two scales (different for K and V) every dequantised
    value is exact in fp16, so the FP8 decode must equal the pinned 16-bit
    decode run on a pool holding those values, bit for bit."""
    rng = np.random.default_rng(5)
    nb, B = 12, 16
    lens = np.array([1, 16, 37, 0, 70], dtype=np.int32)
    maxb = 5
    tables = np.array([rng.permutation(nb)[:maxb] for _ in lens], dtype=np.int32)
    codes = _random_codes(rng, (2, nb, B, Hkv, D))
    ks, vs = 0.125, 4.0
    vals = np.vectorize(oracle.e4m3_to_double)(codes)
    vals[0] *= ks
    vals[1] *= vs
    assert np.all(np.abs(vals) <= 448 * 4)
    if dtype == oracle.F16:
        pool16 = vals.astype(np.float16)
        assert np.array_equal(pool16.astype(np.float64), vals)
        pool16 = pool16.view(np.uint16)
        q = rng.normal(0, 1, (len(lens), Hq, D)).astype(np.float16).view(np.uint16)
    else:
        pool16 = torch.from_numpy(vals).to(torch.bfloat16)
        assert np.array_equal(pool16.double().numpy(), vals)
        pool16 = pool16.view(torch.int16).numpy().view(np.uint16)
        q = torch.randn(len(lens), Hq, D, generator=torch.Generator().manual_seed(1)).to(
            torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    scale = 1 / math.sqrt(D)
    got = oracle.decode_fp8(q, codes, tables, lens, scale, Hq, Hkv, D, nb, B, dtype, ks, vs)
    ref = oracle.decode(q, pool16, tables, lens, scale, Hq, Hkv, D, nb, B, dtype)
    assert np.array_equal(got, ref)
    assert np.all(got[3] == 0)


def test_fp8_decode_scales_k_and_v_separately():
    """Closed forms: one token returns its V row times v_scale whatever K is;
    two tokens with K rows differing by delta in the dot product give the
    weights softmax(scale * k_scale * delta)."""
    D, B, nb = 16, 16, 2
    pool = np.zeros((2, nb, B, 1, D), dtype=np.uint8)
    pool[0, 1, 0, 0, :] = 0x38          # K token 0: all 1.0
    pool[1, 1, 0, 0, :] = 0x40          # V token 0: all 2.0
    pool[0, 1, 1, 0, :] = 0x00          # K token 1: all 0
    pool[1, 1, 1, 0, :] = 0x00          # V token 1: all 0
    q = np.full((1, 1, D), 1.0, dtype=np.float16).view(np.uint16)
    tables = np.array([[1]], np.int32)
    one = oracle.decode_fp8(q, pool, tables, np.array([1], np.int32), 0.1, 1, 1, D, nb, B,
                            oracle.F16, 7.0, 3.0)
    assert np.allclose(one[0, 0], 2.0 * 3.0, rtol=0, atol=1e-15)
    two = oracle.decode_fp8(q, pool, tables, np.array([2], np.int32), 0.1, 1, 1, D, nb, B,
                            oracle.F16, 0.5, 3.0)
    x = 0.1 * 0.5 * D  # score of token 0; token 1 scores 0
    w0 = math.exp(x) / (math.exp(x) + 1.0)
    assert np.allclose(two[0, 0], w0 * 6.0, rtol=1e-14, atol=0)


def test_fp8_decode_sampled_equals_full_batch():
    rng = np.random.default_rng(9)
    nb, B, Hq, Hkv, D = 8, 16, 4, 2, 16
    lens = np.array([5, 33, 64], np.int32)
    tables = np.array([rng.permutation(nb)[:4] for _ in lens], np.int32)
    codes = _random_codes(rng, (2, nb, B, Hkv, D))
    q = rng.normal(0, 1, (3, Hq, D)).astype(np.float16).view(np.uint16)
    full = oracle.decode_fp8(q, codes, tables, lens, 0.25, Hq, Hkv, D, nb, B, oracle.F16, 0.3, 0.7)
    si = np.array([2, 0, 1, 2], np.int32)
    hi = np.array([3, 0, 2, 1], np.int32)
    samp = oracle.decode_fp8_sampled(si, hi, q, codes, tables, lens, 0.25, Hq, Hkv, D, nb, B,
                                     oracle.F16, 0.3, 0.7)
    assert np.array_equal(samp, full[si, hi])
