"""GPU parity of the chunked prefill over an FP8 (E4M3) cache
(pa_prefill_fp8) through the C ABI.

Bar: the chunk's codes written by pa_reshape_and_cache_fp8 bit-exact against
the oracle's quantisation; every output row within the 16-bit tolerances of
the query's type (2e-3 fp16 / 1e-2 bf16, max abs) of the fp64 oracle (each
row the FP8 decode definition over its causal prefix); NaN codes in padding
slots and unused blocks change nothing.
"""
import math

import numpy as np
import pytest

import oracle
from oracle.block_manager import BlockManagerModel
from paged_kv_cache_120_gb300 import binding, build, workloads

from harness import TOL, max_abs_err, max_abs_err_bf16_large, u16

pytestmark = pytest.mark.gpu

KS, VS = workloads.FP8_K_SCALE, workloads.FP8_V_SCALE


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.lib()
    assert binding.pa_get_device_error() == 0
    return torch.device("cuda:0")


def u8(t):
    return t.cpu().numpy().view(np.uint8)


class Fp8PrefillCase:
    """As the 16-bit prefill case, on a byte pool: the prefix is E4M3 codes of
    N(0,1)-sized values, the chunk's K/V go in by pa_reshape_and_cache_fp8."""

    def __init__(self, dev, dtype, Hq, Hkv, B, ctx, qlen, seed, spare=8, poison=False, ks=KS, vs=VS, D=128,
                 split=False):
        import torch
        self.dtype, self.Hq, self.Hkv, self.B, self.D, self.ks, self.vs = dtype, Hq, Hkv, B, D, ks, vs
        self.split = split
        self.scale = 1.0 / math.sqrt(D)
        rng = np.random.default_rng(seed)
        nb = sum(-(-L // B) for L in ctx) + spare
        self.nb = nb
        order = rng.permutation(nb)
        alloc = binding.BlockAllocator(nb, B, order)
        model = BlockManagerModel(nb, B, order)
        ids_a, ids_m, slots = [], [], []
        for L, q in zip(ctx, qlen):
            ids_a.append(alloc.add_seq(L - q))
            ids_m.append(model.add_seq(L - q))
        for a, m, q in zip(ids_a, ids_m, qlen):
            for _ in range(q):
                sa, ca = alloc.append_token(a)
                assert (sa, ca) == model.append_token(m)
                slots.append(sa)
        maxblk = max(1, max(len(model.table(m)) for m in ids_m))
        self.bt = alloc.block_tables(ids_a, maxblk)
        self.slots = np.array(slots, np.int32)
        self.seq_lens = alloc.seq_lens(ids_a)
        self.cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
        self.max_q = max(1, max(qlen))
        total = int(self.cu[-1])
        shape = (nb, B, Hkv, D)
        self.pool = torch.empty((2,) + shape, dtype=torch.uint8, device=dev)
        self.pool[0] = workloads.fp8_codes(shape, ks, seed + 1, dev)
        self.pool[1] = workloads.fp8_codes(shape, vs, seed + 5, dev)
        if poison:
            used = set(int(b) for b in self.bt.ravel() if b >= 0)
            for b in range(nb):
                if b not in used:
                    self.pool[:, b] = 0x7F
            for s, L in enumerate(ctx):
                if L % B:
                    self.pool[:, int(self.bt[s, (L - 1) // B]), L % B:] = 0xFF
        self.q = workloads.normal_values((max(total, 1), Hq, D), dtype, seed + 2, dev)[:total]
        self.k = workloads.normal_values((max(total, 1), Hkv, D), dtype, seed + 3, dev)[:total]
        self.v = workloads.normal_values((max(total, 1), Hkv, D), dtype, seed + 4, dev)[:total]
        self.pool_bits = u8(self.pool).copy()
        self.q_bits, self.k_bits, self.v_bits = u16(self.q), u16(self.k), u16(self.v)
        self.dev = dev

    def gpu(self):
        import torch
        t = lambda a: torch.from_numpy(a).to(self.dev)
        self.bt_d, self.sl_d, self.cu_d = t(self.bt), t(self.seq_lens), t(self.cu)
        if len(self.slots):
            binding.pa_reshape_and_cache_fp8(self.k.contiguous(), self.v.contiguous(), self.pool, t(self.slots),
                                             self.ks, self.vs)
        return self.prefill(self.pool, self.bt_d)

    def workspace(self):
        """The K/V-split workspace for this shape, filled with NaN bytes."""
        ws = binding.prefill_workspace(self.q, self.pool, len(self.seq_lens), self.max_q)
        assert ws is not None, "this shape does not split its K/V ranges"
        return ws.fill_(0xFF)

    def prefill(self, pool, bt_d, split=None):
        import torch
        split = self.split if split is None else split
        out = torch.full_like(self.q, float("nan"))
        binding.pa_prefill_fp8(out, self.q.contiguous(), pool, bt_d, self.cu_d, self.sl_d, self.scale,
                               self.max_q, self.ks, self.vs, self.workspace() if split else None)
        torch.cuda.synchronize()
        return out

    def oracle(self):
        if len(self.slots):
            assert oracle.reshape_and_cache_fp8(self.k_bits, self.v_bits, self.pool_bits, self.slots, self.nb,
                                                self.B, self.Hkv, self.D, self.dtype, self.ks,
                                                self.vs) == len(self.slots)
        return oracle.prefill_fp8(self.q_bits, self.pool_bits, self.bt, self.cu, self.seq_lens, self.scale,
                                  self.Hq, self.Hkv, self.D, self.nb, self.B, self.dtype, self.ks, self.vs)

    def check(self, out):
        want = self.oracle()
        assert np.array_equal(u8(self.pool), self.pool_bits), "reshape_and_cache_fp8 is not bit-exact"
        got = oracle.decode_elems(u16(out), self.dtype)
        err = max_abs_err(got, want)
        assert err <= TOL[self.dtype], f"max abs err {err}"
        assert binding.pa_get_device_error() == 0
        return got, want


CTX = [200, 128, 17, 300, 1, 129, 40, 517, 64]
QLEN = [200, 60, 1, 150, 1, 0, 40, 129, 64]
HEADS = [(4, 4), (8, 2), (8, 1), (16, 1), (32, 1), (12, 3), (40, 8)]


@pytest.mark.parametrize("split", [False, True], ids=["whole", "split"])
@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
@pytest.mark.parametrize("heads", HEADS)
def test_prefill_fp8_parity_small(dev, dtype, heads, split):
    Hq, Hkv = heads
    c = Fp8PrefillCase(dev, dtype, Hq, Hkv, 16, CTX, QLEN, seed=700 + Hq + Hkv + dtype, split=split)
    c.check(c.gpu())


@pytest.mark.parametrize("split", [False, True], ids=["whole", "split"])
@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
def test_prefill_fp8_nan_codes_in_padding_change_nothing(dev, dtype, split):
    c = Fp8PrefillCase(dev, dtype, 8, 2, 16, [33, 250, 7], [33, 100, 7], seed=41 + dtype, poison=True,
                       split=split)
    c.check(c.gpu())


@pytest.mark.parametrize("split", [False, True], ids=["whole", "split"])
@pytest.mark.parametrize("B", [32, 64])
def test_prefill_fp8_larger_blocks(dev, B, split):
    c = Fp8PrefillCase(dev, workloads.F16, 8, 2, B, [300, 129, 70], [100, 129, 3], seed=43 + B, split=split)
    c.check(c.gpu())


def test_prefill_fp8_single_token_chunks_match_fp8_decode(dev):
    """q_len = 1 everywhere: every row is the FP8 decode; the prefill kernel
    and pa_decode_fp8 must both be within tolerance of the same oracle."""
    import torch
    c = Fp8PrefillCase(dev, workloads.BF16, 16, 2, 16, [1, 17, 200, 513], [1, 1, 1, 1], seed=47)
    out = c.gpu()
    got, want = c.check(out)
    ws = binding.decode_fp8_workspace(c.q, c.pool)
    dec = torch.full_like(c.q, float("nan"))
    binding.pa_decode_fp8(dec, c.q.contiguous(), c.pool, c.bt_d, c.sl_d, c.scale, c.ks, c.vs, ws)
    torch.cuda.synchronize()
    assert max_abs_err(oracle.decode_elems(u16(dec), c.dtype), want) <= TOL[c.dtype]


def test_prefill_fp8_llama13b_shaped_batch_sampled(dev):
    """Llama-2-13B heads (40 x 128, fp16) over an FP8 cache: 4 x 512-token
    chunks after prefixes up to 1536, sampled rows against the oracle."""
    import torch
    ctx, ql = [2048, 1000, 700, 1536], [512, 512, 200, 512]
    c = Fp8PrefillCase(dev, workloads.F16, 40, 40, 16, ctx, ql, seed=49)
    out = c.gpu()
    rng = np.random.default_rng(3)
    if len(c.slots):
        oracle.reshape_and_cache_fp8(c.k_bits, c.v_bits, c.pool_bits, c.slots, c.nb, c.B, c.Hkv, c.D, c.dtype,
                                     c.ks, c.vs)
    assert np.array_equal(u8(c.pool), c.pool_bits)
    rows = rng.choice(int(c.cu[-1]), size=24, replace=False)
    got = oracle.decode_elems(u16(out), c.dtype)
    for r in rows:
        s = int(np.searchsorted(c.cu, r, side="right") - 1)
        i = int(r - c.cu[s])
        vis = int(c.seq_lens[s]) - int(c.cu[s + 1] - c.cu[s]) + i + 1
        heads = rng.choice(40, size=4, replace=False).astype(np.int32)
        want = oracle.decode_fp8_sampled(np.zeros(4, np.int32), heads, c.q_bits[r:r + 1], c.pool_bits,
                                         c.bt[s:s + 1], np.array([vis], np.int32), c.scale, 40, 40, 128, c.nb,
                                         c.B, c.dtype, c.ks, c.vs)
        assert max_abs_err(got[r, heads], want) <= TOL[c.dtype], f"row {r}"
    assert binding.pa_get_device_error() == 0


@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
@pytest.mark.parametrize("heads", [(4, 4), (8, 2), (16, 1), (12, 3)])
def test_prefill_fp8_head_size_64(dev, dtype, heads):
    """Head size 64 over an FP8 cache: 64-byte code rows staged without a
    swizzle and widened into one 64-dim chunk per row."""
    Hq, Hkv = heads
    c = Fp8PrefillCase(dev, dtype, Hq, Hkv, 16, CTX, QLEN, seed=950 + Hq + Hkv + dtype, D=64)
    c.check(c.gpu())


def test_prefill_fp8_head_size_64_nan_padding_and_large_blocks(dev):
    c = Fp8PrefillCase(dev, workloads.BF16, 8, 2, 32, [33, 250, 7, 600], [33, 100, 7, 300], seed=97,
                       poison=True, D=64)
    c.check(c.gpu())


@pytest.mark.parametrize("D", [128, 64])
def test_prefill_fp8_bf16_queries_beyond_the_fp16_range(dev, D):
    """bf16 query rows scaled by 2^24, 2^-24 and 2^100, and rows with one
    huge and many tiny elements: the FP8-cache kernel moves each row to
    fp16 under its own power-of-two scale, so none overflows and the outputs
    stay within the bf16 tolerance of the oracle."""
    import torch
    c = Fp8PrefillCase(dev, workloads.BF16, 8, 2, 16, [200, 77, 300], [200, 77, 150], seed=61, D=D)
    q = c.q.float()
    q[0::5] *= 2.0 ** 24
    q[1::5] *= 2.0 ** -24
    q[2::5] *= 2.0 ** 100
    q[3::5, :, 0] = 3.0e5
    q[3::5, :, 1:] *= 2.0 ** -30
    c.q = q.to(torch.bfloat16)
    c.q_bits = u16(c.q)
    assert np.isfinite(oracle.decode_elems(c.q_bits, c.dtype)).all()
    out = c.gpu()
    want = c.oracle()
    assert np.array_equal(u8(c.pool), c.pool_bits)
    # Most rows are one-hot (the output is one V row): bf16 outputs >= 4 are
    # held to the oracle rounded to bf16.
    assert max_abs_err_bf16_large(oracle.decode_elems(u16(out), c.dtype), want) <= TOL[c.dtype]
    assert binding.pa_get_device_error() == 0
