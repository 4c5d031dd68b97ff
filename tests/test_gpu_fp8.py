"""GPU parity of the FP8 (E4M3) cache path through the C ABI against the oracle.

Bars: pa_reshape_and_cache_fp8 and pa_copy_blocks on byte pools bit-exact;
pa_decode_fp8 within max-abs 2e-3 (fp16 activations) / 1e-2 (bf16) of the
oracle's fp64 attention over the dequantised cache (every code widened
exactly, so the kernel's error budget is that of the 16-bit path);
bit-identical under any permutation of physical block placement.
"""
import math

import numpy as np
import pytest

import oracle
from oracle.block_manager import BlockManagerModel
from paged_kv_cache_120_gb300 import binding, build, step, workloads

from harness import TOL, max_abs_err, max_abs_err_bf16_large, oracle_plan, u16

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
    return t.detach().contiguous().cpu().numpy().view(np.uint8)


def _finite_codes(gen, shape, dev, low=0, high=0x7F):
    """Uniform codes among sign x [low, high) magnitudes (0x7F, the NaN, excluded)."""
    import torch
    mag = torch.randint(low, high, shape, generator=gen, dtype=torch.int32)
    sign = torch.randint(0, 2, shape, generator=gen, dtype=torch.int32) * 0x80
    return (mag | sign).to(torch.uint8).to(dev)


class Fp8Case:
    """A small case on an FP8 pool: product allocator for the GPU, oracle
    model for the oracle; codes drawn by ``codes`` ("normal": N(0, 1) under
    the scales; "uniform": every finite code; "subnormal": codes 0..7)."""

    def __init__(self, dev, dtype, D, Hq, Hkv, B, lens, seed, spare=8, poison=False,
                 codes="normal", k_scale=KS, v_scale=VS, kv_mult=1.0):
        import torch
        self.dtype, self.D, self.Hq, self.Hkv, self.B = dtype, D, Hq, Hkv, B
        self.k_scale, self.v_scale = k_scale, v_scale
        self.lens = list(lens)
        self.scale = 1.0 / math.sqrt(D)
        rng = np.random.default_rng(seed)
        nb = sum(-(-L // B) for L in lens) + spare
        self.nb = nb
        order = rng.permutation(nb)
        alloc = binding.BlockAllocator(nb, B, order)
        model = BlockManagerModel(nb, B, order)
        ids_a, ids_m, slots = [], [], []
        for L in lens:
            ids_a.append(alloc.add_seq(max(L - 1, 0)))
            ids_m.append(model.add_seq(max(L - 1, 0)))
        for a, m, L in zip(ids_a, ids_m, lens):
            if L > 0:
                sa, ca = alloc.append_token(a)
                assert (sa, ca) == model.append_token(m)
                slots.append(sa)
            else:
                slots.append(-1)
        maxblk = max(1, max(len(model.table(m)) for m in ids_m))
        self.bt = alloc.block_tables(ids_a, maxblk)
        bt_m = np.full_like(self.bt, -1)
        for i, m in enumerate(ids_m):
            t = model.table(m)
            bt_m[i, :len(t)] = t
        assert np.array_equal(self.bt, bt_m)
        self.slots = np.array(slots, dtype=np.int32)
        self.seq_lens = alloc.seq_lens(ids_a)
        S = len(lens)
        shape = (nb, B, Hkv, D)
        gen = torch.Generator().manual_seed(seed + 1)
        self.pool = torch.empty((2,) + shape, dtype=torch.uint8, device=dev)
        if codes == "normal":
            self.pool[0] = workloads.fp8_codes(shape, k_scale, seed + 1, dev)
            self.pool[1] = workloads.fp8_codes(shape, v_scale, seed + 5, dev)
        elif codes == "uniform":
            self.pool.copy_(_finite_codes(gen, (2,) + shape, dev))
        elif codes == "subnormal":
            self.pool.copy_(_finite_codes(gen, (2,) + shape, dev, 0, 8))
        else:
            raise ValueError(codes)
        if poison:
            used = set(int(b) for b in self.bt.ravel() if b >= 0)
            for b in range(nb):
                if b not in used:
                    self.pool[:, b] = 0x7F
            for s, L in enumerate(lens):
                if L % B:
                    self.pool[:, int(self.bt[s, (L - 1) // B]), L % B:] = 0xFF
        self.q = workloads.normal_values((S, Hq, D), dtype, seed + 2, dev)
        self.k = workloads.normal_values((S, Hkv, D), dtype, seed + 3, dev)
        self.v = workloads.normal_values((S, Hkv, D), dtype, seed + 4, dev)
        if kv_mult != 1.0:
            self.k.mul_(kv_mult)
            self.v.mul_(kv_mult)
        # oracle inputs: snapshot before any libpa kernel runs
        self.pool_bits = u8(self.pool).copy()
        self.q_bits, self.k_bits, self.v_bits = u16(self.q), u16(self.k), u16(self.v)
        self.dev = dev

    def gpu(self, flags=0):
        import torch
        t = lambda a: torch.from_numpy(a).to(self.dev)
        self.bt_d, self.sl_d, self.slots_d = t(self.bt), t(self.seq_lens), t(self.slots)
        binding.pa_reshape_and_cache_fp8(self.k, self.v, self.pool, self.slots_d, self.k_scale,
                                         self.v_scale)
        return self.decode(self.pool, self.bt_d, flags)

    def decode(self, pool, bt_d, flags=0):
        import torch
        out = torch.empty_like(self.q)
        ws = binding.decode_fp8_workspace(self.q, pool)
        binding.pa_decode_fp8(out, self.q, pool, bt_d, self.sl_d, self.scale, self.k_scale,
                              self.v_scale, ws, flags)
        torch.cuda.synchronize()
        return out

    def oracle(self):
        n = oracle.reshape_and_cache_fp8(self.k_bits, self.v_bits, self.pool_bits, self.slots,
                                         self.nb, self.B, self.Hkv, self.D, self.dtype,
                                         self.k_scale, self.v_scale)
        assert n == int((self.slots >= 0).sum())
        return oracle.decode_fp8(self.q_bits, self.pool_bits, self.bt, self.seq_lens, self.scale,
                                 self.Hq, self.Hkv, self.D, self.nb, self.B, self.dtype,
                                 self.k_scale, self.v_scale)

    def check(self, out):
        want = self.oracle()
        assert np.array_equal(u8(self.pool), self.pool_bits), "reshape_and_cache_fp8 is not bit-exact"
        got = oracle.decode_elems(u16(out), self.dtype)
        err = max_abs_err(got, want)
        assert err <= TOL[self.dtype], f"max abs err {err}"
        assert binding.pa_get_device_error() == 0
        return got, want


LENS = [1, 2, 15, 16, 17, 31, 33, 100, 0, 255, 300, 1000]
HEADS = [(4, 4), (8, 2), (8, 1), (12, 3), (16, 1), (32, 1), (64, 2)]


@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("heads", HEADS)
def test_fp8_decode_and_reshape_parity_small(dev, dtype, D, heads):
    Hq, Hkv = heads
    c = Fp8Case(dev, dtype, D, Hq, Hkv, 16, LENS, seed=300 + Hq + D + dtype)
    got, _ = c.check(c.gpu())
    assert np.all(got[LENS.index(0)] == 0.0)


@pytest.mark.parametrize("B", [32, 64])
@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
def test_fp8_larger_block_sizes(dev, B, dtype):
    c = Fp8Case(dev, dtype, 128, 8, 2, B, [1, 31, 32, 33, 64, 65, 129, 700], seed=17 + B)
    c.check(c.gpu())


@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
def test_fp8_every_finite_code(dev, dtype):
    """Codes drawn uniformly over all finite E4M3 values (+-448 and the
    subnormals included) are widened exactly. The scales (1/128) keep the
    values within +-3.5, the magnitude of N(0, 1) draws that the max-abs bars
    are stated for (the rounding of P and of the output scales with |V|)."""
    c = Fp8Case(dev, dtype, 128, 8, 2, 16, [40, 333, 1], seed=41, codes="uniform",
                k_scale=1 / 128, v_scale=1 / 128)
    c.check(c.gpu())


@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
@pytest.mark.parametrize("D", [64, 128])
def test_fp8_subnormal_codes_are_not_flushed(dev, dtype, D):
    """A cache holding only subnormal codes (values 0 .. 7 * 2^-9) under
    large scales (K up to 3.5, V up to 1.75): flushing them to zero would
    change the output by O(1)."""
    c = Fp8Case(dev, dtype, D, 8, 2, 16, [5, 70, 16], seed=43, codes="subnormal",
                k_scale=256.0, v_scale=128.0)
    got, want = c.check(c.gpu())
    assert np.max(np.abs(want)) > 0.25


def test_fp8_bf16_queries_with_wide_dynamic_range(dev):
    """bf16 queries meet fp16-widened K: each query column is moved to fp16
    with its own power-of-two scale. Columns scaled from 2^-30 to 2^12, with
    a few elements 2^-40 below their column's largest, still match."""
    import torch
    c = Fp8Case(dev, workloads.BF16, 128, 16, 2, 16, [5, 70, 16, 1, 300, 33], seed=47)
    gen = torch.Generator().manual_seed(5)
    exps = torch.randint(-30, 13, (1, 16, 1), generator=gen).float()
    q = (c.q.float().cpu() * torch.exp2(exps))
    q[:, :, :3] *= 2.0 ** -40
    c.q = q.to(torch.bfloat16).to(dev)
    c.q_bits = u16(c.q)
    c.check(c.gpu())


def test_fp8_padding_slots_holding_nan_are_ignored(dev):
    c = Fp8Case(dev, workloads.F16, 128, 8, 8, 16, [3, 18, 40, 77, 16], seed=5, poison=True)
    c.check(c.gpu())


@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
def test_fp8_segments_split_across_many_warps(dev, dtype):
    c = Fp8Case(dev, dtype, 128, 8, 1, 16, [30000, 5, 17, 1, 4000], seed=11)
    c.check(c.gpu())


@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
def test_fp8_reshape_saturates_large_values(dev, dtype):
    """New K/V far beyond 448 * scale store +-448 (0x7E / 0xFE), bit for bit
    as the oracle's saturating rounding."""
    c = Fp8Case(dev, dtype, 64, 4, 4, 16, [3, 17, 40], seed=13, kv_mult=20.0)
    c.gpu()
    c.oracle()
    assert np.array_equal(u8(c.pool), c.pool_bits)
    rows = c.pool_bits[:, c.slots // 16, c.slots % 16]
    assert np.isin(rows, [0x7E, 0xFE]).mean() > 0.3


def test_fp8_decode_bit_identical_under_block_permutation(dev):
    import torch
    c = Fp8Case(dev, workloads.BF16, 128, 32, 8, 16, [700, 5, 1234, 16, 999, 2047, 64], seed=19,
                spare=40)
    out1 = c.gpu()
    sigma = np.random.default_rng(98).permutation(c.nb).astype(np.int64)
    pool2 = torch.empty_like(c.pool)
    pool2[:, torch.from_numpy(sigma).to(dev)] = c.pool
    bt2 = np.where(c.bt >= 0, sigma[np.maximum(c.bt, 0)], -1).astype(np.int32)
    out2 = c.decode(pool2, torch.from_numpy(bt2).to(dev))
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    out3 = c.decode(c.pool, c.bt_d, flags=binding.PA_DECODE_SHARED_BLOCKS)
    assert torch.equal(out1.view(torch.int16), out3.view(torch.int16))


def test_fp8_stale_nan_workspace_does_not_leak(dev):
    import torch
    c = Fp8Case(dev, workloads.F16, 128, 8, 2, 16, LENS, seed=77)
    t = lambda a: torch.from_numpy(a).to(dev)
    c.sl_d = t(c.seq_lens)
    binding.pa_reshape_and_cache_fp8(c.k, c.v, c.pool, t(c.slots), c.k_scale, c.v_scale)
    out = torch.empty_like(c.q)
    ws = binding.decode_fp8_workspace(c.q, c.pool)
    ws.fill_(0xFF)
    binding.pa_decode_fp8(out, c.q, c.pool, t(c.bt), c.sl_d, c.scale, c.k_scale, c.v_scale, ws)
    torch.cuda.synchronize()
    c.check(out)


def test_fp8_copy_blocks_bit_exact(dev):
    """A byte pool is copied in 16-byte units; the oracle copies the same
    bytes viewed as 16-bit elements (head_size / 2 of them per head)."""
    import torch
    gen = torch.Generator().manual_seed(3)
    nb, B, H, D = 32, 16, 8, 128
    pools = [_finite_codes(gen, (2, nb, B, H, D), dev) for _ in range(2)]
    before = [u8(p).copy() for p in pools]
    pairs = np.array([[1, 4], [6, 2], [0, 7], [9, 30]], dtype=np.int32)
    binding.pa_copy_blocks(pools, torch.from_numpy(pairs).to(dev))
    as16 = [b.view(np.uint16) for b in before]
    assert oracle.copy_blocks(as16, pairs, nb, B, H, D // 2) == 0
    for p, b in zip(pools, before):
        assert np.array_equal(u8(p), b)
    assert binding.pa_get_device_error() == 0


def test_fp8_bad_block_ids_are_flagged_not_faulted(dev):
    import torch
    c = Fp8Case(dev, workloads.F16, 128, 8, 8, 16, [40, 20], seed=8)
    c.gpu()
    assert binding.pa_get_device_error() == 0
    bt = c.bt.copy()
    bt[0, 1] = c.nb + 5
    c.decode(c.pool, torch.from_numpy(bt).to(dev))
    assert binding.pa_get_device_error() & binding.PA_DEVERR_BLOCK_ID


def test_fp8_wrong_pool_type_is_rejected(dev):
    import torch
    c = Fp8Case(dev, workloads.F16, 64, 4, 4, 16, [20], seed=9)
    out = torch.empty_like(c.q)
    with pytest.raises(TypeError):
        binding.pa_decode_fp8(out, c.q, c.q.view(1, 1, 1, 4, 64).expand(2, 1, 1, 4, 64).contiguous(),
                              torch.zeros(1, 1, dtype=torch.int32, device=dev),
                              torch.ones(1, dtype=torch.int32, device=dev), 1.0, 1.0, 1.0,
                              torch.empty(256, dtype=torch.uint8, device=dev))


# ------------------------------------------------------------ the workloads

@pytest.mark.parametrize("name", ["llama13b", "gqa8b", "longctx", "prefix_cow"])
def test_fp8_workload_full_size(dev, name):
    """Every workload on an FP8 pool at full size: every (seq, head) output
    row against the oracle; the step's written slots and COW copies bit-exact."""
    import torch
    w = workloads.WORKLOADS[name]
    seed = 4
    variant = "fork" if name == "prefix_cow" else "literal"
    plan = step.plan_step(name, seed, variant)
    op = oracle_plan(name, seed, variant)
    assert np.array_equal(plan.block_tables, op["block_tables"])
    assert np.array_equal(plan.slot_mapping, op["slot_mapping"])
    assert np.array_equal(plan.cow_pairs, op["cow_pairs"])
    pool, q, k, v = step.make_device_inputs(name, plan, seed, dev, kv_cache="fp8")
    pool_bits = u8(pool).copy()
    q_bits, k_bits, v_bits = u16(q), u16(k), u16(v)
    st = step.DecodeStep(name, plan, pool, q, k, v, dev)
    assert st.fp8
    st.run()
    torch.cuda.synchronize()
    if len(op["cow_pairs"]):
        assert oracle.copy_blocks([pool_bits.view(np.uint16)], op["cow_pairs"], w.num_blocks,
                                  w.block_size, w.num_kv_heads, w.head_size // 2) == 0
    assert oracle.reshape_and_cache_fp8(k_bits, v_bits, pool_bits, op["slot_mapping"],
                                        w.num_blocks, w.block_size, w.num_kv_heads, w.head_size,
                                        w.dtype, KS, VS) == len(op["slot_mapping"])
    # every (sequence, head) row of the step, element by element
    want = oracle.decode_fp8(q_bits, pool_bits, op["block_tables"], op["seq_lens"], w.scale,
                             w.num_q_heads, w.num_kv_heads, w.head_size, w.num_blocks, w.block_size,
                             w.dtype, KS, VS)
    got = oracle.decode_elems(u16(st.out), w.dtype)
    err = max_abs_err(got, want)
    assert err <= TOL[w.dtype], f"{name}: max abs err {err}"
    touched = set(int(s) // w.block_size for s in plan.slot_mapping if s >= 0)
    touched |= set(int(d) for _, d in plan.cow_pairs)
    idx = torch.tensor(sorted(touched), device=dev)
    assert np.array_equal(u8(pool[:, idx]), pool_bits[:, sorted(touched)])
    assert binding.pa_get_device_error() == 0


@pytest.mark.parametrize("heads", [(8, 2), (16, 1), (4, 4)])
@pytest.mark.parametrize("D", [128, 64])
def test_fp8_decode_bf16_queries_with_huge_scores(dev, heads, D):
    """As for the 16-bit cache: bf16 query rows scaled by 2^100 and 2^-100
    over an FP8 cache (each query column moved to fp16 under its own power
    of two) give one-hot or uniform rows, within the bf16 tolerance."""
    import torch
    Hq, Hkv = heads
    c = Fp8Case(dev, workloads.BF16, D, Hq, Hkv, 16, LENS, seed=73 + Hq + D)
    q = c.q.float()
    q[0::3] *= 2.0 ** 100
    q[1::3] *= 2.0 ** -100
    c.q = q.to(torch.bfloat16).contiguous()
    c.q_bits = u16(c.q)
    out = c.gpu()
    want = c.oracle()
    got = oracle.decode_elems(u16(out), workloads.BF16)
    assert max_abs_err_bf16_large(got, want) <= TOL[workloads.BF16]
