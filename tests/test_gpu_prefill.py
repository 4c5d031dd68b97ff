"""GPU parity of the tcgen05 chunked-prefill kernel through the C ABI.

Bar: every output row within max-abs 2e-3 (fp16) / 1e-2 (bf16) of the fp64
oracle (a prefill row is the decode definition over the causal prefix);
the chunk's K/V written by pa_reshape_and_cache bit-exact; bit-identical
under any permutation of physical block placement.
"""
import math

import numpy as np
import pytest

import oracle
from oracle.block_manager import BlockManagerModel
from paged_kv_cache_120_gb300 import binding, build, workloads

from harness import TOL, max_abs_err, max_abs_err_bf16_large, prefill_tile_samples, u16

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


class PrefillCase:
    """Sequences of total length ctx[s] whose last qlen[s] tokens are this
    step's chunk: the allocator lays out ctx - qlen tokens, then reserves the
    chunk's slots; the chunk's K/V go in by pa_reshape_and_cache."""

    def __init__(self, dev, dtype, Hq, Hkv, B, ctx, qlen, seed, spare=8, poison=False, D=128, split=False):
        import torch
        self.dtype, self.Hq, self.Hkv, self.B, self.D = dtype, Hq, Hkv, B, D
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
        assert self.seq_lens.tolist() == list(ctx)
        self.cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
        self.max_q = max(1, max(qlen))
        total = int(self.cu[-1])
        self.pool = workloads.normal_values((2, nb, B, Hkv, D), dtype, seed + 1, dev)
        if poison:
            nan = torch.tensor(float("nan"), dtype=workloads.torch_dtype(dtype))
            used = set(int(b) for b in self.bt.ravel() if b >= 0)
            for b in range(nb):
                if b not in used:
                    self.pool[:, b] = nan
            for s, L in enumerate(ctx):
                if L % B:
                    self.pool[:, int(self.bt[s, (L - 1) // B]), L % B:] = nan
        self.q = workloads.normal_values((max(total, 1), Hq, D), dtype, seed + 2, dev)[:total]
        self.k = workloads.normal_values((max(total, 1), Hkv, D), dtype, seed + 3, dev)[:total]
        self.v = workloads.normal_values((max(total, 1), Hkv, D), dtype, seed + 4, dev)[:total]
        self.pool_bits = u16(self.pool).copy()
        self.q_bits, self.k_bits, self.v_bits = u16(self.q), u16(self.k), u16(self.v)
        self.dev = dev

    def gpu(self):
        import torch
        t = lambda a: torch.from_numpy(a).to(self.dev)
        self.bt_d, self.sl_d, self.cu_d = t(self.bt), t(self.seq_lens), t(self.cu)
        if len(self.slots):
            binding.pa_reshape_and_cache(self.k.contiguous(), self.v.contiguous(), self.pool,
                                         t(self.slots))
        return self.prefill(self.pool, self.bt_d)

    def workspace(self):
        """The K/V-split workspace for this shape, filled with NaN bytes (its
        contents must not matter); the shape must be one that splits."""
        ws = binding.prefill_workspace(self.q, self.pool, len(self.seq_lens), self.max_q)
        assert ws is not None, "this shape does not split its K/V ranges"
        return ws.fill_(0xFF)

    def prefill(self, pool, bt_d, split=None):
        import torch
        split = self.split if split is None else split
        out = torch.full_like(self.q, float("nan"))
        binding.pa_prefill(out, self.q.contiguous(), pool, bt_d, self.cu_d, self.sl_d, self.scale,
                           self.max_q, self.workspace() if split else None)
        torch.cuda.synchronize()
        return out

    def oracle(self):
        if len(self.slots):
            assert oracle.reshape_and_cache(self.k_bits, self.v_bits, self.pool_bits, self.slots,
                                            self.nb, self.B, self.Hkv, self.D) == len(self.slots)
        return oracle.prefill(self.q_bits, self.pool_bits, self.bt, self.cu, self.seq_lens,
                              self.scale, self.Hq, self.Hkv, self.D, self.nb, self.B, self.dtype)

    def check(self, out):
        want = self.oracle()
        assert np.array_equal(u16(self.pool), self.pool_bits), "reshape_and_cache is not bit-exact"
        got = oracle.decode_elems(u16(out), self.dtype)
        err = max_abs_err(got, want)
        assert err <= TOL[self.dtype], f"max abs err {err}"
        assert binding.pa_get_device_error() == 0
        return got, want


# (context length, chunk length): whole prompts, chunks after a prefix,
# single tokens, empty chunks, lengths across 16-token boxes and 128-token tiles
CTX = [200, 128, 17, 300, 1, 129, 40, 517, 64]
QLEN = [200, 60, 1, 150, 1, 0, 40, 129, 64]
HEADS = [(4, 4), (8, 2), (8, 1), (16, 1), (32, 1), (12, 3), (40, 8), (6, 2)]


@pytest.mark.parametrize("split", [False, True], ids=["whole", "split"])
@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
@pytest.mark.parametrize("heads", HEADS)
def test_prefill_parity_small(dev, dtype, heads, split):
    """Every head layout, with each unit's K/V range whole and (a
    workspace given; these shapes have few units) split across the SMs."""
    Hq, Hkv = heads
    c = PrefillCase(dev, dtype, Hq, Hkv, 16, CTX, QLEN, seed=500 + Hq + Hkv + dtype, split=split)
    c.check(c.gpu())


@pytest.mark.parametrize("split", [False, True], ids=["whole", "split"])
@pytest.mark.parametrize("B", [32, 64, 48])
def test_prefill_block_sizes(dev, B, split):
    c = PrefillCase(dev, workloads.BF16, 8, 2, B, [33, 300, 129, 64], [33, 100, 129, 1], seed=9 + B, split=split)
    c.check(c.gpu())


@pytest.mark.parametrize("split", [False, True], ids=["whole", "split"])
def test_prefill_padding_slots_holding_nan_are_ignored(dev, split):
    c = PrefillCase(dev, workloads.F16, 8, 8, 16, [3, 18, 140, 77], [3, 5, 140, 20], seed=5, poison=True,
                    split=split)
    c.check(c.gpu())


@pytest.mark.parametrize("split", [False, True], ids=["whole", "split"])
@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
def test_prefill_long_context_chunk(dev, dtype, split):
    c = PrefillCase(dev, dtype, 8, 1, 16, [5000, 2100], [300, 2100], seed=21, split=split)
    c.check(c.gpu())


def test_single_token_chunks_agree_with_decode(dev):
    """q_len = 1 everywhere is decode: both kernels against the oracle, and
    against each other."""
    import torch
    c = PrefillCase(dev, workloads.F16, 32, 8, 16, [5, 100, 1000, 16, 2049], [1] * 5, seed=31)
    out = c.gpu()
    c.check(out)
    dec = torch.empty_like(c.q)
    ws = binding.decode_workspace(c.q, c.pool)
    binding.pa_decode(dec, c.q, c.pool, c.bt_d, c.sl_d, c.scale, ws)
    torch.cuda.synchronize()
    d = oracle.decode_elems(u16(dec), workloads.F16)
    p = oracle.decode_elems(u16(out), workloads.F16)
    assert np.max(np.abs(d - p)) <= 2 * TOL[workloads.F16]


def test_prefill_bit_identical_under_block_permutation(dev):
    import torch
    c = PrefillCase(dev, workloads.BF16, 32, 8, 16, [700, 5, 1234, 16], [300, 5, 129, 16], seed=17,
                    spare=40)
    out1 = c.gpu()
    sigma = np.random.default_rng(99).permutation(c.nb).astype(np.int64)
    pool2 = torch.empty_like(c.pool)
    pool2[:, torch.from_numpy(sigma).to(dev)] = c.pool
    bt2 = np.where(c.bt >= 0, sigma[np.maximum(c.bt, 0)], -1).astype(np.int32)
    out2 = c.prefill(pool2, torch.from_numpy(bt2).to(dev))
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_prefill_rows_outside_chunks_are_untouched_and_bad_inputs_flagged(dev):
    import torch
    c = PrefillCase(dev, workloads.F16, 8, 2, 16, [40, 20], [10, 20], seed=8)
    c.gpu()
    assert binding.pa_get_device_error() == 0
    # a length shorter than the chunk: that sequence is skipped and flagged
    sl = torch.from_numpy(np.array([40, 5], np.int32)).to(dev)
    out = torch.full_like(c.q, float("nan"))
    binding.pa_prefill(out, c.q, c.pool, c.bt_d, c.cu_d, sl, c.scale, c.max_q)
    torch.cuda.synchronize()
    assert binding.pa_get_device_error() & binding.PA_DEVERR_SEQ_LEN
    assert torch.isnan(out[10:].float()).all() and not torch.isnan(out[:10].float()).any()
    # a block id outside the pool reads as zeros and is flagged
    bt = c.bt.copy()
    bt[0, 1] = c.nb + 3
    binding.pa_prefill(out, c.q, c.pool, torch.from_numpy(bt).to(dev), c.cu_d, c.sl_d, c.scale, c.max_q)
    assert binding.pa_get_device_error() & binding.PA_DEVERR_BLOCK_ID
    # a chunk longer than the max_seqlen_q hint: that sequence is skipped and
    # flagged, not written in part
    out = torch.full_like(c.q, float("nan"))
    binding.pa_prefill(out, c.q, c.pool, c.bt_d, c.cu_d, c.sl_d, c.scale, 15)
    torch.cuda.synchronize()
    assert binding.pa_get_device_error() == binding.PA_DEVERR_SEQ_LEN
    assert torch.isnan(out[10:].float()).all() and not torch.isnan(out[:10].float()).any()


def test_prefill_sampled_rows_at_llama13b_shape(dev):
    """A Llama-2-13B layer chunked-prefill batch (40 heads, d=128, fp16):
    8 sequences with cached prefixes of up to 2048 tokens and 512-token
    chunks; sampled rows against the oracle (each row is the decode over its
    causal prefix)."""
    rng = np.random.default_rng(77)
    pref = rng.integers(0, 2049, size=8)
    q = np.full(8, 512)
    c = PrefillCase(dev, workloads.F16, 40, 40, 16, list(pref + q), list(q), seed=77)
    out = c.gpu()
    assert oracle.reshape_and_cache(c.k_bits, c.v_bits, c.pool_bits, c.slots, c.nb, c.B, c.Hkv,
                                    c.D) == len(c.slots)
    assert np.array_equal(u16(c.pool), c.pool_bits)
    n = 64
    s = rng.integers(0, 8, size=n)
    i = rng.integers(0, 512, size=n)
    i[:8] = 511
    s[:8] = np.arange(8)
    hq = rng.integers(0, 40, size=n)
    rows = c.cu[s] + i
    want = oracle.decode_sampled(np.arange(n, dtype=np.int32), hq.astype(np.int32), c.q_bits[rows],
                                 c.pool_bits, c.bt[s], (c.seq_lens[s] - 512 + i + 1).astype(np.int32),
                                 c.scale, 40, 40, 128, c.nb, 16, workloads.F16)
    got = oracle.decode_elems(u16(out), workloads.F16)[rows, hq]
    assert max_abs_err(got, want) <= TOL[workloads.F16]
    assert binding.pa_get_device_error() == 0


def test_prefill_replayed_from_a_cuda_graph_is_bit_identical(dev):
    """The work-unit counter a launch uses is fixed when it is captured; the
    last CTA of every run resets it, so replays (interleaved with eager
    launches that use other counters) give the eager outputs bit for bit."""
    import torch
    c = PrefillCase(dev, workloads.BF16, 16, 2, 16, [300, 129, 517, 64], [150, 129, 200, 64], seed=77)
    eager = c.gpu()
    c.check(eager)
    ref = eager.clone()
    out = torch.full_like(c.q, float("nan"))
    q = c.q.contiguous()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.pa_prefill(out, q, c.pool, c.bt_d, c.cu_d, c.sl_d, c.scale, c.max_q)   # warm-up on s
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        binding.pa_prefill(out, q, c.pool, c.bt_d, c.cu_d, c.sl_d, c.scale, c.max_q)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        again = c.prefill(c.pool, c.bt_d)          # an eager launch between replays
        assert torch.equal(again.view(torch.int16), ref.view(torch.int16))
    assert binding.pa_get_device_error() == 0


@pytest.mark.parametrize("split", [False, True], ids=["whole", "split"])
@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
@pytest.mark.parametrize("heads", [(4, 4), (8, 2), (16, 1), (32, 1)])
def test_prefill_head_size_64(dev, dtype, heads, split):
    """Head size 64: one 64-dim chunk per row, four score MMAs per tile,
    P V with N = 64; same cases as the head-size-128 grid."""
    Hq, Hkv = heads
    c = PrefillCase(dev, dtype, Hq, Hkv, 16, CTX, QLEN, seed=900 + Hq + Hkv + dtype, D=64, split=split)
    c.check(c.gpu())


def test_prefill_head_size_64_nan_padding_and_large_blocks(dev):
    c = PrefillCase(dev, workloads.BF16, 8, 2, 32, [33, 250, 7, 600], [33, 100, 7, 300], seed=93, poison=True, D=64)
    c.check(c.gpu())


@pytest.mark.parametrize("kv", ["16bit", "fp8"])
@pytest.mark.parametrize("name", ["prefill_llama13b", "prefill_gqa8b"])
def test_prefill_workload_full_size(dev, name, kv):
    """The prefill step bench.py times (same plan, seed and launch: 8 x
    1024-token chunks after seeded prefixes), run once: the allocator's plan
    against the block-manager model, the chunk's K/V writes bit-exact against
    the oracle over the whole pool, and a row of every query tile of every
    kv head (both tiles of every work unit) plus the last row of every chunk
    against the oracle's decode over the row's causal prefix."""
    import torch
    from paged_kv_cache_120_gb300 import step
    w = workloads.PREFILL_WORKLOADS[name]
    seed = 0
    plan = step.plan_prefill(name, seed)
    model = BlockManagerModel(plan.num_blocks, w.block_size, workloads.free_order(plan.num_blocks, seed))
    pref = workloads.prefill_prefixes(name, seed)
    ids = [model.add_seq(int(p)) for p in pref]
    slots = [model.append_token(sid)[0] for sid in ids for _ in range(w.chunk)]
    assert np.array_equal(np.asarray(slots, np.int32), plan.slot_mapping)
    for k, sid in enumerate(ids):
        t = model.table(sid)
        assert list(plan.block_tables[k, :len(t)]) == list(t)
    st = step.PrefillStep(name, plan, seed, dev, kv)
    fp8 = kv == "fp8"
    pool_bits = st.pool.cpu().numpy().copy() if fp8 else u16(st.pool).copy()
    k_bits, v_bits, q_bits = u16(st.key_new), u16(st.value_new), u16(st.query)
    st.run()
    torch.cuda.synchronize()
    assert binding.pa_get_device_error() == 0
    geo = (plan.num_blocks, w.block_size, w.num_kv_heads, w.head_size)
    if fp8:
        n = oracle.reshape_and_cache_fp8(k_bits, v_bits, pool_bits, plan.slot_mapping, *geo, w.dtype,
                                         st.k_scale, st.v_scale)
        assert np.array_equal(st.pool.cpu().numpy(), pool_bits)
    else:
        n = oracle.reshape_and_cache(k_bits, v_bits, pool_bits, plan.slot_mapping, *geo)
        assert np.array_equal(u16(st.pool), pool_bits)
    assert n == len(plan.slot_mapping)
    s, i, hq = prefill_tile_samples(plan, w, np.random.default_rng(11))
    m = len(s)
    rows = plan.cu_seqlens_q[s] + i
    vis = (plan.seq_lens[s] - w.chunk + i + 1).astype(np.int32)
    args = (np.arange(m, dtype=np.int32), hq, q_bits[rows], pool_bits, plan.block_tables[s], vis, w.scale,
            w.num_q_heads, w.num_kv_heads, w.head_size, plan.num_blocks, w.block_size, w.dtype)
    want = (oracle.decode_fp8_sampled(*args, st.k_scale, st.v_scale) if fp8 else oracle.decode_sampled(*args))
    got = oracle.decode_elems(u16(st.out)[rows, hq], w.dtype)
    assert max_abs_err(got, want) <= TOL[w.dtype]


@pytest.mark.parametrize("D", [128, 64])
def test_prefill_bf16_queries_with_huge_scores(dev, D):
    """bf16 query rows scaled by 2^100 and 2^-100 over a 16-bit cache:
    scores far beyond 2^32 in base 2 give one-hot rows, not overflow (the
    exponent argument rounds the product before subtracting the reference,
    so the largest score's P stays 2^0 .. 2^8)."""
    import torch
    c = PrefillCase(dev, workloads.BF16, 8, 2, 16, [200, 77, 300], [200, 77, 150], seed=63, D=D)
    q = c.q.float()
    q[0::3] *= 2.0 ** 100
    q[1::3] *= 2.0 ** -100
    c.q = q.to(torch.bfloat16)
    c.q_bits = u16(c.q)
    out = c.gpu()
    assert torch.isfinite(out.float()).all()
    want = c.oracle()
    assert max_abs_err_bf16_large(oracle.decode_elems(u16(out), c.dtype), want) <= TOL[c.dtype]
    assert binding.pa_get_device_error() == 0


@pytest.mark.parametrize("scale", [0.0, -0.3, 2.0])
@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
def test_prefill_zero_negative_and_large_scales(dev, scale, dtype):
    """Causally masked scores must weigh exactly nothing whatever the scale:
    0 (every visible token weighs the same), negative (the row minimum is
    the reference), and large; padding slots hold NaN."""
    c = PrefillCase(dev, dtype, 8, 2, 16, [300, 129, 77, 1], [200, 129, 40, 1], seed=61, poison=True)
    c.scale = scale
    out = c.gpu()
    c.check(out)
