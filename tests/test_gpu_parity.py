"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Bars: reshape_and_cache and copy_blocks bit-exact; decode within max-abs
2e-3 (fp16) / 1e-2 (bf16) of the oracle; decode bit-identical under any
permutation of physical block placement.
"""
import math

import numpy as np
import pytest

import oracle
from oracle.block_manager import BlockManagerModel
from paged_kv_cache_120_gb300 import binding, build, step, workloads

from harness import TOL, max_abs_err, max_abs_err_bf16_large, oracle_plan, oracle_step, u16

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


def _tdt(dtype):
    return workloads.torch_dtype(dtype)


class Case:
    """A custom small case: product allocator for the GPU, oracle model for the oracle."""

    def __init__(self, dev, dtype, D, Hq, Hkv, B, lens, seed, spare=8, poison=False):
        import torch
        self.dtype, self.D, self.Hq, self.Hkv, self.B = dtype, D, Hq, Hkv, B
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
                sm, cm = model.append_token(m)
                assert (sa, ca) == (sm, cm)
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
        assert self.seq_lens.tolist() == [max(L, 0) for L in lens]
        S = len(lens)
        self.pool = workloads.normal_values((2, nb, B, Hkv, D), dtype, seed + 1, dev)
        if poison:
            nan = torch.tensor(float("nan"), dtype=_tdt(dtype))
            used = set(int(b) for b in self.bt.ravel() if b >= 0)
            for b in range(nb):
                if b not in used:
                    self.pool[:, b] = nan
            for s, L in enumerate(lens):
                if L % B:
                    self.pool[:, int(self.bt[s, (L - 1) // B]), L % B:] = nan
        self.q = workloads.normal_values((S, Hq, D), dtype, seed + 2, dev)
        self.k = workloads.normal_values((S, Hkv, D), dtype, seed + 3, dev)
        self.v = workloads.normal_values((S, Hkv, D), dtype, seed + 4, dev)
        # oracle inputs: snapshot before any libpa kernel runs
        self.pool_bits = u16(self.pool).copy()
        self.q_bits, self.k_bits, self.v_bits = u16(self.q), u16(self.k), u16(self.v)
        self.dev = dev

    def gpu(self):
        import torch
        t = lambda a: torch.from_numpy(a).to(self.dev)
        self.bt_d, self.sl_d, self.slots_d = t(self.bt), t(self.seq_lens), t(self.slots)
        binding.pa_reshape_and_cache(self.k, self.v, self.pool, self.slots_d)
        out = torch.empty_like(self.q)
        ws = binding.decode_workspace(self.q, self.pool)
        binding.pa_decode(out, self.q, self.pool, self.bt_d, self.sl_d, self.scale, ws)
        torch.cuda.synchronize()
        return out

    def oracle(self):
        n = oracle.reshape_and_cache(self.k_bits, self.v_bits, self.pool_bits, self.slots, self.nb,
                                     self.B, self.Hkv, self.D)
        assert n == int((self.slots >= 0).sum())
        return oracle.decode(self.q_bits, self.pool_bits, self.bt, self.seq_lens, self.scale,
                             self.Hq, self.Hkv, self.D, self.nb, self.B, self.dtype)


LENS = [1, 2, 15, 16, 17, 31, 33, 100, 0, 255, 300, 1000]
HEADS = [(4, 4), (8, 2), (8, 1), (12, 3), (16, 1), (12, 1), (32, 1), (64, 2)]


@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("heads", HEADS)
def test_decode_and_reshape_parity_small(dev, dtype, D, heads):
    Hq, Hkv = heads
    c = Case(dev, dtype, D, Hq, Hkv, 16, LENS, seed=100 + Hq + D + dtype)
    out = c.gpu()
    want = c.oracle()
    assert np.array_equal(u16(c.pool), c.pool_bits), "reshape_and_cache is not bit-exact"
    got = oracle.decode_elems(u16(out), dtype)
    err = max_abs_err(got, want)
    assert err <= TOL[dtype], f"max abs err {err}"
    assert np.all(got[LENS.index(0)] == 0.0)
    assert binding.pa_get_device_error() == 0


@pytest.mark.parametrize("B", [32, 64])
@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
def test_larger_block_sizes(dev, B, dtype):
    c = Case(dev, dtype, 128, 8, 2, B, [1, 31, 32, 33, 64, 65, 129, 700], seed=7 + B)
    out = c.gpu()
    want = c.oracle()
    assert np.array_equal(u16(c.pool), c.pool_bits)
    assert max_abs_err(oracle.decode_elems(u16(out), dtype), want) <= TOL[dtype]


def test_padding_slots_holding_nan_are_ignored(dev):
    c = Case(dev, workloads.F16, 128, 8, 8, 16, [3, 18, 40, 77, 16], seed=5, poison=True)
    out = c.gpu()
    want = c.oracle()
    got = oracle.decode_elems(u16(out), workloads.F16)
    assert max_abs_err(got, want) <= TOL[workloads.F16]


@pytest.mark.parametrize("dtype", [workloads.F16, workloads.BF16])
def test_segments_split_across_many_warps(dev, dtype):
    """One long sequence among short ones: the long segment is cut into many
    pieces that the reduce kernel merges."""
    c = Case(dev, dtype, 128, 8, 1, 16, [30000, 5, 17, 1, 4000], seed=11)
    out = c.gpu()
    want = c.oracle()
    assert max_abs_err(oracle.decode_elems(u16(out), dtype), want) <= TOL[dtype]


@pytest.mark.parametrize("heads", [(8, 2), (32, 8), (12, 1)])
def test_stale_nan_workspace_does_not_leak(dev, heads):
    """The workspace needs no initialisation: fill it with NaN bytes first
    (what a reused buffer may hold) and the output must still match."""
    import torch
    Hq, Hkv = heads
    c = Case(dev, workloads.F16, 64, Hq, Hkv, 16, LENS, seed=77 + Hq)
    t = lambda a: torch.from_numpy(a).to(dev)
    binding.pa_reshape_and_cache(c.k, c.v, c.pool, t(c.slots))
    out = torch.empty_like(c.q)
    ws = binding.decode_workspace(c.q, c.pool)
    ws.fill_(0xFF)  # every float in it is a NaN
    binding.pa_decode(out, c.q, c.pool, t(c.bt), t(c.seq_lens), c.scale, ws)
    torch.cuda.synchronize()
    want = c.oracle()
    assert max_abs_err(oracle.decode_elems(u16(out), workloads.F16), want) <= TOL[workloads.F16]


def test_single_token_sequences_return_value_rows(dev):
    """L = 1 everywhere: the output is the stored V row rounded once (exact)."""
    c = Case(dev, workloads.F16, 64, 4, 2, 16, [1] * 9, seed=3)
    out = c.gpu()
    want = c.oracle()
    assert np.array_equal(oracle.decode_elems(u16(out), workloads.F16), want)


def test_decode_bit_identical_under_block_permutation(dev):
    import torch
    c = Case(dev, workloads.BF16, 128, 32, 8, 16, [700, 5, 1234, 16, 999, 2047, 64], seed=17, spare=40)
    out1 = c.gpu()
    rng = np.random.default_rng(99)
    sigma = rng.permutation(c.nb).astype(np.int64)
    pool2 = torch.empty_like(c.pool)
    pool2[:, torch.from_numpy(sigma).to(dev)] = c.pool
    bt2 = np.where(c.bt >= 0, sigma[np.maximum(c.bt, 0)], -1).astype(np.int32)
    out2 = torch.empty_like(c.q)
    ws = binding.decode_workspace(c.q, pool2)
    binding.pa_decode(out2, c.q, pool2, torch.from_numpy(bt2).to(dev), c.sl_d, c.scale, ws)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_shared_blocks_flag_changes_speed_not_results(dev):
    """PA_DECODE_SHARED_BLOCKS only changes an L2 cache hint: bit-identical output."""
    import torch
    c = Case(dev, workloads.BF16, 128, 32, 8, 16, [700, 5, 1234, 16, 999], seed=23)
    out0 = c.gpu()
    out1 = torch.empty_like(c.q)
    ws = binding.decode_workspace(c.q, c.pool)
    binding.pa_decode(out1, c.q, c.pool, c.bt_d, c.sl_d, c.scale, ws,
                      flags=binding.PA_DECODE_SHARED_BLOCKS)
    torch.cuda.synchronize()
    assert torch.equal(out0.view(torch.int16), out1.view(torch.int16))
    with pytest.raises(binding.PAError) as e:
        binding.pa_decode(out1, c.q, c.pool, c.bt_d, c.sl_d, c.scale, ws, flags=4)
    assert e.value.code == binding.PA_ERR_INVALID_ARG


def test_lengths_written_by_the_kernel_just_before_the_decode(dev):
    """Book §4.5: this step's lengths (its token included) are final before
    attention reads them. A serving loop may compute them on the device, in
    the kernel enqueued just before pa_decode; by default the decode waits for
    that kernel before its first read of seq_lens, so the output is that of
    the new lengths, not of what the buffer held before."""
    import torch
    lens = [2000, 1500, 37, 900, 16, 1, 1200, 640, 333, 1999, 64, 700, 5, 1024, 17, 300]
    c = Case(dev, workloads.BF16, 128, 32, 8, 16, lens, seed=41)
    want = c.oracle()
    t = lambda a: torch.from_numpy(a).to(dev)
    binding.pa_reshape_and_cache(c.k, c.v, c.pool, t(c.slots))
    bt = t(c.bt)
    sl = torch.empty(len(lens), dtype=torch.int32, device=dev)
    # A slow kernel (a row sum over 256 MB) whose outputs are the lengths.
    big = torch.zeros((len(lens), 1 << 22), dtype=torch.int32, device=dev)
    big[:, 0] = t(c.seq_lens)
    ws = binding.decode_workspace(c.q, c.pool)
    for _ in range(3):
        out = torch.full_like(c.q, float("nan"))
        sl.fill_(1)                                             # stale lengths
        torch.cuda.synchronize()
        torch.sum(big, dim=1, dtype=torch.int32, out=sl)       # the kernel just before the decode
        binding.pa_decode(out, c.q, c.pool, bt, sl, c.scale, ws)
        torch.cuda.synchronize()
        assert sl.cpu().numpy().tolist() == lens
        err = max_abs_err(oracle.decode_elems(u16(out), c.dtype), want)
        assert err <= TOL[c.dtype], f"max abs err {err}"
    # With PA_DECODE_LENS_READY the lengths come from a host copy (complete
    # before the kernel ahead of the decode starts): the same bits.
    host = torch.from_numpy(c.seq_lens).pin_memory()
    out2 = torch.empty_like(c.q)
    sl.fill_(1)
    sl.copy_(host, non_blocking=True)
    binding.pa_reshape_and_cache(c.k, c.v, c.pool, t(c.slots))
    binding.pa_decode(out2, c.q, c.pool, bt, sl, c.scale, ws, flags=binding.PA_DECODE_LENS_READY)
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    assert binding.pa_get_device_error() == 0


def test_unknown_decode_flags_are_rejected(dev):
    import torch
    c = Case(dev, workloads.F16, 64, 4, 4, 16, [20], seed=9)
    out = torch.empty_like(c.q)
    ws = binding.decode_workspace(c.q, c.pool)
    with pytest.raises(binding.PAError) as e:
        binding.pa_decode(out, c.q, c.pool, torch.from_numpy(c.bt).to(dev),
                          torch.from_numpy(c.seq_lens).to(dev), c.scale, ws, flags=4)
    assert e.value.code == binding.PA_ERR_INVALID_ARG


def test_copy_blocks_bit_exact_and_conflicts_rejected(dev):
    import torch
    rng = np.random.default_rng(4)
    nb, B, H, D = 32, 16, 8, 128
    pools = [workloads.normal_values((2, nb, B, H, D), workloads.F16, 40 + l, dev) for l in range(3)]
    before = [u16(p).copy() for p in pools]
    pairs = np.array([[1, 4], [6, 2], [0, 7], [9, 30]], dtype=np.int32)
    binding.pa_copy_blocks(pools, torch.from_numpy(pairs).to(dev))
    assert oracle.copy_blocks(before, pairs, nb, B, H, D) == 0
    for p, b in zip(pools, before):
        assert np.array_equal(u16(p), b)
    assert binding.pa_get_device_error() == 0
    # a dst that is also a src, and a repeated dst: those pairs are skipped and flagged
    snap = [u16(p).copy() for p in pools]
    bad = np.array([[3, 5], [5, 8], [10, 12], [11, 12], [13, 14]], dtype=np.int32)
    binding.pa_copy_blocks(pools, torch.from_numpy(bad).to(dev))
    assert binding.pa_get_device_error() & binding.PA_DEVERR_PAIR
    assert oracle.copy_blocks(snap, bad[[1, 4]], nb, B, H, D) == 0   # only the clean pairs
    for p, s in zip(pools, snap):
        assert np.array_equal(u16(p), s)


def test_reshape_skips_negative_and_flags_out_of_range_slots(dev):
    import torch
    nb, B, H, D = 4, 16, 2, 64
    pool = workloads.normal_values((2, nb, B, H, D), workloads.BF16, 5, dev)
    key = workloads.normal_values((3, H, D), workloads.BF16, 6, dev)
    val = workloads.normal_values((3, H, D), workloads.BF16, 7, dev)
    snap = u16(pool).copy()
    slots = np.array([5, -1, nb * B], dtype=np.int32)
    binding.pa_reshape_and_cache(key, val, pool, torch.from_numpy(slots).to(dev))
    assert binding.pa_get_device_error() & binding.PA_DEVERR_SLOT
    assert oracle.reshape_and_cache(u16(key), u16(val), snap, slots[:2], nb, B, H, D) == 1
    assert np.array_equal(u16(pool), snap)


def test_bad_block_ids_and_lengths_are_flagged_not_faulted(dev):
    import torch
    c = Case(dev, workloads.F16, 128, 8, 8, 16, [40, 20], seed=8)
    c.gpu()
    assert binding.pa_get_device_error() == 0
    bt = c.bt.copy()
    bt[0, 1] = c.nb + 5            # outside the pool
    sl = np.array([40, 10 ** 6], dtype=np.int32)  # longer than the table
    out = torch.empty_like(c.q)
    ws = binding.decode_workspace(c.q, c.pool)
    binding.pa_decode(out, c.q, c.pool, torch.from_numpy(bt).to(dev),
                      torch.from_numpy(sl).to(dev), c.scale, ws)
    bits = binding.pa_get_device_error()
    assert bits & binding.PA_DEVERR_BLOCK_ID and bits & binding.PA_DEVERR_SEQ_LEN


def test_workspace_too_small_is_rejected(dev):
    import torch
    c = Case(dev, workloads.F16, 64, 4, 4, 16, [20], seed=9)
    out = torch.empty_like(c.q)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    with pytest.raises(binding.PAError) as e:
        binding.pa_decode(out, c.q, c.pool, torch.from_numpy(c.bt).to(dev),
                          torch.from_numpy(c.seq_lens).to(dev), c.scale, ws)
    assert e.value.code == binding.PA_ERR_WORKSPACE


# ------------------------------------------------------------ the workloads

def _run_workload(dev, name, seed, variant="literal", n_sample=48):
    import torch
    w = workloads.WORKLOADS[name]
    plan = step.plan_step(name, seed, variant)
    op = oracle_plan(name, seed, variant)
    assert np.array_equal(plan.block_tables, op["block_tables"])
    assert np.array_equal(plan.slot_mapping, op["slot_mapping"])
    assert np.array_equal(plan.cow_pairs, op["cow_pairs"])
    assert np.array_equal(plan.seq_lens, op["seq_lens"])
    pool, q, k, v = step.make_device_inputs(name, plan, seed, dev)
    pool_bits = u16(pool).copy()
    q_bits, k_bits, v_bits = u16(q), u16(k), u16(v)
    st = step.DecodeStep(name, plan, pool, q, k, v, dev)
    st.run()
    torch.cuda.synchronize()
    S = len(plan.seq_ids)
    rng = np.random.default_rng(seed + 5)
    if n_sample is None or n_sample >= S * w.num_q_heads:
        seqs = np.repeat(np.arange(S), w.num_q_heads)
        heads = np.tile(np.arange(w.num_q_heads), S)
    else:
        seqs = rng.integers(0, S, size=n_sample)
        heads = rng.integers(0, w.num_q_heads, size=n_sample)
        seqs[:2] = [int(np.argmax(plan.seq_lens)), int(np.argmin(plan.seq_lens))]
    want = oracle_step(w, op, pool_bits, q_bits, k_bits, v_bits, sample=(seqs, heads))
    got = oracle.decode_elems(u16(st.out), w.dtype)[seqs, heads]
    err = max_abs_err(got, want)
    assert err <= TOL[w.dtype], f"{name}: max abs err {err}"
    # writes and copies: compare the touched blocks bit for bit
    touched = set(int(s) // w.block_size for s in plan.slot_mapping if s >= 0)
    touched |= set(int(d) for _, d in plan.cow_pairs)
    idx = torch.tensor(sorted(touched), device=dev)
    assert np.array_equal(u16(pool[:, idx]), pool_bits[:, sorted(touched)])
    assert binding.pa_get_device_error() == 0
    # pool_bits now holds the oracle's own post-step pool
    return st, plan, op, pool_bits, q_bits


def test_workload_toy_worked_example(dev):
    """Worked example: write one token each (slots 121/159/76), decode all
    three, then grow B by 20 tokens (into blocks 11 and 12), decoding every step."""
    import torch
    w = workloads.WORKLOADS["toy"]
    st, plan, op, pool_bits, q_bits = _run_workload(dev, "toy", 0, n_sample=None)
    assert plan.slot_mapping.tolist() == [121, 159, 76]
    assert plan.block_tables.tolist() == [[3, 7, -1], [0, 5, 9], [4, -1, -1]]
    alloc = plan.allocator
    model = op["model"]
    pool = st.pool
    for i in range(workloads.TOY_GROWTH_TOKENS):
        sid, mid = plan.seq_ids[1], op["ids"][1]
        slot, cow = alloc.append_token(sid)
        assert (slot, cow) == model.append_token(mid)
        k = workloads.normal_values((1, w.num_kv_heads, w.head_size), w.dtype, 500 + i, dev)
        v = workloads.normal_values((1, w.num_kv_heads, w.head_size), w.dtype, 600 + i, dev)
        kb, vb = u16(k), u16(v)
        binding.pa_reshape_and_cache(k, v, pool, torch.tensor([slot], dtype=torch.int32, device=dev))
        assert oracle.reshape_and_cache(kb, vb, pool_bits, [slot], w.num_blocks, w.block_size,
                                        w.num_kv_heads, w.head_size) == 1
        bt = alloc.block_tables(plan.seq_ids, 5)
        sl = alloc.seq_lens(plan.seq_ids)
        if sl[1] == 49:
            assert bt[1, :4].tolist() == [0, 5, 9, 11]
        out = torch.empty_like(st.query)
        ws = binding.decode_workspace(st.query, pool)
        binding.pa_decode(out, st.query, pool, torch.from_numpy(bt).to(dev),
                          torch.from_numpy(sl).to(dev), w.scale, ws)
        torch.cuda.synchronize()
        want = oracle.decode(q_bits, pool_bits, bt, sl, w.scale, w.num_q_heads,
                             w.num_kv_heads, w.head_size, w.num_blocks, w.block_size, w.dtype)
        assert max_abs_err(oracle.decode_elems(u16(out), w.dtype), want) <= TOL[w.dtype]
        assert np.array_equal(u16(pool), pool_bits)
    assert alloc.table(plan.seq_ids[1]) == [0, 5, 9, 11, 12]


@pytest.mark.parametrize("name", ["llama13b", "gqa8b", "longctx"])
def test_workload_full_size(dev, name):
    """The whole step at full size; every (sequence, head) output row against
    the oracle, element by element."""
    _run_workload(dev, name, seed=1, n_sample=None)


@pytest.mark.parametrize("variant", ["literal", "fork"])
def test_workload_prefix_sharing_cow(dev, variant):
    st, plan, *_ = _run_workload(dev, "prefix_cow", seed=2, variant=variant, n_sample=None)
    if variant == "fork":
        assert len(plan.cow_pairs) == workloads.PREFIX_GROUPS * (workloads.PREFIX_GROUP_SIZE - 1)
    else:
        assert len(plan.cow_pairs) == 0


def test_full_size_permutation_bit_identity(dev):
    """Llama-2-13B shape: moving every block elsewhere in the pool leaves the
    step's decode output bit-identical."""
    import torch
    name = "llama13b"
    plan = step.plan_step(name, 3)
    pool, q, k, v = step.make_device_inputs(name, plan, 3, dev)
    st = step.DecodeStep(name, plan, pool, q, k, v, dev)
    st.run()
    out1 = st.out.clone()
    w = workloads.WORKLOADS[name]
    sigma = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(5)).to(dev)
    pool2 = torch.empty_like(pool)
    pool2[:, sigma] = pool
    sig = sigma.cpu().numpy()
    bt2 = np.where(plan.block_tables >= 0, sig[np.maximum(plan.block_tables, 0)], -1).astype(np.int32)
    out2 = torch.empty_like(q)
    ws = binding.decode_workspace(q, pool2)
    binding.pa_decode(out2, q, pool2, torch.from_numpy(bt2).to(dev), st.seq_lens, w.scale, ws)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_cow_leaves_other_sharers_unchanged(dev):
    """Digest "写时复制": after a fork, one sibling's write clones the shared
    partial block; every other sibling's decode output is bit-identical to
    before, and the writer's output matches the oracle."""
    import torch
    B, H, D, Hq, nb = 16, 8, 128, 32, 128
    dt = workloads.F16
    alloc = binding.BlockAllocator(nb, B, np.random.default_rng(1).permutation(nb))
    parent = alloc.add_seq(1024 + 7)
    sibs = [parent] + [alloc.fork(parent) for _ in range(3)]
    pool = workloads.normal_values((2, nb, B, H, D), dt, 70, dev)
    q = workloads.normal_values((4, Hq, D), dt, 71, dev)
    pool_bits, q_bits = u16(pool).copy(), u16(q)       # oracle inputs, before any kernel
    scale = 1.0 / math.sqrt(D)
    ws = binding.decode_workspace(q, pool)

    def decode():
        bt = torch.from_numpy(alloc.block_tables(sibs, 70)).to(dev)
        sl = torch.from_numpy(alloc.seq_lens(sibs)).to(dev)
        out = torch.empty_like(q)
        binding.pa_decode(out, q, pool, bt, sl, scale, ws)
        torch.cuda.synchronize()
        return out

    before = decode()
    slot, cow = alloc.append_token(sibs[0])
    assert cow is not None and alloc.ref_count(cow[0]) == 3
    binding.pa_copy_blocks([pool], torch.tensor([cow], dtype=torch.int32, device=dev))
    k = workloads.normal_values((1, H, D), dt, 72, dev)
    v = workloads.normal_values((1, H, D), dt, 73, dev)
    binding.pa_reshape_and_cache(k, v, pool, torch.tensor([slot], dtype=torch.int32, device=dev))
    after = decode()
    assert torch.equal(before[1:].view(torch.int16), after[1:].view(torch.int16))
    assert oracle.copy_blocks([pool_bits], [cow], nb, B, H, D) == 0
    assert oracle.reshape_and_cache(u16(k), u16(v), pool_bits, [slot], nb, B, H, D) == 1
    assert np.array_equal(u16(pool), pool_bits)
    bt = alloc.block_tables(sibs, 70)
    want = oracle.decode(q_bits, pool_bits, bt, alloc.seq_lens(sibs), scale, Hq, H, D, nb, B, dt)
    assert max_abs_err(oracle.decode_elems(u16(after), dt), want) <= TOL[dt]


@pytest.mark.parametrize("heads", [(8, 2), (16, 1), (4, 4)])
@pytest.mark.parametrize("D", [128, 64])
def test_decode_bf16_queries_with_huge_scores(dev, heads, D):
    """bf16 query rows scaled by 2^100 and 2^-100: scores far beyond 2^32 in
    base 2 give one-hot rows (bf16 outputs >= 4 held to the oracle rounded
    to bf16), near-zero scores give the mean of V; nothing overflows."""
    import torch
    Hq, Hkv = heads
    c = Case(dev, workloads.BF16, D, Hq, Hkv, 16, LENS, seed=71 + Hq + D)
    q = c.q.float()
    q[0::3] *= 2.0 ** 100
    q[1::3] *= 2.0 ** -100
    c.q = q.to(torch.bfloat16).contiguous()
    c.q_bits = u16(c.q)
    out = c.gpu()
    want = c.oracle()
    got = oracle.decode_elems(u16(out), workloads.BF16)
    assert max_abs_err_bf16_large(got, want) <= TOL[workloads.BF16]
