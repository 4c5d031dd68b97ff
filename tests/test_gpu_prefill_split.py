"""GPU parity of chunked prefill with the work units' K/V ranges split across
the SMs (stream-K) and the pieces merged, through the C ABI.

A launch with few work units (a few long sequences with short chunks) and a
workspace deals the units' K/V tiles out to the SMs in equal contiguous
shares; each piece of a unit stores its partial softmax state (reference
maximum, row sum, unnormalised output) and a merge kernel combines them in a
fixed order, the online-softmax merge of the book's §4.6 over disjoint token
ranges. Bar: the tolerances of the whole-unit prefill (max abs 2e-3 fp16 /
1e-2 bf16 against the fp64 oracle), NaN padding ignored, results that do not
depend on the workspace's previous contents or on which piece finishes last
(bit-identical reruns and graph replays), bad sequences flagged and skipped.
"""
import numpy as np
import pytest

import oracle
from paged_kv_cache_120_gb300 import binding, build, workloads

from harness import TOL, max_abs_err, prefill_tile_samples, u16
from test_gpu_prefill import PrefillCase
from test_gpu_prefill_fp8 import Fp8PrefillCase

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


def both_modes(c):
    """Split and whole-unit outputs of the case, each against one oracle
    run; returns the split output."""
    split = c.gpu()
    whole = c.prefill(c.pool, c.bt_d, split=False)
    want = c.oracle()
    for out in (split, whole):
        err = max_abs_err(oracle.decode_elems(u16(out), c.dtype), want)
        assert err <= TOL[c.dtype], f"max abs err {err}"
    assert binding.pa_get_device_error() == 0
    return split


# (q heads, kv heads, dtype, head size, context lengths, chunk lengths):
# MHA with two long sequences, GQA with a short chunk, one unit cut into
# pieces by every CTA (16 query heads on one kv head: tiles of 16 heads x 8
# tokens; the merge then spreads each row's pieces over 8 threads), the same
# at head size 64 in bf16, head size 64 with a short sequence beside a long
# one, and the Llama-2-13B head count.
LONG = [
    (8, 8, workloads.F16, 128, [6000, 9100], [100, 256]),
    (32, 8, workloads.BF16, 128, [7000, 3000], [300, 64]),
    (16, 1, workloads.F16, 128, [20000], [8]),
    (16, 1, workloads.BF16, 64, [30000], [8]),
    (8, 2, workloads.BF16, 64, [12000, 40], [77, 40]),
    (40, 40, workloads.F16, 128, [4500, 4100], [256, 129]),
]


@pytest.mark.parametrize("case", LONG, ids=lambda c: f"{c[0]}x{c[1]}-d{c[3]}-{len(c[4])}seq")
def test_split_long_context_parity(dev, case):
    Hq, Hkv, dtype, D, ctx, ql = case
    c = PrefillCase(dev, dtype, Hq, Hkv, 16, ctx, ql, seed=1200 + Hq + D, poison=True, D=D, split=True)
    both_modes(c)


def test_split_many_short_sequences(dev):
    """200 sequences (contexts up to 400 tokens, chunks of 0 to 3 tokens,
    some chunks the whole sequence) over 8/2 heads: 400 units, few enough to
    split. The plan scans the sequences 32 at a time and walks hundreds of
    one- and two-tile units, so shares start and end in every kind of place."""
    rng = np.random.default_rng(1306)
    ql = rng.integers(0, 4, size=200)
    ctx = np.maximum(ql, rng.integers(1, 401, size=200))
    ctx[::17] = ql[::17]  # chunks that are the whole sequence
    c = PrefillCase(dev, workloads.F16, 8, 2, 16, [int(x) for x in ctx], [int(x) for x in ql], seed=1306,
                    poison=True, split=True)
    both_modes(c)


def test_split_fp8_long_context_parity(dev):
    c = Fp8PrefillCase(dev, workloads.BF16, 40, 40, 16, [5000, 3000], [200, 128], seed=1300, poison=True,
                       split=True)
    c.check(c.gpu())
    c.split = False
    c.check(c.prefill(c.pool, c.bt_d))


def test_split_fp8_single_unit(dev):
    """One work unit over an FP8 cache, cut into a piece per SM: the merge
    folds each row's pieces on 8 threads and applies the V scale."""
    c = Fp8PrefillCase(dev, workloads.F16, 16, 1, 16, [20000], [16], seed=1305, poison=True, split=True)
    c.check(c.gpu())


def test_split_is_deterministic_whatever_the_workspace_held(dev):
    """The pieces are combined in a fixed order whichever finishes last, and
    every piece writes its state before any is read: reruns with the
    workspace holding NaN bytes, zeros or random bytes give the same bits."""
    import torch
    c = PrefillCase(dev, workloads.F16, 32, 8, 16, [9000, 7000, 300], [200, 64, 300], seed=1301, split=True)
    first = c.gpu()
    ws = c.workspace()
    g = torch.Generator(device=dev).manual_seed(5)
    for fill in ("nan", "zero", "random"):
        if fill == "zero":
            ws.zero_()
        elif fill == "random":
            ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device=dev, generator=g))
        out = torch.full_like(c.q, float("nan"))
        binding.pa_prefill(out, c.q, c.pool, c.bt_d, c.cu_d, c.sl_d, c.scale, c.max_q, ws)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), first.view(torch.int16)), fill
    c.check(first)


def test_split_replayed_from_a_cuda_graph_is_bit_identical(dev):
    """A split launch is two kernels (the pieces, then the merge, launched
    with programmatic dependent launch); replayed from a CUDA graph between
    eager launches it gives the eager bits."""
    import torch
    c = PrefillCase(dev, workloads.BF16, 16, 2, 16, [8000, 2000], [150, 129], seed=1302, split=True)
    ref = c.gpu()
    c.check(ref)
    ws = c.workspace()
    out = torch.full_like(c.q, float("nan"))
    q = c.q.contiguous()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.pa_prefill(out, q, c.pool, c.bt_d, c.cu_d, c.sl_d, c.scale, c.max_q, ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        binding.pa_prefill(out, q, c.pool, c.bt_d, c.cu_d, c.sl_d, c.scale, c.max_q, ws)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        again = c.prefill(c.pool, c.bt_d)
        assert torch.equal(again.view(torch.int16), ref.view(torch.int16))
    assert binding.pa_get_device_error() == 0


def test_split_skips_and_flags_bad_sequences_then_recovers(dev):
    """A sequence whose length is shorter than its chunk gets no tiles: its
    rows stay untouched and PA_DEVERR_SEQ_LEN is set; the other sequence's
    rows are right, and so is the next launch."""
    import torch
    c = PrefillCase(dev, workloads.F16, 8, 2, 16, [6000, 3000], [64, 40], seed=1303, split=True)
    good = c.gpu()
    got, want = c.check(good)
    sl = torch.from_numpy(np.array([6000, 10], np.int32)).to(dev)
    out = torch.full_like(c.q, float("nan"))
    binding.pa_prefill(out, c.q, c.pool, c.bt_d, c.cu_d, sl, c.scale, c.max_q, c.workspace())
    torch.cuda.synchronize()
    assert binding.pa_get_device_error() == binding.PA_DEVERR_SEQ_LEN
    assert torch.isnan(out[64:].float()).all()
    # (the other sequence's pieces are cut elsewhere now: same tolerance, not the same bits)
    assert max_abs_err(oracle.decode_elems(u16(out[:64]), c.dtype), want[:64]) <= TOL[c.dtype]
    again = c.prefill(c.pool, c.bt_d)
    assert torch.equal(again.view(torch.int16), good.view(torch.int16))
    assert binding.pa_get_device_error() == 0


def test_split_workspace_rules(dev):
    """Size query: 0 for a shape with many work units; for few, per CTA two
    slots of two 128-row tiles of (head_size fp32 + 2 fp32) and a 16-byte job
    record. A workspace that is too small or misaligned is refused; none at
    all means whole units."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert binding.pa_prefill_workspace_size(8, 1024, 40, 40, 128) == 0        # 1280 units
    n = binding.pa_prefill_workspace_size(2, 512, 40, 40, 128)                  # 160 units
    assert n == sms * 2 * 2 * 128 * (128 * 4 + 8) + sms * 16
    assert binding.pa_prefill_workspace_size(1, 8, 16, 1, 64) == sms * 2 * 2 * 128 * (64 * 4 + 8) + sms * 16
    c = PrefillCase(dev, workloads.F16, 8, 2, 16, [3000, 100], [50, 100], seed=1304)
    c.gpu()
    ws = c.workspace()
    out = torch.empty_like(c.q)
    with pytest.raises(binding.PAError) as e:
        binding.pa_prefill(out, c.q, c.pool, c.bt_d, c.cu_d, c.sl_d, c.scale, c.max_q, ws[:-256])
    assert e.value.code == binding.PA_ERR_WORKSPACE
    big = torch.empty(ws.numel() + 256, dtype=torch.uint8, device=dev)
    with pytest.raises(binding.PAError) as e:
        binding.pa_prefill(out, c.q, c.pool, c.bt_d, c.cu_d, c.sl_d, c.scale, c.max_q, big[16:])
    assert e.value.code == binding.PA_ERR_WORKSPACE
    assert binding.pa_get_device_error() == 0


@pytest.mark.parametrize("name", ["prefill_longctx_llama13b", "prefill_longctx_gqa8b"])
def test_split_workload_full_size(dev, name):
    """The long-context steps bench.py times (same plan, seed and launch,
    which splits): the chunk's writes bit-exact, and a row of every query
    tile of every kv head (so both tiles of every work unit, wherever the
    split cut it) plus the last row of every chunk, against the oracle's
    decode over the row's causal prefix; the split and whole-unit launches
    both."""
    import torch
    from paged_kv_cache_120_gb300 import step
    w = workloads.PREFILL_WORKLOADS[name]
    plan = step.plan_prefill(name, 0)
    st = step.PrefillStep(name, plan, 0, dev)
    assert st.workspace is not None
    pool_bits = u16(st.pool).copy()
    k_bits, v_bits, q_bits = u16(st.key_new), u16(st.value_new), u16(st.query)
    st.run()
    torch.cuda.synchronize()
    split = st.out.clone()
    st.workspace, ws = None, st.workspace
    st.prefill()
    torch.cuda.synchronize()
    whole = st.out.clone()
    st.workspace = ws
    assert binding.pa_get_device_error() == 0
    geo = (plan.num_blocks, w.block_size, w.num_kv_heads, w.head_size)
    assert oracle.reshape_and_cache(k_bits, v_bits, pool_bits, plan.slot_mapping, *geo) == len(plan.slot_mapping)
    assert np.array_equal(u16(st.pool), pool_bits)
    s, i, hq = prefill_tile_samples(plan, w, np.random.default_rng(13))
    m = len(s)
    rows = plan.cu_seqlens_q[s] + i
    vis = (plan.seq_lens[s] - w.chunk + i + 1).astype(np.int32)
    want = oracle.decode_sampled(np.arange(m, dtype=np.int32), hq, q_bits[rows], pool_bits, plan.block_tables[s],
                                 vis, w.scale, w.num_q_heads, w.num_kv_heads, w.head_size, plan.num_blocks,
                                 w.block_size, w.dtype)
    for out in (split, whole):
        got = oracle.decode_elems(u16(out)[rows, hq], w.dtype)
        assert max_abs_err(got, want) <= TOL[w.dtype]
