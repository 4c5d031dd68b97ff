"""GPU checks of the multi-layer step: copy-on-write at model scale (one
pa_copy_blocks call over every layer pool: a complete block spans all
layers) and a decode step over several layer pools, eagerly and replayed
from a CUDA graph. Bars: copies and writes bit-exact in every layer,
sampled decode rows within the 16-bit tolerances, graph replay
bit-identical to the eager step."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_120_gb300 import binding, build, step, workloads

from harness import TOL, max_abs_err, oracle_plan, u16

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


def test_copy_blocks_across_40_layer_pools(dev):
    """Llama-2-13B heads (40 x 128, fp16): 40 layer pools, 96 COW pairs; every
    layer copied bit for bit (checked against the oracle on five layers, and
    every pair's destination against its source in all layers)."""
    import torch
    nb, B, H, D, layers = 256, 16, 40, 128, 40
    pools = [workloads.normal_values((2, nb, B, H, D), workloads.F16, 900 + l, dev) for l in range(layers)]
    rng = np.random.default_rng(12)
    ids = rng.permutation(nb)[:192].astype(np.int32)
    pairs = ids.reshape(96, 2)
    check = [0, 1, 17, 38, 39]
    before = {l: u16(pools[l]).copy() for l in check}
    binding.pa_copy_blocks(pools, torch.from_numpy(pairs).to(dev))
    torch.cuda.synchronize()
    assert binding.pa_get_device_error() == 0
    for l in check:
        assert oracle.copy_blocks([before[l]], pairs, nb, B, H, D) == 0
        assert np.array_equal(u16(pools[l]), before[l])
    src = torch.from_numpy(pairs[:, 0].astype(np.int64)).to(dev)
    dst = torch.from_numpy(pairs[:, 1].astype(np.int64)).to(dev)
    for pool in pools:
        assert torch.equal(pool[:, dst].view(torch.int16), pool[:, src].view(torch.int16))


@pytest.mark.parametrize("name,variant,kv", [("prefix_cow", "fork", "16bit"), ("llama13b", "literal", "16bit"),
                                             ("prefix_cow", "fork", "fp8")])
def test_model_step_over_layer_pools_and_graph_replay(dev, name, variant, kv):
    import torch
    w = workloads.WORKLOADS[name]
    seed, layers = 6, 3
    plan = step.plan_step(name, seed, variant)
    op = oracle_plan(name, seed, variant)
    assert np.array_equal(plan.block_tables, op["block_tables"])
    assert np.array_equal(plan.cow_pairs, op["cow_pairs"])
    ms = step.ModelStep(name, plan, layers, seed, dev, kv)
    fp8 = kv == "fp8"
    bits = (lambda t: t.cpu().numpy()) if fp8 else u16
    snaps = [bits(p).copy() for p in ms.pools]
    st0 = ms.layers[0]
    q_bits, k_bits, v_bits = u16(st0.query), u16(st0.key_new), u16(st0.value_new)
    ms.run_eager()
    torch.cuda.synchronize()
    assert binding.pa_get_device_error() == 0
    rng = np.random.default_rng(seed)
    S = len(plan.seq_ids)
    seqs = rng.integers(0, S, size=24)
    heads = rng.integers(0, w.num_q_heads, size=24)
    for l, st in enumerate(ms.layers):
        pb = snaps[l]
        if len(op["cow_pairs"]):
            view = pb.view(np.uint16)
            dh = w.head_size // 2 if fp8 else w.head_size
            assert oracle.copy_blocks([view], op["cow_pairs"], w.num_blocks, w.block_size,
                                      w.num_kv_heads, dh) == 0
        if fp8:
            oracle.reshape_and_cache_fp8(k_bits, v_bits, pb, op["slot_mapping"], w.num_blocks, w.block_size,
                                         w.num_kv_heads, w.head_size, w.dtype, st.k_scale, st.v_scale)
            want = oracle.decode_fp8_sampled(seqs, heads, q_bits, pb, op["block_tables"], op["seq_lens"],
                                             w.scale, w.num_q_heads, w.num_kv_heads, w.head_size,
                                             w.num_blocks, w.block_size, w.dtype, st.k_scale, st.v_scale)
        else:
            oracle.reshape_and_cache(k_bits, v_bits, pb, op["slot_mapping"], w.num_blocks, w.block_size,
                                     w.num_kv_heads, w.head_size)
            want = oracle.decode_sampled(seqs, heads, q_bits, pb, op["block_tables"], op["seq_lens"],
                                         w.scale, w.num_q_heads, w.num_kv_heads, w.head_size, w.num_blocks,
                                         w.block_size, w.dtype)
        got = oracle.decode_elems(u16(st.out), w.dtype)[seqs, heads]
        assert max_abs_err(got, want) <= TOL[w.dtype], f"layer {l}"
        touched = sorted(set(int(s) // w.block_size for s in plan.slot_mapping if s >= 0)
                         | set(int(d) for _, d in plan.cow_pairs))
        idx = torch.tensor(touched, device=dev)
        assert np.array_equal(bits(ms.pools[l][:, idx]), pb[:, touched]), f"layer {l} writes/copies"
    outs = [st.out.clone() for st in ms.layers]
    pools_after = [p.clone() for p in ms.pools]
    for st in ms.layers:
        st.out.zero_()
    ms.capture()
    ms.run()
    torch.cuda.synchronize()
    assert binding.pa_get_device_error() == 0
    for a, st in zip(outs, ms.layers):
        assert torch.equal(a.view(torch.int16), st.out.view(torch.int16))
    for a, p in zip(pools_after, ms.pools):
        assert torch.equal(a.view(torch.uint8) if fp8 else a.view(torch.int16),
                           p.view(torch.uint8) if fp8 else p.view(torch.int16))


@pytest.mark.parametrize("name,variant", [("llama13b", "literal"), ("prefix_cow", "fork")])
def test_pinned_host_step_matches_the_eager_step(dev, name, variant):
    """The packed pinned-host path (one copy each way, the libpa calls
    replayed from a CUDA graph) leaves the pool and the output bit for bit
    as the eager step does, and a new query written into the host view is
    the one the next step attends with."""
    import torch
    w = workloads.WORKLOADS[name]
    plan = step.plan_step(name, 3, variant)
    pool, q, k, v = step.make_device_inputs(name, plan, 3, dev)
    eager = step.DecodeStep(name, plan, pool.clone(), q.clone(), k.clone(), v.clone(), dev)
    pinned = step.DecodeStep(name, plan, pool, q, k, v, dev)
    host = pinned.pin_host()
    out = host.pop("out")
    assert pinned.pinned_bytes() >= sum(t.numel() * t.element_size() for t in host.values())
    eager.run()
    pinned.run_pinned()
    assert torch.equal(out.view(torch.int16), eager.out.cpu().view(torch.int16))
    assert torch.equal(pinned.pool.view(torch.int16), eager.pool.view(torch.int16))
    first = out.clone()
    q2 = workloads.normal_values(tuple(q.shape), w.dtype, 77, dev)
    eager.query.copy_(q2)
    host["query"].copy_(q2.cpu())
    eager.run()
    pinned.run_pinned()
    assert torch.equal(out.view(torch.int16), eager.out.cpu().view(torch.int16))
    assert not torch.equal(out.view(torch.int16), first.view(torch.int16))
    assert binding.pa_get_device_error() == 0


def test_host_step_paths_agree_for_prefill(dev):
    """The chunked-prefill step (GQA-8B shapes, 8 x 1024-token chunks) gives
    the same output bits eagerly, from separate pinned host tensors
    (run_host) and from the packed pinned buffer (run_pinned)."""
    import torch
    plan = step.plan_prefill("prefill_gqa8b", 5)
    st = step.PrefillStep("prefill_gqa8b", plan, 5, dev)
    loose = {n: getattr(st, n).cpu().pin_memory() for n in st._INPUTS}
    st.run()
    torch.cuda.synchronize()
    want = st.out.cpu().view(torch.int16).clone()
    out_loose = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    st.run_host(loose, out_loose)
    assert torch.equal(out_loose.view(torch.int16), want)
    host = st.pin_host()
    out = host.pop("out")
    st.run_pinned()
    st.run_pinned()
    assert torch.equal(out.view(torch.int16), want)
    assert binding.pa_get_device_error() == 0
