"""pa_decode_static_scratch: decode for callers that cannot allocate.

Some callers of this library may not call cudaMalloc at all: a framework
whose caching allocator owns every byte of device memory, a plugin held to a
fixed memory budget, or a latency-critical loop where an allocation (which
can synchronise the device) is forbidden. For them the library offers an
entry point whose split-K scratch is a static device array inside the
library. These tests call it through the C ABI and require the same output
bits as pa_decode with a caller workspace, on two calls in a row that follow
a call of another shape (each call finds the previous call's contents in the
shared array), no change in free device memory across the second call, and a
clear refusal for a shape whose scratch would not fit.

This file is collected last on purpose, and it also passes on its own in a
fresh process (its first call does the one-time address lookup).
"""
import math

import numpy as np
import pytest

from paged_kv_cache_120_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu

TOL = {workloads.F16: 2e-3, workloads.BF16: 1e-2}


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.lib()
    return torch.device("cuda:0")


def _case(dev, dtype, Hq, Hkv, D, lens, seed):
    import torch
    B = 16
    rng = np.random.default_rng(seed)
    nblk = [-(-L // B) for L in lens]
    nb = sum(nblk) + 4
    perm = rng.permutation(nb).astype(np.int32)
    maxblk = max(nblk)
    bt = np.full((len(lens), maxblk), -1, dtype=np.int32)
    i = 0
    for s, n in enumerate(nblk):
        bt[s, :n] = perm[i:i + n]
        i += n
    pool = workloads.normal_values((2, nb, B, Hkv, D), dtype, seed + 1, dev)
    q = workloads.normal_values((len(lens), Hq, D), dtype, seed + 2, dev)
    return (pool, q, torch.from_numpy(bt).to(dev),
            torch.from_numpy(np.array(lens, dtype=np.int32)).to(dev), 1.0 / math.sqrt(D))


@pytest.mark.parametrize("dtype,Hq,Hkv", [(workloads.F16, 40, 40), (workloads.BF16, 32, 8)])
def test_static_scratch_matches_workspace_decode_on_two_calls(dev, dtype, Hq, Hkv):
    import torch
    D = 128
    # long sequences so that segments span many warps and the scratch is used
    lens = [20000, 3, 777, 4096, 1, 12345, 640, 9000]
    pool, q, bt, sl, scale = _case(dev, dtype, Hq, Hkv, D, lens, seed=31 + Hq)
    ref = torch.empty_like(q)
    binding.pa_decode(ref, q, pool, bt, sl, scale, binding.decode_workspace(q, pool))
    # Leave a different shape's records in the shared array first: a later
    # call must not pick any of them up.
    o_pool, o_q, o_bt, o_sl, _ = _case(dev, dtype, Hq, Hkv, D, [30000, 70, 5000], seed=77)
    binding.pa_decode_static_scratch(torch.empty_like(o_q), o_q, o_pool, o_bt, o_sl, 0.3)
    outs = [torch.full_like(q, float("nan")) for _ in range(2)]
    torch.cuda.synchronize()
    for call, out in enumerate(outs):
        free_before = torch.cuda.mem_get_info(dev)[0]
        binding.pa_decode_static_scratch(out, q, pool, bt, sl, scale)
        torch.cuda.synchronize()
        if call == 1:
            # the array was set up by the earlier calls; this call allocates nothing
            assert torch.cuda.mem_get_info(dev)[0] == free_before
        # the same kernels and the same split as pa_decode: the same bits
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call}"
    # (so within the tests' decode tolerance of it too)
    got = outs[1].float().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert float(np.max(np.abs(got - ref.float().cpu().numpy()))) <= TOL[dtype]
    assert binding.pa_get_device_error() == 0


def test_static_scratch_refuses_a_shape_that_does_not_fit(dev):
    import torch
    pool, q, bt, sl, scale = _case(dev, workloads.F16, 32, 1, 128, [100, 200], seed=5)
    need = binding.pa_decode_workspace_size(2, 32, 1, 128, 16, workloads.F16)
    assert need > 16 << 20
    out = torch.empty_like(q)
    with pytest.raises(binding.PAError) as e:
        binding.pa_decode_static_scratch(out, q, pool, bt, sl, scale)
    assert e.value.code == binding.PA_ERR_WORKSPACE
    assert "static" in str(e.value)
