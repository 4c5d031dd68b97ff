"""CPU checks of the C ABI: the library loads, exports every function that
include/pa.h declares, rejects bad arguments on the host (before any CUDA
call), and its host allocator agrees op-for-op with the oracle's model."""
import os
import re

import numpy as np
import pytest

from oracle.block_manager import BlockManagerModel, OutOfBlocks
from paged_kv_cache_120_gb300 import binding, build, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_\w+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 23
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pa.h but not exported"
    assert sorted(n for n, _, _ in binding.SIGNATURES) == names


def test_exported_set_is_exactly_the_declared_set(lib):
    """No pa_* function leaves the library without a declaration in pa.h."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", build.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = sorted({line.split()[-1] for line in out.splitlines()
                       if line.split() and line.split()[-1].startswith("pa_") and " T " in line})
    assert exported == _declared_functions()


def test_version(lib):
    assert binding.pa_version() == 10000


def test_host_side_validation_without_a_gpu(lib):
    null = None
    # dtype, head size and group checks come before any CUDA call
    assert lib.pa_decode(null, null, null, null, 1, null, 4, 1.0, 8, 8, 128, 10, 16, 7, null, 0, 0, null) \
        == binding.PA_ERR_UNSUPPORTED
    assert lib.pa_decode(null, null, null, null, 1, null, 4, 1.0, 8, 8, 96, 10, 16, 0, null, 0, 0, null) \
        == binding.PA_ERR_UNSUPPORTED
    assert lib.pa_decode(null, null, null, null, 1, null, 4, 1.0, 8, 3, 128, 10, 16, 0, null, 0, 0, null) \
        == binding.PA_ERR_INVALID_ARG
    assert lib.pa_decode(null, null, null, null, 1, null, 4, 1.0, 40, 2, 128, 10, 16, 0, null, 0, 0, null) \
        == binding.PA_ERR_UNSUPPORTED          # group 20: neither <= 16 nor a multiple of 16
    assert lib.pa_decode(null, null, null, null, 1, null, 4, 1.0, 8, 8, 128, 10, 24, 0, null, 0, 0, null) \
        == binding.PA_ERR_INVALID_ARG          # block_size not a multiple of 16
    assert "block_size" in binding.pa_last_error()
    assert lib.pa_decode(null, null, null, null, 1, null, 4, 1.0, 8, 8, 128, 10, 16, 0, null, 0, 0, null) \
        == binding.PA_ERR_INVALID_ARG          # null pointers
    assert lib.pa_decode(null, null, null, null, 1, null, 0, 1.0, 8, 8, 128, 10, 16, 0, null, 0, 0, null) \
        == binding.PA_OK                       # empty batch is a no-op
    assert lib.pa_reshape_and_cache(null, null, null, null, 3, 10, 16, 8, 128, 0, null) \
        == binding.PA_ERR_INVALID_ARG
    assert lib.pa_reshape_and_cache(null, null, null, null, 0, 10, 16, 8, 128, 0, null) == binding.PA_OK
    assert lib.pa_copy_blocks(null, 0, null, 1, 10, 16, 8, 128, 0, null) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_copy_blocks(null, 1, null, 0, 10, 16, 8, 128, 0, null) == binding.PA_OK
    assert lib.pa_copy_blocks(null, 1, null, 0, 10, 16, 1, 8, binding.PA_FP8_E4M3, null) \
        == binding.PA_ERR_INVALID_ARG          # an 8-byte FP8 row cannot be copied in 16-byte units
    assert lib.pa_copy_blocks(null, 1, null, 0, 10, 16, 8, 128, 3, null) == binding.PA_ERR_UNSUPPORTED


def test_prefill_host_side_validation_without_a_gpu(lib):
    null = None
    ok_args = dict(bt=null, maxb=4, cu=null, sl=null, S=2, total=10, maxq=8, scale=0.1, hq=8, hkv=2,
                   d=128, nb=16, bs=16, dt=0)

    def call(**kw):
        a = dict(ok_args, **kw)
        return lib.pa_prefill(null, null, null, a["bt"], a["maxb"], a["cu"], a["sl"], a["S"], a["total"],
                              a["maxq"], a["scale"], a["hq"], a["hkv"], a["d"], a["nb"], a["bs"], a["dt"],
                              null, 0, null)
    assert call(d=96) == binding.PA_ERR_UNSUPPORTED
    assert call(d=64) == binding.PA_ERR_INVALID_ARG              # head size 64 is built: null pointers
    assert call(dt=2) == binding.PA_ERR_UNSUPPORTED
    assert call(hq=40, hkv=2) == binding.PA_ERR_UNSUPPORTED      # group 20
    assert call(hkv=3) == binding.PA_ERR_INVALID_ARG
    assert call(bs=24) == binding.PA_ERR_INVALID_ARG
    assert call(scale=float("inf")) == binding.PA_ERR_INVALID_ARG
    assert call() == binding.PA_ERR_INVALID_ARG                  # null pointers
    assert call(S=0) == binding.PA_OK
    assert call(total=0) == binding.PA_OK
    assert call(maxq=0) == binding.PA_OK


def test_prefill_workspace_size_validation_without_a_gpu(lib):
    import ctypes
    n = ctypes.c_size_t(99)
    assert lib.pa_prefill_workspace_size(2, 64, 8, 2, 128, None) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_prefill_workspace_size(2, 64, 8, 2, 96, ctypes.byref(n)) == binding.PA_ERR_UNSUPPORTED
    assert n.value == 0
    assert lib.pa_prefill_workspace_size(2, 64, 8, 3, 128, ctypes.byref(n)) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_prefill_workspace_size(2, 64, 40, 2, 128, ctypes.byref(n)) == binding.PA_ERR_UNSUPPORTED
    assert lib.pa_prefill_workspace_size(-1, 64, 8, 2, 128, ctypes.byref(n)) == binding.PA_ERR_INVALID_ARG
    n.value = 99
    assert lib.pa_prefill_workspace_size(0, 64, 8, 2, 128, ctypes.byref(n)) == binding.PA_OK
    assert n.value == 0
    n.value = 99
    assert lib.pa_prefill_workspace_size(3, 0, 8, 2, 128, ctypes.byref(n)) == binding.PA_OK
    assert n.value == 0


def test_prefill_fp8_host_side_validation_without_a_gpu(lib):
    null = None
    ok_args = dict(maxb=4, S=2, total=10, maxq=8, scale=0.1, hq=8, hkv=2, d=128, nb=16, bs=16, dt=0,
                   ks=0.02, vs=0.05)

    def call(**kw):
        a = dict(ok_args, **kw)
        return lib.pa_prefill_fp8(null, null, null, null, a["maxb"], null, null, a["S"], a["total"], a["maxq"],
                                  a["scale"], a["hq"], a["hkv"], a["d"], a["nb"], a["bs"], a["dt"], a["ks"],
                                  a["vs"], null, 0, null)
    assert call(ks=0.0) == binding.PA_ERR_INVALID_ARG
    assert call(vs=float("nan")) == binding.PA_ERR_INVALID_ARG
    assert call(ks=-1.0) == binding.PA_ERR_INVALID_ARG
    assert call(d=96) == binding.PA_ERR_UNSUPPORTED
    assert call(d=64) == binding.PA_ERR_INVALID_ARG                      # built; null pointers
    assert call(dt=binding.PA_FP8_E4M3) == binding.PA_ERR_UNSUPPORTED  # dtype is the query's type
    assert call(bs=24) == binding.PA_ERR_INVALID_ARG
    assert call() == binding.PA_ERR_INVALID_ARG                          # null pointers
    assert call(S=0) == binding.PA_OK


def test_fp8_host_side_validation_without_a_gpu(lib):
    null = None
    args = (null, null, null, null, 1, null, 4, 1.0, 8, 8, 128, 10, 16)
    # dtype is the activations' type: E4M3 is not a query type
    assert lib.pa_decode_fp8(*args, binding.PA_FP8_E4M3, 1.0, 1.0, null, 0, 0, null) \
        == binding.PA_ERR_UNSUPPORTED
    for ks, vs in ((0.0, 1.0), (1.0, -2.0), (float("inf"), 1.0), (1.0, float("nan"))):
        assert lib.pa_decode_fp8(*args, 0, ks, vs, null, 0, 0, null) == binding.PA_ERR_INVALID_ARG
        assert "k_scale" in binding.pa_last_error()
        assert lib.pa_reshape_and_cache_fp8(null, null, null, null, 3, 10, 16, 8, 128, 0, ks, vs,
                                            null) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_decode_fp8(*args, 0, 1.0, 1.0, null, 0, 0, null) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_decode_fp8(null, null, null, null, 1, null, 0, 1.0, 8, 8, 128, 10, 16, 1, 0.5,
                             2.0, null, 0, 0, null) == binding.PA_OK
    assert lib.pa_reshape_and_cache_fp8(null, null, null, null, 0, 10, 16, 8, 128, 1, 1.0, 1.0,
                                        null) == binding.PA_OK
    assert lib.pa_reshape_and_cache_fp8(null, null, null, null, 3, 10, 16, 8, 128, 2, 1.0, 1.0,
                                        null) == binding.PA_ERR_UNSUPPORTED


def _both(nb, bs, order):
    return binding.BlockAllocator(nb, bs, order), BlockManagerModel(nb, bs, order)


def test_allocator_reproduces_the_worked_example(lib):
    a = binding.BlockAllocator(64, 16, workloads.toy_free_order())
    ids = [a.add_seq(n) for n in workloads.TOY_LENGTHS]
    assert [a.table(i) for i in ids] == [[3, 7], [0, 5, 9], [4]]
    assert a.num_free() == 58
    assert [a.append_token(i)[0] for i in ids] == [121, 159, 76]
    while a.seq_len(ids[1]) < 49:
        a.append_token(ids[1])
    assert a.table(ids[1]) == [0, 5, 9, 11]


def test_allocator_matches_the_oracle_model_on_random_operations(lib):
    rng = np.random.default_rng(21)
    for trial in range(4):
        nb, bs = int(rng.integers(8, 80)), int(rng.choice([16, 32]))
        order = rng.permutation(nb)
        a, m = _both(nb, bs, order)
        live = []
        for step in range(1500):
            op = int(rng.integers(0, 5))
            if op == 0 or not live:
                n = int(rng.integers(0, 4 * bs))
                try:
                    sm = m.add_seq(n)
                except OutOfBlocks:
                    with pytest.raises(binding.PAError) as e:
                        a.add_seq(n)
                    assert e.value.code == binding.PA_ERR_OUT_OF_BLOCKS
                    continue
                sa = a.add_seq(n)
                live.append((sa, sm))
            elif op == 1:
                sa, sm = live[int(rng.integers(len(live)))]
                live.append((a.fork(sa), m.fork(sm)))
            elif op in (2, 3):
                sa, sm = live[int(rng.integers(len(live)))]
                try:
                    want = m.append_token(sm)
                except OutOfBlocks:
                    with pytest.raises(binding.PAError) as e:
                        a.append_token(sa)
                    assert e.value.code == binding.PA_ERR_OUT_OF_BLOCKS
                    continue
                assert a.append_token(sa) == want
            else:
                sa, sm = live.pop(int(rng.integers(len(live))))
                a.free_seq(sa)
                m.free_seq(sm)
            assert a.num_free() == m.num_free()
        for sa, sm in live:
            assert a.table(sa) == m.table(sm)
            assert a.seq_len(sa) == m.seq_len(sm)
        assert [a.ref_count(b) for b in range(nb)] == m.ref


def test_allocator_block_tables_and_errors(lib):
    a = binding.BlockAllocator(16, 16)
    s0, s1 = a.add_seq(20), a.add_seq(0)
    bt = a.block_tables([s0, s1], 3)
    assert bt.tolist() == [[0, 1, -1], [-1, -1, -1]]
    assert a.seq_lens([s0, s1]).tolist() == [20, 0]
    with pytest.raises(binding.PAError) as e:
        a.block_tables([s0], 1)
    assert e.value.code == binding.PA_ERR_INVALID_ARG
    with pytest.raises(binding.PAError) as e:
        a.free_seq(99)
    assert e.value.code == binding.PA_ERR_NOT_FOUND
    with pytest.raises(binding.PAError):
        binding.BlockAllocator(4, 16, [0, 1, 1, 2])
