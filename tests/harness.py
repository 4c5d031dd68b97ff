"""Test-side helpers: the oracle's half of every parity case.

The oracle side never takes an input from the CUDA path: its block tables,
slots and COW pairs come from the oracle's own block-manager model driven by
the same operation sequence as the product allocator, and its K/V/Q values
are the seeded generator's output, snapshotted before any libpa kernel runs.
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle.block_manager import BlockManagerModel
from paged_kv_cache_120_gb300 import workloads

TOL = {workloads.F16: 2e-3, workloads.BF16: 1e-2}


def oracle_plan(name: str, seed: int, variant: str = "literal"):
    """Same operation sequence as paged_kv_cache_120_gb300.step.plan_step, on the model."""
    w = workloads.WORKLOADS[name]
    order = workloads.toy_free_order() if name == "toy" else workloads.free_order(w.num_blocks, seed)
    m = BlockManagerModel(w.num_blocks, w.block_size, order)
    slots, pairs = [], []

    def step_token(sid):
        slot, cow = m.append_token(sid)
        slots.append(slot)
        if cow is not None:
            pairs.append(cow)

    if name == "prefix_cow":
        lens = workloads.seq_lens(name, seed)
        extra = workloads.prefix_fork_extra(seed)
        ids = []
        for gi in range(workloads.PREFIX_GROUPS):
            prompt = workloads.PREFIX_PROMPT + (int(extra[gi]) if variant == "fork" else 0)
            parent = m.add_seq(prompt)
            ids += [parent] + [m.fork(parent) for _ in range(workloads.PREFIX_GROUP_SIZE - 1)]
        if variant == "literal":
            for k, sid in enumerate(ids):
                for _ in range(int(lens[k]) - 1 - m.seq_len(sid)):
                    m.append_token(sid)
    else:
        lens = workloads.seq_lens(name, seed)
        ids = [m.add_seq(int(L) if name == "toy" else int(L) - 1) for L in lens]
    for sid in ids:
        step_token(sid)
    max_blocks = max(1, max(len(m.table(s)) for s in ids))
    bt = np.full((len(ids), max_blocks), -1, dtype=np.int32)
    for i, s in enumerate(ids):
        t = m.table(s)
        bt[i, :len(t)] = t
    return dict(model=m, ids=ids, block_tables=bt,
                seq_lens=np.array([m.seq_len(s) for s in ids], dtype=np.int32),
                slot_mapping=np.array(slots, dtype=np.int32),
                cow_pairs=np.array(pairs, dtype=np.int32).reshape(-1, 2))


def u16(t):
    """torch CPU/GPU tensor (fp16/bf16) -> numpy uint16 bit patterns on the host."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def values(t, dtype):
    return oracle.decode_elems(u16(t), dtype)


def oracle_step(w, op, pool_bits, q_bits, k_bits, v_bits, sample=None):
    """Apply the step (COW copies, writes, decode) on the oracle's host copy.
    Returns decode outputs [S, Hq, D] (or [n, D] for sampled (seq, head) pairs)."""
    if len(op["cow_pairs"]):
        assert oracle.copy_blocks([pool_bits], op["cow_pairs"], w.num_blocks, w.block_size,
                                  w.num_kv_heads, w.head_size) == 0
    n = oracle.reshape_and_cache(k_bits, v_bits, pool_bits, op["slot_mapping"], w.num_blocks,
                                 w.block_size, w.num_kv_heads, w.head_size)
    assert n == (op["slot_mapping"] >= 0).sum()
    if sample is None:
        return oracle.decode(q_bits, pool_bits, op["block_tables"], op["seq_lens"], w.scale,
                             w.num_q_heads, w.num_kv_heads, w.head_size, w.num_blocks,
                             w.block_size, w.dtype)
    seqs, heads = sample
    return oracle.decode_sampled(seqs, heads, q_bits, pool_bits, op["block_tables"],
                                 op["seq_lens"], w.scale, w.num_q_heads, w.num_kv_heads,
                                 w.head_size, w.num_blocks, w.block_size, w.dtype)


def max_abs_err(got, want):
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), "non-finite GPU output"
    return float(np.max(np.abs(got - want))) if got.size else 0.0


def rne_bf16(x):
    """float64 values rounded to the nearest bf16 value, ties to even (normal
    range: 8 significant bits)."""
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def max_abs_err_bf16_large(got, want):
    """The bf16 tolerance reading for outputs of magnitude >= 4, where bf16's
    half-ulp (2^-6) exceeds 1e-2: those elements are compared with the
    oracle rounded to bf16, the rest with the oracle itself."""
    return max_abs_err(got, np.where(np.abs(want) >= 4.0, rne_bf16(want), want))


def prefill_tile_samples(plan, w, rng):
    """(sequence, chunk token, query head) samples covering every query tile
    of every kv head of a prefill batch: the kernel's work unit is a pair of
    tiles of (up to 16 query heads of a kv head) x (128 / heads tokens), so
    one random row per (sequence, tile, kv head) checks both tiles of every
    unit, and with them every place a split can cut a unit's K/V range. The
    last row of every chunk is added."""
    group = w.num_q_heads // w.num_kv_heads
    hpc = min(group, 16)
    rows = (128 // hpc) & ~7
    s_l, i_l, h_l = [], [], []
    for s in range(len(plan.chunk_lens)):
        q_len = int(plan.chunk_lens[s])
        for t0 in range(0, q_len, rows):
            for h in range(w.num_kv_heads):
                s_l.append(s)
                i_l.append(int(rng.integers(t0, min(q_len, t0 + rows))))
                h_l.append(h * group + int(rng.integers(0, group)))
        s_l.append(s)
        i_l.append(q_len - 1)
        h_l.append(int(rng.integers(0, w.num_q_heads)))
    return np.array(s_l), np.array(i_l), np.array(h_l, dtype=np.int32)
