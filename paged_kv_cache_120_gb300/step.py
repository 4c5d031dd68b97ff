"""One decode step of the hot path on synthetic inputs.

``plan_step`` uses the host block allocator (libpa's ``pa_alloc_*``) to lay
out a workload's sequences in the pool and to reserve the slot of each
sequence's new token; it returns the block tables, slot mapping, decode
lengths and copy-on-write pairs of the step. ``DecodeStep`` holds the device
buffers and runs the step as the pages order it (vLLM book chapter 4, §4.5:
write this step's K/V by slot, then read the history through the block
table), preceded by the COW copies the allocator asked for:

    pa_copy_blocks(cow pairs) -> pa_reshape_and_cache(new K/V) -> pa_decode

A pool of E4M3 codes (uint8) selects the FP8 cache calls instead
(pa_reshape_and_cache_fp8, pa_decode_fp8) with the workload's per-tensor
scales.

Everything here is marshalling around libpa calls; no arithmetic of the
method runs in Python.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import binding, workloads


@dataclasses.dataclass
class StepPlan:
    seq_ids: list
    seq_lens: np.ndarray        # decode lengths (this step's token included)
    block_tables: np.ndarray    # [S, max_blocks] int32, padded with -1
    slot_mapping: np.ndarray    # [S] int32: one new token per sequence
    cow_pairs: np.ndarray       # [P, 2] int32 (src, dst)
    allocator: object


def _finish(alloc, ids, slots, pairs, block_size):
    nblk = max(alloc.num_blocks_of(s) for s in ids)
    max_blocks = max(1, nblk)
    return StepPlan(
        seq_ids=list(ids),
        seq_lens=alloc.seq_lens(ids),
        block_tables=alloc.block_tables(ids, max_blocks),
        slot_mapping=np.asarray(slots, dtype=np.int32),
        cow_pairs=np.asarray(pairs, dtype=np.int32).reshape(-1, 2),
        allocator=alloc,
    )


def plan_step(name: str, seed: int, variant: str = "literal") -> StepPlan:
    """Allocate a workload's sequences and reserve this step's slots.

    Standard workloads: each sequence is created with L-1 tokens and then
    appends its step token (decode length L). ``toy``: lengths 25/47/12 at
    the worked example's placement, then one token each. ``prefix_cow``:
    16 groups of 8 forked from a 1024-token prompt; ``variant="literal"``
    gives each sibling its private tail first, ``variant="fork"`` makes the
    prompt 1024 + r tokens (r in 1..15) so the step's first writes hit the
    shared, partly filled last block and are copied on write.
    """
    w = workloads.WORKLOADS[name]
    if name == "toy":
        order = workloads.toy_free_order()
    else:
        order = workloads.free_order(w.num_blocks, seed)
    alloc = binding.BlockAllocator(w.num_blocks, w.block_size, order)
    slots, pairs = [], []

    def step_token(sid):
        slot, cow = alloc.append_token(sid)
        slots.append(slot)
        if cow is not None:
            pairs.append(cow)

    if name == "prefix_cow":
        lens = workloads.seq_lens(name, seed)
        extra = workloads.prefix_fork_extra(seed)
        ids = []
        for gi in range(workloads.PREFIX_GROUPS):
            prompt = workloads.PREFIX_PROMPT + (int(extra[gi]) if variant == "fork" else 0)
            parent = alloc.add_seq(prompt)
            group = [parent] + [alloc.fork(parent) for _ in range(workloads.PREFIX_GROUP_SIZE - 1)]
            ids += group
        if variant == "literal":
            for k, sid in enumerate(ids):
                for _ in range(int(lens[k]) - 1 - alloc.seq_len(sid)):
                    alloc.append_token(sid)
        for sid in ids:
            step_token(sid)
        return _finish(alloc, ids, slots, pairs, w.block_size)

    lens = workloads.seq_lens(name, seed)
    if name == "toy":
        ids = [alloc.add_seq(int(L)) for L in lens]
    else:
        ids = [alloc.add_seq(int(L) - 1) for L in lens]
    for sid in ids:
        step_token(sid)
    return _finish(alloc, ids, slots, pairs, w.block_size)


class PinnedHostStep:
    """A step that can run from one packed pinned host buffer. The class
    names its device inputs in ``_INPUTS`` and runs its libpa calls in
    ``run()``; ``out`` is its output tensor."""

    def pin_host(self) -> dict:
        """Stage the step's inputs through one packed pinned host buffer.

        The step's device inputs become views of one device buffer, and the
        returned dict holds pinned host views of the same layout, filled with
        the current inputs, plus a pinned ``out``. A caller writes the next
        step's inputs into those views and calls run_pinned(). The libpa calls
        are then replayed from a CUDA graph recorded on the first
        run_pinned(), which holds this batch's launch configuration: call
        pin_host() again when the batch's shape or lengths change."""
        import torch
        names = [n for n in self._INPUTS if getattr(self, n, None) is not None]
        offs, size = {}, 0
        for n in names:
            t = getattr(self, n)
            size = (size + 255) & ~255
            offs[n] = size
            size += t.numel() * t.element_size()
        dev_buf = torch.empty(size, dtype=torch.uint8, device=self.out.device)
        host_buf = torch.empty(size, dtype=torch.uint8).pin_memory()
        views = {}
        for n in names:
            t = getattr(self, n)
            nbytes = t.numel() * t.element_size()
            d = dev_buf[offs[n]:offs[n] + nbytes].view(t.dtype).view(t.shape)
            d.copy_(t)
            setattr(self, n, d)
            views[n] = host_buf[offs[n]:offs[n] + nbytes].view(t.dtype).view(t.shape)
            views[n].copy_(t)
        views["out"] = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        torch.cuda.synchronize(self.out.device)
        self._pinned = (host_buf, dev_buf, views["out"])
        self._pinned_graph = None
        return views

    def pinned_bytes(self) -> int:
        """Bytes one run_pinned() copies to the device (the packed inputs)."""
        return self._pinned[0].numel()

    def run_pinned(self) -> None:
        """One step from the buffers of pin_host(): one host-to-device copy
        of the packed inputs, the step's libpa calls (graph replay), one
        device-to-host copy of the output; returns once the output is on the
        host."""
        import torch
        host_buf, dev_buf, out_host = self._pinned
        if self._pinned_graph is None:
            self.run()  # first calls set up kernel attributes and tensor maps
            torch.cuda.synchronize(self.out.device)
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
                    self.run()
            torch.cuda.current_stream().wait_stream(s)
            self._pinned_graph = g
        dev_buf.copy_(host_buf, non_blocking=True)
        self._pinned_graph.replay()
        out_host.copy_(self.out, non_blocking=True)
        torch.cuda.current_stream().synchronize()


class DecodeStep(PinnedHostStep):
    """Device buffers of one step and the three libpa calls that run it."""

    def __init__(self, name: str, plan: StepPlan, pool, query, key_new, value_new, device,
                 k_scale: float = workloads.FP8_K_SCALE, v_scale: float = workloads.FP8_V_SCALE):
        import torch
        self.w = workloads.WORKLOADS[name]
        self.fp8 = pool.dtype == torch.uint8
        self.k_scale, self.v_scale = k_scale, v_scale
        self.pool = pool
        self.query, self.key_new, self.value_new = query, key_new, value_new
        self.block_tables = torch.from_numpy(plan.block_tables).to(device)
        self.seq_lens = torch.from_numpy(plan.seq_lens).to(device)
        self.slot_mapping = torch.from_numpy(plan.slot_mapping).to(device)
        self.cow_pairs = (torch.from_numpy(plan.cow_pairs).to(device)
                          if len(plan.cow_pairs) else None)
        self.out = torch.empty_like(query)
        self.workspace = (binding.decode_fp8_workspace(query, pool) if self.fp8
                          else binding.decode_workspace(query, pool))
        # Blocks that appear in more than one table are shared (prefix / fork):
        # then K/V keep normal L2 priority, else they are streamed.
        ids = plan.block_tables[plan.block_tables >= 0]
        self.flags = binding.PA_DECODE_SHARED_BLOCKS if len(np.unique(ids)) < len(ids) else 0
        # seq_lens only ever arrives by a host-to-device copy, which completes
        # before the reshape kernel that precedes the decode starts.
        self.flags |= binding.PA_DECODE_LENS_READY

    def launches_per_step(self) -> int:
        # copy_blocks (if any COW pairs) + reshape_and_cache + decode (stream + merge)
        return (1 if self.cow_pairs is not None else 0) + 1 + 2

    def run(self, stream=None) -> None:
        if self.cow_pairs is not None:
            binding.pa_copy_blocks([self.pool], self.cow_pairs, stream)
        self.reshape(stream)
        self.decode(stream)

    def reshape(self, stream=None) -> None:
        if self.fp8:
            binding.pa_reshape_and_cache_fp8(self.key_new, self.value_new, self.pool,
                                             self.slot_mapping, self.k_scale, self.v_scale, stream)
        else:
            binding.pa_reshape_and_cache(self.key_new, self.value_new, self.pool,
                                         self.slot_mapping, stream)

    def run_host(self, host: dict, out_host, stream=None) -> None:
        """The step end to end from pinned host buffers: copy this step's
        inputs to the device, run the three calls, copy the output back and
        wait for it. ``host`` holds pinned tensors named like the device
        buffers (query, key_new, value_new, slot_mapping, block_tables,
        seq_lens and, if the step has COW pairs, cow_pairs)."""
        import torch
        for name in ("query", "key_new", "value_new", "slot_mapping", "block_tables", "seq_lens",
                     "cow_pairs"):
            if name in host:
                getattr(self, name).copy_(host[name], non_blocking=True)
        self.run(stream)
        out_host.copy_(self.out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    _INPUTS = ("query", "key_new", "value_new", "slot_mapping", "block_tables", "seq_lens", "cow_pairs")

    def decode(self, stream=None) -> None:
        if self.fp8:
            binding.pa_decode_fp8(self.out, self.query, self.pool, self.block_tables,
                                  self.seq_lens, self.w.scale, self.k_scale, self.v_scale,
                                  self.workspace, self.flags, stream)
        else:
            binding.pa_decode(self.out, self.query, self.pool, self.block_tables, self.seq_lens,
                              self.w.scale, self.workspace, self.flags, stream)


class ModelStep:
    """One decode step of a whole model: `layers` layer pools (each its own
    (2, num_blocks, B, Hkv, D) cache, as the book's §4.3.1 allocates one per
    layer) sharing the block tables, slots and COW pairs of one allocator.
    The step copies every COW pair in all layer pools with one
    pa_copy_blocks call (a complete block spans every layer), then writes and
    decodes layer after layer. `capture()` records the step in a CUDA graph;
    `run()` then replays it."""

    def __init__(self, name: str, plan: StepPlan, layers: int, seed: int, device,
                 kv_cache: str = "16bit"):
        import torch
        self.w = workloads.WORKLOADS[name]
        self.layers = []
        pool0, q, k, v = make_device_inputs(name, plan, seed, device, kv_cache)
        pools = [pool0]
        for l in range(1, layers):
            pool, _, _, _ = make_device_inputs(name, plan, seed + 97 * l, device, kv_cache)
            pools.append(pool)
        for pool in pools:
            self.layers.append(DecodeStep(name, plan, pool, q, k, v, device))
        self.pools = pools
        self.cow_pairs = self.layers[0].cow_pairs
        self.graph = None

    def launches_per_step(self) -> int:
        return (1 if self.cow_pairs is not None else 0) + 3 * len(self.layers)

    def run_eager(self, stream=None) -> None:
        if self.cow_pairs is not None:
            binding.pa_copy_blocks(self.pools, self.cow_pairs, stream)
        for st in self.layers:
            st.reshape(stream)
            st.decode(stream)

    def capture(self) -> None:
        import torch
        self.run_eager()  # first calls set up kernel attributes and tensor maps
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
                self.run_eager()
        torch.cuda.current_stream().wait_stream(s)
        self.graph = g

    def run(self, stream=None) -> None:
        if self.graph is not None:
            self.graph.replay()
        else:
            self.run_eager(stream)


def make_device_inputs(name: str, plan: StepPlan, seed: int, device, kv_cache: str = "16bit"):
    """Pool, queries and new K/V: seeded N(0, 1) values on ``device``.
    ``kv_cache="fp8"`` gives a pool of E4M3 codes of N(0, 1) draws under the
    workload's FP8 scales (K half with FP8_K_SCALE, V half with FP8_V_SCALE)."""
    import torch
    w = workloads.WORKLOADS[name]
    s = len(plan.seq_ids)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_size)
    if kv_cache == "fp8":
        pool = torch.empty((2,) + shape, dtype=torch.uint8, device=device)
        pool[0] = workloads.fp8_codes(shape, workloads.FP8_K_SCALE, seed + 10, device)
        pool[1] = workloads.fp8_codes(shape, workloads.FP8_V_SCALE, seed + 14, device)
    elif kv_cache == "16bit":
        pool = workloads.normal_values((2,) + shape, w.dtype, seed + 10, device)
    else:
        raise ValueError(f"kv_cache must be '16bit' or 'fp8', not {kv_cache!r}")
    query = workloads.normal_values((s, w.num_q_heads, w.head_size), w.dtype, seed + 11, device)
    key_new = workloads.normal_values((s, w.num_kv_heads, w.head_size), w.dtype, seed + 12, device)
    value_new = workloads.normal_values((s, w.num_kv_heads, w.head_size), w.dtype, seed + 13, device)
    return pool, query, key_new, value_new


# ------------------------------------------------------------------ prefill

@dataclasses.dataclass
class PrefillPlan:
    seq_ids: list
    seq_lens: np.ndarray        # prefix + chunk per sequence
    chunk_lens: np.ndarray      # query tokens per sequence
    cu_seqlens_q: np.ndarray    # [S + 1]
    block_tables: np.ndarray
    slot_mapping: np.ndarray    # [total_q]: the chunk's slots, sequence-major
    num_blocks: int
    allocator: object


def plan_prefill(name: str, seed: int) -> PrefillPlan:
    """Lay out each sequence's cached prefix, then reserve its chunk's slots."""
    w = workloads.PREFILL_WORKLOADS[name]
    pref = workloads.prefill_prefixes(name, seed)
    chunk = np.full(w.num_seqs, w.chunk, dtype=np.int32)
    need = int(((pref + chunk + w.block_size - 1) // w.block_size).sum())
    num_blocks = need + 64
    alloc = binding.BlockAllocator(num_blocks, w.block_size,
                                   workloads.free_order(num_blocks, seed))
    ids = [alloc.add_seq(int(p)) for p in pref]
    slots = [alloc.append_token(sid)[0] for sid in ids for _ in range(w.chunk)]
    lens = alloc.seq_lens(ids)
    max_blocks = max(1, max(alloc.num_blocks_of(sid) for sid in ids))
    return PrefillPlan(seq_ids=ids, seq_lens=lens, chunk_lens=chunk,
                       cu_seqlens_q=np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32),
                       block_tables=alloc.block_tables(ids, max_blocks),
                       slot_mapping=np.asarray(slots, dtype=np.int32), num_blocks=num_blocks,
                       allocator=alloc)


class PrefillStep(PinnedHostStep):
    """Device buffers of one chunked-prefill step: the chunk's K/V are written
    by slot (pa_reshape_and_cache), then pa_prefill reads the whole causal
    context of every query through the block table."""

    def __init__(self, name: str, plan: PrefillPlan, seed: int, device, kv_cache: str = "16bit"):
        import torch
        self.w = w = workloads.PREFILL_WORKLOADS[name]
        total = int(plan.cu_seqlens_q[-1])
        self.fp8 = kv_cache == "fp8"
        shape = (plan.num_blocks, w.block_size, w.num_kv_heads, w.head_size)
        if self.fp8:
            self.k_scale, self.v_scale = workloads.FP8_K_SCALE, workloads.FP8_V_SCALE
            self.pool = torch.empty((2,) + shape, dtype=torch.uint8, device=device)
            self.pool[0] = workloads.fp8_codes(shape, self.k_scale, seed + 20, device)
            self.pool[1] = workloads.fp8_codes(shape, self.v_scale, seed + 24, device)
        else:
            self.pool = workloads.normal_values((2,) + shape, w.dtype, seed + 20, device)
        self.query = workloads.normal_values((total, w.num_q_heads, w.head_size), w.dtype, seed + 21, device)
        self.key_new = workloads.normal_values((total, w.num_kv_heads, w.head_size), w.dtype, seed + 22, device)
        self.value_new = workloads.normal_values((total, w.num_kv_heads, w.head_size), w.dtype, seed + 23,
                                                 device)
        t = lambda a: torch.from_numpy(a).to(device)
        self.block_tables, self.seq_lens = t(plan.block_tables), t(plan.seq_lens)
        self.cu_seqlens_q, self.slot_mapping = t(plan.cu_seqlens_q), t(plan.slot_mapping)
        self.max_seqlen_q = int(plan.chunk_lens.max())
        self.out = torch.empty_like(self.query)
        # None unless the shape has few enough work units to split K/V ranges.
        self.workspace = binding.prefill_workspace(self.query, self.pool, len(plan.seq_ids), self.max_seqlen_q)

    _INPUTS = ("query", "key_new", "value_new", "slot_mapping", "block_tables", "seq_lens", "cu_seqlens_q")

    def launches_per_step(self) -> int:
        return 2  # reshape_and_cache + prefill

    def run(self, stream=None) -> None:
        self.reshape(stream)
        self.prefill(stream)

    def reshape(self, stream=None) -> None:
        if self.fp8:
            binding.pa_reshape_and_cache_fp8(self.key_new, self.value_new, self.pool, self.slot_mapping,
                                             self.k_scale, self.v_scale, stream)
        else:
            binding.pa_reshape_and_cache(self.key_new, self.value_new, self.pool, self.slot_mapping, stream)

    def prefill(self, stream=None) -> None:
        if self.fp8:
            binding.pa_prefill_fp8(self.out, self.query, self.pool, self.block_tables, self.cu_seqlens_q,
                                   self.seq_lens, self.w.scale, self.max_seqlen_q, self.k_scale, self.v_scale,
                                   self.workspace, stream)
        else:
            binding.pa_prefill(self.out, self.query, self.pool, self.block_tables, self.cu_seqlens_q,
                               self.seq_lens, self.w.scale, self.max_seqlen_q, self.workspace, stream)

    def run_host(self, host: dict, out_host, stream=None) -> None:
        """The step from pinned host buffers (query, key_new, value_new,
        slot_mapping, block_tables, seq_lens, cu_seqlens_q), output back."""
        import torch
        for name in ("query", "key_new", "value_new", "slot_mapping", "block_tables", "seq_lens",
                     "cu_seqlens_q"):
            getattr(self, name).copy_(host[name], non_blocking=True)
        self.run(stream)
        out_host.copy_(self.out, non_blocking=True)
        torch.cuda.current_stream().synchronize()


def prefill_flops(plan: PrefillPlan, num_q_heads: int, head_size: int) -> int:
    """Causal attention flops of a step: every (query, head) row attends to its
    p + 1 visible tokens with a dot product and a weighted sum (4 D flops per
    token)."""
    total = 0
    for L, q in zip(plan.seq_lens.tolist(), plan.chunk_lens.tolist()):
        first = L - q + 1  # visible tokens of the chunk's first query
        total += (first + L) * q // 2
    return 4 * head_size * num_q_heads * total
