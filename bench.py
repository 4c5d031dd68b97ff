#!/usr/bin/env python3
"""Benchmark of the PagedAttention hot path on GB300.

A decode step is one pass of the whole hot path over one batch:
    pa_copy_blocks (COW pairs, if the workload has any)
    -> pa_reshape_and_cache (one new token per sequence)
    -> pa_decode (stream kernel + split-K merge kernel)
Default workload: the Llama-2-13B layer (64 sequences, 40/40 heads,
head_dim 128, fp16, lengths uniform in [1, 2048], 9000-block pool).

Prints one JSON line (rank 0). ``value`` is the step's algorithmic HBM bytes
per second (GB/s) over exactly --steps timed steps; ``seq_steps_per_s`` is
sequences decoded per second. Each kernel family is also timed alone: a
block of back-to-back launches (at least 50), every launch bracketed by CUDA
events, summarised by its median; the roofline fraction comes from that
median. The default run adds a ``configs`` record with the same measurements
for every other large workload: GQA-8B, long context, prefix sharing with
copy-on-write (L2 flushed between iterations and not), the FP8 (E4M3) cache
on the three decode shapes, and chunked prefill.

``--kv-cache fp8`` runs a step on a cache of E4M3 codes (one byte per K/V
element, per-tensor scales): pa_reshape_and_cache_fp8 and pa_decode_fp8.
``--workload prefill_llama13b|prefill_gqa8b`` times a chunked-prefill step
(pa_reshape_and_cache of each sequence's 1024-token chunk, then the tcgen05
pa_prefill): ``value`` is causal attention TFLOP/s against the tensor-core
roofline. ``--impl reference`` times the fp64 CPU oracle on the host cores.
Under torchrun every rank runs its own replica of the workload (weak
scaling: sequences are independent, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_120_gb300 import workloads  # noqa: E402

NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20
METRIC = "paged-decode attention achieved HBM GB/s (% of GB300 peak); seq-steps/s"
PREFILL_METRIC = "paged chunked-prefill causal attention TFLOP/s"
# Launches per kernel in a per-launch timing block (each bracketed by events).
LAUNCHES = 200


# ------------------------------------------------------------ bytes of a step

def algorithmic_bytes(w, seq_lens, num_pairs: int, num_new_tokens: int, kv_elem: int = 2) -> dict:
    """Bytes a step must move at minimum: every valid K/V element once per kv
    head (padding slots of partial blocks not counted), Q, the output, block
    table entries and lengths; the new K/V rows read (16-bit) and written
    (kv_elem bytes per element); each COW pair's K and V block read and
    written. kv_elem is 2 for a 16-bit cache, 1 for an FP8 cache."""
    e = 2
    L = np.asarray(seq_lens, dtype=np.int64)
    S = len(L)
    kv = int((2 * L * w.num_kv_heads * w.head_size * kv_elem).sum())
    tables = int((4 * ((L + w.block_size - 1) // w.block_size)).sum())
    qo = 2 * S * w.num_q_heads * w.head_size * e
    decode = kv + qo + tables + 4 * S
    reshape = num_new_tokens * (2 * w.num_kv_heads * w.head_size * (e + kv_elem) + 4)
    copy = num_pairs * 2 * 2 * w.block_size * w.num_kv_heads * w.head_size * kv_elem + 8 * num_pairs
    return dict(decode=decode, kv=kv, reshape=reshape, copy=copy, step=decode + reshape + copy)


def unique_kv_bytes(w, seq_lens, block_tables, kv_elem: int = 2) -> int:
    """K/V bytes of the distinct physical blocks the tables reach, each block
    counted once with its largest valid-token count over the sequences that
    share it: what a decode launch must read from HBM at least when blocks
    are shared (the logical count re-reads shared blocks, which L2 serves)."""
    valid = {}
    B = w.block_size
    for s, L in enumerate(np.asarray(seq_lens, dtype=np.int64)):
        for j in range(int((L + B - 1) // B)):
            b = int(block_tables[s][j])
            valid[b] = max(valid.get(b, 0), int(min(B, L - j * B)))
    return int(sum(valid.values())) * 2 * w.num_kv_heads * w.head_size * kv_elem


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy-based)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (MEASURED_PEAKS.json absent)"


def measured_tensor_peak():
    """Sustained dense bf16 TFLOP/s (the prefill kernel runs inside long
    loops); fp16 runs at the same nominal rate."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured (MEASURED_PEAKS.json bf16_tflops_sustained, cuBLAS)"
    except Exception:
        return 1700.0, "fallback 1.7 PFLOP/s sustained (MEASURED_PEAKS.json absent)"


KERNEL_SOURCES = {
    "decode": ("pa_kernels.cu", "pa_device.cuh"),
    "decode_fp8": ("pa_kernels.cu", "pa_device.cuh"),
    "prefill": ("pa_prefill.cu", "pa_device.cuh"),
    "prefill_fp8": ("pa_prefill.cu", "pa_device.cuh"),
}


def kernel_source_hash(tag: str) -> str:
    """SHA-256 over the code of the CUDA sources a kernel family is built
    from, in order, comments and blank lines removed (a comment edit does not
    change the kernel that an ncu summary measured)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[tag]:
        with open(os.path.join(ROOT, "paged_kv_cache_120_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        code = "\n".join(line.rstrip() for line in src.splitlines() if line.strip())
        h.update(code.encode())
    return h.hexdigest()


def traffic_record(tag: str, workload: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    summary (profiles/<tag>_<workload>_traffic.txt), if the summary was taken
    on the current sources (their hash matches); else None."""
    path = os.path.join(ROOT, "profiles", f"{tag}_{workload}_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256") != kernel_source_hash(tag):
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling in the background for the whole run; summaries
    are taken over the windows in which GPU work was timed."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def close(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        try:
            os.unlink(self.file.name)
        except OSError:
            pass

    def _rows(self):
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts + frac, float(parts[2]), float(parts[3]), parts[6:10]))
                except Exception:
                    continue
        return rows

    def summary(self, t0: float, t1: float):
        """Median SM clock, max clock and active throttle reasons of the
        samples taken in [t0, t1] (all samples so far if none fell inside)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)   # let the sampler write the window's last line
        rows = self._rows()
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in use for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(inside),
                "window": ("timed steps, per-launch blocks and e2e steps" if inside
                           else "whole run (timed window too short to sample)")}


# --------------------------------------------------------------- distributed

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 0, 1
    import torch.distributed as dist
    backend = os.environ.get("BENCH_DIST_BACKEND", "nccl")
    dist.init_process_group(backend=backend)
    return dist.get_rank(), int(os.environ.get("LOCAL_RANK", "0")), dist.get_world_size()


def dist_max(value: float, world: int, device=None) -> float:
    """Max of a host float over ranks (the slowest rank's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# -------------------------------------------------------------- GPU timing

def gpu_lead(dev):
    """Keep the GPU busy for about a millisecond (a spin kernel, outside any
    timed interval) so that the host has enqueued the first timed launches
    before the start event is reached: the interval then holds device time
    only, not the host's first launch latency."""
    import torch
    torch.cuda._sleep(2_000_000)


def timed_steps(fn, K: int, world: int, dev) -> float:
    """Exactly K calls of fn between two events, bracketed by a barrier and a
    device synchronisation on both sides; milliseconds, max over ranks."""
    import torch
    stream = torch.cuda.current_stream(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world, dev)
    torch.cuda.synchronize(dev)
    gpu_lead(dev)
    start.record(stream)
    for _ in range(K):
        fn()
    end.record(stream)
    torch.cuda.synchronize(dev)
    dist_barrier(world, dev)
    return dist_max(start.elapsed_time(end), world, dev)


def per_launch(fn, n: int, world: int, dev, before=None) -> dict:
    """n calls of fn, each bracketed by its own pair of events (``before``,
    if given, runs outside the events ahead of each call). Returns the
    median, mean and spread in ms (median max over ranks)."""
    import torch
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    dist_barrier(world, dev)
    torch.cuda.synchronize(dev)
    gpu_lead(dev)
    for a, b in ev:
        if before is not None:
            before()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize(dev)
    dist_barrier(world, dev)
    ms = sorted(a.elapsed_time(b) for a, b in ev)
    q = lambda f: ms[min(len(ms) - 1, int(f * len(ms)))]
    return {"median_ms": dist_max(statistics.median(ms), world, dev), "mean_ms": statistics.mean(ms),
            "p10_ms": q(0.1), "p90_ms": q(0.9), "launches": n}


class L2Flush:
    """Writes a buffer twice the size of L2, evicting whatever the previous
    launch left there (a torch fill kernel, run outside the timed events)."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
        self.i = 0

    def __call__(self):
        self.i += 1
        self.buf.fill_(self.i)


def check_device_error(where: str):
    from paged_kv_cache_120_gb300 import binding
    err = binding.pa_get_device_error()
    if err:
        raise RuntimeError(f"device error word {err} set during {where}")


# ------------------------------------------------------------ oracle timing

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def pool_host_bits(t):
    """Host copy of a tensor's bits: uint16 patterns, or the E4M3 bytes."""
    import torch
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def compact_decode_inputs(w, plan, pool, query, cap_bytes: float, kv_elem: int) -> dict:
    """The oracle's host inputs for the first sequences of a batch (in order,
    until their K/V bytes reach cap_bytes): their blocks gathered into a
    small pool (shared blocks once), their tables renumbered into it, their
    queries. The oracle then walks exactly the blocks the GPU walks."""
    import torch
    B = w.block_size
    L = np.asarray(plan.seq_lens, dtype=np.int64)
    take, tot = [], 0
    for s in range(len(L)):
        take.append(s)
        tot += int(2 * L[s] * w.num_kv_heads * w.head_size * kv_elem)
        if tot >= cap_bytes:
            break
    nblk = [int((L[s] + B - 1) // B) for s in take]
    ids = np.concatenate([plan.block_tables[s, :n] for s, n in zip(take, nblk)]).astype(np.int64)
    uniq, inv = np.unique(ids, return_inverse=True)
    bt = np.full((len(take), max(1, max(nblk))), -1, dtype=np.int32)
    o = 0
    for i, n in enumerate(nblk):
        bt[i, :n] = inv[o:o + n]
        o += n
    idx = torch.from_numpy(uniq).to(pool.device)
    sub = pool.index_select(1, idx)
    sel = torch.tensor(take, dtype=torch.long, device=query.device)
    return {"pool": pool_host_bits(sub), "q": pool_host_bits(query.index_select(0, sel)), "bt": bt,
            "lens": L[take].astype(np.int32), "num_blocks": int(len(uniq)), "seqs": len(take),
            "seq_bytes": [algorithmic_bytes(w, [L[s]], 0, 0, kv_elem)["decode"] for s in take]}


def oracle_decode_rate(w, h, fp8: bool, budget_s: float, threads: int, batch: int, start: int = 0):
    """Time the oracle's decode on (sequence, q-head) rows of the compacted
    inputs h, ``batch`` rows per call, cycling through them, until about
    budget_s of wall time. A row is credited 1/Hq of its sequence's
    algorithmic bytes. Returns (seconds, bytes, rows, next start)."""
    import oracle
    oracle.set_threads(threads)
    Hq = w.num_q_heads
    P = h["seqs"] * Hq
    t, b, n, k = 0.0, 0.0, 0, start
    while t < budget_s:
        r = (np.arange(k, k + batch) % P)
        seqs, heads = (r // Hq).astype(np.int32), (r % Hq).astype(np.int32)
        t0 = time.perf_counter()
        if fp8:
            oracle.decode_fp8_sampled(seqs, heads, h["q"], h["pool"], h["bt"], h["lens"], w.scale, Hq,
                                      w.num_kv_heads, w.head_size, h["num_blocks"], w.block_size, w.dtype,
                                      workloads.FP8_K_SCALE, workloads.FP8_V_SCALE)
        else:
            oracle.decode_sampled(seqs, heads, h["q"], h["pool"], h["bt"], h["lens"], w.scale, Hq,
                                  w.num_kv_heads, w.head_size, h["num_blocks"], w.block_size, w.dtype)
        t += time.perf_counter() - t0
        b += sum(h["seq_bytes"][s] for s in seqs) / Hq
        n += batch
        k += batch
    return t, b, n, k


def decode_cpu_baseline(w, h, fp8: bool, budget_s: float) -> dict:
    """The oracle as it stands, on the machine's host cores: single-threaded and
    on every core (rows spread over OpenMP threads), GB/s of the metric."""
    import oracle
    cores = host_cores()
    t1, b1, n1, _ = oracle_decode_rate(w, h, fp8, budget_s / 2, 1, 1)
    tn, bn, nn, _ = oracle_decode_rate(w, h, fp8, budget_s / 2, cores, 4 * cores)
    oracle.set_threads(cores)
    what = (f"(sequence, q-head) rows of the first {h['seqs']} sequences of the same batch, "
            f"each credited 1/{w.num_q_heads} of its sequence's bytes")
    return {"value": bn / tn / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{nn} {what} ({tn:.1f} s on {cores} threads, fp64 C with OpenMP over rows)",
            "single_thread": {"value": b1 / t1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"{n1} rows ({t1:.1f} s)"},
            "host_cores": cores}


def prefill_rows_inputs(plan, pool, query) -> dict:
    """Host copies for the prefill oracle: the pool, the queries and, per
    chunk row, its sequence and number of visible tokens."""
    cu = plan.cu_seqlens_q
    rows = int(cu[-1])
    seq = (np.searchsorted(cu, np.arange(rows), side="right") - 1).astype(np.int64)
    vis = (plan.seq_lens[seq] - plan.chunk_lens[seq] + (np.arange(rows) - cu[seq]) + 1).astype(np.int32)
    return {"pool": pool_host_bits(pool), "q": pool_host_bits(query), "seq": seq, "vis": vis, "rows": rows}


def oracle_prefill_rate(w, plan, h, fp8_scales, budget_s: float, threads: int, batch: int, start: int = 0):
    """Time the oracle on prefill query rows (all heads of each row; a row is
    the decode definition over its visible tokens), ``batch`` rows per call,
    rows visited in a scattered fixed order. Returns (seconds, flops, rows,
    next start)."""
    import oracle
    oracle.set_threads(threads)
    Hq = w.num_q_heads
    t, fl, n, k = 0.0, 0, 0, start
    while t < budget_s:
        r = (np.arange(k, k + batch) * 7919) % h["rows"]
        bt = plan.block_tables[h["seq"][r]]
        vis = h["vis"][r]
        seqs = np.repeat(np.arange(batch, dtype=np.int32), Hq)
        heads = np.tile(np.arange(Hq, dtype=np.int32), batch)
        t0 = time.perf_counter()
        if fp8_scales is None:
            oracle.decode_sampled(seqs, heads, h["q"][r], h["pool"], bt, vis, w.scale, Hq, w.num_kv_heads,
                                  w.head_size, plan.num_blocks, w.block_size, w.dtype)
        else:
            oracle.decode_fp8_sampled(seqs, heads, h["q"][r], h["pool"], bt, vis, w.scale, Hq,
                                      w.num_kv_heads, w.head_size, plan.num_blocks, w.block_size, w.dtype,
                                      *fp8_scales)
        t += time.perf_counter() - t0
        fl += int(4 * w.head_size * Hq * vis.astype(np.int64).sum())
        n += batch
        k += batch
    return t, fl, n, k


def prefill_cpu_baseline(w, plan, h, fp8_scales, budget_s: float) -> dict:
    import oracle
    cores = host_cores()
    t1, f1, n1, _ = oracle_prefill_rate(w, plan, h, fp8_scales, budget_s / 2, 1, 1)
    tn, fn, nn, _ = oracle_prefill_rate(w, plan, h, fp8_scales, budget_s / 2, cores, cores)
    oracle.set_threads(cores)
    return {"value": fn / tn / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{nn} query rows x {w.num_q_heads} heads of the same batch ({tn:.1f} s on {cores} "
                      "threads, fp64 C with OpenMP over rows)",
            "single_thread": {"value": f1 / t1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                              "sample": f"{n1} rows ({t1:.1f} s)"},
            "host_cores": cores}


# -------------------------------------------------------------- configs

def workload_config(name, plan, kv_cache="16bit"):
    w = workloads.WORKLOADS[name]
    fp8 = kv_cache == "fp8"
    ab = algorithmic_bytes(w, plan.seq_lens, len(plan.cow_pairs), int((plan.slot_mapping >= 0).sum()),
                           1 if fp8 else 2)
    cache = (f"fp8 e4m3, k_scale {workloads.FP8_K_SCALE}, v_scale {workloads.FP8_V_SCALE}" if fp8
             else ("f16" if w.dtype == workloads.F16 else "bf16"))
    return {"workload": f"{name}: {w.description}" + (" [FP8 E4M3 cache]" if fp8 else ""),
            "kv_cache": cache, "num_seqs": int(len(plan.seq_lens)),
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_size": w.head_size,
            "block_size": w.block_size, "num_blocks": w.num_blocks,
            "mean_seq_len": float(np.mean(plan.seq_lens)), "cow_pairs": int(len(plan.cow_pairs)),
            "kv_bytes_per_step": ab["kv"], "step_bytes": ab["step"],
            "l2": ("inputs larger than L2: %.2f GB of K/V read per step vs 129 MB L2, no flush"
                   % (ab["kv"] / 1e9))}


def prefill_config(name, plan, kv_cache="16bit"):
    w = workloads.PREFILL_WORKLOADS[name]
    kvb = 2 * int(plan.seq_lens.sum()) * w.num_kv_heads * w.head_size * (1 if kv_cache == "fp8" else 2)
    return {"workload": f"{name}: {w.description}", "num_seqs": w.num_seqs,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_size": w.head_size,
            "block_size": w.block_size, "num_blocks": int(plan.num_blocks),
            "seq_lens": [int(x) for x in plan.seq_lens], "chunk": w.chunk,
            "kv_cache": "fp8_e4m3" if kv_cache == "fp8" else "16bit",
            "l2": "inputs larger than L2: %.0f MB of K/V read per step vs 129 MB L2, no flush" % (kvb / 1e6)}


def dtype_name(w) -> str:
    return "f16" if w.dtype == workloads.F16 else "bf16"


# ------------------------------------------------------------------ decode

def measure_decode(args, rank, world, dev, clocks, name, kv_cache="16bit", variant="literal",
                   cpu_budget=0.0, l2_variants=False) -> dict:
    """One decode workload: exactly args.steps timed steps, then per-launch
    blocks (the decode alone, the reshape alone, the decode right behind its
    reshape), then steps end to end from pinned host memory, then (rank 0)
    the oracle on the host cores. With l2_variants the steps and the decode
    are also timed with L2 flushed before every iteration."""
    import torch
    from paged_kv_cache_120_gb300 import step as stepmod
    w = workloads.WORKLOADS[name]
    seed = args.seed + 1000 * rank
    plan = stepmod.plan_step(name, seed, variant)
    pool, q, k, v = stepmod.make_device_inputs(name, plan, seed, dev, kv_cache)
    st = stepmod.DecodeStep(name, plan, pool, q, k, v, dev)
    kv_elem = 1 if st.fp8 else 2
    n_tokens = int((plan.slot_mapping >= 0).sum())
    ab = algorithmic_bytes(w, plan.seq_lens, len(plan.cow_pairs), n_tokens, kv_elem)
    kv_u = unique_kv_bytes(w, plan.seq_lens, plan.block_tables, kv_elem)
    roof_bytes = ab["decode"] - ab["kv"] + kv_u
    K = args.steps

    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize(dev)
    check_device_error("warm-up")

    def before_decode():
        if st.cow_pairs is not None:
            from paged_kv_cache_120_gb300 import binding
            binding.pa_copy_blocks([st.pool], st.cow_pairs)
        st.reshape()

    w0 = time.time()
    step_ms = timed_steps(st.run, K, world, dev) / K
    dec = per_launch(st.decode, LAUNCHES, world, dev)
    resh = per_launch(st.reshape, LAUNCHES, world, dev)
    in_step = per_launch(st.decode, 50, world, dev, before=before_decode)
    flushed = None
    if l2_variants:
        fl = L2Flush(dev)
        st_fl = per_launch(st.run, max(K, 50), world, dev, before=fl)
        dec_fl = per_launch(st.decode, LAUNCHES, world, dev, before=fl)
        del fl
        flushed = {"step_ms": st_fl["mean_ms"], "steps": st_fl["launches"],
                   "value": world * ab["step"] / (st_fl["mean_ms"] / 1e3) / 1e9,
                   "decode_only": dict(dec_fl, gbs=ab["decode"] / (dec_fl["median_ms"] / 1e3) / 1e9),
                   "roofline_achieved_gbs": roof_bytes / (dec_fl["median_ms"] / 1e3) / 1e9}
    torch.cuda.synchronize(dev)
    check_device_error("the timed region")

    # End to end through the public step API from pinned host memory: every
    # step copies all of its inputs (one packed buffer) to the device, runs
    # the libpa calls and reads the output back before the next step starts.
    host = st.pin_host()
    out_host = host.pop("out")
    h2d = st.pinned_bytes()
    d2h = out_host.numel() * out_host.element_size()
    for _ in range(3):
        st.run_pinned()
    dist_barrier(world, dev)
    torch.cuda.synchronize(dev)
    ke = max(1, min(K, 200))
    t0 = time.perf_counter()
    for _ in range(ke):
        st.run_pinned()
    e2e_s = dist_max(time.perf_counter() - t0, world, dev)
    w1 = time.time()
    dist_barrier(world, dev)
    if rank != 0:
        return {}

    peak, peak_note = measured_peak()
    dec_ms = dec["median_ms"]
    achieved = roof_bytes / (dec_ms / 1e3) / 1e9
    value = world * ab["step"] / (step_ms / 1e3) / 1e9
    tag = "decode_fp8" if st.fp8 else "decode"
    rec = {
        "value": value, "unit": "GB/s", "steps": K, "ms_per_step": step_ms,
        "dtype": dtype_name(w),
        "config": workload_config(name, plan, kv_cache),
        "seq_steps_per_s": world * len(plan.seq_lens) / (step_ms / 1e3),
        "pct_of_nominal_8TBps": 100.0 * value / NOMINAL_HBM_GBS,
        "pct_of_measured_peak": 100.0 * value / peak,
        "decode_only": dict(dec, gbs=ab["decode"] / (dec_ms / 1e3) / 1e9,
                            pct_of_nominal_8TBps=100.0 * ab["decode"] / (dec_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                            seq_steps_per_s=len(plan.seq_lens) / (dec_ms / 1e3)),
        "reshape_only": resh,
        "decode_in_step": dict(in_step, note="decode launches each bracketed right behind this step's "
                                             "reshape: the event between them stops the decode's prologue "
                                             "from overlapping the reshape"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic_record(tag, name + ("_fork" if variant == "fork" else "")),
                     "kernel": ("pa_decode_fp8" if st.fp8 else "pa_decode")
                               + " (paged_decode_kernel + paged_decode_reduce_kernel)",
                     "duration": f"median of {dec['launches']} back-to-back launches, CUDA events",
                     "peak_source": peak_note, "bytes_per_launch": roof_bytes,
                     "bytes_basis": ("unique physical blocks (shared blocks once); logical "
                                     f"{ab['decode']} B per launch") if kv_u < ab["kv"] else "logical = unique"},
        "kv_l2_policy": "normal (blocks shared)" if st.flags & 1 else "evict-first (no block shared)",
        "e2e": {"value": world * ab["step"] * ke / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3 / ke,
                "steps": ke},
        "gpu_launches": st.launches_per_step() * K,
        "clocks": clocks.summary(w0, w1) if clocks else None,
    }
    if flushed is not None:
        rec["config"]["l2"] = ("unflushed: the shared prompt's K/V (64 MB) stay in L2 across steps; "
                               "see l2_flushed for the same step with L2 flushed before every iteration")
        rec["l2_flushed"] = dict(flushed, note="a 258 MB buffer written before every iteration, outside the events")
    if cpu_budget > 0:
        h = compact_decode_inputs(w, plan, st.pool, st.query, 1.0e9, kv_elem)
        rec["cpu_baseline"] = decode_cpu_baseline(w, h, st.fp8, cpu_budget)
    return rec


# ----------------------------------------------------------------- prefill

def measure_prefill(args, rank, world, dev, clocks, name, kv_cache="16bit", cpu_budget=0.0) -> dict:
    """One chunked-prefill workload: exactly args.steps timed steps
    (reshape + prefill), a per-launch block of the prefill alone, steps end
    to end from pinned host memory, then (rank 0) the oracle."""
    import torch
    from paged_kv_cache_120_gb300 import step as stepmod
    w = workloads.PREFILL_WORKLOADS[name]
    seed = args.seed + 1000 * rank
    plan = stepmod.plan_prefill(name, seed)
    st = stepmod.PrefillStep(name, plan, seed, dev, kv_cache)
    flops = stepmod.prefill_flops(plan, w.num_q_heads, w.head_size)
    K = args.steps
    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize(dev)
    check_device_error("warm-up")
    w0 = time.time()
    step_ms = timed_steps(st.run, K, world, dev) / K
    pre = per_launch(st.prefill, LAUNCHES, world, dev)
    whole = None
    if st.workspace is not None:
        # Few work units: the step splits K/V ranges across the SMs. The same
        # launches with each unit's range whole, for comparison.
        ws, st.workspace = st.workspace, None
        whole = per_launch(st.prefill, LAUNCHES, world, dev)
        st.workspace = ws
    torch.cuda.synchronize(dev)
    check_device_error("the timed region")
    host = st.pin_host()
    out_host = host.pop("out")
    h2d = st.pinned_bytes()
    d2h = out_host.numel() * out_host.element_size()
    for _ in range(3):
        st.run_pinned()
    dist_barrier(world, dev)
    torch.cuda.synchronize(dev)
    ke = max(1, min(K, 200))
    t0 = time.perf_counter()
    for _ in range(ke):
        st.run_pinned()
    e2e_s = dist_max(time.perf_counter() - t0, world, dev)
    w1 = time.time()
    dist_barrier(world, dev)
    if rank != 0:
        return {}
    peak, peak_note = measured_tensor_peak()
    achieved = flops / (pre["median_ms"] / 1e3) / 1e12
    value = world * flops / (step_ms / 1e3) / 1e12
    tag = "prefill_fp8" if st.fp8 else "prefill"
    rec = {
        "value": value, "unit": "TFLOP/s", "steps": K, "ms_per_step": step_ms, "dtype": dtype_name(w),
        "config": prefill_config(name, plan, kv_cache),
        "tokens_per_s": world * int(plan.cu_seqlens_q[-1]) / (step_ms / 1e3),
        "prefill_only": dict(pre, tflops=achieved),
        "kv_split": None if whole is None else {
            "whole_units": dict(whole, tflops=flops / (whole["median_ms"] / 1e3) / 1e12),
            "speedup": whole["median_ms"] / pre["median_ms"],
            "workspace_bytes": st.workspace.numel()},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic_record(tag, name[len("prefill_"):]),
                     "kernel": ("pa_prefill_fp8" if st.fp8 else "pa_prefill") + " (paged_prefill_kernel)",
                     "duration": f"median of {pre['launches']} back-to-back launches, CUDA events",
                     "peak_source": peak_note, "flops_per_launch": flops},
        "e2e": {"value": world * flops * ke / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3 / ke,
                "steps": ke},
        "gpu_launches": st.launches_per_step() * K,
        "clocks": clocks.summary(w0, w1) if clocks else None,
    }
    if cpu_budget > 0:
        h = prefill_rows_inputs(plan, st.pool, st.query)
        rec["cpu_baseline"] = prefill_cpu_baseline(w, plan, h, (st.k_scale, st.v_scale) if st.fp8 else None,
                                                   cpu_budget)
    return rec


# The default run's other workloads: (key, kind, workload, cache, variant, L2 variants).
EXTRA_CONFIGS = (
    ("gqa8b", "decode", "gqa8b", "16bit", "literal", False),
    ("longctx", "decode", "longctx", "16bit", "literal", False),
    ("prefix_cow", "decode", "prefix_cow", "16bit", "literal", True),
    ("prefix_cow_fork", "decode", "prefix_cow", "16bit", "fork", True),
    ("llama13b_fp8", "decode", "llama13b", "fp8", "literal", False),
    ("gqa8b_fp8", "decode", "gqa8b", "fp8", "literal", False),
    ("longctx_fp8", "decode", "longctx", "fp8", "literal", False),
    ("prefill_llama13b", "prefill", "prefill_llama13b", "16bit", None, False),
    ("prefill_gqa8b", "prefill", "prefill_gqa8b", "16bit", None, False),
    ("prefill_llama13b_fp8", "prefill", "prefill_llama13b", "fp8", None, False),
    ("prefill_gqa8b_fp8", "prefill", "prefill_gqa8b", "fp8", None, False),
    ("prefill_longctx_llama13b", "prefill", "prefill_longctx_llama13b", "16bit", None, False),
    ("prefill_longctx_gqa8b", "prefill", "prefill_longctx_gqa8b", "16bit", None, False),
)


def top_line(rec: dict, args, world, metric, data) -> dict:
    """The contract's JSON line around a measured record."""
    line = {"metric": metric, "value": rec["value"], "unit": rec["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": rec["dtype"],
            "data": data, "config": rec["config"]}
    for k, v in rec.items():
        if k not in line and k not in ("steps",):
            line[k] = v
    return line


def run_ours(args, rank, local_rank, world):
    import torch
    from paged_kv_cache_120_gb300 import build
    build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    clocks = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    try:
        if args.layers > 1:
            from paged_kv_cache_120_gb300 import step as stepmod
            plan = stepmod.plan_step(args.workload, args.seed + 1000 * rank, args.variant)
            return run_model_step(args, rank, world, dev, clocks, args.workload, plan, args.seed + 1000 * rank)
        prefill = args.workload in workloads.PREFILL_WORKLOADS
        if prefill:
            rec = measure_prefill(args, rank, world, dev, clocks, args.workload, args.kv_cache, args.cpu_budget)
            metric, data = PREFILL_METRIC, "synthetic (seeded N(0,1) values, seeded block placement)"
        else:
            rec = measure_decode(args, rank, world, dev, clocks, args.workload, args.kv_cache, args.variant,
                                 args.cpu_budget, l2_variants=args.workload == "prefix_cow")
            metric, data = METRIC, "synthetic (seeded N(0,1) values, seeded block placement)"
        configs = {}
        default_run = (args.workload == "llama13b" and args.kv_cache == "16bit" and args.variant == "literal"
                       and not args.no_configs)
        if default_run:
            for key, kind, name, kv, variant, l2v in EXTRA_CONFIGS:
                torch.cuda.empty_cache()
                budget = args.cpu_budget * 0.4
                if kind == "decode":
                    configs[key] = measure_decode(args, rank, world, dev, clocks, name, kv, variant, budget, l2v)
                else:
                    configs[key] = measure_prefill(args, rank, world, dev, clocks, name, kv, budget)
        if rank == 0:
            line = top_line(rec, args, world, metric, data)
            if configs:
                line["configs"] = configs
            print(json.dumps(line), flush=True)
    finally:
        if clocks:
            clocks.close()


# ------------------------------------------------------------- model step

def run_model_step(args, rank, world, dev, clocks, name, plan, seed):
    """A decode step of a whole model: COW copies in every layer pool (one
    pa_copy_blocks call), then reshape_and_cache + decode for each of
    args.layers layers, eagerly or replayed from a CUDA graph (--graph)."""
    import torch
    from paged_kv_cache_120_gb300 import step as stepmod
    w = workloads.WORKLOADS[name]
    ms = stepmod.ModelStep(name, plan, args.layers, seed, dev, args.kv_cache)
    fp8 = ms.layers[0].fp8
    n_tokens = int((plan.slot_mapping >= 0).sum())
    ab = algorithmic_bytes(w, plan.seq_lens, len(plan.cow_pairs), n_tokens, 1 if fp8 else 2)
    step_bytes = args.layers * ab["step"]
    for _ in range(args.warmup):
        ms.run()
    if args.graph:
        ms.capture()
        for _ in range(3):
            ms.run()
    torch.cuda.synchronize(dev)
    check_device_error("warm-up")
    K = args.steps
    w0 = time.time()
    t_s = timed_steps(ms.run, K, world, dev) / 1e3
    w1 = time.time()
    check_device_error("the timed region")
    if rank != 0:
        return
    peak, peak_note = measured_peak()
    kv_u = unique_kv_bytes(w, plan.seq_lens, plan.block_tables, 1 if fp8 else 2)
    roof_bytes = args.layers * (ab["step"] - ab["kv"] + kv_u)
    achieved = roof_bytes / (t_s / K) / 1e9
    copy_bytes = args.layers * ab["copy"]
    line = {
        "metric": METRIC, "value": world * step_bytes * K / t_s / 1e9, "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": t_s * 1e3 / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_name(w),
        "data": "synthetic (seeded N(0,1) values per layer, seeded block placement)",
        "config": dict(workload_config(name, plan, args.kv_cache), layers=args.layers,
                       launch="CUDA graph replay" if args.graph else "eager",
                       cow_bytes_per_step=copy_bytes,
                       complete_block_bytes=2 * args.layers * w.block_size * w.num_kv_heads * w.head_size
                       * (1 if fp8 else 2)),
        "seq_steps_per_s": world * len(plan.seq_lens) * K / t_s,
        "ms_per_layer": t_s * 1e3 / K / args.layers,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "whole model step (copy_blocks + per-layer reshape and decode)",
                     "peak_source": peak_note, "bytes_per_step": roof_bytes,
                     "bytes_basis": ("unique physical blocks (shared blocks once); logical "
                                     f"{step_bytes} B per step") if kv_u < ab["kv"] else "logical = unique"},
        "gpu_launches": ms.launches_per_step() * K,
        "clocks": clocks.summary(w0, w1) if clocks else None,
    }
    print(json.dumps(line), flush=True)


def run_prefix_cache(args, rank, local_rank, world):
    """A serving wave per step: SHARED_PROMPT["requests"] requests with a common
    system prompt and private suffixes arrive; the prefix cache hands out
    tables (cached system blocks shared), only uncached tokens are written
    (pa_reshape_and_cache) and prefilled (pa_prefill); the requests are then
    freed (their blocks stay cached). --no-prefix-cache computes every
    prompt in full. Host bookkeeping and device time are reported apart."""
    import torch
    from paged_kv_cache_120_gb300 import binding, build
    build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = workloads.SHARED_PROMPT
    R, B, D = cfg["requests"], cfg["block_size"], cfg["head_size"]
    Hq, Hkv, dt = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["dtype"]
    system, g = workloads.shared_prompt_tokens(args.seed + 1000 * rank)
    max_tok = R * (cfg["system"] + cfg["suffix_hi"])
    nb = 4 * (max_tok // B + R) + 1
    pool = workloads.normal_values((2, nb, B, Hkv, D), dt, 51, dev)
    q = workloads.normal_values((max_tok, Hq, D), dt, 52, dev)
    k = workloads.normal_values((max_tok, Hkv, D), dt, 53, dev)
    v = workloads.normal_values((max_tok, Hkv, D), dt, 54, dev)
    out = torch.empty_like(q)
    use_cache = not args.no_prefix_cache
    pc = binding.PrefixCache(nb, B)
    flags = 0 if use_cache else binding.PA_PCACHE_NO_CACHE
    maxb = (cfg["system"] + cfg["suffix_hi"] + B - 1) // B
    # The admission writes the wave's device inputs into one pinned staging
    # buffer (cu_seqlens_q, seq_lens, slot_mapping, block tables), moved to
    # the device with one copy into views of the same layout.
    parts = (("cu_seqlens_q", R + 1), ("seq_lens", R), ("slot_mapping", max_tok), ("block_tables", R * maxb))
    stage = torch.empty(sum(n for _, n in parts), dtype=torch.int32).pin_memory()
    d_stage = torch.empty(stage.numel(), dtype=torch.int32, device=dev)
    host = {"seq_ids": torch.empty(R, dtype=torch.int32), "num_cached": torch.empty(R, dtype=torch.int32)}
    dview, off = {}, 0
    for name, n in parts:
        host[name], dview[name] = stage[off:off + n], d_stage[off:off + n]
        off += n
    d_cu, d_sl, d_slots = dview["cu_seqlens_q"], dview["seq_lens"], dview["slot_mapping"]
    d_bt = dview["block_tables"].view(R, maxb)
    copied = torch.cuda.Event()
    copied.record()
    scale = D ** -0.5
    stream = torch.cuda.current_stream(dev)
    events = None

    def wave(w, times):
        """One wave (tokens, cu_tokens, prompt tokens); returns (tokens computed, cached tokens per
        request, new tokens per request)."""
        tokens, cu_tokens, served = w
        copied.synchronize()        # the previous wave's pinned inputs are on the device
        t0 = time.perf_counter()
        count, _ = pc.admit(tokens, cu_tokens, maxb, flags, host)
        if count != R:
            raise RuntimeError(f"pool admitted {count} of {R} requests")
        cu = host["cu_seqlens_q"].numpy()
        news = int(cu[R])
        t1 = time.perf_counter()
        d_stage.copy_(stage, non_blocking=True)
        copied.record()
        binding.pa_reshape_and_cache(k[:news], v[:news], pool, d_slots[:news])
        if events is not None:
            events.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
            events[-1][0].record(stream)
        binding.pa_prefill(out[:news], q[:news], pool, d_bt, d_cu, d_sl, scale, int(np.diff(cu).max()))
        if events is not None:
            events[-1][1].record(stream)
        t2 = time.perf_counter()
        pc.free_seqs(host["seq_ids"])
        times[0] += (t1 - t0) + (time.perf_counter() - t2)
        return news, host["num_cached"].numpy().copy(), np.diff(cu)

    def prompts_for_wave():
        prompts = [np.concatenate([system, g.integers(0, cfg["vocab"], size=int(g.integers(
            cfg["suffix_lo"], cfg["suffix_hi"] + 1)))]).astype(np.int32) for _ in range(R)]
        cu_tokens = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
        return np.concatenate(prompts), cu_tokens, int(cu_tokens[-1])

    # 64 distinct waves, cycled: a wave's private blocks are long evicted
    # (about 20 waves of allocation refill the pool) before it comes round again
    waves = [prompts_for_wave() for _ in range(64)]
    def wave_flops(hits, n_new):
        hits, n_new = hits.astype(np.int64), n_new.astype(np.int64)
        return int((4 * D * Hq * ((2 * hits + 1 + n_new) * n_new // 2)).sum())

    host_s = [0.0]
    for i in range(args.warmup):
        wave(waves[i % len(waves)], host_s)
    torch.cuda.synchronize(dev)
    if binding.pa_get_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")
    host_s = [0.0]
    K = args.steps
    clocks = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    w0 = time.time()
    dist_barrier(world, dev)
    torch.cuda.synchronize(dev)
    computed = served = 0
    events, counts = [], []
    t0 = time.perf_counter()
    for i in range(K):
        w = waves[(args.warmup + i) % len(waves)]
        a, hits, n_new = wave(w, host_s)
        computed, served = computed + a, served + w[2]
        counts.append((hits, n_new))
    torch.cuda.synchronize(dev)
    t_s = dist_max(time.perf_counter() - t0, world, dev)
    flops = sum(wave_flops(h, n) for h, n in counts)
    dist_barrier(world, dev)
    w1 = time.time()
    if binding.pa_get_device_error():
        raise RuntimeError("device error word set during the timed region")
    if clocks:
        summary = clocks.summary(w0, w1)
        clocks.close()
    if rank != 0:
        return
    pre_ms = sum(a.elapsed_time(b) for a, b in events) / K
    achieved = flops / K / (pre_ms * 1e-3) / 1e12
    peak, peak_note = measured_tensor_peak()
    cpu = prefix_wave_cpu_baseline(args, cfg, waves, host, pool, q, maxb, scale)
    line = {
        "metric": "prefix-cache serving wave: prompt tokens served/s", "value": world * served / t_s,
        "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": t_s * 1e3 / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic (seeded token ids and N(0,1) values)",
        "config": {"workload": f"prefix-cache serving wave: {R} requests, {cfg['system']}-token system prompt "
                               f"+ suffix U[{cfg['suffix_lo']},{cfg['suffix_hi']}], 40/40 heads, d=128, fp16",
                   "prefix_cache": use_cache, "num_blocks": nb, "waves": len(waves),
                   "l2": "the shared prompt K/V (21 MB) is re-read by every request and may stay in L2; no flush"},
        "computed_tokens_per_s": world * computed / t_s,
        "computed_fraction": computed / served,
        "host_bookkeeping_us_per_request": 1e6 * host_s[0] / (K * R),
        "prefill_tflops_per_s": world * flops / t_s / 1e12,
        "prefill_only": {"ms_per_wave": pre_ms, "tflops": achieved},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None, "kernel": "pa_prefill (paged_prefill_kernel)",
                     "peak_source": peak_note, "flops_per_launch": flops / K},
        "cpu_baseline": cpu,
        "gpu_launches": 2 * K,
        "clocks": summary,
    }
    print(json.dumps(line), flush=True)


def prefix_wave_cpu_baseline(args, cfg, waves, host, pool, q, maxb, scale):
    """The oracle on the serving wave: the prefix-cache pool model admits and
    frees whole waves (timed), and the attention oracle runs query rows of the
    last timed wave (all heads of one row at a time) for the rest of the
    budget; a wave's CPU time = its admission time + its causal flops at the
    oracle's measured flop rate."""
    import torch
    import oracle
    from oracle.prefix_cache import PrefixCacheModel
    R, B = cfg["requests"], cfg["block_size"]
    Hq, Hkv, D = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_size"]
    budget = args.cpu_budget
    m = PrefixCacheModel(pool.shape[1], B)
    t_adm, n_adm, i = 0.0, 0, 0
    while (t_adm < budget / 3 or n_adm < 2) and n_adm < len(waves):
        tokens, cu_tokens, _ = waves[i % len(waves)]
        t0 = time.perf_counter()
        ids = [m.add_seq(tokens[cu_tokens[r]:cu_tokens[r + 1]],
                         cache=not args.no_prefix_cache)[0] for r in range(R)]
        for sid in ids:
            m.free_seq(sid)
        dt = time.perf_counter() - t0
        if i > 0:              # the first wave fills the cache
            t_adm, n_adm = t_adm + dt, n_adm + 1
        i += 1
    pool_bits = pool.view(torch.int16).cpu().numpy().view(np.uint16)
    q_bits = q.view(torch.int16).cpu().numpy().view(np.uint16)
    cu = host["cu_seqlens_q"].numpy().copy()
    sl = host["seq_lens"].numpy().copy()
    bt = host["block_tables"].numpy().reshape(R, maxb).copy()
    heads = np.arange(Hq, dtype=np.int32)
    cores = host_cores()
    oracle.set_threads(cores)
    rows = int(cu[R])
    t_att, fl, n, k = 0.0, 0, 0, 0
    while t_att < budget * 2 / 3 and n < rows:
        row = (k * 7919) % rows
        s = int(np.searchsorted(cu, row, side="right") - 1)
        vis = int(sl[s]) - int(cu[s + 1] - cu[s]) + (row - int(cu[s])) + 1
        t0 = time.perf_counter()
        oracle.decode_sampled(np.zeros(Hq, np.int32), heads, q_bits[row:row + 1], pool_bits, bt[s:s + 1],
                              np.array([vis], np.int32), scale, Hq, Hkv, D, pool.shape[1], B, cfg["dtype"])
        t_att += time.perf_counter() - t0
        fl += 4 * D * Hq * vis
        n, k = n + 1, k + 1
    # causal flops of the average timed wave, from the last wave's admission
    hits = host["num_cached"].numpy().astype(np.int64)
    n_new = np.diff(cu).astype(np.int64)
    last_flops = float((4 * D * Hq * ((2 * hits + 1 + n_new) * n_new // 2)).sum())
    served = float(sl.astype(np.int64).sum())
    wave_s = t_adm / n_adm + last_flops / (fl / t_att)
    return {"value": served / wave_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"pool model (one thread) over {n_adm} whole waves ({1e3 * t_adm / n_adm:.1f} ms/wave) + "
                      f"attention oracle (heads of a row over {cores} threads) on {n} query rows of the last "
                      f"wave x {Hq} heads ({fl / t_att / 1e9:.2f} GFLOP/s), scaled to that wave's "
                      f"{last_flops / 1e9:.1f} GFLOP"}


# ---------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle on the host cores (every core,
    rows over OpenMP threads), each step a bounded sample of the workload."""
    if rank != 0:
        return
    import torch
    from paged_kv_cache_120_gb300 import step as stepmod
    name = args.workload
    per_step = max(0.05, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    dev = torch.device("cuda:0") if torch.cuda.is_available() else torch.device("cpu")
    cores = host_cores()
    if name in workloads.PREFILL_WORKLOADS:
        w = workloads.PREFILL_WORKLOADS[name]
        plan = stepmod.plan_prefill(name, args.seed)
        st = stepmod.PrefillStep(name, plan, args.seed, dev, args.kv_cache)
        h = prefill_rows_inputs(plan, st.pool, st.query)
        scales = (st.k_scale, st.v_scale) if st.fp8 else None
        del st
        rate = lambda b, k: oracle_prefill_rate(w, plan, h, scales, b, cores, cores, k)
        metric, unit, scale_unit = PREFILL_METRIC, "TFLOP/s", 1e12
        config = prefill_config(name, plan, args.kv_cache)
        what = f"query rows x {w.num_q_heads} heads of the {name} batch"
    else:
        w = workloads.WORKLOADS[name]
        plan = stepmod.plan_step(name, args.seed, args.variant)
        pool, q, _, _ = stepmod.make_device_inputs(name, plan, args.seed, dev, args.kv_cache)
        fp8 = args.kv_cache == "fp8"
        h = compact_decode_inputs(w, plan, pool, q, 1.0e9, 1 if fp8 else 2)
        del pool, q
        rate = lambda b, k: oracle_decode_rate(w, h, fp8, b, cores, 4 * cores, k)
        metric, unit, scale_unit = METRIC, "GB/s", 1e9
        config = workload_config(name, plan, args.kv_cache)
        what = (f"(sequence, q-head) rows of the first {h['seqs']} sequences of the {name} batch, each "
                f"credited 1/{w.num_q_heads} of its sequence's bytes")
    nxt = 0
    for _ in range(args.warmup):
        _, _, _, nxt = rate(per_step, nxt)
    tot_t, tot_x, tot_n = 0.0, 0.0, 0
    for _ in range(args.steps):
        t, x, n, nxt = rate(per_step, nxt)
        tot_t, tot_x, tot_n = tot_t + t, tot_x + x, tot_n + n
    v = tot_x / tot_t / scale_unit
    sample = (f"{tot_n} {what}, about {per_step:.2f} s per step on {cores} threads "
              "(fp64 C, OpenMP over rows)")
    line = {"impl": "reference", "metric": metric, "value": v, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": config,
            "cpu_baseline": {"value": v, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# (q heads, kv heads, dtype, context of each sequence, chunk of each sequence)
SPLIT_SWEEP = (
    [(40, 40, workloads.F16, [8192 + 37 * i for i in range(n)], [512] * n) for n in (1, 2, 3, 4, 6)]
    + [(32, 8, workloads.BF16, [16384 + 101 * i for i in range(n)], [1024] * n) for n in (1, 2)]
    + [(32, 8, workloads.BF16, [32768], [64]), (8, 1, workloads.F16, [32768], [256]),
       (16, 1, workloads.F16, [65536], [16])])


def run_split_sweep(args, rank) -> None:
    """pa_prefill kernel time with each work unit's K/V range whole (no
    workspace) and split across the SMs (workspace), over shapes from many
    to very few units (head size 128, 16-token blocks, seeded placement and
    N(0,1) values): 10 launches replayed from a CUDA graph, median of 7
    replays. One JSON line per shape."""
    import torch
    from paged_kv_cache_120_gb300 import binding, build
    if rank != 0:
        return
    build.build()
    dev = torch.device("cuda:0")
    D, B = 128, 16

    def graph_us(call):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(3):
                call(s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            for _ in range(10):
                call(s)
        ts = []
        for _ in range(7):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 10 * 1e3)
        return sorted(ts)[3]

    for k, (hq, hkv, dt, ctx, ql) in enumerate(SPLIT_SWEEP):
        rng = np.random.default_rng(args.seed + k)
        nblk = [-(-L // B) for L in ctx]
        nb = sum(nblk) + 4
        perm = rng.permutation(nb).astype(np.int32)
        bt = np.full((len(ctx), max(nblk)), -1, np.int32)
        o = 0
        for i, n in enumerate(nblk):
            bt[i, :n] = perm[o:o + n]
            o += n
        cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
        pool = workloads.normal_values((2, nb, B, hkv, D), dt, args.seed + 100 + k, dev)
        q = workloads.normal_values((int(cu[-1]), hq, D), dt, args.seed + 200 + k, dev)
        out = torch.empty_like(q)
        t = lambda a: torch.from_numpy(a).to(dev)
        bt_d, cu_d, sl_d = t(bt), t(cu), t(np.array(ctx, np.int32))
        ws = binding.prefill_workspace(q, pool, len(ctx), max(ql))
        run = lambda w: (lambda s: binding.pa_prefill(out, q, pool, bt_d, cu_d, sl_d, D ** -0.5, max(ql), w, s))
        whole = graph_us(run(None))
        split = graph_us(run(ws)) if ws is not None else None
        check_device_error("the split sweep")
        group = hq // hkv
        hpc = min(group, 16)
        rows = (128 // hpc) & ~7
        units = (-(-(-(-max(ql) // rows)) // 2)) * len(ctx) * hkv * (group // hpc)
        print(json.dumps({"heads": f"{hq}/{hkv}", "contexts": ctx, "chunks": ql, "units": units,
                          "whole_us": round(whole, 1), "split_us": None if split is None else round(split, 1),
                          "speedup": None if split is None else round(whole / split, 3)}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama13b",
                    choices=sorted(workloads.WORKLOADS) + sorted(workloads.PREFILL_WORKLOADS)
                    + ["prefix_cache_prefill"])
    ap.add_argument("--no-prefix-cache", action="store_true",
                    help="prefix_cache_prefill: compute every prompt in full")
    ap.add_argument("--variant", default="literal", choices=["literal", "fork"])
    ap.add_argument("--kv-cache", default="16bit", choices=["16bit", "fp8"],
                    help="cache element type: the workload's 16-bit type, or E4M3 codes")
    ap.add_argument("--layers", type=int, default=1,
                    help="decode workloads: layers per model step (one pool per layer)")
    ap.add_argument("--graph", action="store_true",
                    help="with --layers: replay the model step from a CUDA graph")
    ap.add_argument("--no-configs", action="store_true",
                    help="default workload: skip the records of the other workloads")
    ap.add_argument("--pool-blocks", type=int, default=0,
                    help="decode workloads: pool of this many blocks instead of the workload's (the same "
                         "sequences and lengths, placement drawn from fewer blocks): small profiling cases")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--split-sweep", action="store_true",
                    help="print pa_prefill kernel times with K/V ranges whole and split over a range of "
                         "unit counts, then exit")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for the main cpu_baseline (0.4x for each other config)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.pool_blocks > 0 and args.workload in workloads.WORKLOADS:
        import dataclasses
        w = workloads.WORKLOADS[args.workload]
        workloads.WORKLOADS[args.workload] = dataclasses.replace(w, num_blocks=args.pool_blocks)
        args.no_configs = True
    rank, local_rank, world = dist_setup()
    if args.split_sweep:
        run_split_sweep(args, rank)
    elif args.workload == "prefix_cache_prefill":
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the prefix-cache wave is host "
                                  "bookkeeping plus pa_prefill; its oracle arm is the prefill one"}))
        else:
            run_prefix_cache(args, rank, local_rank, world)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local_rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
