"""Seeded synthetic inputs for the five PagedAttention decode workloads.

This module serves both the CUDA path and the oracle, so it holds none of the
method's arithmetic: no block counts, no slots, no attention. It only fixes
shapes, draws sequence lengths from the stated distributions, draws the
physical-block free-list order, and draws N(0, 1) values (and, for the FP8
cache variant, E4M3 codes of N(0, 1) draws rounded by PyTorch's cast).

Workloads (shapes follow the PagedAttention pages: the Llama-2-13B shape of
the vLLM book chapter "第4章 PagedAttention：虚拟内存的启示" §4.1.1/§4.3.1;
the 64-block worked example of "PagedAttention: virtual memory for the KV
cache", section "具体实例演示"):

  toy          64 blocks x 16, lengths 25/47/12 placed at [3,7], [0,5,9], [4],
               4 q heads = 4 kv heads, head_dim 64, fp16, scale 1/8
  llama13b     40 q = 40 kv heads, head_dim 128, fp16, 64 seqs,
               lengths uniform in [1, 2048], 9000-block pool
  gqa8b        32 q over 8 kv heads, head_dim 128, bf16, 256 seqs,
               lengths lognormal (median 800, sigma 1.0) clipped to [16, 8192],
               160000-block pool
  longctx      64 q over 8 kv heads, head_dim 128, bf16, 8 seqs,
               lengths uniform in [32768, 131072], 70000-block pool
  prefix_cow   16 groups x 8 seqs sharing a 1024-token prompt, private tails
               uniform in [1, 512], 32 q over 8 kv heads, head_dim 128, fp16,
               16384-block pool; the fork variant adds 1..15 prompt tokens per
               group so the last prompt block is shared and partly filled.

Sequence lengths are the lengths the decode step sees (the step's own new
token included), except for the toy, whose 25/47/12 are the lengths before
its first step (the worked example's numbers).
"""
from __future__ import annotations

import dataclasses

import numpy as np

F16 = 0
BF16 = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_blocks: int
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    dtype: int
    num_seqs: int
    scale: float
    description: str


WORKLOADS = {
    "toy": Workload("toy", 64, 16, 4, 4, 64, F16, 3, 1.0 / 8.0,
                    "worked example: 64 blocks x 16, lengths 25/47/12, 4/4 heads, d=64, fp16"),
    "llama13b": Workload("llama13b", 9000, 16, 40, 40, 128, F16, 64, 128 ** -0.5,
                         "Llama-2-13B layer: 40/40 heads, d=128, fp16, 64 seqs, L~U[1,2048]"),
    "gqa8b": Workload("gqa8b", 160000, 16, 32, 8, 128, BF16, 256, 128 ** -0.5,
                      "GQA 8B: 32/8 heads, d=128, bf16, 256 seqs, L~lognormal(800,1) in [16,8192]"),
    "longctx": Workload("longctx", 70000, 16, 64, 8, 128, BF16, 8, 128 ** -0.5,
                        "long context split-K: 64/8 heads, d=128, bf16, 8 seqs, L~U[32768,131072]"),
    "prefix_cow": Workload("prefix_cow", 16384, 16, 32, 8, 128, F16, 128, 128 ** -0.5,
                           "prefix sharing + COW: 16x8 seqs, 1024-token shared prompt, tails U[1,512]"),
}

# Chunked-prefill workloads (many queries per sequence, causal): each
# sequence holds a cached prefix of U[min_prefix, max_prefix] tokens and this
# step brings a chunk of `chunk` new tokens whose K/V are written first, as
# the varlen read of the book's §4.5 receives them. The long-context ones are
# few long sequences with short chunks (the late chunks of long prompts):
# few work units, so each unit's K/V range is split across the SMs.
@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    dtype: int
    num_seqs: int
    max_prefix: int
    chunk: int
    scale: float
    description: str
    min_prefix: int = 0


PREFILL_WORKLOADS = {
    "prefill_llama13b": PrefillWorkload(
        "prefill_llama13b", 16, 40, 40, 128, F16, 8, 2048, 1024, 128 ** -0.5,
        "Llama-2-13B layer chunked prefill: 40/40 heads, d=128, fp16, 8 seqs, "
        "prefix U[0,2048] + 1024-token chunk"),
    "prefill_gqa8b": PrefillWorkload(
        "prefill_gqa8b", 16, 32, 8, 128, BF16, 8, 4096, 1024, 128 ** -0.5,
        "GQA 8B chunked prefill: 32/8 heads, d=128, bf16, 8 seqs, prefix U[0,4096] + 1024-token chunk"),
    "prefill_longctx_llama13b": PrefillWorkload(
        "prefill_longctx_llama13b", 16, 40, 40, 128, F16, 2, 16384, 512, 128 ** -0.5,
        "Llama-2-13B layer, long context: 40/40 heads, d=128, fp16, 2 seqs, "
        "prefix U[12288,16384] + 512-token chunk", min_prefix=12288),
    "prefill_longctx_gqa8b": PrefillWorkload(
        "prefill_longctx_gqa8b", 16, 32, 8, 128, BF16, 1, 65536, 2048, 128 ** -0.5,
        "GQA 8B, long prompt: 32/8 heads, d=128, bf16, 1 seq, prefix U[57344,65536] + 2048-token chunk",
        min_prefix=57344),
}


# Prefix-cache serving wave: requests sharing a system prompt, each with a
# private suffix; Llama-2-13B layer shape (40/40 heads, d=128, fp16).
SHARED_PROMPT = dict(requests=16, system=1024, suffix_lo=64, suffix_hi=512, num_q_heads=40,
                     num_kv_heads=40, head_size=128, dtype=F16, block_size=16, vocab=32000)


def shared_prompt_tokens(seed: int):
    """The system prompt's token ids and a generator of request suffixes."""
    g = rng(seed + 5)
    system = g.integers(0, SHARED_PROMPT["vocab"], size=SHARED_PROMPT["system"]).astype(np.int32)
    return system, g


def prefill_prefixes(name: str, seed: int) -> np.ndarray:
    """Cached prefix length of every sequence of a prefill workload."""
    w = PREFILL_WORKLOADS[name]
    return rng(seed + 3).integers(w.min_prefix, w.max_prefix + 1, size=w.num_seqs).astype(np.int32)


TOY_LENGTHS = (25, 47, 12)
TOY_PLACEMENT = ((3, 7), (0, 5, 9), (4,))
TOY_GROWTH_BLOCKS = (11, 12)      # B's next blocks as it grows by 20 tokens
TOY_GROWTH_TOKENS = 20

PREFIX_GROUPS = 16
PREFIX_GROUP_SIZE = 8
PREFIX_PROMPT = 1024


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def toy_free_order() -> np.ndarray:
    """Free-list order that makes a pop-from-head allocator reproduce the
    worked example's placement, then B's growth blocks, then the rest."""
    head = [b for t in TOY_PLACEMENT for b in t] + list(TOY_GROWTH_BLOCKS)
    rest = [b for b in range(WORKLOADS["toy"].num_blocks) if b not in head]
    return np.array(head + rest, dtype=np.int32)


def free_order(num_blocks: int, seed: int) -> np.ndarray:
    """A seeded permutation of 0..num_blocks-1: the order in which a
    pop-from-head allocator hands out physical blocks, so that block tables
    are random non-repeating physical ids."""
    return rng(seed).permutation(num_blocks).astype(np.int32)


def seq_lens(name: str, seed: int) -> np.ndarray:
    """Decode lengths drawn from the workload's stated distribution."""
    g = rng(seed + 1)
    w = WORKLOADS[name]
    if name == "toy":
        return np.array(TOY_LENGTHS, dtype=np.int32)
    if name == "llama13b":
        return g.integers(1, 2049, size=w.num_seqs).astype(np.int32)
    if name == "gqa8b":
        x = np.round(g.lognormal(mean=np.log(800.0), sigma=1.0, size=w.num_seqs))
        return np.clip(x, 16, 8192).astype(np.int32)
    if name == "longctx":
        return g.integers(32768, 131073, size=w.num_seqs).astype(np.int32)
    if name == "prefix_cow":
        tails = g.integers(1, 513, size=w.num_seqs)
        return (PREFIX_PROMPT + tails).astype(np.int32)
    raise KeyError(name)


def prefix_fork_extra(seed: int) -> np.ndarray:
    """Per-group extra prompt tokens (1..15) for the fork variant."""
    return rng(seed + 2).integers(1, 16, size=PREFIX_GROUPS).astype(np.int32)


def normal_values(shape, dtype: int, seed: int, device="cpu"):
    """N(0, 1) draws rounded to fp16/bf16 (a torch tensor on ``device``)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    tdt = torch.float16 if dtype == F16 else torch.bfloat16
    out = torch.empty(tuple(shape), dtype=tdt, device=device)
    flat = out.view(-1)
    step = 1 << 26
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=gen, device=device, dtype=torch.float32).to(tdt)
    return out


# Per-tensor scales of the FP8 (E4M3) cache variant of every workload: a code
# c stands for e4m3(c) * scale. N(0, 1) draws use the E4M3 range down to
# about 2^-6 * scale and saturate beyond 448 * scale (5.6 for K, 4.48 for V).
FP8_K_SCALE = 0.0125
FP8_V_SCALE = 0.01


def fp8_codes(shape, scale: float, seed: int, device="cpu"):
    """E4M3 codes (uint8 tensor on ``device``) of N(0, 1) draws for a cache
    with the given per-tensor scale: draws of N(0, 1 / scale^2), clipped to
    +-448, rounded by PyTorch's float8_e4m3fn cast. An input generator only:
    it is not the write path's quantisation (that is an fp32 division by the
    scale, done by the kernel and by the oracle)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    out = torch.empty(tuple(shape), dtype=torch.uint8, device=device)
    flat = out.view(-1)
    step = 1 << 26
    sigma = 1.0 / float(scale)
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        x = torch.randn(n, generator=gen, device=device, dtype=torch.float32) * sigma
        flat[i:i + n] = x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def torch_dtype(dtype: int):
    import torch
    return torch.float16 if dtype == F16 else torch.bfloat16
