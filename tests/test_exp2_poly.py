"""The FMA-pipe 2^x of the prefill softmax: its coefficients are the ones
the Remez fit in paged_kv_cache_120_gb300/exp2_poly.py produces (the kernel
quotes them as hex floats), and the kernel's fp32 sequence, emulated step by
step, stays within the fit's error bound over the range the softmax uses."""
import os
import re

import numpy as np

from paged_kv_cache_120_gb300 import exp2_poly

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _kernel_constants():
    src = open(os.path.join(ROOT, "paged_kv_cache_120_gb300", "csrc", "pa_prefill.cu")).read()
    body = src[src.index("__device__ __forceinline__ void exp2_poly2"):]
    body = body[:body.index("float p0, p1, j0, j1;")]
    deg4 = body[body.index("if constexpr (DEG == 4)"):body.index("} else {")]
    deg3 = body[body.index("} else {"):]
    hexes = lambda t: [float.fromhex(h[:-1]) for h in re.findall(r"0x1\.[0-9a-f]+p-?\d+f", t)]
    # pk2(c, c) lists every constant twice, in Horner order (highest first)
    return {4: hexes(deg4)[::2][::-1], 3: hexes(deg3)[::2][::-1]}


def test_kernel_coefficients_are_the_remez_fit():
    k = _kernel_constants()
    for d in (3, 4):
        assert k[d] == exp2_poly.fp32_coefficients(d), d


def test_fit_levels_the_relative_error():
    for d, bound in ((3, 7.6e-5), (4, 2.7e-6)):
        c, e = exp2_poly.remez_relative(d)
        assert e < bound
        # a minimax fit beats the Taylor polynomial of the same degree
        taylor = [np.log(2.0) ** i / np.prod(range(1, i + 1)) for i in range(d + 1)]
        f = np.linspace(-0.5, 0.5, 10001)
        t_err = np.max(np.abs(np.polyval(taylor[::-1], f) / np.exp2(f) - 1))
        assert e < t_err / 4


def test_fp32_sequence_within_bound_and_special_values():
    # results with a normal exponent (x >= -125); below that the value is
    # under 2^-124, which the 16-bit P rounds to zero (fp16) or carries as a
    # negligible subnormal next to the row's largest weight (>= 1)
    xs = np.concatenate([np.linspace(-125.0, 8.5, 3000001, dtype=np.float32),
                         np.array([0.0, -0.5, 0.5, -1.0, 1.0, 8.0, -124.5], np.float32)])
    for d, bound in ((3, 7.6e-5), (4, 2.8e-6)):
        got = exp2_poly.emulate(xs, exp2_poly.fp32_coefficients(d)).astype(np.float64)
        rel = np.abs(got / np.exp2(xs.astype(np.float64)) - 1.0)
        assert rel.max() < bound, (d, rel.max())
        # below the clamp: tiny and non-negative, never garbage
        low = exp2_poly.emulate(np.array([-125.5, -126.0, -127.0, -200.0, -1e30, -np.inf], np.float32),
                                exp2_poly.fp32_coefficients(d))
        assert np.all(low >= 0) and np.all(low <= 2.0 ** -124)
        assert np.isnan(exp2_poly.emulate(np.array([np.nan], np.float32), exp2_poly.fp32_coefficients(d)))[0]
