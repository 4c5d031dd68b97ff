"""Mutation check of the pins: plant one plausible slip at a time in a copy
of the oracle (on the CPU, in a scratch copy of the tree) and require the
pin suite to fail. A mutant that survives means a part of the oracle is not
actually pinned."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (file, original text, planted slip, pin file expected to catch it)
MUTANTS = [
    ("oracle/oracle.c", "expo - 25);", "expo - 24);", "test_oracle_pins.py"),          # f16 bias
    ("oracle/oracle.c", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)", "test_oracle_pins.py"),
    ("oracle/oracle.c", "expo - 134);", "expo - 133);", "test_oracle_pins.py"),        # bf16 bias
    ("oracle/oracle.c", "long long offset = pos % block_size;",
     "long long offset = pos / block_size;", "test_oracle_pins.py"),                   # slot offset
    ("oracle/oracle.c", "* block_size + t) * num_kv_heads + h)",
     "* num_kv_heads + h) * block_size + t)", "test_oracle_pins.py"),                 # pool dims
    ("oracle/oracle.c",
     "pool[pool_index(0, b, off, h, d, num_blocks, block_size, num_kv_heads, head_size)] = key[src];",
     "pool[pool_index(0, b, off, h, d, num_blocks, block_size, num_kv_heads, head_size)] = value[src];",
     "test_oracle_pins.py"),                                                           # K/V swap
    ("oracle/oracle.c", "for (int c = 0; c < 2; ++c)", "for (int c = 0; c < 1; ++c)",
     "test_oracle_pins.py"),                                                           # copy K only
    ("oracle/oracle.c", "x[i] = scale * dot;", "x[i] = dot;", "test_oracle_pins.py"),  # no scale
    ("oracle/oracle.c", "denom += x[i];", "denom += 1.0;", "test_oracle_pins.py"),     # bad normaliser
    ("oracle/oracle.c", "int kv_head = q_head / group;", "int kv_head = q_head % num_kv_heads;",
     "test_oracle_pins.py"),                                                           # GQA mapping
    ("oracle/oracle.c", "int b = table[i / block_size];", "int b = table[i % block_size];",
     "test_oracle_pins.py"),                                                           # table walk
    ("oracle/oracle.c", "double a_old = exp(m - m_new);", "double a_old = exp(m_new - m);",
     "test_oracle_pins.py"),                                                           # merge sign
    ("oracle/oracle.c", "s = s * a_old + sp * a_new;", "s = s * a_old + sp;",
     "test_oracle_pins.py"),                                                           # merge term
    ("oracle/block_manager.py", "self.free.insert(0, b)", "self.free.append(b)",
     "test_block_manager.py"),                                                         # free to tail
    ("oracle/block_manager.py", "                self.ref[last] -= 1\n", "",
     "test_block_manager.py"),                                                         # COW ref leak
    ("oracle/block_manager.py", "if self.ref[last] > 1:", "if self.ref[last] > 0:",
     "test_block_manager.py"),                                                         # COW always
    ("oracle/block_manager.py", "self.block_size + pos % self.block_size",
     "self.block_size + self.lens[sid] % self.block_size", "test_block_manager.py"),  # slot off by one
    ("oracle/block_manager.py", "need = -(-num_tokens // self.block_size)",
     "need = num_tokens // self.block_size + 1", "test_block_manager.py"),            # ceil
]


def _copy_tree(dst):
    for d in ("oracle", "tests", "paged_kv_cache_120_gb300"):
        shutil.copytree(os.path.join(ROOT, d), os.path.join(dst, d),
                        ignore=shutil.ignore_patterns("_build", "__pycache__", "*.so", "csrc"))
    shutil.copy(os.path.join(ROOT, "pytest.ini"), dst)


@pytest.mark.parametrize("idx", range(len(MUTANTS)))
def test_planted_slip_is_caught(tmp_path, idx):
    path, old, new, pins = MUTANTS[idx]
    _copy_tree(str(tmp_path))
    target = os.path.join(str(tmp_path), path)
    src = open(target).read()
    assert src.count(old) == 1, f"mutation anchor not unique in {path}: {old!r}"
    open(target, "w").write(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", os.path.join("tests", pins)],
                       cwd=str(tmp_path), capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {idx} ({new!r}) survived the pins:\n{r.stdout[-2000:]}"
