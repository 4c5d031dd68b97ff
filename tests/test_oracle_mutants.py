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

# The gather prologue of the 16-bit and the FP8 decode (they differ in the
# type of the K/V buffers): {0} is the q-head -> kv-head map, {1} the
# logical-block index of token i.
_GATHER = """    int kv_head = {0};
    const int32_t *table = block_tables + (long long)seq * max_blocks_per_seq;
    size_t n = seq_len > 0 ? (size_t)seq_len * head_size : 1;
    %s *k = (%s *)malloc(sizeof(%s) * n);
    %s *v = (%s *)malloc(sizeof(%s) * n);
"""
_GATHER16 = (_GATHER % (("uint16_t",) * 6)) + """    for (int i = 0; i < seq_len; ++i) {{
        int b = table[{1}];"""
_GATHER8 = (_GATHER % (("double",) * 6)) + """    double *q = (double *)malloc(sizeof(double) * (size_t)head_size);
    for (int i = 0; i < seq_len; ++i) {{
        int b = table[{1}];"""

# (file, original text, planted slip, pin file expected to catch it)
# the query-row and call lines that follow the visible length in the prefill
# row loops (16-bit and FP8; they differ only in the call)
_ROW_TAIL = ("\n        const uint16_t *q_row = query + (long long)r * num_q_heads * head_size;"
             "\n        for (int hq = 0; hq < num_q_heads; ++hq)\n            %s(")
_PREFILL16 = _ROW_TAIL % "oracle_decode_one"
_PREFILL8 = _ROW_TAIL % "oracle_decode_fp8_one"
_VISIBLE = "int32_t visible = seq_lens[s] - q_len + i + 1; /* tokens 0..p */"
# the row -> sequence search that opens each prefill row
_ROW_SEARCH = ("while (cu_seqlens_q[s + 1] <= r) /* the sequence whose chunk holds row r */\n"
               "            ++s;\n        int q0 = cu_seqlens_q[s];\n"
               "        int q_len = cu_seqlens_q[s + 1] - q0;\n        int i = r - q0;\n"
               "        const int32_t *table = block_tables + (long long)s * max_blocks_per_seq;\n        ")

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
    ("oracle/oracle.c", _GATHER16.format("q_head / group", "i / block_size"),
     _GATHER16.format("q_head % num_kv_heads", "i / block_size"),
     "test_oracle_pins.py"),                                                           # GQA mapping
    ("oracle/oracle.c", _GATHER16.format("q_head / group", "i / block_size"),
     _GATHER16.format("q_head / group", "i % block_size"),
     "test_oracle_pins.py"),                                                           # table walk
    ("oracle/oracle.c", _GATHER8.format("q_head / group", "i / block_size"),
     _GATHER8.format("q_head % num_kv_heads", "i / block_size"),
     "test_oracle_fp8_pins.py"),                                                       # fp8 GQA mapping
    ("oracle/oracle.c", _GATHER8.format("q_head / group", "i / block_size"),
     _GATHER8.format("q_head / group", "i % block_size"),
     "test_oracle_fp8_pins.py"),                                                       # fp8 table walk
    ("oracle/oracle.c", "double a_old = exp(m - m_new);", "double a_old = exp(m_new - m);",
     "test_oracle_pins.py"),                                                           # merge sign
    ("oracle/oracle.c", "s = s * a_old + sp * a_new;", "s = s * a_old + sp;",
     "test_oracle_pins.py"),                                                           # merge term
    ("oracle/oracle.c", "mag = ldexp((double)(8 + frac), expo - 10);",
     "mag = ldexp((double)(8 + frac), expo - 9);", "test_oracle_fp8_pins.py"),       # e4m3 bias
    ("oracle/oracle.c", "mag = ldexp((double)frac, -9);", "mag = ldexp((double)frac, -10);",
     "test_oracle_fp8_pins.py"),                                                      # subnormals
    ("oracle/oracle.c", "(c & 1) == 0 && (best & 1) == 1", "(c & 1) == 1 && (best & 1) == 0",
     "test_oracle_fp8_pins.py"),                                                      # ties to odd
    ("oracle/oracle.c", "return sign | 0x7E;", "return sign | 0x7F;",
     "test_oracle_fp8_pins.py"),                                                      # no saturation
    ("oracle/oracle.c", "float y = v / scale;", "float y = v * scale;",
     "test_oracle_fp8_pins.py"),                                                      # scale inverted
    ("oracle/oracle.c", "oracle_quantize_e4m3(value[src], dtype, v_scale);",
     "oracle_quantize_e4m3(value[src], dtype, k_scale);", "test_oracle_fp8_pins.py"), # V with K scale
    ("oracle/oracle.c", "v[(long long)i * head_size + d] = oracle_e4m3_to_double(vc) * v_scale;",
     "v[(long long)i * head_size + d] = oracle_e4m3_to_double(vc) * k_scale;",
     "test_oracle_fp8_pins.py"),                                                      # decode scale swap
    ("oracle/oracle.c", _VISIBLE + _PREFILL16, _VISIBLE.replace("i + 1;", "i + 2;") + _PREFILL16,
     "test_oracle_prefill_pins.py"),                                                  # sees p+1
    ("oracle/oracle.c", _VISIBLE + _PREFILL16, _VISIBLE.replace("i + 1;", "1;") + _PREFILL16,
     "test_oracle_prefill_pins.py"),                                                  # not causal in i
    ("oracle/oracle.c", _PREFILL16, _PREFILL16.replace("(long long)r *", "(long long)i *"),
     "test_oracle_prefill_pins.py"),                                                  # wrong query row
    ("oracle/oracle.c", _ROW_SEARCH + _VISIBLE + _PREFILL16,
     _ROW_SEARCH.replace("<= r)", "< r)") + _VISIBLE + _PREFILL16,
     "test_oracle_prefill_pins.py"),                                                  # row -> sequence off by one
    ("oracle/oracle.c", "dtype, k_scale, v_scale);\n    }\n}\n\n/* ---- the online-softmax",
     "dtype, v_scale, k_scale);\n    }\n}\n\n/* ---- the online-softmax",
     "test_oracle_prefill_pins.py"),                                                  # FP8 prefill scales swapped
    ("oracle/oracle.c", _VISIBLE + _PREFILL8, _VISIBLE.replace("i + 1;", "i + 2;") + _PREFILL8,
     "test_oracle_prefill_pins.py"),                                                  # FP8 prefill row sees one more
    ("oracle/prefix_cache.py", "if (i + 1) * B > n - 1 or h not in self.cached:",
     "if (i + 1) * B > n or h not in self.cached:", "test_prefix_cache_model.py"),   # hit limit
    ("oracle/prefix_cache.py", "                    self.free.append(b)",
     "                    self.free.insert(0, b)", "test_prefix_cache_model.py"),    # cached to head
    ("oracle/prefix_cache.py", "for b in reversed(s[\"table\"]):", "for b in s[\"table\"]:",
     "test_prefix_cache_model.py"),                                                   # free order
    ("oracle/prefix_cache.py", "        self._evict(b)\n        self.ref[b] = 1",
     "        self.ref[b] = 1", "test_prefix_cache_model.py"),                         # no eviction
    ("oracle/prefix_cache.py", 'parent = s["hashes"][-1] if s["hashes"] else NONE_HASH',
     "parent = NONE_HASH", "test_prefix_cache_model.py"),                             # chain broken
    ("oracle/prefix_cache.py", "            if self.ref[b] == 0:\n                self.free.remove(b)\n",
     "", "test_prefix_cache_model.py"),                                                # no touch
    ("oracle/prefix_cache.py", "hashes = chain_hashes(tokens, B) if cache else []",
     "hashes = chain_hashes(tokens, B)", "test_prefix_cache_model.py"),              # caching never off
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
