"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch every one of them.  Each mutant is a text substitution in a copy of the
oracle's C source, compiled to a temporary library and exercised in a child
process (a mutant may index out of bounds)."""
import os
import subprocess
import sys

import pytest

from oracle import build as obuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "page_from_offset": ("return table_row[j / B];", "return table_row[j % B];"),
    "offset_wrong": ("*offset = j % B;", "*offset = (j + 1) % B;"),
    "gqa_interleaved": ("  int g = h / G;\n  int ctx = context_lens[s];", "  int g = h % Hkv;\n  int ctx = context_lens[s];"),
    "scale_dropped": ("x[j] = scale * dot;", "x[j] = dot;"),
    "no_max_subtraction": ("x[j] = exp(x[j] - m);", "x[j] = exp(x[j]);"),
    "unnormalised": ("out[d] = acc / denom;", "out[d] = acc;"),
    "k_for_v": ("acc += x[j] * V[(size_t)j * D + d];", "acc += x[j] * K[(size_t)j * D + d];"),
    "head_major_pool": ("size_t base = (((size_t)p * Hkv + g) * B + o) * (size_t)D;",
                        "size_t base = (((size_t)g * num_blocks + p) * B + o) * (size_t)D;"),
    "causal_off_by_one": ("int n = pos + 1;", "int n = pos;"),
    "chunk_position": ("int pos = ctx - C + i;", "int pos = i;"),
    "combine_drops_l": ("double w = l[p] * exp(m[p] - mx);", "double w = exp(m[p] - mx);"),
    "cache_offset": ("int64_t p = slot / B, o = slot % B;", "int64_t p = slot / B, o = (slot + 1) % B;"),
    "cache_negative_slot_written": ("if (slot < 0) continue;", "if (slot < 0) slot = 0;"),
    "copy_reversed": ("int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];",
                      "int64_t dst = pairs[2 * i], src = pairs[2 * i + 1];"),
    "swap_reversed": ("int64_t from = pairs[2 * i], to = pairs[2 * i + 1];",
                      "int64_t to = pairs[2 * i], from = pairs[2 * i + 1];"),
    "swap_bound_of_other_pool": ("from >= src_blocks || to < 0 || to >= dst_blocks",
                                 "from >= dst_blocks || to < 0 || to >= src_blocks"),
    "sizing_one_tensor": ("return 2 * layers * kv_heads * head_dim * elem_bytes;",
                          "return layers * kv_heads * head_dim * elem_bytes;"),
}

RUNNER = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle, pins
o = oracle.Oracle({lib!r})
failed = []
for p in pins.ALL_PINS:
    try:
        p(o)
    except Exception as e:
        failed.append(p.__name__)
print("FAILED:" + ",".join(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/found"
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src.replace(old, new))
    lib = obuild.build(force=True, src=str(msrc), out=str(tmp_path / "libmutant.so"))
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    caught = r.returncode != 0 or ("FAILED:" in r.stdout and r.stdout.strip().split("FAILED:")[-1] != "")
    assert caught, f"mutant {name} passed every pin:\n{r.stdout}\n{r.stderr}"
