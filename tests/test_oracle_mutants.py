"""Planted mistakes in the oracle must each trip at least one pin (CPU only).

Each mutant is a one-line edit of a copy of ``oracle/oracle.c`` (a dropped
term, a wrong index, a swapped operand, an off-by-one, a wrong sign). The copy
is compiled into a temporary directory and the whole pin battery of
``tests/oracle_pins.py`` runs against it in a child process (a mutant may
crash; that counts as caught). The real oracle is never modified.
"""
import json
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle as oracle_pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, original text, replacement); the original must occur in oracle.c and
# only its first occurrence is replaced.
MUTANTS = [
    ("gqa_modulo_grouping", "const int32_t kv = h / group;",
     "const int32_t kv = h % a->num_kv_heads;"),
    ("scale_dropped", "const double s = a->scale * dot;", "const double s = dot;"),
    ("causal_excludes_self", "int64_t hi = pos + 1;", "int64_t hi = pos;"),
    ("causal_top_left", "const int64_t pos = (int64_t)a->seq_lens[i] - query_len + j;",
     "const int64_t pos = j;"),
    ("key_offset_uses_block_index", "const int64_t offset = p % a->block_size;",
     "const int64_t offset = (p / a->block_size) % a->block_size;"),
    ("v_read_from_k_half", "const uint16_t *vrow = a->pool + pool_index(1,",
     "const uint16_t *vrow = a->pool + pool_index(0,"),
    ("query_uses_kv_head", "const uint16_t *qrow = a->q + ((size_t)t * a->num_heads + h) * D;",
     "const uint16_t *qrow = a->q + ((size_t)t * a->num_heads + kv) * D;"),
    ("lse_drops_max", "*lse = m + log(sum);", "*lse = log(sum);"),
    ("softmax_not_normalised", "const double prob = exp(scores[p - lo] - m) / sum;",
     "const double prob = exp(scores[p - lo] - m);"),
    ("normaliser_drops_max", "sum += exp(scores[p - lo] - m);", "sum += exp(scores[p - lo]);"),
    ("merge_weight_sign", "const double w = exp(l - M);", "const double w = exp(M - l);"),
    ("merge_not_normalised", "o[d] /= wsum;", "o[d] /= 1.0;"),
    ("merge_lse_drops_max", "out_lse[r] = M + log(wsum);", "out_lse[r] = log(wsum);"),
    ("write_k_gets_v", "dst_k[d] = src_k[d];", "dst_k[d] = src_v[d];"),
    ("write_offset_off_by_one", "const int64_t offset = s % block_size;",
     "const int64_t offset = (s + 1) % block_size;"),
    ("request_lookup_inclusive", "if (cu_seqlens[i] <= t && t < cu_seqlens[i + 1]) return i;",
     "if (cu_seqlens[i] <= t && t <= cu_seqlens[i + 1]) return i;"),
    ("sizing_drops_kv_factor", "return 2 * num_layers * num_kv_heads * head_dim * bytes_per_element;",
     "return num_layers * num_kv_heads * head_dim * bytes_per_element;"),
    ("table_row_of_request_zero", "const int32_t *table = a->block_table + (size_t)i * a->max_blocks;",
     "const int32_t *table = a->block_table;"),
]

_CHILD = r"""
import json, sys
sys.path.insert(0, {root!r})
import oracle
from tests import oracle_pins
o = oracle.Oracle({lib!r})
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(o)
    except Exception as e:  # any failure of a pin counts
        failed.append(pin.__name__)
print("FAILED=" + json.dumps(failed))
"""


def _run_mutant(tmp_dir, name, old, new):
    with open(oracle_pkg.SOURCE) as f:
        src = f.read()
    assert old in src, f"mutant {name}: text not found in oracle.c"
    mutated = src.replace(old, new, 1)
    c_path = os.path.join(tmp_dir, f"{name}.c")
    with open(c_path, "w") as f:
        f.write(mutated)
    lib = oracle_pkg.compile_oracle(c_path, os.path.join(tmp_dir, f"lib{name}.so"))
    env = dict(os.environ, OMP_NUM_THREADS="2")
    proc = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT, lib=lib)],
                          capture_output=True, text=True, timeout=600, env=env)
    if proc.returncode != 0:
        return name, ["<crashed %d>" % proc.returncode]
    line = [ln for ln in proc.stdout.splitlines() if ln.startswith("FAILED=")][-1]
    return name, json.loads(line[len("FAILED="):])


def test_every_planted_mistake_is_caught(tmp_path):
    with ThreadPoolExecutor(max_workers=4) as pool:
        results = list(pool.map(lambda m: _run_mutant(str(tmp_path), *m), MUTANTS))
    survivors = [name for name, failed in results if not failed]
    report = {name: failed for name, failed in results}
    assert not survivors, f"mutants not caught by any pin: {survivors}\n{json.dumps(report, indent=1)}"


def test_unmodified_copy_passes(tmp_path):
    name, failed = _run_mutant(str(tmp_path), "identity", "#include <math.h>", "#include <math.h>")
    assert failed == [], failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_text_present(name, old, new):
    with open(oracle_pkg.SOURCE) as f:
        assert old in f.read()
