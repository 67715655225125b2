"""The pins must catch plausible mistakes in the oracle.

Each case compiles a copy of oracle.c with one planted mistake (CPU only),
runs the pin suite against it in a fresh process and requires that suite to
fail.  The planted mistakes live only in these temporary copies.
"""
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "gqa_head_mapping": ("tables + (int64_t)b * max_blocks, len, V);\n"
                         "        for (int d = 0; d < head_dim; ++d)\n"
                         "            qd[d] = load_elem(q, ((int64_t)b * num_q_heads + hq) * head_dim + d, q_dtype);\n"
                         "        oracle_attend(qd, K, V, len, num_kv_heads, hq / group,",
                         "tables + (int64_t)b * max_blocks, len, V);\n"
                         "        for (int d = 0; d < head_dim; ++d)\n"
                         "            qd[d] = load_elem(q, ((int64_t)b * num_q_heads + hq) * head_dim + d, q_dtype);\n"
                         "        oracle_attend(qd, K, V, len, num_kv_heads, hq % num_kv_heads,"),
    "no_normalisation": ("for (int d = 0; d < head_dim; ++d) o[d] /= l;",
                         "for (int d = 0; d < head_dim; ++d) o[d] /= 1.0;"),
    "causal_off_by_one": ("oracle_attend(qd, K, V, pos + 1,", "oracle_attend(qd, K, V, pos,"),
    "block_offset": ("int64_t offset = j % block_size;", "int64_t offset = (j + 1) % block_size;"),
    "lse_without_log_sum": ("*lse = m + log(l);", "*lse = m;"),
    "missing_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "no_max_subtraction": ("double w = exp(s[j] - m);", "double w = exp(s[j]);"),
    "slot_split_swapped": ("int64_t block = slot / block_size, offset = slot % block_size;",
                           "int64_t block = slot % block_size, offset = slot / block_size;"),
    "half_exponent_bias": ("v = ldexp((double)(1024 + frac), expo - 25);",
                           "v = ldexp((double)(1024 + frac), expo - 24);"),
    "half_subnormal_as_normal": ("        v = ldexp((double)frac, -24);",
                                 "        v = ldexp((double)(1024 + frac), -24);"),
}


@pytest.fixture(scope="module")
def gcc():
    g = shutil.which("gcc")
    if not g:
        pytest.skip("gcc not available")
    return g


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name, gcc, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run([gcc, "-O1", "-std=c11", "-fPIC", "-shared", str(mutant), "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"the pins did not notice the planted mistake '{name}'"
