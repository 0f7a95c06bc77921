"""The pins reject a plausible mistake anywhere in the C oracle.

Each case plants one mistake in a copy of oracle/oracle.c (a textual substitution, so the oracle
itself stays as it is), builds it, and runs the oracle pin suites against that build in a separate
process (PKV_ORACLE_LIB points the oracle's loader at it): at least one pin must fail. Every planted
mistake keeps the oracle's reads and writes inside its buffers. The substituted text must occur in
oracle.c exactly as often as stated, so a change to the oracle that moves it fails here loudly.
"""
import os
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
SRC = ROOT / "oracle" / "oracle.c"
PINS = ["tests/test_oracle_pins.py", "tests/test_prefill_oracle_pins.py"]

# (name, text, replacement, occurrences in oracle.c, which occurrence to replace: 0-based, or None = all)
MUTANTS = [
    # decode attention ("La idea de PagedAttention", step 5, then dense softmax attention)
    ("decode: query head mapped to the wrong KV head", "const int g = h / group;", "const int g = h % n_kv;", 2, 0),
    ("decode: row offset inside a block shifted", "orc_row(phys, g, j % block_size, n_kv, block_size, head_dim)",
     "orc_row(phys, g, (j + 1) % block_size, n_kv, block_size, head_dim)", 2, 0),
    ("decode: K gathered from the V pool", "kc[(size_t)j * head_dim + i] = orc_load(dtype, k_pool, row + i);",
     "kc[(size_t)j * head_dim + i] = orc_load(dtype, v_pool, row + i);", 2, 0),
    ("decode: scale dropped", "z[j] = scale * acc;", "z[j] = acc;", 2, 0),
    ("decode: max subtraction dropped", "z[j] = exp(z[j] - m);", "z[j] = exp(z[j]);", 2, 0),
    ("decode: normalisation dropped", "acc += (z[j] / zsum) * vc[(size_t)j * head_dim + i];",
     "acc += z[j] * vc[(size_t)j * head_dim + i];", 2, 0),
    # prefill attention ("01 - Conceito", paragraph 5: a chunk of new tokens, causal)
    ("prefill: query head mapped to the wrong KV head", "const int g = h / group;", "const int g = h % n_kv;", 2, 1),
    ("prefill: causal mask dropped", "j <= pos", "j < c", 3, None),
    ("prefill: a query does not see its own key", "const int pos = c - n_new + t;",
     "const int pos = c - n_new + t - 1;", 1, 0),
    ("prefill: chunk rows read in reverse", "const size_t qrow = ((size_t)(query_start[s] + t) * n_q + h) * head_dim;",
     "const size_t qrow = ((size_t)(query_start[s] + (n_new - 1 - t)) * n_q + h) * head_dim;", 1, 0),
    ("prefill: normalisation dropped", "acc += (z[j] / zsum) * vc[(size_t)j * head_dim + i];",
     "acc += z[j] * vc[(size_t)j * head_dim + i];", 2, 1),
    # append, copy-on-write copy, byte formula, decoders
    ("append: slot offset shifted", "int off = (int)(slot % block_size);", "int off = (int)((slot + 1) % block_size);",
     1, 0),
    ("copy: V block copied from the K pool",
     "memcpy((char*)v_pool + l * layer_bytes + dst, (const char*)v_pool + l * layer_bytes + src, block_bytes);",
     "memcpy((char*)v_pool + l * layer_bytes + dst, (const char*)k_pool + l * layer_bytes + src, block_bytes);", 1, 0),
    ("bytes per token: K or V only", "return 2ull * (uint64_t)n_layers", "return 1ull * (uint64_t)n_layers", 1, 0),
    ("bf16 decoder: exponent bias off by one", "e - 134", "e - 133", 1, 0),
    ("fp16 decoder: subnormal scale off by one", "ldexp((double)f, -24)", "ldexp((double)f, -23)", 1, 0),
]


def _mutate(text: str, old: str, new: str, count: int, which):
    assert text.count(old) == count, f"oracle.c holds {text.count(old)} copies of {old!r}, expected {count}"
    if which is None:
        return text.replace(old, new)
    parts = text.split(old)
    return old.join(parts[: which + 1]) + new + old.join(parts[which + 1:])


@pytest.mark.parametrize("name,old,new,count,which", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_planted_mistake(tmp_path, name, old, new, count, which):
    src = tmp_path / "oracle_mutant.c"
    src.write_text(_mutate(SRC.read_text(), old, new, count, which))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-fopenmp", str(src), "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, PKV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "not gpu", *PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"{name}: the pins did not fail (exit {r.returncode})\n{r.stdout[-2000:]}"
    assert " failed" in r.stdout


def test_unmutated_copy_passes_the_pins(tmp_path):
    """The same procedure on an unchanged copy passes, so a failure above is the planted mistake."""
    src = tmp_path / "oracle_copy.c"
    src.write_text(SRC.read_text())
    lib = tmp_path / "liboracle_copy.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-fopenmp", str(src), "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, PKV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "not gpu", *PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
