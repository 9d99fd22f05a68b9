"""The oracle's pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of ``oracle/hs_oracle.c`` (a wrong
exponent bias, a dropped term, a reversed order, an index off by one, ...),
builds that copy into a temporary library, points the ``oracle`` package at
it in a child process and runs the pins of ``test_oracle_pins.py`` that
cover the function: at least one of them must fail.  The unchanged copy,
built the same way, must pass the same pins.  Nothing here runs on a GPU
and the oracle's own source is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "hs_oracle.c")
PINS = os.path.join("tests", "test_oracle_pins.py")

FORMATS = "e4m3 or bf16 or dequant or generator_rows"
INDEXER = "indexer and not identity"
TOPK = "topk"
RESOLVE = "resolve or page_resident or zero_residency or hot_buffer"
ATTENTION = "attention or zero_residency"

# (name, text in hs_oracle.c, planted replacement, pins that must catch it)
MUTANTS = [
    ("e4m3 exponent bias 8 instead of 7",
     "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)", FORMATS),
    ("e4m3 subnormals scaled by 2^-7",
     "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)", FORMATS),
    ("group scale of the next group",
     "hso_e4m3(row[i]) * (double)sc[i / 128]", "hso_e4m3(row[i]) * (double)sc[(i / 128 + 1) & 3]",
     FORMATS),
    ("rope read two bytes early",
     "memcpy(&h, row + 528 + 2 * i, 2);", "memcpy(&h, row + 526 + 2 * i, 2);", FORMATS),
    ("indexer gate without the ReLU",
     "#define HSO_GATE(x) ((x) > 0.0 ? (x) : 0.0)", "#define HSO_GATE(x) (x)", INDEXER),
    ("indexer key scale dropped",
     "x = (double)sigma[t] * dot;", "x = dot;", INDEXER),
    ("indexer visibility one token short",
     "int visible = N - nq + j + 1;", "int visible = N - nq + j;", INDEXER),
    ("indexer head weights of query 0 for every query",
     "acc += (double)w[j * Hi + h] * HSO_GATE(x);", "acc += (double)w[h] * HSO_GATE(x);", INDEXER),
    ("top-K ties to the higher token",
     "return (x->t > y->t) - (x->t < y->t);", "return (x->t < y->t) - (x->t > y->t);", TOPK),
    ("top-K padding 0 instead of -1",
     "out[t] = -1;", "out[t] = 0;", TOPK),
    ("resolve: union keeps duplicates",
     "if (i == 0 || U[i] != U[i - 1])", "if (1)", RESOLVE),
    ("resolve: a hit does not refresh its stamp",
     "            stamp[hot_map[u]] = step;\n", "", RESOLVE),
    ("resolve: most recently used slots evicted first",
     "if (x->stamp != y->stamp) return x->stamp < y->stamp ? -1 : 1;",
     "if (x->stamp != y->stamp) return x->stamp > y->stamp ? -1 : 1;", RESOLVE),
    ("resolve: equal stamps evicted highest slot first",
     "    return (x->slot > y->slot) - (x->slot < y->slot);",
     "    return (x->slot < y->slot) - (x->slot > y->slot);", RESOLVE),
    ("resolve: slots used in this step may be evicted",
     "if (stamp[i] < step) {", "if (stamp[i] <= step) {", RESOLVE),
    ("resolve: victims matched to misses in LRU order, not slot order",
     "    qsort(victim, (size_t)m, sizeof(int32_t), cmp_i32);\n", "", RESOLVE),
    ("attention: softmax scale dropped",
     "z[rr] = tau * dot;", "z[rr] = dot;", ATTENTION),
    ("attention: values read 64 dims late",
     "o[(size_t)h * HSO_NOPE + i] += p * kv[(size_t)rr * HSO_LATENT + i];",
     "o[(size_t)h * HSO_NOPE + i] += p * kv[(size_t)rr * HSO_LATENT + i + 64];", ATTENTION),
    ("attention: scores without the rope dims",
     "            for (i = 0; i < HSO_LATENT; i++)\n                dot += qh[i]",
     "            for (i = 0; i < HSO_NOPE; i++)\n                dot += qh[i]", ATTENTION),
    ("attention: log-sum-exp in base 2",
     "lse[h] = mx + log(l);", "lse[h] = mx + log2(l);", ATTENTION),
]


def _run_pins(src_text, workdir, selection):
    """Build src_text as the oracle library in workdir and run the selected
    pins against it in a child process; returns (exit code, output tail)."""
    os.makedirs(workdir, exist_ok=True)
    src = os.path.join(workdir, "hs_oracle.c")
    lib = os.path.join(workdir, "liboracle.so")
    with open(src, "w") as f:
        f.write(src_text)
    code = (
        "import sys, oracle\n"
        f"oracle._SRC = {src!r}\n"
        f"oracle._LIB = {lib!r}\n"
        "oracle.build()\n"
        "import pytest\n"
        "sys.exit(pytest.main(['-x', '-q', '-p', 'no:cacheprovider', '-m', 'not gpu', "
        f"{PINS!r}, '-k', {selection!r}]))\n"
    )
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    return r.returncode, (r.stdout + r.stderr)[-1500:]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_unchanged_copy_passes_every_selection(source, tmp_path):
    selection = " or ".join(f"({s})" for s in sorted({m[3] for m in MUTANTS}))
    rc, tail = _run_pins(source, str(tmp_path / "control"), selection)
    assert rc == 0, tail


@pytest.mark.parametrize("name,old,new,selection", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(source, tmp_path, name, old, new, selection):
    assert source.count(old) == 1, f"the text to mutate is not unique in hs_oracle.c: {old!r}"
    rc, tail = _run_pins(source.replace(old, new), str(tmp_path / "mutant"), selection)
    assert rc == 1, f"no pin caught '{name}' (pytest exit {rc}):\n{tail}"
    shutil.rmtree(str(tmp_path / "mutant"), ignore_errors=True)
