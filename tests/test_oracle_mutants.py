"""The oracle's pins catch plausible mistakes in the oracle.

Each case plants one mistake (a wrong exponent bias, a dropped term, a
reversed order, an index off by one, ...) in a copy of the ``oracle``
package, in its C arithmetic or in its Python readings, imports that copy
in a child process (its C part built there) and runs the pins of
``test_oracle_pins.py`` that cover the function: at least one of them must
fail.  The unchanged copy, built the same way, must pass the same pins.
Nothing here runs on a GPU and the oracle's own files are never modified.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")
C_SRC, PY_SRC = "hs_oracle.c", "__init__.py"
PINS = os.path.join("tests", "test_oracle_pins.py")

FORMATS = "e4m3 or bf16 or dequant or generator_rows"
INDEXER = "indexer and not identity"
TOPK = "topk"
RESOLVE = "resolve or page_resident or zero_residency or hot_buffer"
ATTENTION = "attention or zero_residency"
PRESSURE = "pressure or page_resident"

# (name, file, text in it, planted replacement, pins that must catch it)
MUTANTS = [
    ("e4m3 exponent bias 8 instead of 7", C_SRC,
     "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)", FORMATS),
    ("e4m3 subnormals scaled by 2^-7", C_SRC,
     "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)", FORMATS),
    ("group scale of the next group", C_SRC,
     "hso_e4m3(row[i]) * (double)sc[i / 128]", "hso_e4m3(row[i]) * (double)sc[(i / 128 + 1) & 3]",
     FORMATS),
    ("rope read two bytes early", C_SRC,
     "memcpy(&h, row + 528 + 2 * i, 2);", "memcpy(&h, row + 526 + 2 * i, 2);", FORMATS),
    ("indexer gate without the ReLU", C_SRC,
     "#define HSO_GATE(x) ((x) > 0.0 ? (x) : 0.0)", "#define HSO_GATE(x) (x)", INDEXER),
    ("indexer key scale dropped", C_SRC,
     "x = (double)sigma[t] * dot;", "x = dot;", INDEXER),
    ("indexer visibility one token short", C_SRC,
     "int visible = N - nq + j + 1;", "int visible = N - nq + j;", INDEXER),
    ("indexer head weights of query 0 for every query", C_SRC,
     "acc += (double)w[j * Hi + h] * HSO_GATE(x);", "acc += (double)w[h] * HSO_GATE(x);", INDEXER),
    ("top-K ties to the higher token", C_SRC,
     "return (x->t > y->t) - (x->t < y->t);", "return (x->t < y->t) - (x->t > y->t);", TOPK),
    ("top-K padding 0 instead of -1", C_SRC,
     "out[t] = -1;", "out[t] = 0;", TOPK),
    ("resolve: union keeps duplicates", C_SRC,
     "if (i == 0 || U[i] != U[i - 1])", "if (1)", RESOLVE),
    ("resolve: a hit does not refresh its stamp", C_SRC,
     "            stamp[hot_map[u]] = step;\n", "", RESOLVE),
    ("resolve: most recently used slots evicted first", C_SRC,
     "if (x->stamp != y->stamp) return x->stamp < y->stamp ? -1 : 1;",
     "if (x->stamp != y->stamp) return x->stamp > y->stamp ? -1 : 1;", RESOLVE),
    ("resolve: equal stamps evicted highest slot first", C_SRC,
     "    return (x->slot > y->slot) - (x->slot < y->slot);",
     "    return (x->slot < y->slot) - (x->slot > y->slot);", RESOLVE),
    ("resolve: slots used in this step may be evicted", C_SRC,
     "if (stamp[i] < step) {", "if (stamp[i] <= step) {", RESOLVE),
    ("resolve: victims matched to misses in LRU order, not slot order", C_SRC,
     "    qsort(victim, (size_t)m, sizeof(int32_t), cmp_i32);\n", "", RESOLVE),
    ("attention: softmax scale dropped", C_SRC,
     "z[rr] = tau * dot;", "z[rr] = dot;", ATTENTION),
    ("attention: values read 64 dims late", C_SRC,
     "o[(size_t)h * HSO_NOPE + i] += p * kv[(size_t)rr * HSO_LATENT + i];",
     "o[(size_t)h * HSO_NOPE + i] += p * kv[(size_t)rr * HSO_LATENT + i + 64];", ATTENTION),
    ("attention: scores without the rope dims", C_SRC,
     "            for (i = 0; i < HSO_LATENT; i++)\n                dot += qh[i]",
     "            for (i = 0; i < HSO_NOPE; i++)\n                dot += qh[i]", ATTENTION),
    ("attention: log-sum-exp in base 2", C_SRC,
     "lse[h] = mx + log(l);", "lse[h] = mx + log2(l);", ATTENTION),
    ("f32 rows read with swapped neighbours", C_SRC,
     "memcpy(&f, row + 4 * i, 4);", "memcpy(&f, row + 4 * (i ^ 1), 4);", FORMATS),
    ("bf16 shifted by 15 bits", C_SRC,
     "uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;", FORMATS),
    ("e4m3 NaN for the whole top binade", C_SRC,
     "if (e == 15 && m == 7)", "if (e == 15)", FORMATS),
    ("top-K indices left in score order", C_SRC,
     "    qsort(out, (size_t)m, sizeof(int32_t), cmp_i32);\n", "", TOPK),
    ("resolve: the evicted token stays in the hot map", C_SRC,
     "            hot_map[slot_token[c]] = -1;\n", "", RESOLVE),
    ("resolve: a copied row keeps its slot's old stamp", C_SRC,
     "        stamp[c] = step;\n", "", RESOLVE),
    ("attention: the mask ignored", C_SRC,
     "if (mask && !mask[rr]) {", "if (0) {", ATTENTION),
    ("attention: softmax not normalised", C_SRC,
     "            o[(size_t)h * HSO_NOPE + i] /= l;\n", "", ATTENTION),
    ("visibility one token short (Python reading)", PY_SRC,
     "    return N - nq + j + 1\n", "    return N - nq + j\n", INDEXER + " or visibility"),
    ("tail window drops its partial first page", PY_SRC,
     "        first = max(N - T, 0) // P\n", "        first = max(N - T, 0) // P + 1\n", RESOLVE),
    ("full residency charged a hot buffer", PY_SRC,
     "(0 if mode == FULL else hot_pages)", "hot_pages", PRESSURE),
    ("pressure flips the request with the fewest pages", PY_SRC,
     "most = max((self.N[x] + self.P - 1) // self.P for x in cands)",
     "most = min((self.N[x] + self.P - 1) // self.P for x in cands)", PRESSURE),
    ("pressure ties flip the higher id", PY_SRC,
     "x = min(x for x in cands if (self.N[x] + self.P - 1) // self.P == most)",
     "x = max(x for x in cands if (self.N[x] + self.P - 1) // self.P == most)", PRESSURE),
    ("pressure flips requests whose flip frees nothing", PY_SRC,
     "\n                     and self.blocks(x, MIXED) < self.blocks(x, FULL)]", "]", PRESSURE),
    ("relief returns the first flipped first", PY_SRC,
     "x = self.flipped[-1]", "x = self.flipped[0]", PRESSURE),
    ("relief without the per-request margin", PY_SRC,
     "if self.cap - self.used() < need + len(self.mode):", "if self.cap - self.used() < need:",
     PRESSURE),
]


def _sources():
    out = {}
    for name in (C_SRC, PY_SRC):
        with open(os.path.join(ORACLE, name)) as f:
            out[name] = f.read()
    return out


def _run_pins(files, workdir, selection):
    """Write the oracle package `files` under workdir/oracle, import it in a
    child process ahead of the real one (its C part built there), and run
    the selected pins against it; returns (exit code, output tail)."""
    pkg = os.path.join(workdir, "oracle")
    os.makedirs(pkg, exist_ok=True)
    for name, text in files.items():
        with open(os.path.join(pkg, name), "w") as f:
            f.write(text)
    code = (
        "import sys\n"
        f"sys.path.insert(0, {workdir!r})\n"
        "import oracle\n"
        f"assert oracle.__file__.startswith({pkg!r}), oracle.__file__\n"
        "oracle.build()\n"
        "import pytest\n"
        "sys.exit(pytest.main(['-x', '-q', '-p', 'no:cacheprovider', '-m', 'not gpu', "
        f"{PINS!r}, '-k', {selection!r}]))\n"
    )
    env = dict(os.environ, OMP_NUM_THREADS="1")  # the children run side by side
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=600, env=env)
    return r.returncode, (r.stdout + r.stderr)[-1500:]


CONTROL = "unchanged copy"


@pytest.fixture(scope="module")
def runs(tmp_path_factory):
    """Every child run at once (they are independent): name -> (exit code,
    output tail), the unchanged copy under CONTROL; None for a mutant whose
    text is missing or not unique."""
    base = tmp_path_factory.mktemp("oracle_mutants")
    jobs = {CONTROL: (_sources(), " or ".join(f"({s})" for s in sorted({m[4] for m in MUTANTS})))}
    out = {}
    for i, (name, fname, old, new, selection) in enumerate(MUTANTS):
        files = _sources()
        if files[fname].count(old) != 1:
            out[name] = None
            continue
        files[fname] = files[fname].replace(old, new)
        jobs[name] = (files, selection)
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        futs = {name: ex.submit(_run_pins, files, str(base / f"run{i}"), sel)
                for i, (name, (files, sel)) in enumerate(jobs.items())}
        out.update({name: f.result() for name, f in futs.items()})
    return out


def test_unchanged_copy_passes_every_selection(runs):
    rc, tail = runs[CONTROL]
    assert rc == 0, tail


@pytest.mark.parametrize("name,fname,old,new,selection", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(runs, name, fname, old, new, selection):
    assert runs[name] is not None, f"the text to mutate is not unique in {fname}: {old!r}"
    rc, tail = runs[name]
    assert rc == 1, f"no pin caught '{name}' (pytest exit {rc}):\n{tail}"
