"""Planted mistakes in the oracle, on the CPU: every mutant copy of the oracle's sources must fail at least
one of the pins in test_oracle.py.

Each mutant changes one expression of the oracle: a dropped term, a wrong sign, index or operand, an
off-by-one mask or count.  It is built from a copy of the sources in a temporary folder (gcc, the
oracle's own flags) and loaded as a module of its own, so the real oracle is untouched.  The pins are
called on it one by one until one of them fails.  A mutant that no pin rejects would be a mistake the
pins cannot see.
"""
import importlib.util
import itertools
import os
import shutil
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")

# (file, original text, planted text, what the mistake is)
MUTANTS = [
    # explicit form (la_oracle.c)
    ("la_oracle.c", "long jend = causal ? i + 1 : N;", "long jend = causal ? i : N;",
     "causal mask without the diagonal"),
    ("la_oracle.c", "long jend = causal ? i + 1 : N;", "long jend = i + 1;",
     "non-causal calls masked as causal"),
    ("la_oracle.c", "w[j] = c + dot(q + i * D, k + j * D, D);", "w[j] = dot(q + i * D, k + j * D, D);",
     "constant c dropped from the weights"),
    ("la_oracle.c", "gi += w[j];", "gi += w[j] * w[j];",
     "normaliser not the row sum of the weights"),
    ("la_oracle.c", "double a = w[j] / gi; /* A_ij */", "double a = w[j]; /* A_ij */",
     "output not normalised"),
    ("la_oracle.c", "double dW = (dot(dO + i * D, v + j * D, D) - delta) / gi; /* dW_ij */",
     "double dW = (dot(dO + i * D, v + j * D, D) + delta) / gi; /* dW_ij */",
     "sign of the delta term in dW"),
    ("la_oracle.c", "double dW = (dot(dO + i * D, v + j * D, D) - delta) / gi; /* dW_ij */",
     "double dW = dot(dO + i * D, v + j * D, D) / gi; /* dW_ij */",
     "delta term dropped from dW"),
    ("la_oracle.c", "double dW = (dot(dO + i * D, v + j * D, D) - delta) / gi; /* dW_ij */",
     "double dW = (dot(dO + i * D, v + j * D, D) - delta); /* dW_ij */",
     "division by g_i dropped from dW"),
    ("la_oracle.c", "dq[i * D + d] += dW * k[j * D + d]; /* dQ_i = sum_j dW_ij k_j */",
     "dq[i * D + d] += dW * k[i * D + d]; /* dQ_i = sum_j dW_ij k_j */",
     "wrong row index in dQ"),
    ("la_oracle.c", "dk[j * D + d] += dW * q[i * D + d]; /* dK_j = sum_i dW_ij q_i */",
     "dk[j * D + d] += dW * k[i * D + d]; /* dK_j = sum_i dW_ij q_i */",
     "k in place of q in dK"),
    ("la_oracle.c", "dv[j * D + d] += Aij * dO[i * D + d]; /* dV_j = sum_i A_ij dO_i */",
     "dv[i * D + d] += Aij * dO[j * D + d]; /* dV_j = sum_i A_ij dO_i */",
     "transposed weights in dV"),
    ("la_oracle.c", "        double delta = dot(dO + i * D, o, D);                              /* delta_i = dO_i . O_i */",
     "        double delta = dot(dO + i * D, v + i * D, D);                      /* delta_i = dO_i . O_i */",
     "v_i in place of O_i in delta"),
    ("la_oracle.c", "    for (long i = a->causal ? j : 0; i < N; ++i) {",
     "    for (long i = a->causal ? j + 1 : 0; i < N; ++i) {",
     "sampled dK/dV rows skip the diagonal"),
    ("la_oracle.c", "        for (long d = 0; d < D; ++d) dq[d] += dW * k[j * D + d];",
     "        for (long d = 0; d < D; ++d) dq[d] += dW * k[i * D + d];",
     "sampled dQ rows with the wrong key index"),
    # running-state form (la_prefix.c)
    ("la_prefix.c", "            n = i + 1;\n        }\n        double gi = jb->c * (double)n;",
     "            n = i;\n        }\n        double gi = jb->c * (double)n;",
     "prefix forward count off by one"),
    ("la_prefix.c", "dk[j * D + d] = s - y[d];", "dk[j * D + d] = s + y[d];",
     "sign of y in the prefix dK"),
    ("la_prefix.c", "double s = c * ev[e];", "double s = ev[e];",
     "constant c dropped from the prefix dV"),
    ("la_prefix.c", "P[d * D + e] += q[j * D + d] * (dO[j * D + e] / gv[j]);",
     "P[d * D + e] += q[j * D + d] * dO[j * D + e];",
     "1/g dropped from the causal reverse sum P"),
    ("la_prefix.c", "dq[i * D + d] = s - dt[i] * z[d];", "dq[i * D + d] = s - dt[i] * a[d];",
     "a in place of z in the prefix dQ"),
    # recurrent form (__init__.py)
    ("__init__.py", 'S2 = _f64(S) + np.einsum("bhtd,bhte->bhde", K, V)',
     'S2 = _f64(S) + np.einsum("bhtd,bhte->bhed", K, V)', "transposed decode state"),
    ("__init__.py", 'g = c * n2 + np.einsum("bhd,bhd->bh", q, z2)',
     'g = c * n2 + np.einsum("bhd,bhd->bh", q, _f64(z))', "decode normaliser from the state before the token"),
    ("__init__.py", "n2 = np.asarray(n, dtype=np.int64) + K.shape[2]",
     "n2 = np.asarray(n, dtype=np.int64) + 1", "decode count advances by one per append"),
]


def _mutant(tmp_path, idx, fname, old, new):
    d = tmp_path / f"oracle_mutant_{idx}"
    d.mkdir()
    for f in ("la_oracle.c", "la_prefix.c", "__init__.py"):
        shutil.copy(os.path.join(ORACLE, f), d / f)
    src = (d / fname).read_text()
    assert src.count(old) == 1, f"mutation site not unique in {fname}: {old!r}"
    (d / fname).write_text(src.replace(old, new))
    name = f"oracle_mutant_{idx}"
    spec = importlib.util.spec_from_file_location(name, str(d / "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod
    spec.loader.exec_module(mod)
    mod.build(force=True)
    return mod


def _pins():
    """Every pin of test_oracle.py that takes the oracle as its first argument, with each parameter set."""
    import inspect

    import test_oracle as T
    # cheap pins first; the finite-difference pin (every input entry, twice) last
    for name, fn in sorted(vars(T).items(), key=lambda kv: ("central_differences" in kv[0], kv[0])):
        if not name.startswith("test_") or not callable(fn):
            continue
        if list(inspect.signature(fn).parameters)[:1] != ["oracle_lib"]:
            continue
        grids = []
        for m in getattr(fn, "pytestmark", []):
            if m.name == "parametrize":
                names = [s.strip() for s in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
                vals = [v if len(names) > 1 else (v,) for v in m.args[1]]
                grids.append([dict(zip(names, v)) for v in vals])
        for combo in itertools.product(*grids) if grids else [()]:
            kw = {}
            for part in combo:
                kw.update(part)
            yield name, fn, kw


def test_the_real_oracle_passes_every_pin(oracle_lib):
    """The harness itself: the unmodified oracle passes every pin it will run on the mutants."""
    n = 0
    for _, fn, kw in _pins():
        fn(oracle_lib, **kw)
        n += 1
    assert n >= 30


@pytest.mark.parametrize("idx", range(len(MUTANTS)), ids=[m[3].replace(" ", "_") for m in MUTANTS])
def test_a_planted_mistake_fails_a_pin(tmp_path, idx):
    fname, old, new, what = MUTANTS[idx]
    mod = _mutant(tmp_path, idx, fname, old, new)
    caught = None
    with np.errstate(all="ignore"):
        for name, fn, kw in _pins():
            try:
                fn(mod, **kw)
            except (AssertionError, ArithmeticError, ValueError, RuntimeError) as e:
                caught = (name, kw, type(e).__name__)
                break
    assert caught is not None, f"no pin fails for the planted mistake: {what}"
