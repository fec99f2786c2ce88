"""The fp64 oracle against its pins, and the pins against planted mistakes.

CPU only.  ``test_pin`` runs every pin in ``oracle_pins`` on the real oracle.
``test_planted_mistake_is_caught`` builds copies of the oracle source with one
plausible mistake each (a dropped term, a wrong sign or index, a transposed
operand, an off-by-one mask) and checks that at least one pin fails on each.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
from tests import oracle_pins

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# (label, exact text in attn_oracle.c, replacement).  Each replaces the first
# occurrence only.
MUTANTS = [
    ("scale dropped", "S[(long)i * c->Skv + j] = c->scale * dot;", "S[(long)i * c->Skv + j] = dot;"),
    ("causal off by one", "if (c->causal && j > i + (c->Skv - c->Sq))", "if (c->causal && j >= i + (c->Skv - c->Sq))"),
    ("causal top-left", "if (c->causal && j > i + (c->Skv - c->Sq))", "if (c->causal && j > i)"),
    ("gqa map modulo", "int G = c->Hq / c->Hkv, hk = hq / G;\n    int i, j, t;", "int G = c->Hq / c->Hkv, hk = hq % c->Hkv;\n    int i, j, t;"),
    ("P not normalised", "p = exp(Srow[j] - m) / l;", "p = exp(Srow[j] - m);"),
    ("LSE without max", "c->lse[((long)b * c->Hq + hq) * c->Sq + i] = m + log(l);", "c->lse[((long)b * c->Hq + hq) * c->Sq + i] = log(l);"),
    ("exp sign flipped", "for (j = 0; j < c->Skv; ++j) l += exp(Srow[j] - m);", "for (j = 0; j < c->Skv; ++j) l += exp(m - Srow[j]);"),
    ("K read from V", "const double* k_row = kb + (long)j * kv_row_stride;\n            for (t = 0; t < c->d; ++t) dot", "const double* k_row = vb + (long)j * kv_row_stride;\n            for (t = 0; t < c->d; ++t) dot"),
    ("q row stride uses Hkv", "long q_row_stride = (long)c->Hq * c->d;\n    long kv_row_stride", "long q_row_stride = (long)c->Hkv * c->d;\n    long kv_row_stride"),
    ("split LSE without max", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("split mask off by one", "if (j > jmax) {", "if (j >= jmax) {"),
    ("merge not normalised", "for (t = 0; t < d; ++t) orow[t] /= wsum;", "for (t = 0; t < d; ++t) orow[t] /= 1.0;"),
    ("merge LSE missing sum", "lse[row] = M + log(wsum);", "lse[row] = M;"),
    ("merge weight sign", "w = exp(pl[s] - M);", "w = exp(M - pl[s]);"),
    ("split rule ignores min rows", "if (chunk < min_rows) chunk = min_rows;", ""),
    ("split rule floor", "chunk = ((long)L + n_splits - 1) / n_splits;", "chunk = (long)L / n_splits;"),
    ("decode gqa map modulo", "int G = c->Hq / c->Hkv, hk = hq / G, s, L = c->kv_lens[b];", "int G = c->Hq / c->Hkv, hk = hq % c->Hkv, s, L = c->kv_lens[b];"),
    ("rows: causal bound top-left", "int jmax = c->causal ? i + (c->Skv - c->Sq) : c->Skv - 1;", "int jmax = c->causal ? i : c->Skv - 1;"),
    ("window off by one", "j <= i + (c->Skv - c->Sq) - c->window)", "j < i + (c->Skv - c->Sq) - c->window)"),
    ("window sinks ignored", "if (c->window > 0 && j >= c->n_sink &&", "if (c->window > 0 && j >= 0 &&"),
    ("window rows: lower bound off by one", "int jlo = c->window > 0 ? i + (c->Skv - c->Sq) - c->window + 1 : 0;", "int jlo = c->window > 0 ? i + (c->Skv - c->Sq) - c->window : 0;"),
]


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("label,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(label, old, new, mutant_dir):
    src = open(ORACLE_SRC).read()
    assert old in src, f"mutation site for '{label}' not found in the oracle source"
    mutated = src.replace(old, new, 1)
    tag = "".join(ch if ch.isalnum() else "_" for ch in label)
    c_path = os.path.join(mutant_dir, f"m_{tag}.c")
    so_path = os.path.join(mutant_dir, f"m_{tag}.so")
    with open(c_path, "w") as f:
        f.write(mutated)
    subprocess.check_call(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-o", so_path, c_path,
                           "-lm", "-lpthread"])
    lib = oracle.load_variant(so_path)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake '{label}' passed every pin"
