"""Planted mistakes: each mutant is a copy of the oracle's C source with one
plausible error, compiled into a temporary library on the CPU.  The pins must
reject every one of them, which shows they constrain the oracle rather than
restate it.  Mutants stay memory-safe (no index is moved out of bounds)."""
import os
import shutil

import numpy as np
import pytest

import oracle
from conftest import make_tree_batch, rel_fro
from gated_deltanet_verification_gb300 import inputs as I
from pins_lib import closed_form_batch, commit_from_factors

SRC = os.path.join(os.path.dirname(oracle.__file__), "bole_oracle.c")

MUTANTS = {
    "no_decay": ("Si[e] = g * Sp[e];", "Si[e] = Sp[e];"),
    "no_write_gate": ("u[c] = bt * (v[c] - acc);", "u[c] = (v[c] - acc);"),
    "wrong_sign": ("u[c] = bt * (v[c] - acc);", "u[c] = bt * (v[c] + acc);"),
    "readout_with_k": ("acc += Si[(size_t)r * dv + c] * q[r];",
                       "acc += Si[(size_t)r * dv + c] * k[r];"),
    "sibling_leak": ("const double *Sp = (p < 0) ? S0 : snap + (size_t)p * dk * dv;",
                     "const double *Sp = (i == 0) ? S0 : snap + (size_t)(i - 1) * dk * dv;"),
    "decay_not_cumulative": ("P[i] = g * (p < 0 ? 1.0 : P[p]);", "P[i] = g;"),
    "commit_reverse_path": ("for (int t = L - 1; t >= 0; --t) {", "for (int t = 0; t < L; ++t) {"),
    "commit_skips_decay": ("for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] *= g;", ";"),
}


def _pins_pass(lib) -> bool:
    """The pin set (golden example + dense Theorem 1 + Eq. (10)) on two trees."""
    import json
    with open(os.path.join(os.path.dirname(__file__), "golden", "worked_tree3.json")) as f:
        g = json.load(f)
    gb = make_tree_batch([g["parent"]], g["S_pre"], g["q"], g["k"], g["v"], g["gamma"],
                         g["beta"])
    O, U, logP = oracle.verify(gb, nthreads=1, lib=lib)
    if not (np.allclose(O[:, 0], g["expected"]["o"], atol=1e-12)
            and np.allclose(U[:, 0], g["expected"]["u"], atol=1e-12)
            and np.allclose(np.exp(logP[:, 0]), g["expected"]["P"], atol=1e-12)):
        return False
    for a, S_exp in g["expected"]["S_commit"].items():
        S = oracle.commit(gb, accepted=np.array([int(a)], np.int32), nthreads=1, lib=lib)
        if not np.allclose(S[0, 0], S_exp, atol=1e-12):
            return False
    b = I.random_batch(5, 2, 2, 4, 6, [11, 7], 4, dtype="f32", accept="deepest")
    O, U, logP = oracle.verify(b, nthreads=1, lib=lib)
    Oc, Uc, logPc = closed_form_batch(b)
    if rel_fro(O, Oc) > 1e-10 or rel_fro(U, Uc) > 1e-10 or rel_fro(logP, logPc) > 1e-10:
        return False
    S = oracle.commit(b, nthreads=1, lib=lib)
    if rel_fro(S, commit_from_factors(b, Uc, logPc)) > 1e-10:
        return False
    return True


def test_unmodified_oracle_passes_pin_set():
    assert _pins_pass(oracle.load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"mut_{name}.c"
    path.write_text(src.replace(old, new))
    so = oracle.build(str(path), str(tmp_path / f"libmut_{name}.so"))
    lib = oracle.load(so)
    assert not _pins_pass(lib), f"pins did not catch mutant {name}"
