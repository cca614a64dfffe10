"""The oracle's pins must reject a plausible mistake.

Each case plants one mistake in a temporary copy of the oracle's C source
(on the CPU), compiles it, and checks that the hand-derived worked examples
and the single-token closed form no longer hold.
"""
import json
import os
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "kda_oracle.c")

MUTANTS = {
    "dropped_write": ("S[i * dv + j] += kt[i] * p[j];", "S[i * dv + j] += 0.0 * kt[i] * p[j];"),
    "decay_on_columns": ("S[i * dv + j] *= a[i];", "S[i * dv + j] *= a[j];"),
    "wrong_sign": ("p[j] = bt * (ld(v, xv + j, f64) - p[j]);",
                   "p[j] = bt * (ld(v, xv + j, f64) + p[j]);"),
    "transposed_prediction": ("p[j] += S[i * dv + j] * kt[i];", "p[j] += S[j * dv + i] * kt[i];"),
    "missing_beta": ("p[j] = bt * (ld(v, xv + j, f64) - p[j]);",
                     "p[j] = (ld(v, xv + j, f64) - p[j]);"),
    "missing_scale": ("ot[j] *= scale;", "ot[j] *= 1.0;"),
    "gate_not_exponentiated": ("a[i] = exp(ld(g, xk + i, f64));", "a[i] = ld(g, xk + i, f64);"),
}


def _golden_ok(oracle, lib):
    ok = True
    for name in ("scalar_two_token.json", "matrix_two_token.json"):
        d = json.load(open(os.path.join(HERE, "golden", name)))
        dk, dv = d["dk"], d["dv"]
        S = np.array(d["h0"], dtype=np.float64).reshape(1, 1, dk, dv)
        scales = d["scale"] if isinstance(d["scale"], list) else [d["scale"]] * len(d["beta"])
        for t in range(len(d["beta"])):
            row = lambda key: np.array(d[key][t], dtype=np.float64).reshape(1, 1, -1)
            o, S = oracle.recurrent(row("q"), row("k"), row("v"), np.log(row("alpha")),
                                    np.array([[d["beta"][t]]]), cu_seqlens=np.array([0, 1]),
                                    h0=S, scale=scales[t], lib=lib)
            ok &= np.allclose(o.reshape(-1), d["o"][t], rtol=0, atol=1e-12)
        ok &= np.allclose(S.reshape(dk, dv), d["hT"], rtol=0, atol=1e-12)
    return bool(ok)


def test_unmutated_copy_passes(oracle_mod, tmp_path):
    so = tmp_path / "orig.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", SRC, "-o", str(so), "-lm"],
                   check=True)
    assert _golden_ok(oracle_mod, oracle_mod.load_library(str(so)))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_rejected(oracle_mod, tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    c = tmp_path / f"{name}.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"],
                   check=True)
    assert not _golden_ok(oracle_mod, oracle_mod.load_library(str(so)))
