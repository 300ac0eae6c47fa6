"""The pins are sharp enough: each planted slip in the oracle fails one of them.

Each case copies ``oracle/kda_oracle.c`` to a temporary directory, applies one
textual change that a careless restatement could make, compiles the copy with
gcc on the CPU, and runs the pin checks against it.  At least one check must
fail for every mutant; the unmodified source must pass them all.
"""
import json
import os
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kda_oracle.c")
GOLDEN = os.path.join(ROOT, "tests", "golden", "hand_2x2.json")

MUTANTS = {
    "decay is exp(log_alpha)": ("a[i] = exp(-exp((double)log_alpha[t * dk + i]));",
                                "a[i] = exp(-((double)log_alpha[t * dk + i]));"),
    "scalar decay is exp(log_alpha)": ("a[i] = exp(-exp((double)log_alpha[t]));",
                                       "a[i] = exp((double)log_alpha[t]);"),
    "beta dropped": ("u[j] = bt * ((double)vt[j] - u[j]);", "u[j] = ((double)vt[j] - u[j]);"),
    "correction sign flipped": ("u[j] = bt * ((double)vt[j] - u[j]);",
                                "u[j] = bt * ((double)vt[j] + u[j]);"),
    "decay on the value axis": ("for (int j = 0; j < dv; ++j) row[j] *= a[i];",
                                "for (int j = 0; j < dv; ++j) row[j] *= a[j % dk];"),
    "read before decay": ("for (int j = 0; j < dv; ++j) u[j] += kd[i] * row[j];",
                          "for (int j = 0; j < dv; ++j) u[j] += kd[i] * row[j] / a[i];"),
    "write decayed again": ("for (int j = 0; j < dv; ++j) row[j] += kd[i] * u[j];",
                            "for (int j = 0; j < dv; ++j) row[j] += kd[i] * u[j] * a[i];"),
    "read-out uses the key": ("const double qi = (double)qt[i];", "const double qi = kd[i];"),
    "read-out of the transposed state": (
        "for (int j = 0; j < dv; ++j) ot[j] += qi * row[j];",
        "for (int j = 0; j < dv; ++j) ot[j] += qi * S[(size_t)(j % dk) * dv + (i % dv)];"),
}


def _compile(src_text, tmp_path, name):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src_text)
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), str(c), "-lm"], check=True)
    return oracle.open_library(str(so))


def _pins_pass(lib):
    """The pin checks of test_oracle_pins, as booleans, against ``lib``."""
    ok = []
    g = json.load(open(GOLDEN))
    inp = g["inputs"]
    q, k, v = (np.array(inp[n], np.float32) for n in ("q", "k", "v"))
    beta = np.array(inp["beta"], np.float32)
    o, hT = oracle.recurrent(q, k, v, beta, lib=lib)
    ok.append(np.allclose(o, g["no_decay"]["o"], atol=1e-6) and
              np.allclose(hT, g["no_decay"]["hT"], atol=1e-6))
    la = np.array([[float(x) for x in row] for row in inp["log_alpha_channel"]], np.float32)
    o, hT = oracle.recurrent(q, k, v, beta, la, lib=lib)
    ok.append(np.allclose(o, g["channel_decay"]["o"], atol=1e-6) and
              np.allclose(hT, g["channel_decay"]["hT"], atol=1e-6))
    # recurrent vs chunked, channel and scalar decay, with h0
    rng = np.random.default_rng(0)
    T, dk, dv = 32, 6, 9
    q = rng.standard_normal((T, dk)).astype(np.float32)
    k = rng.standard_normal((T, dk))
    k = (k / np.linalg.norm(k, axis=1, keepdims=True)).astype(np.float32)
    v = rng.standard_normal((T, dv)).astype(np.float32)
    b = rng.uniform(0.1, 0.9, T).astype(np.float32)
    h0 = 0.1 * rng.standard_normal((dk, dv))
    for la in ((-2 + 0.5 * rng.standard_normal((T, dk))).astype(np.float32),
               (-2 + 0.5 * rng.standard_normal(T)).astype(np.float32)):
        o_r, h_r = oracle.recurrent(q, k, v, b, la, h0, lib=lib)
        o_c, h_c = oracle.chunked(q, k, v, b, la, h0, C=8)
        ok.append(np.abs(o_r - o_c).max() <= 1e-12 * np.abs(o_c).max() and
                  np.abs(h_r - h_c).max() <= 1e-12 * np.abs(h_c).max())
    # pure decay closed form
    la = (-1 + 0.5 * rng.standard_normal((T, dk))).astype(np.float32)
    o, hT = oracle.recurrent(q, k, v, np.zeros(T, np.float32), la, h0, lib=lib)
    ok.append(np.allclose(hT, np.exp(-np.exp(la.astype(np.float64)).sum(0))[:, None] * h0,
                          rtol=1e-12, atol=1e-15))
    # unit-key full write reads back for any decay
    o, _ = oracle.recurrent(k, k, v, np.ones(T, np.float32), la, h0, lib=lib)
    ok.append(np.allclose(o, v, atol=2e-6))
    return ok


def test_unmodified_oracle_passes_every_check(tmp_path):
    lib = _compile(open(SRC).read(), tmp_path, "orig")
    assert all(_pins_pass(lib))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_slip_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name!r} not found once"
    lib = _compile(src.replace(old, new), tmp_path, "mut")
    assert not all(_pins_pass(lib)), f"no pin caught: {name}"
