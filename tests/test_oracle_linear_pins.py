"""Pins for the oracle's linear-attention loop and input maps.

Linear attention ("22,580: From GPT-2 to Kimi K3" (yichencityu.github.io),
section 6.2): S = Diag(a_t) S + k_t v_t^T, o_t = S^T q_t.  Pinned by closed
forms written with matrix products (no decay: o = Q h0 + tril(Q K^T) V and
hT = h0 + K^T V; per-channel decay: the same sums weighted by exp(g_t - g_s)),
by the pages' chunked form for several chunk sizes, and by planted slips in a
copy of the C source that these checks must catch.

Input maps (same page, section 5.2: q = normalize(silu(q)), k = normalize(silu(k)),
beta = sigmoid(.)): pinned against torch's own silu, normalize and sigmoid in
float64.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kda_oracle.c")


def _head(rng, T=40, dk=6, dv=5, mode="channel", h0=True):
    q = rng.standard_normal((T, dk)).astype(np.float32)
    k = rng.standard_normal((T, dk)).astype(np.float32)
    v = rng.standard_normal((T, dv)).astype(np.float32)
    la = None
    if mode == "channel":
        la = (-2.0 + 0.5 * rng.standard_normal((T, dk))).astype(np.float32)
    elif mode == "scalar":
        la = (-2.0 + 0.5 * rng.standard_normal(T)).astype(np.float32)
    s0 = 0.3 * rng.standard_normal((dk, dv)) if h0 else None
    return q, k, v, la, s0


def _closed_form(q, k, v, la, h0):
    """o_t = sum_{s<=t} sum_c q_tc k_sc e^{g_tc - g_sc} v_s + sum_c q_tc e^{g_tc} h0[c];
    hT = sum_s diag(e^{g_T - g_s}) k_s v_s^T + diag(e^{g_T}) h0, g = running sum of -exp(la)."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    T, dk = q.shape
    if la is None:
        g = np.zeros((T, dk))
    else:
        la = np.asarray(la, np.float64)
        step = -np.exp(la if la.ndim == 2 else np.repeat(la[:, None], dk, axis=1))
        g = np.cumsum(step, axis=0)
    w = np.exp(g[:, None, :] - g[None, :, :])          # [t, s, c]
    mask = np.tril(np.ones((T, T)))[:, :, None]
    scores = np.einsum("tc,sc,tsc->ts", q, k, w * mask)
    o = scores @ v
    hT = np.einsum("sc,sd,sc->cd", k, v, np.exp(g[-1][None, :] - g))
    if h0 is not None:
        o += (q * np.exp(g)) @ h0
        hT += np.exp(g[-1])[:, None] * h0
    return o, hT


def _chunked_pages_form(q, k, v, h0, C):
    """The pages' chunk loop with no decay: o = q_c S + tril(q_c k_c^T) v_c, then S += k_c^T v_c."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    T = q.shape[0]
    S = np.zeros((q.shape[1], v.shape[1])) if h0 is None else np.array(h0, np.float64)
    out = []
    for i in range(0, T, C):
        qc, kc, vc = q[i:i + C], k[i:i + C], v[i:i + C]
        out.append(qc @ S + np.tril(qc @ kc.T) @ vc)
        S = S + kc.T @ vc
    return np.concatenate(out), S


def _close(a, b, rel=1e-12):
    return np.abs(a - b).max() <= rel * max(np.abs(b).max(), 1e-300)


@pytest.mark.parametrize("mode", ["none", "scalar", "channel"])
@pytest.mark.parametrize("h0", [False, True])
def test_linear_matches_closed_form(mode, h0):
    rng = np.random.default_rng(7 + len(mode) + h0)
    q, k, v, la, s0 = _head(rng, mode=mode, h0=h0)
    o, hT = oracle.linear(q, k, v, la, s0)
    o_c, h_c = _closed_form(q, k, v, la, s0)
    assert _close(o, o_c) and _close(hT, h_c)


def test_linear_no_decay_is_plain_matrix_products():
    rng = np.random.default_rng(3)
    q, k, v, _, _ = _head(rng, mode="none", h0=False)
    o, hT = oracle.linear(q, k, v)
    q64, k64, v64 = (x.astype(np.float64) for x in (q, k, v))
    assert _close(o, np.tril(q64 @ k64.T) @ v64)
    assert _close(hT, k64.T @ v64)


@pytest.mark.parametrize("C", [1, 3, 8, 40])
def test_linear_equals_pages_chunked_form(C):
    rng = np.random.default_rng(11)
    q, k, v, _, s0 = _head(rng, mode="none", h0=True)
    o, hT = oracle.linear(q, k, v, None, s0)
    o_c, h_c = _chunked_pages_form(q, k, v, s0, C)
    assert _close(o, o_c) and _close(hT, h_c)


def test_linear_scalar_decay_is_channel_broadcast():
    rng = np.random.default_rng(5)
    q, k, v, la, s0 = _head(rng, mode="scalar")
    o1, h1 = oracle.linear(q, k, v, la, s0)
    o2, h2 = oracle.linear(q, k, v, np.repeat(la[:, None], q.shape[1], axis=1), s0)
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)


def test_input_maps_match_torch():
    rng = np.random.default_rng(9)
    x = 2.0 * rng.standard_normal((4, 17, 32))
    x[0, 0] = 0.0  # an all-zero row stays zero
    b = 3.0 * rng.standard_normal((4, 17))
    mq, mk, mb = oracle.input_maps(x, -x, b)
    tx = torch.from_numpy(x)
    ref_q = torch.nn.functional.normalize(torch.nn.functional.silu(tx), dim=-1, eps=1e-12)
    ref_k = torch.nn.functional.normalize(torch.nn.functional.silu(-tx), dim=-1, eps=1e-12)
    assert np.allclose(mq, ref_q.numpy(), rtol=1e-13, atol=1e-15)
    assert np.allclose(mk, ref_k.numpy(), rtol=1e-13, atol=1e-15)
    assert np.allclose(mb, torch.sigmoid(torch.from_numpy(b)).numpy(), rtol=1e-14, atol=0)
    norms = np.linalg.norm(mq, axis=-1)
    assert np.allclose(norms[norms > 0], 1.0, rtol=1e-13) and np.all(mq[0, 0] == 0)


# ---------------------------------------------------------------- planted slips

LINEAR_MUTANTS = {
    "decay also scales the new write": (
        "srow[e] = decay * srow[e] + kc * (double)v[t * dv + e];",
        "srow[e] = decay * (srow[e] + kc * (double)v[t * dv + e]);"),
    "decay read as exp(log_alpha)": (
        "decay = exp(-exp((double)log_alpha[t * dk + c]));",
        "decay = exp(-((double)log_alpha[t * dk + c]));"),
    "read-out with the key": (
        "acc += (double)q[t * dk + c] * state[(size_t)c * dv + e];",
        "acc += (double)k[t * dk + c] * state[(size_t)c * dv + e];"),
    "value index transposed": (
        "srow[e] = decay * srow[e] + kc * (double)v[t * dv + e];",
        "srow[e] = decay * srow[e] + kc * (double)v[t * dv + (e + c) % dv];"),
}


def _linear_pins_pass(lib):
    ok = []
    for mode, h0 in (("none", True), ("channel", True), ("scalar", False)):
        rng = np.random.default_rng(21 + len(mode))
        q, k, v, la, s0 = _head(rng, mode=mode, h0=h0)
        o, hT = oracle.linear(q, k, v, la, s0, lib=lib)
        o_c, h_c = _closed_form(q, k, v, la, s0)
        ok.append(_close(o, o_c) and _close(hT, h_c))
    return ok


def _compile(text, tmp_path, name):
    c, so = tmp_path / f"{name}.c", tmp_path / f"{name}.so"
    c.write_text(text)
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), str(c), "-lm"], check=True)
    return oracle.open_library(str(so))


def test_unmodified_linear_oracle_passes(tmp_path):
    assert all(_linear_pins_pass(_compile(open(SRC).read(), tmp_path, "orig")))


@pytest.mark.parametrize("name", sorted(LINEAR_MUTANTS))
def test_planted_linear_slip_is_caught(tmp_path, name):
    old, new = LINEAR_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name!r} not found once"
    lib = _compile(src.replace(old, new), tmp_path, "mut")
    assert not all(_linear_pins_pass(lib)), f"no pin caught: {name}"
