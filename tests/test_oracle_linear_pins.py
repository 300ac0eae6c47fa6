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


# ---------------------------------------------------------------- normalised form
#
# The linear attention of the same page's section 04 with its normaliser: z = a_t z + k_t,
# o_t = S^T q_t / (q_t . z).  Pinned by the explicit causal ratio of kernel
# sums, o_t = sum_{s<=t} w_ts v_s / sum_{s<=t} w_ts with
# w_ts = sum_c q_tc k_sc e^{g_tc - g_sc} (the closed form above, evaluated for
# v and for a value of all ones), by invariants that hold for any positive
# weights, and by planted slips.


def _mapped_head(rng, T=40, dk=6, dv=5, mode="channel"):
    q, k, v, la, _ = _head(rng, T=T, dk=dk, dv=dv, mode=mode, h0=False)
    mq, mk, _ = oracle.input_maps(q, k, qk_map="elu1")
    return mq.astype(np.float32), mk.astype(np.float32), v, la


def _kernel_ratio(q, k, v, la):
    num, _ = _closed_form(q, k, v, la, None)
    den, _ = _closed_form(q, k, np.ones((q.shape[0], 1)), la, None)
    return num / den


@pytest.mark.parametrize("mode", ["none", "scalar", "channel"])
def test_linear_norm_matches_kernel_ratio(mode):
    rng = np.random.default_rng(31 + len(mode))
    q, k, v, la = _mapped_head(rng, mode=mode)
    o, _, _ = oracle.linear_norm(q, k, v, la)
    assert _close(o, _kernel_ratio(q, k, v, la))


def test_linear_norm_state_and_normaliser_closed_forms():
    rng = np.random.default_rng(37)
    q, k, v, la = _mapped_head(rng, mode="channel")
    _, hT, zT = oracle.linear_norm(q, k, v, la)
    _, h_c = _closed_form(q, k, v, la, None)
    _, z_c = _closed_form(q, k, np.ones((q.shape[0], 1)), la, None)
    assert _close(hT, h_c) and _close(zT, z_c[:, 0])


def test_linear_norm_constant_values_are_returned():
    rng = np.random.default_rng(41)
    q, k, _, la = _mapped_head(rng, mode="channel")
    c = np.array([0.5, -2.0, 3.0], np.float32)
    o, _, _ = oracle.linear_norm(q, k, np.tile(c, (q.shape[0], 1)), la)
    assert np.abs(o - c).max() <= 1e-12 * np.abs(c).max()


def test_linear_norm_first_token_reads_its_own_value():
    rng = np.random.default_rng(43)
    q, k, v, la = _mapped_head(rng, T=1, mode="channel")
    o, _, _ = oracle.linear_norm(q, k, v, la)
    assert np.abs(o[0] - v[0]).max() <= 1e-13 * np.abs(v[0]).max()


def test_elu1_map_matches_torch():
    rng = np.random.default_rng(47)
    x = 3.0 * rng.standard_normal((3, 11, 16))
    x[0, 0, :4] = 0.0
    mq, mk, _ = oracle.input_maps(x, -x, qk_map="elu1")
    tx = torch.from_numpy(x)
    # torch forms elu(x) + 1 as expm1(x) + 1: about 1e-16 absolute below zero
    assert np.allclose(mq, (torch.nn.functional.elu(tx) + 1).numpy(), rtol=1e-14, atol=1e-15)
    assert np.allclose(mk, (torch.nn.functional.elu(-tx) + 1).numpy(), rtol=1e-14, atol=1e-15)
    assert np.all(mq > 0) and np.all(mq[0, 0, :4] == 1.0)


LINEAR_NORM_MUTANTS = {
    "normaliser not decayed": ("zT[i] = ai * zT[i] + (double)kt[i];",
                               "zT[i] = zT[i] + (double)kt[i];"),
    "normaliser read with the key": ("den += (double)qt[i] * zT[i];",
                                     "den += (double)kt[i] * zT[i];"),
    "normaliser decays the new key": ("zT[i] = ai * zT[i] + (double)kt[i];",
                                      "zT[i] = ai * (zT[i] + (double)kt[i]);"),
    "no division": ("o[t * dv + j] = num / den;", "o[t * dv + j] = num;"),
    "state decays the new write": ("Si[j] = ai * Si[j] + (double)kt[i] * (double)vt[j];",
                                   "Si[j] = ai * (Si[j] + (double)kt[i] * (double)vt[j]);"),
}


def _linear_norm_pins_pass(lib):
    ok = []
    for mode in ("none", "channel", "scalar"):
        rng = np.random.default_rng(51 + len(mode))
        q, k, v, la = _mapped_head(rng, mode=mode)
        o, _, zT = oracle.linear_norm(q, k, v, la, lib=lib)
        _, z_c = _closed_form(q, k, np.ones((q.shape[0], 1)), la, None)
        ok.append(_close(o, _kernel_ratio(q, k, v, la)) and _close(zT, z_c[:, 0]))
    return ok


def test_unmodified_linear_norm_oracle_passes(tmp_path):
    assert all(_linear_norm_pins_pass(_compile(open(SRC).read(), tmp_path, "orig_n")))


@pytest.mark.parametrize("name", sorted(LINEAR_NORM_MUTANTS))
def test_planted_linear_norm_slip_is_caught(tmp_path, name):
    old, new = LINEAR_NORM_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name!r} not found once"
    lib = _compile(src.replace(old, new), tmp_path, "mut_n")
    assert not all(_linear_norm_pins_pass(lib)), f"no pin caught: {name}"


def test_linear_norm_hand_worked_golden():
    """Exact rational example (golden/hand_linear_norm_2tok.json): the
    normaliser's accumulation, its decay and the division after the write."""
    import json
    with open(os.path.join(ROOT, "tests", "golden", "hand_linear_norm_2tok.json")) as f:
        g = json.load(f)
    inp = g["inputs"]
    q, k, v = (np.array(inp[n], np.float32) for n in ("q", "k", "v"))
    num = lambda x: float("-inf") if x == "-inf" else float(x)
    la = np.array([[num(x) for x in row] for row in inp["log_alpha_channel"]], np.float32)
    for case, log_alpha in (("no_decay", None), ("channel_decay", la)):
        o, hT, zT = oracle.linear_norm(q, k, v, log_alpha)
        np.testing.assert_allclose(o, g[case]["o"], rtol=0, atol=1e-6)
        np.testing.assert_allclose(hT, g[case]["hT"], rtol=0, atol=1e-6)
        np.testing.assert_allclose(zT, g[case]["zT"], rtol=0, atol=1e-6)
