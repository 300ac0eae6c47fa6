"""Pins for the float64 oracle: each test ties it to something other than itself.

- a hand-worked example in exact rationals (golden fixture),
- closed forms (pure decay, identity),
- exact read-back facts the pages state for unit keys,
- the chunk-wise restatement, which must agree with the token-by-token loop
  for every chunk size (the pages suggest exactly this check),
- the matrix inverse for the forward substitution.

A plausible slip in the oracle (decay applied after the read, decay on the
value axis, exp(log_alpha) instead of exp(-exp(log_alpha)), a missing beta,
read-out before the write, a transposed state, a sign error in the
correction) changes at least one of these results.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_head(rng, T, dk, dv, mode, h0=False, la_mu=-3.0):
    q = rng.standard_normal((T, dk))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    k = rng.standard_normal((T, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    la = None
    if mode == "scalar":
        la = la_mu + 0.5 * rng.standard_normal(T)
    elif mode == "channel":
        la = la_mu + 0.5 * rng.standard_normal((T, dk))
    H0 = 0.1 * rng.standard_normal((dk, dv)) if h0 else None
    f = lambda a: None if a is None else a.astype(np.float32)
    return f(q), f(k), f(v), f(beta), f(la), H0


def _num(x):
    return float("-inf") if x == "-inf" else float(x)


def test_hand_worked_2x2_golden(oracle_lib):
    """Exact rational example (golden/hand_2x2.json): pins the decay order,
    the decay axis, beta, the sign of the correction and that the read-out
    follows the write."""
    with open(os.path.join(GOLDEN, "hand_2x2.json")) as f:
        g = json.load(f)
    inp = g["inputs"]
    q, k, v = (np.array(inp[n], np.float32) for n in ("q", "k", "v"))
    beta = np.array(inp["beta"], np.float32)
    o, hT = oracle.recurrent(q, k, v, beta)
    np.testing.assert_allclose(o, g["no_decay"]["o"], rtol=0, atol=1e-6)
    np.testing.assert_allclose(hT, g["no_decay"]["hT"], rtol=0, atol=1e-6)
    la = np.array([[_num(x) for x in row] for row in inp["log_alpha_channel"]], np.float32)
    o, hT = oracle.recurrent(q, k, v, beta, la)
    np.testing.assert_allclose(o, g["channel_decay"]["o"], rtol=0, atol=1e-6)
    np.testing.assert_allclose(hT, g["channel_decay"]["hT"], rtol=0, atol=1e-6)


@pytest.mark.parametrize("C", [1, 2, 5, 16, 64])
def test_forward_substitution_inverts_unit_lower(C):
    rng = np.random.default_rng(C)
    A = np.tril(rng.standard_normal((C, C)) * 0.3, -1)
    Tm = oracle.forward_substitution(A)
    np.testing.assert_allclose(Tm, np.linalg.inv(np.eye(C) + A), rtol=1e-10, atol=1e-12)
    assert np.allclose(np.triu(Tm, 1), 0.0) and np.allclose(np.diag(Tm), 1.0)


@pytest.mark.parametrize("mode", ["none", "scalar", "channel"])
@pytest.mark.parametrize("with_h0", [False, True])
@pytest.mark.parametrize("C", [1, 2, 4, 16, 64])
def test_recurrent_equals_chunked(oracle_lib, mode, with_h0, C):
    """Recurrent and chunk-wise forms agree for every chunk size, C = 1 (pure
    recurrence) through C = T (one chunk)."""
    rng = np.random.default_rng(1000 + C)
    T, dk, dv = 64, 8, 12
    q, k, v, beta, la, h0 = _rand_head(rng, T, dk, dv, mode, with_h0)
    o_r, h_r = oracle.recurrent(q, k, v, beta, la, h0)
    o_c, h_c = oracle.chunked(q, k, v, beta, la, h0, C=C)
    so, sh = np.abs(o_r).max(), np.abs(h_r).max()
    assert np.abs(o_r - o_c).max() <= 1e-12 * so
    assert np.abs(h_r - h_c).max() <= 1e-12 * sh


def test_identity_when_nothing_is_written_or_forgotten(oracle_lib):
    """beta = 0 and no decay leave S_T = h0 and o_t = h0^T q_t exactly."""
    rng = np.random.default_rng(7)
    q, k, v, beta, _, h0 = _rand_head(rng, 40, 6, 9, "none", True)
    o, hT = oracle.recurrent(q, k, v, np.zeros_like(beta), None, h0)
    np.testing.assert_array_equal(hT, h0)
    np.testing.assert_allclose(o, q.astype(np.float64) @ h0, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("mode", ["scalar", "channel"])
def test_pure_decay_closed_form(oracle_lib, mode):
    """beta = 0: S_t = Diag(prod_s exp(-exp(log_alpha_s))) h0, per key channel
    (rows of S); o_t = S_t^T q_t.  dk != dv so a decay on the wrong axis fails."""
    rng = np.random.default_rng(11)
    T, dk, dv = 30, 5, 7
    q, k, v, beta, la, h0 = _rand_head(rng, T, dk, dv, mode, True, la_mu=-1.0)
    o, hT = oracle.recurrent(q, k, v, np.zeros_like(beta), la, h0)
    lad = la.astype(np.float64)
    if mode == "scalar":
        lad = np.repeat(lad[:, None], dk, axis=1)
    logdecay = -np.cumsum(np.exp(lad), axis=0)            # [T, dk]
    for t in range(T):
        St = np.exp(logdecay[t])[:, None] * h0
        np.testing.assert_allclose(o[t], St.T @ q[t].astype(np.float64), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(hT, np.exp(logdecay[-1])[:, None] * h0, rtol=1e-12, atol=1e-15)


def test_decay_to_zero(oracle_lib):
    """Large log_alpha (alpha -> 0) with beta = 0 clears the state."""
    rng = np.random.default_rng(3)
    q, k, v, beta, _, h0 = _rand_head(rng, 8, 4, 4, "none", True)
    la = np.full((8, 4), 3.0, np.float32)    # alpha = exp(-e^3) ~ 2e-9 per step
    o, hT = oracle.recurrent(q, k, v, np.zeros_like(beta), la, h0)
    assert np.abs(hT).max() < 1e-60 and np.abs(o[-1]).max() < 1e-60


def test_orthonormal_keys_read_back_exactly(oracle_lib):
    """Unit keys, beta = 1, no decay: with orthonormal keys every written value
    reads back exactly, k_j^T S_T = v_j^T, whatever h0 held."""
    rng = np.random.default_rng(5)
    dk, dv, n = 16, 10, 12
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:n].astype(np.float32)                      # orthonormal rows
    v = rng.standard_normal((n, dv)).astype(np.float32)
    h0 = rng.standard_normal((dk, dv))
    o, hT = oracle.recurrent(keys, keys, v, np.ones(n, np.float32), None, h0)
    kd = keys.astype(np.float64)
    tol = 1e-6  # keys are float32-rounded, so orthonormality holds to ~1e-7
    np.testing.assert_allclose(kd @ hT, v, atol=tol)
    np.testing.assert_allclose(o, v, atol=tol)              # q_t = k_t reads v_t


@pytest.mark.parametrize("mode", ["none", "scalar", "channel"])
def test_unit_key_full_write_reads_back_for_any_decay(oracle_lib, mode):
    """beta_t = 1 and |k_t| = 1 give k_t^T S_t = v_t^T for any decay and any
    prior state, so q_t = k_t returns v_t: the read uses the decayed state and
    the write replaces exactly that component."""
    rng = np.random.default_rng(9)
    T, dk, dv = 50, 8, 6
    _, k, v, _, la, h0 = _rand_head(rng, T, dk, dv, mode, True, la_mu=-0.5)
    kd = k.astype(np.float64)
    k = (kd / np.linalg.norm(kd, axis=1, keepdims=True)).astype(np.float32)
    o, _ = oracle.recurrent(k, k, v, np.ones(T, np.float32), la, h0)
    np.testing.assert_allclose(o, v, atol=2e-6)


def test_repeated_key_replaces_value(oracle_lib):
    """Two full-strength writes to one key: reading it returns the second value."""
    k = np.array([[0.6, 0.8, 0.0], [0.6, 0.8, 0.0]], np.float32)
    v = np.array([[1.0, -2.0], [3.0, 0.5]], np.float32)
    o, hT = oracle.recurrent(k, k, v, np.ones(2, np.float32))
    kd = k[0].astype(np.float64)
    np.testing.assert_allclose(hT.T @ kd, v[1], atol=1e-6)


def test_scalar_decay_equals_broadcast_channel_decay(oracle_lib):
    rng = np.random.default_rng(13)
    q, k, v, beta, la, h0 = _rand_head(rng, 33, 7, 5, "scalar", True)
    o1, h1 = oracle.recurrent(q, k, v, beta, la, h0)
    o2, h2 = oracle.recurrent(q, k, v, beta, np.repeat(la[:, None], 7, axis=1), h0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(h1, h2)


def test_minus_inf_log_alpha_is_no_decay(oracle_lib):
    rng = np.random.default_rng(17)
    q, k, v, beta, _, h0 = _rand_head(rng, 20, 4, 3, "none", True)
    o1, h1 = oracle.recurrent(q, k, v, beta, None, h0)
    o2, h2 = oracle.recurrent(q, k, v, beta, np.full((20, 4), -np.inf, np.float32), h0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(h1, h2)


def test_split_and_resume(oracle_lib):
    """Running [0, T1) then [T1, T) from the carried state equals one run."""
    rng = np.random.default_rng(19)
    q, k, v, beta, la, h0 = _rand_head(rng, 48, 6, 6, "channel", True)
    o, hT = oracle.recurrent(q, k, v, beta, la, h0)
    oa, ha = oracle.recurrent(q[:20], k[:20], v[:20], beta[:20], la[:20], h0)
    ob, hb = oracle.recurrent(q[20:], k[20:], v[20:], beta[20:], la[20:], ha)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(hb, hT, rtol=1e-13, atol=1e-14)


def test_empty_sequence_returns_initial_state(oracle_lib):
    h0 = np.arange(6, dtype=np.float64).reshape(2, 3)
    e = np.zeros((0, 2), np.float32)
    o, hT = oracle.recurrent(e, e, np.zeros((0, 3), np.float32), np.zeros(0, np.float32), None, h0)
    assert o.shape == (0, 3)
    np.testing.assert_array_equal(hT, h0)


def test_heads_and_decode_wrappers_match_single_head(oracle_lib):
    rng = np.random.default_rng(23)
    B, H, T, dk, dv = 2, 3, 10, 4, 5
    arr = lambda *s: rng.standard_normal(s).astype(np.float32)
    q, k, v = arr(B, H, T, dk), arr(B, H, T, dk), arr(B, H, T, dv)
    beta = rng.uniform(0, 1, (B, H, T)).astype(np.float32)
    la = (arr(B, H, T, dk) - 2).astype(np.float32)
    h0 = rng.standard_normal((B, H, dk, dv))
    o, hT = oracle.recurrent_heads(q, k, v, beta, la, h0, threads=3)
    o1, h1 = oracle.recurrent(q[1, 2], k[1, 2], v[1, 2], beta[1, 2], la[1, 2], h0[1, 2])
    np.testing.assert_array_equal(o.reshape(B, H, T, dv)[1, 2], o1)
    np.testing.assert_array_equal(hT.reshape(B, H, dk, dv)[1, 2], h1)
    # decode = one token of the recurrence from the given state
    od, Sd = oracle.decode_step(q[:, :, 0], k[:, :, 0], v[:, :, 0], beta[:, :, 0], la[:, :, 0], h0)
    o2, h2 = oracle.recurrent(q[0, 1, :1], k[0, 1, :1], v[0, 1, :1], beta[0, 1, :1], la[0, 1, :1], h0[0, 1])
    np.testing.assert_array_equal(od[1], o2[0])
    np.testing.assert_array_equal(Sd[1], h2)
