"""Seeded input generator: deterministic, per-head independent, exact in the
storage dtype, and shaped like each workload's stated distribution."""
import numpy as np
import pytest

import workloads as W


def test_bf16_rounding_is_nearest_even_and_idempotent():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-9, -2.5, 3.14159, 1e-3], np.float32)
    r = W.round_bf16(x)
    assert r[0] == 1.0
    assert r[1] == 1.0                                         # 1 + 2^-8 ties to 1.0 (even)
    assert r[2] == 1.0 + 2**-7                                 # 1 + 3*2^-9 rounds up
    np.testing.assert_array_equal(W.round_bf16(r), r)
    assert np.all((r.view(np.uint32) & 0xFFFF) == 0)


def test_heads_are_independent_and_deterministic():
    w = W.DELTANET_BF16.with_(B=2, H=3, T=128)
    full = W.prefill_inputs(w, threads=2)
    sub = W.prefill_inputs(w, heads=[(1, 2), (0, 1)], threads=1)
    np.testing.assert_array_equal(sub["q"][0], full["q"][1, 2])
    np.testing.assert_array_equal(sub["v"][1], full["v"][0, 1])
    again = W.prefill_inputs(w, threads=3)
    for key in ("q", "k", "v", "beta"):
        np.testing.assert_array_equal(again[key], full[key])


@pytest.mark.parametrize("name", ["tiny_kda_fp32", "gdn_bf16", "kda_prefill_bf16"])
def test_distributions_match_the_workload(name):
    w = W.WORKLOADS[name]
    w = w.with_(T=min(w.T, 2048))
    d = W.prefill_head(w, 0, 0)
    assert d["q"].shape == (w.T, w.dk) and d["v"].shape == (w.T, w.dv)
    np.testing.assert_allclose(np.linalg.norm(d["k"], axis=1), 1.0, atol=2e-2 if w.dtype == "bf16" else 1e-6)
    assert np.all((d["beta"] > 0) & (d["beta"] < 1))
    la = d["log_alpha"]
    assert la.shape == ((w.T,) if w.alpha == "scalar" else (w.T, w.dk))
    assert abs(la.mean() - w.la_mu) < 0.05 and abs(la.std() - w.la_sd) < 0.05
    if w.dtype == "bf16":
        for key in ("q", "k", "v"):
            np.testing.assert_array_equal(W.round_bf16(d[key]), d[key])
    assert (d["h0"] is None) == (w.h0_sd == 0)


def test_decode_pool_and_state():
    w = W.KDA_DECODE_BF16.with_(N=4, H=2)
    S = W.decode_state(w, threads=2)
    assert S.shape == (4, 2, 128, 128) and abs(S.std() - 0.02) < 1e-3
    t0, t1 = W.decode_tokens(w, 0), W.decode_tokens(w, 1)
    assert t0["q"].shape == (4, 2, 128) and t0["log_alpha"].shape == (4, 2, 128)
    assert not np.array_equal(t0["k"], t1["k"])
    np.testing.assert_array_equal(W.decode_tokens(w, 0)["v"], t0["v"])
