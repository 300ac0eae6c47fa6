"""kda_chunk_fwd_rule on the GPU against the float64 oracle.

- KDA_RULE_LINEAR: linear attention (S = Diag(a) S + k v^T, o = S^T q) on the
  d = 128 tensor path, every decay mode, ragged last chunk, initial state.
- input maps: q, k = normalize(silu(.)) and beta = sigmoid(.) applied inside
  the prep kernel to raw projections; the oracle applies the same maps in
  float64 to the same stored values, then runs its token loop.
- KDA_RULE_LINEAR_NORM with KDA_MAP_QK_ELU1: the same linear attention with
  the ELU + 1 feature map on q, k and the normaliser (o = S^T q / q.z),
  against the oracle's normalised loop on the same stored values.
- argument checks of the new entry point.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_wise_gb300 as kda
import oracle
import workloads as W
from _gpu_helpers import DEV, TOL_BF16, device_inputs, put, rel_err
from _margins import case_name, record

pytestmark = pytest.mark.gpu


def _run_rule(d, C, rule, maps, with_hT=True):
    q = d["q"]
    B, H, T, dk = q.shape
    dv = d["v"].shape[-1]
    o = torch.empty((B, H, T, dv), dtype=q.dtype, device=DEV)
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=DEV) if with_hT else None
    ws = kda.workspace_for(q, d["v"], C, d["log_alpha"], kda.KDA_PATH_TENSOR)
    kda.kda_chunk_fwd_rule(q, d["k"], d["v"], d.get("beta"), d["log_alpha"], d["h0"], o, hT, C,
                           ws, rule, maps)
    kda.kda_chunk_fwd_status(ws)
    return o, hT


def _err(w, qty, got, ref):
    """rel_err of got against the oracle's ref, recorded as a parity margin."""
    return record(case_name(w), qty, rel_err(got, ref), TOL_BF16)


def _prefill(name, T, alpha, h0_sd, seed, H=2, B=1):
    return W.Prefill(name, B=B, H=H, T=T, dk=128, dv=128, C=64, dtype="bf16", alpha=alpha,
                     la_mu=-3.5, h0_sd=h0_sd, seed=seed)


@pytest.mark.parametrize("alpha", ["none", "scalar", "channel"])
def test_linear_attention_matches_oracle(alpha):
    w = _prefill("lin", 3 * 64 + 33, alpha, 0.05, seed=31 + len(alpha))
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    d["beta"] = None
    o, hT = _run_rule(d, w.C, kda.KDA_RULE_LINEAR, 0)
    ro, rh = oracle.linear_heads(x["q"], x["k"], x["v"], x["log_alpha"], x["h0"])
    eo = _err(w, "o", o.float().cpu().numpy().reshape(ro.shape), ro)
    eh = _err(w, "hT", hT.cpu().numpy().reshape(rh.shape), rh)
    assert eo <= TOL_BF16 and eh <= TOL_BF16, (eo, eh)


def test_linear_attention_long_sequence():
    """Many chunks: the state keeps growing without the delta correction; 512
    chunk-heads, more than the prep's persistent grid, so CTAs take several."""
    w = _prefill("lin_long", 4096, "channel", 0.0, seed=41, H=8)
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    d["beta"] = None
    o, hT = _run_rule(d, w.C, kda.KDA_RULE_LINEAR, 0)
    ro, rh = oracle.linear_heads(x["q"], x["k"], x["v"], x["log_alpha"], x["h0"])
    assert _err(w, "o", o.float().cpu().numpy().reshape(ro.shape), ro) <= TOL_BF16
    assert _err(w, "hT", hT.cpu().numpy().reshape(rh.shape), rh) <= TOL_BF16


def test_linear_attention_many_heads():
    """48 heads: the scan takes two 64-column CTAs per head (four 32-column
    ones would need two rounds of the SMs); every head against the oracle."""
    w = _prefill("lin_heads", 64 * 5 + 9, "channel", 0.05, seed=43, H=24, B=2)
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    d["beta"] = None
    o, hT = _run_rule(d, w.C, kda.KDA_RULE_LINEAR, 0)
    ro, rh = oracle.linear_heads(x["q"], x["k"], x["v"], x["log_alpha"], x["h0"])
    assert _err(w, "o", o.float().cpu().numpy().reshape(ro.shape), ro) <= TOL_BF16
    assert _err(w, "hT", hT.cpu().numpy().reshape(rh.shape), rh) <= TOL_BF16


def _raw_projections(w, seed, raw_qk=True):
    """Raw (pre-map) q, k in bf16 with a spread that exercises silu's both sides
    (only with raw_qk: unmapped keys must stay unit-norm for the delta rule to
    be stable), beta logits in float32; decay, v and h0 from the workload
    generator."""
    x = W.prefill_inputs(w)
    rng = np.random.default_rng(seed)
    shp = (w.B, w.H, w.T, w.dk)
    if raw_qk:
        x["q"] = W.round_bf16((1.5 * rng.standard_normal(shp)).astype(np.float32))
        x["k"] = W.round_bf16((1.5 * rng.standard_normal(shp) + 0.3).astype(np.float32))
    x["beta"] = (1.5 * rng.standard_normal((w.B, w.H, w.T))).astype(np.float32)
    return x


@pytest.mark.parametrize("maps", [kda.KDA_MAP_QK_SILU_NORM, kda.KDA_MAP_BETA_SIGMOID,
                                  kda.KDA_MAP_QK_SILU_NORM | kda.KDA_MAP_BETA_SIGMOID])
def test_input_maps_match_oracle(maps):
    w = _prefill("maps", 2 * 64 + 17, "channel", 0.05, seed=51 + maps)
    x = _raw_projections(w, seed=61 + maps, raw_qk=bool(maps & kda.KDA_MAP_QK_SILU_NORM))
    d = device_inputs(w, x)
    if not maps & kda.KDA_MAP_BETA_SIGMOID:  # beta must be a valid write strength then
        x["beta"] = (1.0 / (1.0 + np.exp(-x["beta"].astype(np.float64)))).astype(np.float32)
        d["beta"] = put(x["beta"])
    o, hT = _run_rule(d, w.C, kda.KDA_RULE_DELTA, maps)
    q, k, b = x["q"], x["k"], x["beta"]
    mq, mk, mb = oracle.input_maps(q if maps & 1 else None, k if maps & 1 else None,
                                   b if maps & 2 else None)
    q = mq if mq is not None else q
    k = mk if mk is not None else k
    b = mb if mb is not None else b
    ro, rh = oracle.recurrent_heads(q, k, x["v"], b, x["log_alpha"], x["h0"])
    eo = _err(w, "o", o.float().cpu().numpy().reshape(ro.shape), ro)
    eh = _err(w, "hT", hT.cpu().numpy().reshape(rh.shape), rh)
    assert eo <= TOL_BF16 and eh <= TOL_BF16, (eo, eh)


def test_input_maps_many_chunks():
    """Fused maps on the delta rule over 512 chunk-heads (more than the prep's
    persistent grid): the general prep's multi-chunk path."""
    maps = kda.KDA_MAP_QK_SILU_NORM | kda.KDA_MAP_BETA_SIGMOID
    w = _prefill("maps_long", 4096, "channel", 0.0, seed=161, H=8)
    x = _raw_projections(w, seed=162)
    d = device_inputs(w, x)
    o, hT = _run_rule(d, w.C, kda.KDA_RULE_DELTA, maps)
    mq, mk, mb = oracle.input_maps(x["q"], x["k"], x["beta"])
    ro, rh = oracle.recurrent_heads(mq, mk, x["v"], mb, x["log_alpha"], x["h0"])
    assert _err(w, "o", o.float().cpu().numpy().reshape(ro.shape), ro) <= TOL_BF16
    assert _err(w, "hT", hT.cpu().numpy().reshape(rh.shape), rh) <= TOL_BF16


def test_input_maps_with_linear_rule():
    w = _prefill("maps_lin", 3 * 64, "scalar", 0.0, seed=71)
    x = _raw_projections(w, seed=72)
    d = device_inputs(w, x)
    d["beta"] = None
    o, hT = _run_rule(d, w.C, kda.KDA_RULE_LINEAR, kda.KDA_MAP_QK_SILU_NORM)
    mq, mk, _ = oracle.input_maps(x["q"], x["k"], None)
    ro, rh = oracle.linear_heads(mq, mk, x["v"], x["log_alpha"], x["h0"])
    assert _err(w, "o", o.float().cpu().numpy().reshape(ro.shape), ro) <= TOL_BF16
    assert _err(w, "hT", hT.cpu().numpy().reshape(rh.shape), rh) <= TOL_BF16


def _norm_case(name, T, alpha, seed, H=2):
    """Raw q, k (N(0, 1.5^2), bf16, both signs so that ELU + 1 takes both
    branches), v and decay from the workload generator, zero initial state."""
    w = _prefill(name, T, alpha, 0.0, seed=seed, H=H)
    x = W.prefill_inputs(w)
    rng = np.random.default_rng(seed + 1000)
    shp = (w.B, w.H, w.T, w.dk)
    x["q"] = W.round_bf16((1.5 * rng.standard_normal(shp)).astype(np.float32))
    x["k"] = W.round_bf16((1.5 * rng.standard_normal(shp)).astype(np.float32))
    d = device_inputs(w, x)
    d["beta"] = None
    d["h0"] = None
    return w, x, d


def _norm_reference(x):
    mq, mk, _ = oracle.input_maps(x["q"], x["k"], qk_map="elu1")
    return oracle.linear_norm_heads(mq, mk, x["v"], x["log_alpha"])


@pytest.mark.parametrize("alpha", ["none", "scalar", "channel"])
def test_normalised_linear_attention_matches_oracle(alpha):
    w, x, d = _norm_case("linn", 3 * 64 + 33, alpha, seed=101 + len(alpha))
    o, _ = _run_rule(d, w.C, kda.KDA_RULE_LINEAR_NORM, kda.KDA_MAP_QK_ELU1, with_hT=False)
    ro = _norm_reference(x)
    eo = _err(w, "o", o.float().cpu().numpy().reshape(ro.shape), ro)
    assert eo <= TOL_BF16, eo


@pytest.mark.parametrize("B,H,T", [(1, 1, 1), (1, 2, 33), (2, 2, 64), (2, 3, 2 * 64 + 5)])
def test_normalised_linear_attention_edges(B, H, T):
    """One token, a single partial chunk, exactly one chunk, and batches > 1."""
    w = W.Prefill("linn_edge", B=B, H=H, T=T, dk=128, dv=128, C=64, dtype="bf16",
                  alpha="channel", la_mu=-3.5, h0_sd=0.0, seed=141 + T)
    x = W.prefill_inputs(w)
    rng = np.random.default_rng(151 + T)
    shp = (B, H, T, 128)
    x["q"] = W.round_bf16((1.5 * rng.standard_normal(shp)).astype(np.float32))
    x["k"] = W.round_bf16((1.5 * rng.standard_normal(shp)).astype(np.float32))
    d = device_inputs(w, x)
    d["beta"] = None
    d["h0"] = None
    o, _ = _run_rule(d, w.C, kda.KDA_RULE_LINEAR_NORM, kda.KDA_MAP_QK_ELU1, with_hT=False)
    ro = _norm_reference(x)
    eo = _err(w, "o", o.float().cpu().numpy().reshape(ro.shape), ro)
    assert eo <= TOL_BF16, eo


def test_normalised_linear_attention_long_sequence():
    """Many chunks: the normaliser and the state grow together chunk by chunk;
    512 chunk-heads, so the prep's CTAs take several chunks each."""
    w, x, d = _norm_case("linn_long", 4096, "channel", seed=121, H=8)
    o, _ = _run_rule(d, w.C, kda.KDA_RULE_LINEAR_NORM, kda.KDA_MAP_QK_ELU1, with_hT=False)
    ro = _norm_reference(x)
    assert _err(w, "o", o.float().cpu().numpy().reshape(ro.shape), ro) <= TOL_BF16


def test_normalised_linear_attention_constant_values():
    """v the same vector for every token: every output row is that vector."""
    w, x, d = _norm_case("linn_const", 2 * 64 + 9, "channel", seed=131)
    c = W.round_bf16(np.linspace(-2.0, 2.0, w.dv).astype(np.float32))
    d["v"] = put(np.broadcast_to(c, d["v"].shape).copy()).to(d["v"].dtype)
    o, _ = _run_rule(d, w.C, kda.KDA_RULE_LINEAR_NORM, kda.KDA_MAP_QK_ELU1, with_hT=False)
    got = o.float().cpu().numpy()
    assert np.abs(got - c).max() <= TOL_BF16 * np.abs(c).max()


def test_default_rule_equals_kda_chunk_fwd():
    w = _prefill("rule0", 2 * 64 + 5, "channel", 0.05, seed=81)
    d = device_inputs(w, W.prefill_inputs(w))
    o1, h1 = _run_rule(d, w.C, kda.KDA_RULE_DELTA, 0)
    o2, h2 = kda.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], d["h0"], w.C)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_rule_argument_checks():
    w = _prefill("args", 64, "none", 0.0, seed=91)
    d = device_inputs(w, W.prefill_inputs(w))
    bad = [(kda.KDA_RULE_LINEAR, kda.KDA_MAP_BETA_SIGMOID, kda.KDA_ERR_INVALID_ARG),
           (kda.KDA_RULE_LINEAR_NORM, kda.KDA_MAP_BETA_SIGMOID, kda.KDA_ERR_INVALID_ARG),
           (kda.KDA_RULE_DELTA, kda.KDA_MAP_QK_SILU_NORM | kda.KDA_MAP_QK_ELU1,
            kda.KDA_ERR_INVALID_ARG),
           (3, 0, kda.KDA_ERR_INVALID_ARG),
           (kda.KDA_RULE_DELTA, 8, kda.KDA_ERR_INVALID_ARG),
           (kda.KDA_RULE_DELTA, kda.KDA_MAP_QK_ELU1, kda.KDA_ERR_INVALID_ARG),
           (kda.KDA_RULE_LINEAR_NORM, kda.KDA_MAP_QK_ELU1, kda.KDA_ERR_UNSUPPORTED)]  # hT given
    for rule, maps, code in bad:
        with pytest.raises(kda.KdaError) as e:
            _run_rule(d, w.C, rule, maps)
        assert e.value.status == code, (rule, maps)
    w64 = W.Prefill("args64", B=1, H=1, T=64, dk=64, dv=64, C=64, dtype="bf16", alpha="none",
                    seed=92)
    d64 = device_inputs(w64, W.prefill_inputs(w64))
    with pytest.raises(kda.KdaError) as e:
        _run_rule(d64, 64, kda.KDA_RULE_LINEAR, 0)
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED
