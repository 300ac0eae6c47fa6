"""GPU parity of kda_chunk_fwd against the float64 oracle.

Bar: max|o_gpu - o_ref| <= tol * max|o_ref| and the same for hT, with
tol = 1e-4 for float32 workloads and 2e-2 for bf16-input / float32-state ones.
Small problems are checked on every element; the full-size workloads run on
the GPU in full and are checked on a seeded sample of heads that the oracle
steps through the whole sequence.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_wise_gb300 as kda
import oracle
import workloads as W
from _gpu_helpers import (DEV, TOL_BF16, TOL_F32, device_inputs, device_inputs_streamed, put,
                          rel_err, tdtype, tol_for)
from _margins import case_name, record

pytestmark = pytest.mark.gpu

PATHS = {"auto": kda.KDA_PATH_AUTO, "cuda_core": kda.KDA_PATH_CUDA_CORE,
         "tensor": kda.KDA_PATH_TENSOR, "split": kda.KDA_PATH_TENSOR_SPLIT_SCAN,
         "wide": kda.KDA_PATH_TENSOR_WIDE_SCAN, "pipelined": kda.KDA_PATH_TENSOR_PIPELINED}


def tensor_path_ok(w):
    return kda.kda_chunk_fwd_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.C,
                                            kda.KDA_BF16 if w.dtype == "bf16" else kda.KDA_F32,
                                            {"none": 0, "scalar": 1, "channel": 2}[w.alpha],
                                            kda.KDA_PATH_TENSOR) > 0


def run(w, d, path="auto", hT_out=True, h0=None):
    o, hT = kda.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"],
                          d["h0"] if h0 is None else h0, C=w.C, output_final_state=hT_out,
                          path=PATHS[path])
    torch.cuda.synchronize()
    return o, hT


def check_full(w, path="auto", x=None):
    x = x if x is not None else W.prefill_inputs(w)
    d = device_inputs(w, x)
    o, hT = run(w, d, path)
    o_ref, h_ref = oracle.recurrent_heads(x["q"], x["k"], x["v"], x["beta"], x["log_alpha"],
                                          x["h0"])
    tol = tol_for(w.dtype)
    eo = rel_err(o.float().cpu().numpy().reshape(o_ref.shape), o_ref)
    eh = rel_err(hT.cpu().numpy().reshape(h_ref.shape), h_ref)
    record(case_name(w, path), "o", eo, tol)
    record(case_name(w, path), "hT", eh, tol)
    assert eo <= tol and eh <= tol, f"{w.name} [{path}]: o {eo:.3e} hT {eh:.3e} (tol {tol})"
    return eo, eh


# ---------------------------------------------------------------- the five workloads

def test_tiny_kda_fp32():
    check_full(W.TINY_KDA_FP32)


@pytest.mark.parametrize("path", ["auto", "cuda_core"])
def test_deltanet_bf16(path):
    check_full(W.DELTANET_BF16, path)


def _sampled(w, n_heads, path="auto", seed=0):
    d = device_inputs_streamed(w)
    o, hT = run(w, d, path)
    rng = np.random.default_rng(seed)
    all_heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    pick = [all_heads[i] for i in sorted(rng.choice(len(all_heads), n_heads, replace=False))]
    x = W.prefill_inputs(w, heads=pick)
    o_ref, h_ref = oracle.recurrent_heads(x["q"][:, None], x["k"][:, None], x["v"][:, None],
                                          x["beta"][:, None],
                                          None if x["log_alpha"] is None else x["log_alpha"][:, None],
                                          None if x["h0"] is None else x["h0"][:, None])
    og = torch.stack([o[b, h] for b, h in pick]).float().cpu().numpy()
    hg = torch.stack([hT[b, h] for b, h in pick]).cpu().numpy()
    tol = tol_for(w.dtype)
    eo, eh = rel_err(og, o_ref), rel_err(hg, h_ref)
    case = f"{case_name(w, path)}, {n_heads} sampled heads"
    record(case, "o", eo, tol)
    record(case, "hT", eh, tol)
    # per head as well: the worst head's error is the margin that matters
    for i, (b, h) in enumerate(pick):
        record(case, f"o h{b}.{h}", rel_err(og[i], o_ref[i]), tol)
    assert eo <= tol and eh <= tol, f"{w.name} [{path}] sampled: o {eo:.3e} hT {eh:.3e}"


def test_gdn_bf16_sampled_heads():
    _sampled(W.GDN_BF16, 12)


@pytest.mark.slow
def test_kda_prefill_bf16_full_size_sampled_heads():
    _sampled(W.KDA_PREFILL_BF16, 16, seed=1)


@pytest.mark.slow
def test_kda_prefill_bf16_full_size_wide_scan_sampled_heads():
    """The full KDA workload through the one-CTA-per-head scan (the automatic
    choice takes the split scan for its 32 heads)."""
    _sampled(W.KDA_PREFILL_BF16, 8, path="wide", seed=2)


def test_gdn_bf16_wide_scan_sampled_heads():
    """Gated DeltaNet (128 heads, h0 given) through the one-CTA-per-head scan
    as well (the automatic choice is the value-column split scan)."""
    _sampled(W.GDN_BF16, 6, path="wide", seed=4)


# ---------------------------------------------------------------- the two scans of the tensor path

@pytest.mark.parametrize("alpha", ["none", "scalar", "channel"])
@pytest.mark.parametrize("B,H,T", [(1, 2, 3 * 64 + 33), (2, 3, 64), (1, 1, 1), (1, 5, 700),
                                   (1, 3, 64 * 7 + 63)])
def test_wide_scan_matches_oracle(alpha, B, H, T):
    """One scan CTA per (batch, head): several chunks, ragged last chunk,
    initial state, every decay mode."""
    w = W.Prefill("wide", B=B, H=H, T=T, dk=128, dv=128, C=64, dtype="bf16", alpha=alpha,
                  la_mu=-3.5, h0_sd=0.05, seed=T + 7 * H + len(alpha))
    check_full(w, "wide")


# ---------------------------------------------------------------- the pipelined call

@pytest.mark.parametrize("alpha", ["none", "scalar", "channel"])
@pytest.mark.parametrize("B,H,T", [(1, 3, 64 * 37 + 19), (2, 2, 64 * 16), (1, 2, 64 * 8 + 5),
                                   (1, 1, 64 * 130 + 1)])
def test_pipelined_matches_oracle(alpha, B, H, T):
    """Segments of the sequence, each prep beside the previous segment's
    scan: 4 segments with a short last one and a partial last chunk, 2
    segments, a single segment (9 chunks), and 15 segments (14 of 9 chunks,
    the last of 5 ending in a one-token chunk); initial state, every decay
    mode."""
    w = W.Prefill("pipelined", B=B, H=H, T=T, dk=128, dv=128, C=64, dtype="bf16", alpha=alpha,
                  la_mu=-3.5, h0_sd=0.05, seed=T + 11 * H + len(alpha))
    check_full(w, "pipelined")


def test_pipelined_segment_count():
    """The launches of a pipelined call: prep and scan per segment, the one-CTA-
    per-head scan except for the last segment's split scan."""
    names = kda.kda_chunk_fwd_kernel_names(1, 3, 64 * 37 + 19, 128, 128, 64, kda.KDA_BF16,
                                           kda.KDA_ALPHA_CHANNEL, kda.KDA_PATH_TENSOR_PIPELINED)
    assert names == ["kda_prep_kernel", "kda_scan_wide_kernel"] * 3 + \
        ["kda_prep_kernel", "kda_scan_kernel"]


def test_pipelined_without_final_state():
    """No hT: the state between segments lives in the workspace."""
    w = W.KDA_PREFILL_BF16.with_(B=1, H=2, T=64 * 40 + 3, h0_sd=0.02, seed=31)
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    o, hT = run(w, d, "pipelined", hT_out=False)
    assert hT is None
    o_ref, _ = oracle.recurrent_heads(x["q"], x["k"], x["v"], x["beta"], x["log_alpha"], x["h0"])
    tol = tol_for(w.dtype)
    eo = rel_err(o.float().cpu().numpy().reshape(o_ref.shape), o_ref)
    record(case_name(w, "pipelined") + ", no hT", "o", eo, tol)
    assert eo <= tol, f"o {eo:.3e}"


def test_pipelined_rejected_at_d64():
    w = W.DELTANET_BF16.with_(B=1, H=1, T=64 * 20)
    d = device_inputs(w, W.prefill_inputs(w))
    with pytest.raises(kda.KdaError) as e:
        run(w, d, "pipelined")
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED


@pytest.mark.slow
def test_kda_prefill_bf16_full_size_pipelined_sampled_heads():
    """The full KDA workload as a pipelined call (16 segments of 128 chunks)."""
    _sampled(W.KDA_PREFILL_BF16, 8, path="pipelined", seed=3)


@pytest.mark.parametrize("alpha", ["none", "scalar", "channel"])
def test_split_scan_64_columns_matches_oracle(alpha):
    """48 heads: four 32-column scan CTAs per head would take two rounds of
    the GPU's SMs, so each head gets two 64-column CTAs (two record stages);
    every head against the oracle, ragged last chunk, initial state."""
    w = W.Prefill("split64", B=2, H=24, T=64 * 5 + 7, dk=128, dv=128, C=64, dtype="bf16",
                  alpha=alpha, la_mu=-3.5, h0_sd=0.05, seed=41 + len(alpha))
    check_full(w, "split")
    check_full(w, "pipelined")


def test_wide_scan_long_sequence_many_chunks():
    w = W.KDA_PREFILL_BF16.with_(B=1, H=4, T=64 * 300 + 17, h0_sd=0.02, seed=23)
    check_full(w, "wide")


def test_wide_scan_empty_sequence_copies_initial_state():
    w = W.GDN_BF16.with_(B=2, H=3, T=0)
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    o, hT = run(w, d, "wide")
    np.testing.assert_array_equal(hT.cpu().numpy(), x["h0"])


def test_wide_scan_rejected_at_d64():
    w = W.DELTANET_BF16.with_(B=1, H=1, T=64)
    d = device_inputs(w, W.prefill_inputs(w))
    with pytest.raises(kda.KdaError) as e:
        run(w, d, "wide")
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED


# ---------------------------------------------------------------- shapes and edge cases

SHAPES = [(16, 16, 16), (32, 16, 16), (16, 64, 32), (64, 64, 64), (128, 64, 64),
          (64, 128, 64), (128, 128, 64), (128, 32, 32), (32, 128, 16)]


@pytest.mark.parametrize("dk,dv,C", SHAPES)
@pytest.mark.parametrize("alpha", ["none", "scalar", "channel"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_shapes_modes_ragged_tail(dk, dv, C, alpha, dtype):
    """Several chunks plus a partial last chunk, two heads, initial state."""
    w = W.Prefill("shape", B=1, H=2, T=3 * C + C // 2 + 1, dk=dk, dv=dv, C=C, dtype=dtype,
                  alpha=alpha, la_mu=-3.5, h0_sd=0.05, seed=dk * 7 + dv + C)
    check_full(w, "auto")
    if dtype == "bf16":
        check_full(w, "cuda_core")


@pytest.mark.parametrize("T", [1, 5, 63, 64, 65, 130])
def test_lengths_around_the_chunk(T):
    check_full(W.KDA_PREFILL_BF16.with_(B=2, H=1, T=T, h0_sd=0.02, seed=T))


def test_empty_sequence_copies_initial_state():
    w = W.GDN_BF16.with_(B=2, H=3, T=0)
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    o, hT = run(w, d)
    assert o.numel() == 0
    np.testing.assert_array_equal(hT.cpu().numpy(), x["h0"])


def test_in_place_state_and_split_resume():
    """h0 == hT is allowed; [0, T1) then [T1, T) from the carried state gives
    the oracle's one-pass o and hT (the state is the cache handed from call
    to call)."""
    w = W.KDA_PREFILL_BF16.with_(B=1, H=3, T=320, h0_sd=0.02, seed=77)
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    T1 = 192
    sl = lambda t, a, b: None if t is None else t[:, :, a:b].contiguous()
    S = d["h0"].clone()
    outs = []
    for a, b in ((0, T1), (T1, w.T)):
        part = dict(q=sl(d["q"], a, b), k=sl(d["k"], a, b), v=sl(d["v"], a, b),
                    beta=sl(d["beta"], a, b), log_alpha=sl(d["log_alpha"], a, b))
        o = torch.empty_like(part["v"])
        ws = kda.workspace_for(part["q"], part["v"], w.C, part["log_alpha"])
        kda.kda_chunk_fwd(part["q"], part["k"], part["v"], part["beta"], part["log_alpha"],
                          S, o, S, w.C, ws)           # in place: h0 is hT
        outs.append(o)
    torch.cuda.synchronize()
    o_split = torch.cat(outs, dim=2)
    o_ref, h_ref = oracle.recurrent_heads(x["q"], x["k"], x["v"], x["beta"], x["log_alpha"], x["h0"])
    eo = rel_err(o_split.float().cpu().numpy().reshape(o_ref.shape), o_ref)
    eh = rel_err(S.cpu().numpy().reshape(h_ref.shape), h_ref)
    record(case_name(w) + f", split at {T1}, in place", "o", eo, TOL_BF16)
    record(case_name(w) + f", split at {T1}, in place", "hT", eh, TOL_BF16)
    assert eo <= TOL_BF16 and eh <= TOL_BF16, (eo, eh)


def test_pipelined_in_place_state_and_split_resume():
    """The pipelined call with h0 == hT (its segments then carry the state in
    the caller's buffer), resumed from that state by a second pipelined call."""
    w = W.KDA_PREFILL_BF16.with_(B=1, H=3, T=64 * 36 + 9, h0_sd=0.02, seed=78)
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    T1 = 64 * 20
    sl = lambda t, a, b: None if t is None else t[:, :, a:b].contiguous()
    S = d["h0"].clone()
    outs = []
    for a, b in ((0, T1), (T1, w.T)):
        part = dict(q=sl(d["q"], a, b), k=sl(d["k"], a, b), v=sl(d["v"], a, b),
                    beta=sl(d["beta"], a, b), log_alpha=sl(d["log_alpha"], a, b))
        o = torch.empty_like(part["v"])
        P = kda.KDA_PATH_TENSOR_PIPELINED
        ws = kda.workspace_for(part["q"], part["v"], w.C, part["log_alpha"], P)
        kda.kda_chunk_fwd_ex(part["q"], part["k"], part["v"], part["beta"], part["log_alpha"],
                             S, o, S, w.C, ws, None, P)   # in place: h0 is hT
        outs.append(o)
    torch.cuda.synchronize()
    o_split = torch.cat(outs, dim=2)
    o_ref, h_ref = oracle.recurrent_heads(x["q"], x["k"], x["v"], x["beta"], x["log_alpha"], x["h0"])
    eo = rel_err(o_split.float().cpu().numpy().reshape(o_ref.shape), o_ref)
    eh = rel_err(S.cpu().numpy().reshape(h_ref.shape), h_ref)
    record(case_name(w, "pipelined") + f", split at {T1}, in place", "o", eo, TOL_BF16)
    record(case_name(w, "pipelined") + f", split at {T1}, in place", "hT", eh, TOL_BF16)
    assert eo <= TOL_BF16 and eh <= TOL_BF16, (eo, eh)


@pytest.mark.parametrize("T,B,H", [(129, 2, 2), (64, 1, 3), (200, 1, 2)])
def test_prefill_then_decode_matches_oracle(T, B, H):
    """Prefill of the first T - 1 tokens, then one decode step on the state it
    returned: the decode output is the oracle's o at token T - 1 and the
    state is the oracle's after all T tokens (state in, state out)."""
    w = W.KDA_PREFILL_BF16.with_(B=B, H=H, T=T, seed=5 + T)
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    T0 = w.T - 1
    sl = lambda t: None if t is None else t[:, :, :T0].contiguous()
    o_p, S = kda.chunk_fwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["beta"]), sl(d["log_alpha"]),
                           None, C=w.C)
    last = lambda t: None if t is None else t[:, :, T0].contiguous()
    o_d = kda.decode_step(last(d["q"]), last(d["k"]), last(d["v"]), last(d["beta"]),
                          last(d["log_alpha"]), S)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle.recurrent_heads(x["q"], x["k"], x["v"], x["beta"], x["log_alpha"],
                                          x["h0"])
    o_ref = o_ref.reshape(B, H, T, w.dv)
    case = case_name(w) + ", prefill T-1 then decode"
    ep = record(case, "o prefill", rel_err(o_p.float().cpu().numpy(), o_ref[:, :, :T0]), TOL_BF16)
    ed = record(case, "o decode", rel_err(o_d.float().cpu().numpy(), o_ref[:, :, T0]), TOL_BF16)
    es = record(case, "S", rel_err(S.cpu().numpy().reshape(h_ref.shape), h_ref), TOL_BF16)
    assert ep <= TOL_BF16 and ed <= TOL_BF16 and es <= TOL_BF16, (ep, ed, es)


def test_unzeroed_workspace_header_reports_once_then_clears():
    """The workspace's first 256 bytes are the device error word and must be
    zero before first use.  Left holding other bytes, they make the next
    kda_chunk_fwd_status report an error no call made, and that read clears
    them; the results themselves do not depend on them."""
    w = W.KDA_PREFILL_BF16.with_(B=1, H=2, T=150, seed=9)
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    ws = kda.workspace_for(d["q"], d["v"], w.C, d["log_alpha"])
    ws.fill_(0xA5)
    o = torch.empty_like(d["v"])
    hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=DEV)
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], None, o, hT, w.C, ws)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_chunk_fwd_status(ws)
    assert e.value.status == kda.KDA_ERR_CUDA
    kda.kda_chunk_fwd_status(ws)  # cleared by that read
    o_ref, h_ref = oracle.recurrent_heads(x["q"], x["k"], x["v"], x["beta"], x["log_alpha"])
    assert rel_err(o.float().cpu().numpy().reshape(o_ref.shape), o_ref) <= TOL_BF16
    assert rel_err(hT.cpu().numpy().reshape(h_ref.shape), h_ref) <= TOL_BF16
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], None, o, hT, w.C, ws)
    kda.kda_chunk_fwd_status(ws)  # a zero header stays zero


@pytest.mark.parametrize("path", ["auto", "cuda_core"])
def test_strong_decay(path):
    """Fast-forgetting channels: exp(log_alpha) about 1.7 per token, so one
    64-token chunk decays by about e^-108 per channel.  On the d = 128 tensor
    path the split factors e^g and e^-g are taken from the middle of the
    chunk, which keeps them inside float range up to about e^-87 per half
    chunk; a chunk-start reference would overflow here."""
    w = W.Prefill("strong", B=1, H=2, T=3 * 64 + 20, dk=128, dv=128, C=64, dtype="bf16",
                  alpha="channel", la_mu=0.4, la_sd=0.5, h0_sd=0.05, seed=77)
    check_full(w, path)


def test_identity_and_no_decay_limits():
    """beta = 0 with no decay leaves S = h0; log_alpha = -inf equals no decay."""
    w = W.GDN_BF16.with_(B=1, H=2, T=200, seed=3)
    x = W.prefill_inputs(w)
    x0 = dict(x, beta=np.zeros_like(x["beta"]), log_alpha=None)
    d = device_inputs(w.with_(alpha="none"), x0)
    o, hT = run(w, d)
    np.testing.assert_allclose(hT.cpu().numpy(), x["h0"], rtol=0, atol=1e-6)
    xi = dict(x, log_alpha=np.full_like(x["log_alpha"], -np.inf))
    o1, h1 = run(w, device_inputs(w, xi))
    o2, h2 = run(w.with_(alpha="none"), device_inputs(w.with_(alpha="none"), dict(x, log_alpha=None)))
    assert rel_err(h1.cpu().numpy(), h2.cpu().numpy()) <= 1e-5
    assert rel_err(o1.float().cpu().numpy(), o2.float().cpu().numpy()) <= 1e-2


def test_timeout_selftest_reports_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    kda.kda_selftest_wait_timeout(ws, spin_limit=64)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_chunk_fwd_status(ws)
    assert e.value.status == 4  # KDA_ERR_TIMEOUT
    kda.kda_chunk_fwd_status(ws)  # cleared by the read
    check_full(W.TINY_KDA_FP32)   # the context still works
