"""kda_chunk_fwd_host: the prefill from and to host memory, pipelined over
two copy streams either by segments of the sequence (group_heads = 0: the
state carried from segment to segment in float32) or by groups of heads.
Its results must equal kda_chunk_fwd on device copies of the same inputs bit
for bit (the same kernels run on the same chunks), for segments (ragged last
segment, one segment only, with and without initial and final state) and for
every way of cutting the heads into groups; one case is also held against
the float64 oracle."""
import numpy as np
import pytest
import torch

import gated_delta_rule_wise_gb300 as kda
import oracle
import workloads as W
from _gpu_helpers import DEV, device_inputs, rel_err, tdtype, tol_for
from _margins import case_name, record

pytestmark = pytest.mark.gpu


def _pinned(a, dtype=torch.float32):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).pin_memory()


def _host_inputs(w, x):
    dt = tdtype(w.dtype)
    return dict(q=_pinned(x["q"], dt), k=_pinned(x["k"], dt), v=_pinned(x["v"], dt),
                beta=_pinned(x["beta"]), log_alpha=_pinned(x["log_alpha"]), h0=_pinned(x["h0"]))


def _run_host(w, hx, group_heads, with_hT=True):
    B, H, T = w.B, w.H, w.T
    o = torch.empty((B, H, T, w.dv), dtype=tdtype(w.dtype)).pin_memory()
    hT = torch.empty((B, H, w.dk, w.dv), dtype=torch.float32).pin_memory() if with_hT else None
    buf = kda.host_buffer_for(hx["q"], hx["v"], w.C, hx["log_alpha"], group_heads, DEV)
    stream = torch.cuda.current_stream()
    kda.kda_chunk_fwd_host(hx["q"], hx["k"], hx["v"], hx["beta"], hx["log_alpha"], hx["h0"],
                           o, hT, w.C, buf, group_heads, stream)
    kda.kda_chunk_fwd_status(buf, stream)  # synchronises; raises on a device error
    return o, hT


def _run_device(w, x, with_hT=True):
    d = device_inputs(w, x)
    o, hT = kda.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], d["h0"], w.C,
                          output_final_state=with_hT)
    torch.cuda.synchronize()
    return o.cpu(), (hT.cpu() if hT is not None else None)


CASES = [
    # tensor path, per-channel decay, initial state; 6 heads, partial last chunk
    (W.Prefill("host_tc", B=2, H=3, T=300, dk=128, dv=128, C=64, dtype="bf16", alpha="channel",
               la_mu=-4.0, h0_sd=0.05, seed=11), [1, 2, 4, 0]),
    # CUDA-core path, scalar decay, no initial state; 5 heads
    (W.Prefill("host_ffma", B=1, H=5, T=130, dk=64, dv=32, C=32, dtype="f32", alpha="scalar",
               la_mu=-3.0, h0_sd=0.0, seed=12), [0, 2, 5]),
    # D = 64 tensor path, no decay
    (W.Prefill("host_d64", B=1, H=4, T=256, dk=64, dv=64, C=64, dtype="bf16", alpha="none",
               la_mu=0.0, h0_sd=0.02, seed=13), [0, 3]),
    # a sequence shorter than one segment's chunk (one segment)
    (W.Prefill("host_short", B=1, H=2, T=40, dk=128, dv=128, C=64, dtype="bf16", alpha="channel",
               la_mu=-4.0, h0_sd=0.05, seed=14), [0, 1]),
]


@pytest.mark.parametrize("w,groups", CASES, ids=[c[0].name for c in CASES])
def test_host_api_equals_device_api(w, groups):
    x = W.prefill_inputs(w)
    o_ref, hT_ref = _run_device(w, x)
    hx = _host_inputs(w, x)
    for g in groups:
        o, hT = _run_host(w, hx, g)
        assert torch.equal(o, o_ref), f"group_heads={g}: o differs"
        assert torch.equal(hT, hT_ref), f"group_heads={g}: hT differs"
    for g in sorted({groups[0], 0}):
        o, hT = _run_host(w, hx, g, with_hT=False)
        assert hT is None and torch.equal(o, o_ref), f"group_heads={g}, no hT"


@pytest.mark.parametrize("group_heads", [0, 4])
def test_host_api_against_oracle(group_heads):
    w = CASES[0][0]
    x = W.prefill_inputs(w)
    o, hT = _run_host(w, _host_inputs(w, x), group_heads)
    ro, rh = oracle.recurrent_heads(x["q"], x["k"], x["v"], x["beta"], x["log_alpha"], x["h0"])
    tol = tol_for(w.dtype)
    case = case_name(w, f"host memory, group_heads={group_heads}")
    eo = record(case, "o", rel_err(o.float().numpy().reshape(ro.shape), ro), tol)
    eh = record(case, "hT", rel_err(hT.numpy().reshape(rh.shape), rh), tol)
    assert eo <= tol and eh <= tol, (eo, eh)


@pytest.mark.parametrize("group_heads", [0, 2])
def test_host_api_rejects_small_buffer(group_heads):
    w = CASES[0][0]
    hx = _host_inputs(w, W.prefill_inputs(w))
    need = kda.kda_chunk_fwd_host_buffer_size(w.B, w.H, w.T, w.dk, w.dv, w.C, kda.KDA_BF16,
                                              kda.KDA_ALPHA_CHANNEL, group_heads)
    small = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    o = torch.empty((w.B, w.H, w.T, w.dv), dtype=torch.bfloat16)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_chunk_fwd_host(hx["q"], hx["k"], hx["v"], hx["beta"], hx["log_alpha"], hx["h0"],
                               o, None, w.C, small, group_heads)
    assert e.value.status == kda.KDA_ERR_INVALID_ARG
