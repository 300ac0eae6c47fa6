"""kda_chunk_fwd_noalloc: the prefill entry point for callers that cannot
allocate device memory (it uses a fixed scratch array inside the library
instead of a caller workspace).

Calls it directly through the C ABI, twice in a row on different problems,
and checks each result against kda_chunk_fwd with a caller-allocated
workspace and against the float64 oracle, within the bf16 tolerance of the
other GPU tests.  Also checks that a problem needing more than the fixed
64 MiB is refused before any launch, and that a call with a bad argument
returns before it enqueues anything.  This file is named to be collected
last.
"""
import ctypes
import ctypes.util
import glob
import os

import numpy as np
import pytest
import torch

import gated_delta_rule_wise_gb300 as kda
import oracle
import workloads as W
from _gpu_helpers import TOL_BF16, device_inputs, rel_err
from _margins import case_name, record

pytestmark = pytest.mark.gpu

_P, _I = ctypes.c_void_p, ctypes.c_int


def _noalloc_fn():
    lib = kda.load_library()
    f = lib.kda_chunk_fwd_noalloc
    f.restype = _I
    f.argtypes = [_P] * 8 + [_I] * 8 + [_P]
    return f


def _ptr(t):
    return None if t is None else t.data_ptr()


def _call_noalloc(w, d, o, hT):
    f = _noalloc_fn()
    am = {"none": 0, "scalar": 1, "channel": 2}[w.alpha]
    return f(_ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]), _ptr(d["beta"]), _ptr(d["log_alpha"]),
             _ptr(d["h0"]), _ptr(o), _ptr(hT), w.B, w.H, w.T, w.dk, w.dv, w.C,
             kda.KDA_BF16, am, torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    cases = [W.KDA_PREFILL_BF16.with_(B=2, H=3, T=1000, h0_sd=0.02, seed=41),
             W.DELTANET_BF16.with_(B=1, H=5, T=777, seed=42)]
    for w in cases:
        x = W.prefill_inputs(w)
        d = device_inputs(w, x)
        o = torch.full((w.B, w.H, w.T, w.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
        hT = torch.full((w.B, w.H, w.dk, w.dv), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_noalloc(w, d, o, hT) == 0
        o_ref, h_ref = kda.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], d["h0"],
                                     C=w.C)
        torch.cuda.synchronize()
        assert rel_err(o.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= TOL_BF16
        assert rel_err(hT.cpu().numpy(), h_ref.cpu().numpy()) <= TOL_BF16
        ro, rh = oracle.recurrent_heads(x["q"], x["k"], x["v"], x["beta"], x["log_alpha"],
                                        x["h0"])
        case = case_name(w, "kda_chunk_fwd_noalloc")
        eo = record(case, "o", rel_err(o.float().cpu().numpy().reshape(ro.shape), ro), TOL_BF16)
        eh = record(case, "hT", rel_err(hT.cpu().numpy().reshape(rh.shape), rh), TOL_BF16)
        assert eo <= TOL_BF16 and eh <= TOL_BF16, (eo, eh)


def test_noalloc_refuses_problems_beyond_its_scratch():
    w = W.KDA_PREFILL_BF16.with_(B=1, H=8, T=64 * 93)   # 744 chunk records > 64 MiB
    need = kda.kda_chunk_fwd_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.C, kda.KDA_BF16, 2)
    assert need > (64 << 20)
    fake = 0x7f0000000000   # never dereferenced: the size check comes first
    f = _noalloc_fn()
    rc = f(fake, fake, fake, fake, fake, None, fake, fake, w.B, w.H, w.T, w.dk, w.dv, w.C,
           kda.KDA_BF16, 2, None)
    assert rc == 2   # KDA_ERR_UNSUPPORTED


def _cudart():
    """The CUDA runtime library, for stream-capture introspection (None if absent)."""
    cands = [ctypes.util.find_library("cudart"), "/usr/local/cuda/lib64/libcudart.so"]
    cands += sorted(glob.glob(os.path.join(os.path.dirname(torch.__file__), "lib",
                                           "libcudart*.so*")))
    cands += sorted(glob.glob("/usr/local/cuda/lib64/libcudart.so*"))
    for c in cands:
        if c:
            try:
                return ctypes.CDLL(c)
            except OSError:
                continue
    return None


def test_noalloc_rejected_call_enqueues_nothing():
    """A misaligned output pointer is refused with KDA_ERR_INVALID_ARG before
    the entry point enqueues anything: a stream capture around the refused
    call records no operation (while one around a plain copy records one)."""
    rt = _cudart()
    if rt is None:
        pytest.skip("CUDA runtime library not found for capture introspection")
    w = W.KDA_PREFILL_BF16.with_(B=1, H=2, T=100, seed=43)
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    o = torch.empty((w.B, w.H, w.T, w.dv + 8), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    assert _call_noalloc(w, d, o[..., : w.dv].contiguous(), hT) == 0   # set-up call
    torch.cuda.synchronize()
    f = _noalloc_fn()
    side = torch.cuda.Stream()
    graph = ctypes.c_void_p()
    count = ctypes.c_size_t()

    def capture(fn):
        h = ctypes.c_void_p(side.cuda_stream)
        assert rt.cudaStreamBeginCapture(h, 2) == 0          # relaxed mode
        try:
            fn(h)
        finally:
            assert rt.cudaStreamEndCapture(h, ctypes.byref(graph)) == 0
        assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(count)) == 0
        rt.cudaGraphDestroy(graph)
        return count.value

    bad_o = o.data_ptr() + 2       # not 16-byte aligned
    am = 2
    rcs = []
    nodes = capture(lambda h: rcs.append(
        f(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["beta"].data_ptr(),
          d["log_alpha"].data_ptr(), None, bad_o, hT.data_ptr(), w.B, w.H, w.T, w.dk, w.dv,
          w.C, kda.KDA_BF16, am, h)))
    assert rcs == [kda.KDA_ERR_INVALID_ARG] and nodes == 0
    src = torch.zeros(256, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    rt.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                   ctypes.c_int, ctypes.c_void_p]
    assert capture(lambda h: rt.cudaMemcpyAsync(dst.data_ptr(), src.data_ptr(), 256, 3, h)) == 1
