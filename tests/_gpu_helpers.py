"""Helpers shared by the GPU parity tests: move seeded workload inputs to the
device in their storage dtype, run the library, compare with the oracle."""
import numpy as np
import torch

import workloads as W

DEV = torch.device("cuda:0")
TOL_F32 = 1e-4   # max|o_gpu - o_ref| <= TOL * max|o_ref|, float32 workloads
TOL_BF16 = 2e-2  # same bound for bf16-input / float32-state workloads


def tol_for(dtype):
    return TOL_F32 if dtype == "f32" else TOL_BF16


def tdtype(dtype):
    return torch.float32 if dtype == "f32" else torch.bfloat16


def put(a, dtype=torch.float32):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV).to(dtype)


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def device_inputs(w, x):
    """Device tensors for the arrays returned by workloads.prefill_inputs."""
    dt = tdtype(w.dtype)
    return dict(q=put(x["q"], dt), k=put(x["k"], dt), v=put(x["v"], dt),
                beta=put(x["beta"]), log_alpha=put(x["log_alpha"]), h0=put(x["h0"]))


def device_inputs_streamed(w):
    """Fill full-size device inputs head by head (no full float32 copy on the host)."""
    dt = tdtype(w.dtype)
    B, H, T = w.B, w.H, w.T
    d = dict(q=torch.empty((B, H, T, w.dk), dtype=dt, device=DEV),
             k=torch.empty((B, H, T, w.dk), dtype=dt, device=DEV),
             v=torch.empty((B, H, T, w.dv), dtype=dt, device=DEV),
             beta=torch.empty((B, H, T), dtype=torch.float32, device=DEV))
    if w.alpha == "scalar":
        d["log_alpha"] = torch.empty((B, H, T), dtype=torch.float32, device=DEV)
    elif w.alpha == "channel":
        d["log_alpha"] = torch.empty((B, H, T, w.dk), dtype=torch.float32, device=DEV)
    else:
        d["log_alpha"] = None
    d["h0"] = (torch.empty((B, H, w.dk, w.dv), dtype=torch.float32, device=DEV)
               if w.h0_sd > 0 else None)

    def sink(b, h, hd):
        for key, t in d.items():
            if t is not None:
                t[b, h].copy_(torch.from_numpy(hd[key]).to(t.dtype))

    W.prefill_inputs(w, sink=sink)
    torch.cuda.synchronize()
    return d
