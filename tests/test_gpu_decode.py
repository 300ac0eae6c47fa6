"""GPU parity of kda_decode_step against the float64 oracle.

The full decode workload (256 sequences x 32 heads, d = 128, 1000 in-place
steps over a cycled pool of 16 token sets) runs on the GPU in full; the
oracle follows a seeded sample of 64 states through all 1000 steps.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_wise_gb300 as kda
import oracle
import workloads as W
from _gpu_helpers import DEV, put, rel_err, tdtype, tol_for
from _margins import record

pytestmark = pytest.mark.gpu


def _tokens_dev(w, tk):
    dt = tdtype(w.dtype)
    return dict(q=put(tk["q"], dt), k=put(tk["k"], dt), v=put(tk["v"], dt),
                beta=put(tk["beta"]), log_alpha=put(tk["log_alpha"]))


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 32), (128, 16), (16, 128),
                                   (64, 64), (128, 128)])
@pytest.mark.parametrize("alpha", ["none", "scalar", "channel"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_shapes(dk, dv, alpha, dtype):
    w = W.Decode("dec", N=5, H=3, dk=dk, dv=dv, dtype=dtype, alpha=alpha, la_mu=-2.0,
                 S_sd=0.1, seed=dk + 3 * dv)
    S0 = W.decode_state(w)
    S = put(S0)
    S_ref = S0.astype(np.float64)
    for step in range(3):
        tk = W.decode_tokens(w, step)
        d = _tokens_dev(w, tk)
        o = kda.decode_step(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], S)
        o_ref, S_ref = oracle.decode_step(tk["q"], tk["k"], tk["v"], tk["beta"], tk["log_alpha"],
                                          S_ref)
        S_ref = S_ref.reshape(S0.shape)
        torch.cuda.synchronize()
        tol = tol_for(dtype)
        case = f"decode N=5 H=3 dk={dk} dv={dv} {dtype} {alpha}"
        eo = record(case, "o", rel_err(o.float().cpu().numpy().reshape(o_ref.shape), o_ref), tol)
        es = record(case, "S", rel_err(S.cpu().numpy(), S_ref), tol)
        assert eo <= tol and es <= tol, (step, eo, es)


def test_decode_full_workload_1000_steps_sampled_states():
    w = W.KDA_DECODE_BF16
    S0 = W.decode_state(w)
    S = put(S0)
    pool = [W.decode_tokens(w, i) for i in range(w.pool)]
    pool_dev = [_tokens_dev(w, tk) for tk in pool]
    rng = np.random.default_rng(0)
    flat = sorted(rng.choice(w.N * w.H, 64, replace=False))
    states = [(int(i) // w.H, int(i) % w.H) for i in flat]
    o_dev = torch.empty((w.N, w.H, w.dv), dtype=torch.bfloat16, device=DEV)
    o_last = []
    for step in range(w.steps):
        d = pool_dev[step % w.pool]
        kda.kda_decode_step(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], S, o_dev)
        if step >= w.steps - 3:
            o_last.append(o_dev.clone())
    torch.cuda.synchronize()
    # oracle: the sampled states through all steps
    Sref = np.stack([S0[n, h] for n, h in states]).astype(np.float64)[:, None]   # [64,1,dk,dv]
    o_ref_last = []
    for step in range(w.steps):
        tk = pool[step % w.pool]
        pick = lambda a: None if a is None else np.stack([a[n, h] for n, h in states])[:, None]
        o_ref, Sn = oracle.decode_step(pick(tk["q"]), pick(tk["k"]), pick(tk["v"]),
                                       pick(tk["beta"]), pick(tk["log_alpha"]), Sref)
        Sref = Sn[:, None]
        if step >= w.steps - 3:
            o_ref_last.append(o_ref)
    Sg = np.stack([S[n, h].cpu().numpy() for n, h in states])
    tol = tol_for(w.dtype)
    case = f"{w.name} N={w.N} H={w.H} d={w.dk}, {w.steps} steps, 64 sampled states"
    es = record(case, "S", rel_err(Sg, Sref[:, 0]), tol)
    assert es <= tol, es
    for og, orf in zip(o_last, o_ref_last):
        got = np.stack([og[n, h].float().cpu().numpy() for n, h in states])
        eo = record(case, "o (last 3 steps)", rel_err(got, orf), tol)
        assert eo <= tol, eo
