"""White-box checks of the tensor-core prefill path.

The prep kernel leaves one record per (head, chunk) in the workspace.
D = 64: Ap = -Kbar^T W, Qp = Q*gamma - M W, Kbar^T, M, U^T (bf16 tiles in the
128-byte swizzled K-major operand layout) and gamma_C (float).
D = 128: Ap, Qp (swizzled tiles), B = Kbar^T U and O = M U (plain bf16 in
32-column blocks) and gamma_C.  These tests decode the
records and compare each matrix with a float64 numpy evaluation of its
definition (the chunk-wise form with cumulative decay), then check that the
tensor path and the CUDA-core path agree on o and hT.  End-to-end parity with
the oracle is in test_gpu_prefill.py.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_wise_gb300 as kda
import workloads as W
from _gpu_helpers import TOL_BF16, device_inputs, rel_err

pytestmark = pytest.mark.gpu
C = 64


def sw128_off(row, k, rows):
    katom, kk = k >> 6, k & 63
    return katom * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + (((kk >> 3) ^ (row & 7)) << 4) + (kk & 7) * 2


def untile(buf, rows, K):
    """bf16 tile bytes -> float64 [rows, K]."""
    r = np.arange(rows)[:, None]
    k = np.arange(K)[None, :]
    off = sw128_off(r, k, rows) // 2
    u16 = np.frombuffer(buf, dtype=np.uint16)
    return (u16[off].astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_blocks(buf, rows):
    """[4][rows][32] bf16 blocks of 64-byte rows whose 16-byte chunk q sits at
    position q ^ ((row >> 1) & 3) -> float64 [rows, 128]."""
    u16 = np.frombuffer(buf, dtype=np.uint16).reshape(4, rows, 4, 8)
    r = np.arange(rows)[:, None]
    pos = np.arange(4)[None, :] ^ ((r >> 1) & 3)          # [rows, 4]: position of chunk q
    u16 = u16[:, r, pos, :].reshape(4, rows, 32)
    f = (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.concatenate([f[b] for b in range(4)], axis=1)


def record_layout(D):
    if D == 128:
        return dict(AP=0, QP=32768, BI=49152, OI=81920, GC=98304, BYTES=98816)
    AP = 0
    QP = AP + D * D * 2
    KBT = QP + C * D * 2
    MM = KBT + D * C * 2
    UT = MM + C * C * 2
    GC = UT + D * C * 2
    return dict(AP=AP, QP=QP, KBT=KBT, MM=MM, UT=UT, GC=GC, BYTES=GC + D * 4)


def chunk_reference(q, k, v, beta, la):
    """float64 chunk quantities for one chunk (q, k [C, D]; v [C, D]; la [C, D] or None)."""
    loga = np.zeros_like(k) if la is None else -np.exp(la.astype(np.float64))
    g = np.cumsum(loga, axis=0)
    gam = np.exp(g)
    Kb = beta[:, None] * k * gam
    Kh = k / gam
    Qg = q * gam
    Kbar = k * gam[-1][None, :] / gam
    A = np.tril(Kb @ Kh.T, -1)
    Tm = np.linalg.inv(np.eye(len(k)) + A)
    Wm = Tm @ Kb
    U = Tm @ (beta[:, None] * v)
    M = np.tril(Qg @ Kh.T)
    return dict(AP=-Kbar.T @ Wm, QP=Qg - M @ Wm, KBT=Kbar.T, MM=M, UT=U.T, GC=gam[-1],
                BI=Kbar.T @ U, OI=M @ U)


@pytest.mark.parametrize("D,alpha", [(128, "channel"), (128, "scalar"), (64, "none"), (64, "channel")])
def test_prep_records_match_definitions(D, alpha):
    w = W.Prefill("rec", B=1, H=2, T=2 * C + 37, dk=D, dv=D, C=C, dtype="bf16", alpha=alpha,
                  la_mu=-3.0, h0_sd=0.0, seed=D + len(alpha))
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    ws = kda.workspace_for(d["q"], d["v"], C, d["log_alpha"], kda.KDA_PATH_TENSOR)
    kda.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], None, C=C,
                  path=kda.KDA_PATH_TENSOR, workspace=ws)
    torch.cuda.synchronize()
    L = record_layout(D)
    raw = ws.cpu().numpy().tobytes()
    NC = (w.T + C - 1) // C
    for h in range(w.H):
        for n in range(NC):
            base = 256 + (h * NC + n) * L["BYTES"]
            rec = raw[base: base + L["BYTES"]]
            sl = slice(n * C, min(w.T, (n + 1) * C))
            pad = lambda a: np.concatenate([a, np.zeros((C - a.shape[0],) + a.shape[1:])]) if a.shape[0] < C else a
            la = None
            if alpha == "channel":
                la = pad(x["log_alpha"][0, h, sl].astype(np.float64))
                la[sl.stop - sl.start:] = -np.inf
            elif alpha == "scalar":
                la1 = pad(x["log_alpha"][0, h, sl].astype(np.float64)[:, None])
                la1[sl.stop - sl.start:] = -np.inf
                la = np.repeat(la1, D, axis=1)
            ref = chunk_reference(pad(x["q"][0, h, sl].astype(np.float64)),
                                  pad(x["k"][0, h, sl].astype(np.float64)),
                                  pad(x["v"][0, h, sl].astype(np.float64)),
                                  pad(x["beta"][0, h, sl].astype(np.float64)), la)
            gc = np.frombuffer(rec[L["GC"]:L["BYTES"]], dtype=np.float32).astype(np.float64)
            if D == 128:
                got = dict(AP=untile(rec[L["AP"]:L["QP"]], D, D),
                           QP=untile(rec[L["QP"]:L["BI"]], C, D),
                           BI=bf16_blocks(rec[L["BI"]:L["OI"]], D),
                           OI=bf16_blocks(rec[L["OI"]:L["GC"]], C), GC=gc)
            else:
                got = dict(AP=untile(rec[L["AP"]:L["QP"]], D, D), QP=untile(rec[L["QP"]:L["KBT"]], C, D),
                           KBT=untile(rec[L["KBT"]:L["MM"]], D, C), MM=untile(rec[L["MM"]:L["UT"]], C, C),
                           UT=untile(rec[L["UT"]:L["GC"]], D, C), GC=gc)
            for key in got:
                e = rel_err(got[key], ref[key])
                assert e <= 2e-2, f"D={D} {alpha} head {h} chunk {n}: {key} rel err {e:.3e}"


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("alpha", ["none", "scalar", "channel"])
def test_tensor_path_matches_cuda_core_path(D, alpha):
    w = W.Prefill("cmp", B=2, H=3, T=5 * C + 9, dk=D, dv=D, C=C, dtype="bf16", alpha=alpha,
                  la_mu=-4.0, h0_sd=0.02, seed=3 * D + len(alpha))
    x = W.prefill_inputs(w)
    d = device_inputs(w, x)
    o1, h1 = kda.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], d["h0"], C=C,
                           path=kda.KDA_PATH_TENSOR)
    o2, h2 = kda.chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], d["h0"], C=C,
                           path=kda.KDA_PATH_CUDA_CORE)
    torch.cuda.synchronize()
    assert rel_err(o1.float().cpu().numpy(), o2.float().cpu().numpy()) <= TOL_BF16
    assert rel_err(h1.cpu().numpy(), h2.cpu().numpy()) <= TOL_BF16

