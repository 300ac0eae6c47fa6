"""Seeded synthetic inputs for the gated delta-rule workloads.

This module is shared by the tests, the benchmark and the smoke check.  It
draws random numbers and shapes them into the distributions each workload
names; it holds none of the recurrence's arithmetic (no decay, no state
update, no read-out), so the oracle and the GPU path stay independent.

Every array it returns is float32 and holds values that are exactly
representable in the workload's storage dtype (bf16 values are rounded here,
round-to-nearest-even), so widening them to float64 for the oracle, or
narrowing them to bf16 for the GPU, is exact.

Each (batch, head) of a prefill workload, each sequence of the decode state
and each pre-generated decode token set draws from its own PCG64 stream keyed
by (seed, role, index...), so any subset can be regenerated on its own and the
result does not depend on thread count or platform.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

# stream roles (part of the PCG64 key)
_ROLE_PREFILL, _ROLE_DECODE_STATE, _ROLE_DECODE_TOKENS = 11, 12, 13


@dataclass(frozen=True)
class Prefill:
    """A chunked-prefill workload: B x H heads of T tokens each."""
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    C: int
    dtype: str          # "f32" or "bf16": storage type of q, k, v and o
    alpha: str          # "none" | "scalar" | "channel"
    la_mu: float = 0.0  # log_alpha ~ N(la_mu, la_sd)
    la_sd: float = 0.5
    h0_sd: float = 0.0  # h0 ~ N(0, h0_sd); 0 means h0 = 0 (passed as NULL)
    seed: int = 0
    kind: str = field(default="prefill")

    def with_(self, **kw):
        return replace(self, **kw)


@dataclass(frozen=True)
class Decode:
    """A decode workload: N x H independent states stepped one token at a time."""
    name: str
    N: int
    H: int
    dk: int
    dv: int
    dtype: str
    alpha: str
    la_mu: float = 0.0
    la_sd: float = 0.5
    S_sd: float = 0.02
    steps: int = 1000
    pool: int = 16      # distinct token sets, cycled over the steps
    seed: int = 0
    kind: str = field(default="decode")

    def with_(self, **kw):
        return replace(self, **kw)


TINY_KDA_FP32 = Prefill("tiny_kda_fp32", B=1, H=1, T=64, dk=16, dv=16, C=16, dtype="f32",
                        alpha="channel", la_mu=-3.0, la_sd=0.5, h0_sd=0.0, seed=0)
DELTANET_BF16 = Prefill("deltanet_bf16", B=4, H=8, T=2048, dk=64, dv=64, C=64, dtype="bf16",
                        alpha="none", h0_sd=0.0, seed=1)
GDN_BF16 = Prefill("gdn_bf16", B=8, H=16, T=8192, dk=128, dv=128, C=64, dtype="bf16",
                   alpha="scalar", la_mu=-4.0, la_sd=0.5, h0_sd=0.02, seed=2)
KDA_PREFILL_BF16 = Prefill("kda_prefill_bf16", B=1, H=32, T=131072, dk=128, dv=128, C=64,
                           dtype="bf16", alpha="channel", la_mu=-5.0, la_sd=0.5, h0_sd=0.0,
                           seed=3)
KDA_DECODE_BF16 = Decode("kda_decode_bf16", N=256, H=32, dk=128, dv=128, dtype="bf16",
                         alpha="channel", la_mu=-5.0, la_sd=0.5, S_sd=0.02, steps=1000,
                         pool=16, seed=4)

WORKLOADS = {w.name: w for w in (TINY_KDA_FP32, DELTANET_BF16, GDN_BF16, KDA_PREFILL_BF16,
                                 KDA_DECODE_BF16)}


def round_bf16(x):
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def _store(x, dtype):
    x = np.asarray(x, dtype=np.float32)
    return round_bf16(x) if dtype == "bf16" else np.ascontiguousarray(x)


def _rng(*key):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _unit_rows(g, n, d):
    x = g.standard_normal((n, d), dtype=np.float32)
    nrm = np.sqrt(np.einsum("ij,ij->i", x, x, dtype=np.float32))
    return x / np.maximum(nrm, np.float32(1e-30))[:, None]


def _sigmoid_normal(g, shape):
    z = g.standard_normal(shape, dtype=np.float32)
    return (np.float32(1.0) / (np.float32(1.0) + np.exp(-z))).astype(np.float32)


def prefill_head(w: Prefill, b: int, h: int):
    """Inputs of one (b, h) head: dict with q, k [T, dk], v [T, dv], beta [T],
    log_alpha ([T], [T, dk] or None) and h0 ([dk, dv] or None)."""
    g = _rng(w.seed, _ROLE_PREFILL, b, h)
    q = _store(_unit_rows(g, w.T, w.dk), w.dtype)
    k = _store(_unit_rows(g, w.T, w.dk), w.dtype)
    v = _store(g.standard_normal((w.T, w.dv), dtype=np.float32), w.dtype)
    beta = _sigmoid_normal(g, (w.T,))
    if w.alpha == "none":
        la = None
    else:
        shape = (w.T,) if w.alpha == "scalar" else (w.T, w.dk)
        la = (np.float32(w.la_mu) + np.float32(w.la_sd) *
              g.standard_normal(shape, dtype=np.float32)).astype(np.float32)
    h0 = None
    if w.h0_sd > 0:
        h0 = (np.float32(w.h0_sd) * g.standard_normal((w.dk, w.dv), dtype=np.float32))
    return dict(q=q, k=k, v=v, beta=beta, log_alpha=la, h0=h0)


def _threads(threads):
    return threads or max(1, min(16, os.cpu_count() or 1))


def prefill_inputs(w: Prefill, heads=None, threads=None, sink=None):
    """Inputs of a prefill workload.

    Without ``sink``: returns a dict of float32 arrays shaped [B, H, T, d]
    (log_alpha [B, H, T] / [B, H, T, dk] / None, h0 [B, H, dk, dv] / None)
    holding every head, or only ``heads`` (a list of (b, h)) stacked as
    [n, T, d] in that order.
    With ``sink(b, h, head_dict)``: calls it for every head (from worker
    threads) and returns None; used to fill large device-bound buffers
    without holding the whole workload in float32.
    """
    all_heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    sel = all_heads if heads is None else list(heads)
    if sink is not None:
        with ThreadPoolExecutor(_threads(threads)) as ex:
            list(ex.map(lambda bh: sink(bh[0], bh[1], prefill_head(w, *bh)), sel))
        return None
    n = len(sel)
    out = dict(q=np.empty((n, w.T, w.dk), np.float32), k=np.empty((n, w.T, w.dk), np.float32),
               v=np.empty((n, w.T, w.dv), np.float32), beta=np.empty((n, w.T), np.float32))
    if w.alpha == "scalar":
        out["log_alpha"] = np.empty((n, w.T), np.float32)
    elif w.alpha == "channel":
        out["log_alpha"] = np.empty((n, w.T, w.dk), np.float32)
    else:
        out["log_alpha"] = None
    out["h0"] = np.empty((n, w.dk, w.dv), np.float32) if w.h0_sd > 0 else None

    def put(i):
        d = prefill_head(w, *sel[i])
        for key, arr in out.items():
            if arr is not None:
                arr[i] = d[key]

    with ThreadPoolExecutor(_threads(threads)) as ex:
        list(ex.map(put, range(n)))
    if heads is None:
        for key, arr in list(out.items()):
            if arr is not None:
                out[key] = arr.reshape((w.B, w.H) + arr.shape[1:])
    return out


def decode_state(w: Decode, threads=None):
    """Initial decode state S0 [N, H, dk, dv], float32, N(0, S_sd)."""
    S = np.empty((w.N, w.H, w.dk, w.dv), np.float32)

    def put(n):
        g = _rng(w.seed, _ROLE_DECODE_STATE, n)
        S[n] = np.float32(w.S_sd) * g.standard_normal((w.H, w.dk, w.dv), dtype=np.float32)

    with ThreadPoolExecutor(_threads(threads)) as ex:
        list(ex.map(put, range(w.N)))
    return S


def decode_tokens(w: Decode, set_index: int):
    """Token set ``set_index``: q, k [N, H, dk], v [N, H, dv], beta [N, H],
    log_alpha ([N, H, dk], [N, H] or None)."""
    g = _rng(w.seed, _ROLE_DECODE_TOKENS, set_index)
    NH = w.N * w.H
    q = _store(_unit_rows(g, NH, w.dk), w.dtype).reshape(w.N, w.H, w.dk)
    k = _store(_unit_rows(g, NH, w.dk), w.dtype).reshape(w.N, w.H, w.dk)
    v = _store(g.standard_normal((w.N, w.H, w.dv), dtype=np.float32), w.dtype)
    beta = _sigmoid_normal(g, (w.N, w.H))
    if w.alpha == "none":
        la = None
    else:
        shape = (w.N, w.H) if w.alpha == "scalar" else (w.N, w.H, w.dk)
        la = (np.float32(w.la_mu) + np.float32(w.la_sd) *
              g.standard_normal(shape, dtype=np.float32)).astype(np.float32)
    return dict(q=q, k=k, v=v, beta=beta, log_alpha=la)
