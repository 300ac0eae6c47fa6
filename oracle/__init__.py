"""Float64 CPU oracle for the gated delta rule.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The GPU
library (``gated_delta_rule_wise_gb300``) never imports it and shares no code,
header, table or helper with it; the only thing both sides consume is the
seeded input generator in ``workloads/``, which holds none of the method's
arithmetic.

Contents
--------
``recurrent``          token-by-token recurrence of one head (plain C, float64,
                       ``kda_oracle.c``).  This is the definition every GPU
                       result is compared against.
``recurrent_heads``    the same, over ``[B, H, T, d]`` arrays, one thread per
                       head (the C call releases the GIL).
``decode_step``        one recurrent step for ``[N, H]`` states (the recurrence
                       with T = 1, starting from the given state).
``chunked``            float64 chunk-wise restatement (numpy), used only by the
                       self-checks that pin the recurrent oracle: the two must
                       agree for every chunk size.
``forward_substitution`` the row recursion that inverts a unit lower-triangular
                       matrix, as stated for the chunked DeltaNet form.
``linear``, ``linear_norm`` linear attention without and with the normaliser
                       (plain C, float64); ``input_maps`` the maps applied to
                       the projections (silu + normalise, sigmoid, ELU + 1).

Pins (``tests/test_oracle_pins.py``) tie every function to facts the pages and
the mathematics fix: a hand-worked 2x2 example, closed forms for pure decay,
exact read-back with orthonormal keys, recurrent-versus-chunked equivalence,
and the matrix inverse for the forward substitution.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")

ALPHA_NONE, ALPHA_SCALAR, ALPHA_CHANNEL = 0, 1, 2
_VERSION = 3

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``oracle/_build/libkda_oracle.so``.

    Plain gcc, no architecture flags (the same source builds on x86_64 and on
    aarch64), FMA contraction off so the float64 arithmetic is the written one.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def open_library(path):
    """Load a compiled oracle library from ``path`` and declare its C API."""
    lib = ctypes.CDLL(path)
    lib.kda_oracle_version.restype = ctypes.c_int
    if lib.kda_oracle_version() != _VERSION:
        raise RuntimeError("stale oracle build; rebuild with oracle.build(force=True)")
    f = lib.kda_oracle_recurrent
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p]
    f = lib.kda_oracle_linear
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p]
    f = lib.kda_oracle_linear_norm
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_long, ctypes.c_int,
                                         ctypes.c_int] + [ctypes.c_void_p] * 3
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


def _f32(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data


def alpha_mode_of(log_alpha, T, dk):
    """Infer the decay mode from the shape of ``log_alpha`` for one head."""
    if log_alpha is None:
        return ALPHA_NONE
    la = np.asarray(log_alpha)
    if la.shape == (T,):
        return ALPHA_SCALAR
    if la.shape == (T, dk):
        return ALPHA_CHANNEL
    raise ValueError(f"log_alpha shape {la.shape} fits neither [T] nor [T, dk]")


def recurrent(q, k, v, beta, log_alpha=None, h0=None, lib=None):
    """Token-by-token gated delta rule for one head, in float64.

    q, k: [T, dk]; v: [T, dv]; beta: [T]; log_alpha: None, [T] or [T, dk];
    h0: None or [dk, dv].  Returns (o [T, dv], hT [dk, dv]) as float64.
    ``lib`` selects another build of the same C source (the mutation tests
    use it); by default the package's own build is used.
    """
    lib = lib or _load()
    q, k, v, beta = _f32(q), _f32(k), _f32(v), _f32(beta)
    T, dk = q.shape
    dv = v.shape[1]
    if k.shape != (T, dk) or v.shape != (T, dv) or beta.shape != (T,):
        raise ValueError("shape mismatch")
    mode = alpha_mode_of(log_alpha, T, dk)
    la = _f32(log_alpha)
    h0d = None if h0 is None else np.ascontiguousarray(h0, dtype=np.float64)
    if h0d is not None and h0d.shape != (dk, dv):
        raise ValueError("h0 must be [dk, dv]")
    o = np.empty((T, dv), dtype=np.float64)
    hT = np.empty((dk, dv), dtype=np.float64)
    rc = lib.kda_oracle_recurrent(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(la),
                                  mode, _ptr(h0d), T, dk, dv, _ptr(o), _ptr(hT))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_recurrent failed with {rc}")
    return o, hT


def linear(q, k, v, log_alpha=None, h0=None, lib=None):
    """Token-by-token linear attention for one head, in float64:
    S = Diag(a_t) S + k_t v_t^T, o_t = S^T q_t (see kda_oracle_linear).

    q, k: [T, dk]; v: [T, dv]; log_alpha: None, [T] or [T, dk]; h0: None or
    [dk, dv].  Returns (o [T, dv], hT [dk, dv]) as float64.
    """
    lib = lib or _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    T, dk = q.shape
    dv = v.shape[1]
    if k.shape != (T, dk) or v.shape != (T, dv):
        raise ValueError("shape mismatch")
    mode = alpha_mode_of(log_alpha, T, dk)
    la = _f32(log_alpha)
    h0d = None if h0 is None else np.ascontiguousarray(h0, dtype=np.float64)
    o = np.empty((T, dv), dtype=np.float64)
    hT = np.empty((dk, dv), dtype=np.float64)
    rc = lib.kda_oracle_linear(_ptr(q), _ptr(k), _ptr(v), _ptr(la), mode, _ptr(h0d), T, dk,
                               dv, _ptr(o), _ptr(hT))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_linear failed with {rc}")
    return o, hT


def linear_norm(q, k, v, log_alpha=None, lib=None):
    """Token-by-token normalised linear attention for one head from a zero
    state, in float64: S = Diag(a_t) S + k_t v_t^T, z = a_t z + k_t,
    o_t = S^T q_t / (q_t . z) (see kda_oracle_linear_norm).  q and k are the
    feature-mapped values (``input_maps(..., qk_map="elu1")``).

    Returns (o [T, dv], hT [dk, dv], zT [dk]) as float64.
    """
    lib = lib or _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    T, dk = q.shape
    dv = v.shape[1]
    if k.shape != (T, dk) or v.shape != (T, dv):
        raise ValueError("shape mismatch")
    mode = alpha_mode_of(log_alpha, T, dk)
    la = _f32(log_alpha)
    o = np.empty((T, dv), dtype=np.float64)
    hT = np.empty((dk, dv), dtype=np.float64)
    zT = np.empty(dk, dtype=np.float64)
    rc = lib.kda_oracle_linear_norm(_ptr(q), _ptr(k), _ptr(v), _ptr(la), mode, T, dk, dv,
                                    _ptr(o), _ptr(hT), _ptr(zT))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_linear_norm failed with {rc}")
    return o, hT, zT


def linear_norm_heads(q, k, v, log_alpha=None):
    """``linear_norm`` for every (b, h) of ``[B, H, T, d]`` inputs; o as [B*H, T, dv]."""
    B, H, T, dk = q.shape
    mode = ALPHA_NONE if log_alpha is None else (ALPHA_SCALAR if np.ndim(log_alpha) == 3
                                                 else ALPHA_CHANNEL)
    return np.stack([linear_norm(q[b, h], k[b, h], v[b, h],
                                 _alpha_slice(log_alpha, mode, b, h))[0]
                     for b in range(B) for h in range(H)])


def linear_heads(q, k, v, log_alpha=None, h0=None):
    """``linear`` for every (b, h) of ``[B, H, T, d]`` inputs; (o [B*H, T, dv], hT [B*H, dk, dv])."""
    B, H, T, dk = q.shape
    mode = ALPHA_NONE if log_alpha is None else (ALPHA_SCALAR if np.ndim(log_alpha) == 3
                                                 else ALPHA_CHANNEL)
    os_, hs = [], []
    for b in range(B):
        for h in range(H):
            o, hT = linear(q[b, h], k[b, h], v[b, h], _alpha_slice(log_alpha, mode, b, h),
                           None if h0 is None else h0[b, h])
            os_.append(o)
            hs.append(hT)
    return np.stack(os_), np.stack(hs)


def input_maps(q=None, k=None, beta_logit=None, qk_map="silu_norm"):
    """The maps the pages apply to the projections before the delta rule
    ("22,580: From GPT-2 to Kimi K3" (yichencityu.github.io), section 5.2,
    the DeltaNet forward: q = normalize(silu(q)), k = normalize(silu(k)) along
    the head dimension, beta = sigmoid(w_beta x)), in float64 on the stored
    values.

    silu(x) = x / (1 + exp(-x)); normalize(x) = x / max(||x||_2, 1e-12) over
    the last axis; sigmoid(x) = 1 / (1 + exp(-x)).  With ``qk_map="elu1"`` q
    and k take instead the feature map of the same page's linear attention,
    elu(x) + 1 = x + 1 for x > 0, exp(x) otherwise.  Returns the mapped arrays
    (None for an argument given as None).
    """
    if qk_map not in ("silu_norm", "elu1"):
        raise ValueError(qk_map)
    def silu_norm(x):
        x = np.asarray(x, dtype=np.float64)
        s = x / (1.0 + np.exp(-x))
        n = np.sqrt((s * s).sum(axis=-1, keepdims=True))
        return s / np.maximum(n, 1e-12)

    def elu1(x):
        x = np.asarray(x, dtype=np.float64)
        return np.where(x > 0.0, x + 1.0, np.exp(np.minimum(x, 0.0)))

    fmap = silu_norm if qk_map == "silu_norm" else elu1
    out_q = None if q is None else fmap(q)
    out_k = None if k is None else fmap(k)
    out_b = None if beta_logit is None else 1.0 / (1.0 + np.exp(-np.asarray(beta_logit, np.float64)))
    return out_q, out_k, out_b


def attn_res(V, w, eps=1e-6):
    """Depth mixing of AttnRes ("22,580: From GPT-2 to Kimi K3"
    (yichencityu.github.io), section 12, block_attn_res), in float64.

    V: [N+1, ..., D], the stacked block representations (blocks and the
    partial block); w: [D], the learned scoring vector.  Keys are the
    RMS-normalised values, K_n = V_n / sqrt(mean(V_n^2) + eps) (the pages'
    `norm`, read as the RMSNorm they use elsewhere, without a learned scale);
    logits_n = w . K_n; a = softmax over the block axis; h = sum_n a_n V_n.
    Returns h [..., D] as float64.
    """
    V = np.asarray(V, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    K = V / np.sqrt((V * V).mean(axis=-1, keepdims=True) + eps)
    logits = K @ w                                   # [N+1, ...]
    logits = logits - logits.max(axis=0, keepdims=True)
    a = np.exp(logits)
    a = a / a.sum(axis=0, keepdims=True)
    return (a[..., None] * V).sum(axis=0)


def _alpha_slice(log_alpha, mode, b, h):
    if mode == ALPHA_NONE or log_alpha is None:
        return None
    return log_alpha[b, h]


def recurrent_heads(q, k, v, beta, log_alpha=None, h0=None, heads=None, threads=None):
    """Run ``recurrent`` for every (b, h) of ``[B, H, T, d]`` inputs.

    log_alpha: None, [B, H, T] or [B, H, T, dk]; h0: None or [B, H, dk, dv].
    ``heads`` restricts the work to a list of (b, h) pairs; the result then
    holds only those, in that order, as (o [n, T, dv], hT [n, dk, dv]).
    """
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    heads = list(heads)
    o = np.empty((len(heads), T, dv), dtype=np.float64)
    hT = np.empty((len(heads), dk, dv), dtype=np.float64)
    mode = ALPHA_NONE if log_alpha is None else (ALPHA_SCALAR if log_alpha.ndim == 3 else ALPHA_CHANNEL)

    def one(i):
        b, h = heads[i]
        oi, hi = recurrent(q[b, h], k[b, h], v[b, h], beta[b, h],
                           _alpha_slice(log_alpha, mode, b, h),
                           None if h0 is None else h0[b, h])
        o[i] = oi
        hT[i] = hi

    nthreads = threads or default_threads()
    if nthreads <= 1 or len(heads) <= 1:
        for i in range(len(heads)):
            one(i)
    else:
        with ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(one, range(len(heads))))
    return o, hT


def decode_step(q, k, v, beta, log_alpha, S, states=None, threads=None):
    """One recurrent step for ``[N, H]`` independent states.

    q, k: [N, H, dk]; v: [N, H, dv]; beta: [N, H]; log_alpha: None, [N, H] or
    [N, H, dk]; S: [N, H, dk, dv].  Returns (o, S_new) for the listed
    ``states`` (all by default), shaped [n, dv] and [n, dk, dv].
    """
    N, H, dk = q.shape
    if states is None:
        states = [(n, h) for n in range(N) for h in range(H)]
    la = None
    if log_alpha is not None:
        la = log_alpha[:, :, None] if log_alpha.ndim == 2 else log_alpha[:, :, None, :]
    o, Sn = recurrent_heads(q[:, :, None, :], k[:, :, None, :], v[:, :, None, :],
                            beta[:, :, None], la, S, heads=states, threads=threads)
    return o[:, 0, :], Sn


def default_threads():
    return max(1, os.cpu_count() or 1)


# ---------------------------------------------------------------------------
# Chunk-wise restatement (numpy, float64), used only to pin the recurrence.
# ---------------------------------------------------------------------------

def forward_substitution(A):
    """Invert ``I + A`` for a strictly lower-triangular ``A`` by row recursion.

    This is the per-chunk forward substitution of the chunked DeltaNet form
    ("22,580: From GPT-2 to Kimi K3" (yichencityu.github.io), section 6.3,
    read for one 2-D chunk): start from ``-A``; for each row i in turn, add to
    its first i entries the row-i-weighted sum of the already finished rows;
    finally add the identity.
    """
    A = np.asarray(A, dtype=np.float64)
    C = A.shape[0]
    N = -np.tril(A, -1)
    for i in range(1, C):
        # row i of N still holds -A[i, :]; rows < i are finished.
        N[i, :i] = N[i, :i] + N[i, :] @ N[:, :i]
    return N + np.eye(C)


def chunked(q, k, v, beta, log_alpha=None, h0=None, C=16):
    """Chunk-wise gated delta rule for one head, in float64.

    Within each chunk of C tokens, with g the running sum of log(a) from the
    chunk start and gamma = exp(g) (per key channel):
      A     = strict_lower(diag(beta) (K*gamma) (K/gamma)^T)
      Tm    = (I + A)^-1                       (forward substitution)
      W     = Tm diag(beta) (K*gamma),   U = Tm diag(beta) V
      u     = U - W S
      o     = (Q*gamma) S + lower_incl((Q*gamma) (K/gamma)^T) u
      S     = Diag(gamma_C) S + (K * gamma_C / gamma)^T u
    With no decay this is the chunked DeltaNet loop of "22,580: From GPT-2 to
    Kimi K3" (yichencityu.github.io), section 6.3; the decay factors are the
    cumulative products that the gated form needs ("22580: From GPT-2 to
    Kimi3, Explained" (zharfai.com), "Gated DeltaNet adds controlled
    forgetting").  T must be a multiple of C.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    T, dk = q.shape
    dv = v.shape[1]
    if T % C:
        raise ValueError("T must be a multiple of C")
    mode = alpha_mode_of(log_alpha, T, dk)
    if mode == ALPHA_NONE:
        loga = np.zeros((T, dk))
    elif mode == ALPHA_SCALAR:
        loga = np.repeat(-np.exp(np.asarray(log_alpha, dtype=np.float64))[:, None], dk, axis=1)
    else:
        loga = -np.exp(np.asarray(log_alpha, dtype=np.float64))
    S = np.zeros((dk, dv)) if h0 is None else np.array(h0, dtype=np.float64)
    o = np.empty((T, dv))
    for c0 in range(0, T, C):
        sl = slice(c0, c0 + C)
        Q, K, V, b = q[sl], k[sl], v[sl], beta[sl]
        g = np.cumsum(loga[sl], axis=0)
        gam = np.exp(g)
        Kb = b[:, None] * (K * gam)
        Kh = K / gam
        A = np.tril(Kb @ Kh.T, -1)
        Tm = forward_substitution(A)
        W = Tm @ Kb
        U = Tm @ (b[:, None] * V)
        u = U - W @ S
        Qg = Q * gam
        o[sl] = Qg @ S + np.tril(Qg @ Kh.T) @ u
        S = gam[-1][:, None] * S + (K * (gam[-1][None, :] / gam)).T @ u
    return o, S
