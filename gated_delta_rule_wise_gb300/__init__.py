"""GB300-native gated delta rule (DeltaNet / Gated DeltaNet / KDA).

A thin Python binding over ``libkda.so``, whose C ABI is ``include/kda.h``.
The functions named like the C entry points (``kda_chunk_fwd``,
``kda_decode_step``, ...) only marshal arguments: they read shapes and
device pointers off torch tensors, call the C function on the current (or
given) CUDA stream and turn a non-OK status into ``KdaError``.  Every step of
the computation runs in the library's CUDA kernels; there is no Python or
CPU fallback, and importing a function whose library is missing raises.

``chunk_fwd`` and ``decode_step`` are conveniences that also allocate the
outputs and the workspace with torch.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "KdaError", "library_path", "load_library", "kda_abi_version", "kda_status_string",
    "kda_chunk_fwd", "kda_chunk_fwd_ex", "kda_chunk_fwd_workspace_size",
    "kda_chunk_fwd_status", "kda_decode_step", "kda_selftest_wait_timeout",
    "kda_chunk_fwd_launches", "kda_chunk_fwd_kernel_names", "kernel_sources",
    "kda_chunk_fwd_host", "kda_chunk_fwd_host_buffer_size", "host_buffer_for",
    "kda_chunk_fwd_rule", "KDA_RULE_DELTA", "KDA_RULE_LINEAR", "KDA_RULE_LINEAR_NORM",
    "KDA_MAP_QK_SILU_NORM", "KDA_MAP_BETA_SIGMOID", "KDA_MAP_QK_ELU1", "kda_attn_res", "attn_res",
    "chunk_fwd", "decode_step", "workspace_for",
    "KDA_F32", "KDA_BF16", "KDA_ALPHA_NONE", "KDA_ALPHA_SCALAR", "KDA_ALPHA_CHANNEL",
    "KDA_PATH_AUTO", "KDA_PATH_CUDA_CORE", "KDA_PATH_TENSOR", "KDA_PATH_TENSOR_SPLIT_SCAN",
    "KDA_PATH_TENSOR_WIDE_SCAN", "KDA_PATH_TENSOR_PIPELINED",
]

_PKG = os.path.dirname(os.path.abspath(__file__))

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = range(5)
KDA_F32, KDA_BF16 = 0, 1
KDA_ALPHA_NONE, KDA_ALPHA_SCALAR, KDA_ALPHA_CHANNEL = 0, 1, 2
KDA_PATH_AUTO, KDA_PATH_CUDA_CORE, KDA_PATH_TENSOR = 0, 1, 2
KDA_PATH_TENSOR_SPLIT_SCAN, KDA_PATH_TENSOR_WIDE_SCAN, KDA_PATH_TENSOR_PIPELINED = 3, 4, 5
ABI_VERSION = 1

_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


class KdaError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {kda_status_string(status)}")


def library_path() -> str:
    return os.path.join(_PKG, "_build", "libkda.so")


def load_library():
    """Load libkda.so (built in-tree by ``gated_delta_rule_wise_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m gated_delta_rule_wise_gb300.build`")
        lib = ctypes.CDLL(path)
        lib.kda_abi_version.restype = _I
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [_I]
        lib.kda_chunk_fwd_workspace_size.restype = _SZ
        lib.kda_chunk_fwd_workspace_size.argtypes = [_I] * 8
        lib.kda_chunk_fwd_workspace_size_ex.restype = _SZ
        lib.kda_chunk_fwd_workspace_size_ex.argtypes = [_I] * 9
        chunk_args = [_P] * 8 + [_I] * 8 + [_P, _SZ, _P]
        lib.kda_chunk_fwd.restype = _I
        lib.kda_chunk_fwd.argtypes = chunk_args
        lib.kda_chunk_fwd_ex.restype = _I
        lib.kda_chunk_fwd_ex.argtypes = chunk_args + [_I, ctypes.POINTER(_P), _I]
        lib.kda_chunk_fwd_launches.restype = _I
        lib.kda_chunk_fwd_launches.argtypes = [_I] * 9
        lib.kda_chunk_fwd_kernel_name.restype = ctypes.c_char_p
        lib.kda_chunk_fwd_kernel_name.argtypes = [_I] * 10
        lib.kda_chunk_fwd_status.restype = _I
        lib.kda_chunk_fwd_status.argtypes = [_P, _P]
        lib.kda_decode_step.restype = _I
        lib.kda_decode_step.argtypes = [_P] * 7 + [_I] * 6 + [_P]
        lib.kda_chunk_fwd_rule.restype = _I
        lib.kda_chunk_fwd_rule.argtypes = chunk_args[:16] + [_I, ctypes.c_uint] + chunk_args[16:]
        lib.kda_attn_res.restype = _I
        lib.kda_attn_res.argtypes = [_P, _I, _P, _P, ctypes.c_longlong, _I, _I, ctypes.c_float, _P]
        lib.kda_chunk_fwd_host_buffer_size.restype = _SZ
        lib.kda_chunk_fwd_host_buffer_size.argtypes = [_I] * 9
        lib.kda_chunk_fwd_host.restype = _I
        lib.kda_chunk_fwd_host.argtypes = [_P] * 8 + [_I] * 9 + [_P, _SZ, _P]
        lib.kda_selftest_wait_timeout.restype = _I
        lib.kda_selftest_wait_timeout.argtypes = [_P, _SZ, ctypes.c_uint, _P]
        if lib.kda_abi_version() != ABI_VERSION:
            raise RuntimeError("libkda.so ABI version does not match this binding; rebuild it")
        _lib = lib
        return lib


def kda_abi_version() -> int:
    return load_library().kda_abi_version()


def kda_status_string(status: int) -> str:
    return load_library().kda_status_string(int(status)).decode()


def _check(status, what):
    if status != KDA_OK:
        raise KdaError(status, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libkda takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libkda takes contiguous tensors")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise ValueError(f"q/k/v/o must be float32 or bfloat16, got {t.dtype}")


def _alpha_mode(log_alpha, lead_ndim):
    if log_alpha is None:
        return KDA_ALPHA_NONE
    return KDA_ALPHA_SCALAR if log_alpha.dim() == lead_ndim else KDA_ALPHA_CHANNEL


def kda_chunk_fwd_workspace_size(B, H, T, dk, dv, C, dtype, alpha_mode,
                                 path=KDA_PATH_AUTO) -> int:
    return load_library().kda_chunk_fwd_workspace_size_ex(B, H, T, dk, dv, C, dtype,
                                                          alpha_mode, path)


def kda_chunk_fwd_ex(q, k, v, beta, log_alpha, h0, o, hT, C, workspace, stream=None,
                     path=KDA_PATH_AUTO, events=None):
    """Chunked prefill through the C ABI.  q, k [B,H,T,dk]; v, o [B,H,T,dv];
    beta [B,H,T]; log_alpha None / [B,H,T] / [B,H,T,dk]; h0, hT None or
    [B,H,dk,dv] float32; workspace a uint8 device tensor (or raw pointer
    with its size as a (ptr, nbytes) tuple).  ``events``: optional list of
    recorded-once ``torch.cuda.Event(enable_timing=True)``; events[i] is
    re-recorded before kernel launch i and events[-1] after the last."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if isinstance(workspace, tuple):
        ws_ptr, ws_bytes = workspace
    else:
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    ev_arr, n_ev = None, 0
    if events:
        ev_arr = (_P * len(events))(*[e.cuda_event for e in events])
        n_ev = len(events)
    st = load_library().kda_chunk_fwd_ex(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(log_alpha), _ptr(h0), _ptr(o), _ptr(hT),
        B, H, T, dk, dv, C, _dtype_code(q), _alpha_mode(log_alpha, 3), ws_ptr, ws_bytes,
        _stream(stream), path, ev_arr, n_ev)
    _check(st, "kda_chunk_fwd")


def kda_chunk_fwd(q, k, v, beta, log_alpha, h0, o, hT, C, workspace, stream=None):
    kda_chunk_fwd_ex(q, k, v, beta, log_alpha, h0, o, hT, C, workspace, stream, KDA_PATH_AUTO)


KDA_RULE_DELTA, KDA_RULE_LINEAR, KDA_RULE_LINEAR_NORM = 0, 1, 2
KDA_MAP_QK_SILU_NORM, KDA_MAP_BETA_SIGMOID, KDA_MAP_QK_ELU1 = 1, 2, 4


def kda_chunk_fwd_rule(q, k, v, beta, log_alpha, h0, o, hT, C, workspace, rule=KDA_RULE_DELTA,
                       maps=0, stream=None):
    """``kda_chunk_fwd`` with an update rule (KDA_RULE_DELTA, KDA_RULE_LINEAR,
    KDA_RULE_LINEAR_NORM) and input maps (KDA_MAP_* bits) applied on the fly;
    beta may be None for the linear rules, and KDA_RULE_LINEAR_NORM takes
    h0 = hT = None (its state stays inside the call)."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    st = load_library().kda_chunk_fwd_rule(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(log_alpha), _ptr(h0), _ptr(o), _ptr(hT),
        B, H, T, dk, dv, C, _dtype_code(q), _alpha_mode(log_alpha, 3), rule, maps,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "kda_chunk_fwd_rule")


def kda_attn_res(V, w, h, eps=1e-6, stream=None):
    """AttnRes depth mixing: V [n_blocks, ..., D] (float32 or bf16), w [D]
    float32, h [..., D] of V's dtype (written)."""
    nb, D = V.shape[0], V.shape[-1]
    rows = V[0].numel() // D
    st = load_library().kda_attn_res(_ptr(V), nb, _ptr(w), _ptr(h), rows, D, _dtype_code(V),
                                     float(eps), _stream(stream))
    _check(st, "kda_attn_res")


def attn_res(V, w, eps=1e-6, stream=None):
    """Allocate h and run ``kda_attn_res``; returns h [..., D]."""
    h = torch.empty(V.shape[1:], dtype=V.dtype, device=V.device)
    kda_attn_res(V, w, h, eps, stream)
    return h


def _host_ptr(t):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("kda_chunk_fwd_host takes host tensors")
    if not t.is_contiguous():
        raise ValueError("libkda takes contiguous tensors")
    return t.data_ptr()


def kda_chunk_fwd_host_buffer_size(B, H, T, dk, dv, C, dtype, alpha_mode, group_heads=0) -> int:
    return load_library().kda_chunk_fwd_host_buffer_size(B, H, T, dk, dv, C, dtype, alpha_mode,
                                                         group_heads)


def host_buffer_for(q, v, C, log_alpha=None, group_heads=0, device=None):
    """Device buffer for ``kda_chunk_fwd_host`` on host tensors q [B,H,T,dk], v."""
    B, H, T, dk = q.shape
    n = kda_chunk_fwd_host_buffer_size(B, H, T, dk, v.shape[-1], C, _dtype_code(q),
                                       _alpha_mode(log_alpha, 3), group_heads)
    if n == 0:
        raise KdaError(KDA_ERR_UNSUPPORTED, "kda_chunk_fwd_host_buffer_size")
    buf = torch.empty(n, dtype=torch.uint8, device=device or torch.device("cuda"))
    buf[:256].zero_()
    return buf


def kda_chunk_fwd_host(q, k, v, beta, log_alpha, h0, o, hT, C, dev_buffer, group_heads=0,
                       stream=None):
    """Prefill with q, k, v, beta, log_alpha, h0 and the outputs o, hT in host
    (ideally pinned) memory; ``dev_buffer`` from ``host_buffer_for`` (same
    ``group_heads``).  ``group_heads`` 0 pipelines segments of the sequence,
    > 0 groups of that many (batch, head) pairs.  Returns once enqueued;
    synchronise ``stream`` before reading o / hT."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    st = load_library().kda_chunk_fwd_host(
        _host_ptr(q), _host_ptr(k), _host_ptr(v), _host_ptr(beta), _host_ptr(log_alpha),
        _host_ptr(h0), _host_ptr(o), _host_ptr(hT), B, H, T, dk, dv, C, _dtype_code(q),
        _alpha_mode(log_alpha, 3), group_heads, _ptr(dev_buffer),
        dev_buffer.numel() * dev_buffer.element_size(), _stream(stream))
    _check(st, "kda_chunk_fwd_host")


def kda_chunk_fwd_launches(B, H, T, dk, dv, C, dtype, alpha_mode, path=KDA_PATH_AUTO) -> int:
    return load_library().kda_chunk_fwd_launches(B, H, T, dk, dv, C, dtype, alpha_mode, path)


def kda_chunk_fwd_kernel_names(B, H, T, dk, dv, C, dtype, alpha_mode, path=KDA_PATH_AUTO):
    lib = load_library()
    n = lib.kda_chunk_fwd_launches(B, H, T, dk, dv, C, dtype, alpha_mode, path)
    return [lib.kda_chunk_fwd_kernel_name(B, H, T, dk, dv, C, dtype, alpha_mode, path, i).decode()
            for i in range(max(n, 0))]


# Source files behind each kernel (their hash tells whether a recorded ncu
# measurement still describes the kernel that runs).
_TC_HEADERS = ["kda_internal.cuh", "kda_ptx.cuh", "kda_umma.cuh"]
KERNEL_SOURCES = {
    "chunk_ffma_kernel": ["kda_chunk_ffma.cu", "kda_internal.cuh"],
    "decode_step_kernel": ["kda_decode.cu", "kda_internal.cuh"],
    "kda_prep_kernel": ["kda_chunk_tc.cu"] + _TC_HEADERS,
    "kda_scan_kernel": ["kda_chunk_tc.cu"] + _TC_HEADERS,
    "kda_scan_wide_kernel": ["kda_chunk_tc.cu"] + _TC_HEADERS,
    "attn_res_kernel": ["kda_attnres.cu", "kda_internal.cuh"],
}


def kernel_sources(name):
    return KERNEL_SOURCES[name]


def kda_chunk_fwd_status(workspace, stream=None):
    """Synchronise the stream and return the device status word (raises on error)."""
    st = load_library().kda_chunk_fwd_status(_ptr(workspace), _stream(stream))
    _check(st, "kda_chunk_fwd (device)")


def kda_decode_step(q, k, v, beta, log_alpha, S, o, stream=None):
    """One in-place decode step.  q, k [N,H,dk]; v, o [N,H,dv]; beta [N,H];
    log_alpha None / [N,H] / [N,H,dk]; S [N,H,dk,dv] float32 (updated)."""
    N, H, dk = q.shape
    dv = v.shape[-1]
    st = load_library().kda_decode_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(log_alpha), _ptr(S), _ptr(o),
        N, H, dk, dv, _dtype_code(q), _alpha_mode(log_alpha, 2), _stream(stream))
    _check(st, "kda_decode_step")


def kda_selftest_wait_timeout(workspace, spin_limit=1000, stream=None):
    st = load_library().kda_selftest_wait_timeout(
        _ptr(workspace), workspace.numel() * workspace.element_size(), spin_limit,
        _stream(stream))
    _check(st, "kda_selftest_wait_timeout")


def workspace_for(q, v, C, log_alpha=None, path=KDA_PATH_AUTO):
    B, H, T, dk = q.shape
    n = kda_chunk_fwd_workspace_size(B, H, T, dk, v.shape[-1], C, _dtype_code(q),
                                     _alpha_mode(log_alpha, 3), path)
    if n == 0:
        raise KdaError(KDA_ERR_UNSUPPORTED, "kda_chunk_fwd_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=q.device)
    ws[:256].zero_()
    return ws


def chunk_fwd(q, k, v, beta, log_alpha=None, h0=None, C=64, output_final_state=True,
              path=KDA_PATH_AUTO, stream=None, workspace=None):
    """Allocate o (and hT) and run ``kda_chunk_fwd``; returns (o, hT or None)."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    hT = (torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
          if output_final_state else None)
    ws = workspace if workspace is not None else workspace_for(q, v, C, log_alpha, path)
    kda_chunk_fwd_ex(q, k, v, beta, log_alpha, h0, o, hT, C, ws, stream, path)
    return o, hT


def decode_step(q, k, v, beta, log_alpha, S, stream=None):
    """Allocate o and run one in-place ``kda_decode_step``; returns o."""
    o = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    kda_decode_step(q, k, v, beta, log_alpha, S, o, stream)
    return o
