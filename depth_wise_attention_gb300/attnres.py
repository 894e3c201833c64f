"""Thin ctypes binding of libattnres.so (C ABI in include/attnres.h).

Argument marshalling only: every step of the read runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (torch supplies device memory and the
current stream); each function has the name of the C entry point it calls and
raises ``AttnResError`` when the call does not return ATTNRES_OK.  There is no
fallback: if the library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattnres.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "attnres.h")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = range(5)
F32, BF16 = 0, 1

_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_f = ctypes.c_float
_SIGS = {
    "attnres_full_fwd": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _vp, _vp, _f, _vp, _vp],
    "attnres_block_phase1": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _vp, _i64, _vp, _f, _vp,
                             _vp, _vp],
    "attnres_block_phase2_merge": [_vp, _vp, _vp, _i64, _i64, ctypes.c_int, _vp, _vp, _f, _vp, _vp],
    "attnres_block_phase2_update_merge": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_int, _vp, _vp,
                                          _f, _vp, _vp],
    "mhar_phase2_merge": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_int, _vp, _vp, _f, _vp, _vp],
    "attnres_read_bwd": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _vp, _i64, _vp, _f, _vp, _vp, _i64,
                         ctypes.c_int, _vp, _vp, _vp, ctypes.c_size_t, _vp],
    "attnres_read_bwd_noalloc": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _vp, _i64, _vp, _f, _vp, _vp, _i64,
                                 ctypes.c_int, _vp, _vp, _vp],
    "attnres_read_bwd_workspace_size": [_i64, _i64, _i64, _i64, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
    "attnres_block_phase1_bwd": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _vp, _i64, _vp, _f, _vp, _vp, _vp,
                                 _i64, ctypes.c_int, _vp, _vp, _vp, ctypes.c_size_t, _vp],
    "attnres_block_phase2_bwd": [_vp, _vp, _vp, _i64, _i64, ctypes.c_int, _vp, _vp, _f, _vp, _vp, _vp, _vp,
                                 ctypes.c_int, _vp, _vp, _vp, ctypes.c_size_t, _vp],
    "attnres_block_phase2_bwd_workspace_size": [_i64, _i64, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
    "mhar_read_bwd": [_vp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _vp, _i64, _vp, _f, _vp, _vp, _i64,
                      ctypes.c_int, _vp, _vp, _vp, ctypes.c_size_t, _vp],
    "mhar_read_bwd_workspace_size": [_i64, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
    "mhar_fwd": [_vp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _vp, _i64, _vp, _f, _vp, _vp,
                 _vp],
    "msar_expand_fwd": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _vp, _vp, _f,
                        _vp, _vp, _f, _vp, _vp],
    "msar_expand_fwd_ps": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _i64, _vp, _vp, _f, _vp,
                           _vp, _f, _vp, _vp],
    "msar_block_phase1": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _vp, _i64, _vp, _f, _vp,
                          _vp, _vp],
    "msar_block_phase2": [_vp, _vp, _vp, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _vp, _vp, _f, _vp, _vp, _f,
                          _vp, _vp],
    "msar_expand_fwd_chunk": [_vp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _vp, _vp, _f,
                              _vp, _vp, _f, _vp, _vp],
    "msar_expand_bwd": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _vp, _vp, _f, _vp, _vp, _f,
                        _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp],
    "msar_expand_bwd_workspace_size": [_i64, _i64, _i64, ctypes.c_int, _i64, _vp, ctypes.POINTER(ctypes.c_size_t)],
    "msar_expand_bwd_chunk": [_vp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _vp, _vp, _f, _vp,
                              _vp, _f, _vp, _vp, _i64, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                              _vp],
    "msar_expand_bwd_ps": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _i64, _vp, _vp, _f, _vp, _vp,
                           _f, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp],
    "msar_expand_fwd_ws": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _i64, _vp, _vp, _f, _vp, _vp,
                           _f, _vp, _vp, ctypes.c_size_t, _vp],
    "msar_expand_fwd_ws_workspace_size": [_i64, _i64, _i64, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
    "msar_block_phase1_ws": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _vp, _i64, _vp, _f, _vp,
                             _vp, _vp, ctypes.c_size_t, _vp],
    "msar_block_phase1_ws_workspace_size": [_i64, _i64, _i64, ctypes.c_int, _i64, ctypes.POINTER(ctypes.c_size_t)],
    "msar_block_phase2_ws": [_vp, _vp, _vp, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _vp, _vp, _f, _vp, _vp, _f,
                             _vp, _vp, ctypes.c_size_t, _vp],
    "msar_block_phase2_ws_workspace_size": [_i64, _i64, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
    "msar_block_phase2_bwd": [_vp, _vp, _vp, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _vp, _vp, _f, _vp, _vp, _f,
                              _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp],
    "msar_block_phase2_bwd_workspace_size": [_i64, _i64, ctypes.c_int, _i64, _vp, ctypes.POINTER(ctypes.c_size_t)],
    "msar_block_phase1_bwd": [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _i64, _vp, _vp, _vp, _i64, _vp, _f, _vp,
                              _vp, _vp, _i64, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp],
    "msar_block_phase1_bwd_workspace_size": [_i64, _i64, _i64, ctypes.c_int, _i64, _vp, _i64,
                                             ctypes.POINTER(ctypes.c_size_t)],
    "attnres_status_string": [ctypes.c_int],
    "attnres_last_cuda_error": [],
    "attnres_sync_status": [_vp],
    "attnres_debug_set_wait_timeout_ns": [ctypes.c_uint64],
    "attnres_debug_set_stall_injection": [ctypes.c_int],
    "attnres_debug_set_kernel_variant": [ctypes.c_int],
    "attnres_version": [],
}
_RESTYPES = {"attnres_status_string": ctypes.c_char_p, "attnres_last_cuda_error": ctypes.c_char_p,
             "attnres_version": ctypes.c_char_p, "attnres_debug_set_wait_timeout_ns": None,
             "attnres_debug_set_stall_injection": None,
             "attnres_debug_set_kernel_variant": None}


class AttnResError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn}: {status_string(status)}"
        if status == ERR_CUDA:
            msg += f" ({last_cuda_error()})"
        super().__init__(msg)


def load(path: str = LIB_PATH):
    """Load libattnres.so (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m depth_wise_attention_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, args in _SIGS.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = _RESTYPES.get(name, ctypes.c_int)
        _lib = lib
    return _lib


def header_functions(header: str = HEADER):
    """Names of the functions declared in include/attnres.h."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_0-9]+)\s*\(", text)) - {"defined"})


def status_string(status: int) -> str:
    return load().attnres_status_string(status).decode()


def last_cuda_error() -> str:
    return load().attnres_last_cuda_error().decode()


def version() -> str:
    return load().attnres_version().decode()


def _dt(t):
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _p(t):
    return None if t is None else _vp(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return _vp(s.cuda_stream)


def _check(fn, status):
    if status != OK:
        raise AttnResError(fn, status)


def _src_geometry(src):
    """src [n_src, T, d]: each source contiguous, sources src.stride(0) apart."""
    n_src, T, d = src.shape
    if src.stride(2) != 1 or src.stride(1) != d:
        raise ValueError("each source must be a contiguous [T, d] block")
    return n_src, T, d, src.stride(0)


def attnres_full_fwd(src, query, gain=None, eps=1e-6, out=None, stream=None):
    """Full AttnRes read of one layer: src [n_src,T,d] -> out [T,d]."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    if out is None:
        out = torch.empty((T, d), dtype=src.dtype, device=src.device)
    _check("attnres_full_fwd", load().attnres_full_fwd(
        _p(src), n_src, stride, T, d, _dt(src), _p(query), _p(gain), eps, _p(out), _stream(stream)))
    return out


def attnres_block_phase1(src, queries, gain=None, eps=1e-6, o=None, lse=None, want_lse=True,
                         stream=None):
    """Phase 1: queries [n_q,d] against src [n_src,T,d] -> (o [n_q,T,d], lse [n_q,T])."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    n_q = queries.shape[0]
    if o is None:
        o = torch.empty((n_q, T, d), dtype=src.dtype, device=src.device)
    if lse is None and want_lse:
        lse = torch.empty((n_q, T), dtype=torch.float32, device=src.device)
    _check("attnres_block_phase1", load().attnres_block_phase1(
        _p(src), n_src, stride, T, d, _dt(src), _p(queries), n_q, _p(gain), eps, _p(o), _p(lse),
        _stream(stream)))
    return o, lse


def attnres_block_phase2_merge(o, lse, partial, query, gain=None, eps=1e-6, out=None, stream=None):
    """Phase 2: merge partial [T,d] (or None) into (o [T,d], lse [T]) -> out [T,d]."""
    import torch
    T, d = o.shape
    if out is None:
        out = torch.empty_like(o)
    _check("attnres_block_phase2_merge", load().attnres_block_phase2_merge(
        _p(o), _p(lse), _p(partial), T, d, _dt(o), _p(query), _p(gain), eps, _p(out),
        _stream(stream)))
    return out


def attnres_block_phase2_update_merge(partial, f, o, lse, query, gain=None, eps=1e-6, partial_out=None,
                                      out=None, stream=None):
    """Fused update and merge: partial [T,d] or None, f [T,d] -> (partial + f, merged out).
    partial_out may be partial or f (in place); out may be o."""
    import torch
    T, d = o.shape
    if partial_out is None:
        partial_out = torch.empty_like(f)
    if out is None:
        out = torch.empty_like(o)
    _check("attnres_block_phase2_update_merge", load().attnres_block_phase2_update_merge(
        _p(partial), _p(f), _p(partial_out), _p(o), _p(lse), T, d, _dt(o), _p(query), _p(gain), eps,
        _p(out), _stream(stream)))
    return partial_out, out


def mhar_phase2_merge(o, lse, partial, query, gain=None, eps=1e-6, f=None, partial_out=None, out=None,
                      stream=None):
    """Per-head phase-2 merge: o [T,d], lse [H,T], partial [T,d] or None, query [H,d/H].
    With f, the partial is first updated (returned as partial_out).  Returns out, or
    (partial_out, out) when f is given."""
    import torch
    T, d = o.shape
    H = query.shape[0]
    if f is not None and partial_out is None:
        partial_out = torch.empty_like(f)
    if out is None:
        out = torch.empty_like(o)
    _check("mhar_phase2_merge", load().mhar_phase2_merge(
        _p(o), _p(lse), _p(partial), _p(f), _p(partial_out), T, d, H, _dt(o), _p(query), _p(gain), eps,
        _p(out), _stream(stream)))
    return (partial_out, out) if f is not None else out


def attnres_read_bwd_workspace_size(n_src, T, d, n_q, dtype):
    import torch
    n = ctypes.c_size_t(0)
    dt = BF16 if dtype == torch.bfloat16 else F32
    _check("attnres_read_bwd_workspace_size",
           load().attnres_read_bwd_workspace_size(n_src, T, d, n_q, dt, ctypes.byref(n)))
    return n.value


def attnres_read_bwd(src, queries, dout, gain=None, eps=1e-6, dsrc=None, accumulate=False, dqueries=None,
                     dgain=None, want_dgain=True, workspace=None, stream=None):
    """Backward of the read of queries [n_q,d] over src [n_src,T,d] for output
    gradients dout [n_q,T,d] -> (dsrc, dqueries, dgain).  The workspace is
    allocated here unless given (the library itself allocates nothing)."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    n_q = queries.shape[0]
    if dsrc is None:
        dsrc = torch.empty((n_src, T, d), dtype=src.dtype, device=src.device)
    _, _, _, dstride = _src_geometry(dsrc)
    if dqueries is None:
        dqueries = torch.empty((n_q, d), dtype=torch.float32, device=src.device)
    if dgain is None and want_dgain:
        dgain = torch.empty((d,), dtype=torch.float32, device=src.device)
    if workspace is None:
        nbytes = attnres_read_bwd_workspace_size(n_src, T, d, n_q, src.dtype)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=src.device)
    _check("attnres_read_bwd", load().attnres_read_bwd(
        _p(src), n_src, stride, T, d, _dt(src), _p(queries), n_q, _p(gain), eps, _p(dout), _p(dsrc), dstride,
        1 if accumulate else 0, _p(dqueries), _p(dgain), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return dsrc, dqueries, dgain


def attnres_read_bwd_noalloc(src, queries, dout, gain=None, eps=1e-6, dsrc=None, accumulate=False,
                             dqueries=None, dgain=None, want_dgain=True, stream=None):
    """attnres_read_bwd with the library's built-in scratch instead of a workspace."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    n_q = queries.shape[0]
    if dsrc is None:
        dsrc = torch.empty((n_src, T, d), dtype=src.dtype, device=src.device)
    _, _, _, dstride = _src_geometry(dsrc)
    if dqueries is None:
        dqueries = torch.empty((n_q, d), dtype=torch.float32, device=src.device)
    if dgain is None and want_dgain:
        dgain = torch.empty((d,), dtype=torch.float32, device=src.device)
    _check("attnres_read_bwd_noalloc", load().attnres_read_bwd_noalloc(
        _p(src), n_src, stride, T, d, _dt(src), _p(queries), n_q, _p(gain), eps, _p(dout), _p(dsrc), dstride,
        1 if accumulate else 0, _p(dqueries), _p(dgain), _stream(stream)))
    return dsrc, dqueries, dgain


def attnres_block_phase1_bwd(src, queries, d_o, d_lse=None, gain=None, eps=1e-6, dsrc=None, accumulate=False,
                             dqueries=None, dgain=None, want_dgain=True, workspace=None, stream=None):
    """Backward of Block phase 1 for gradients of its outputs o [n_q,T,d] and
    lse [n_q,T] (None: zero) -> (dsrc, dqueries, dgain)."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    n_q = queries.shape[0]
    if dsrc is None:
        dsrc = torch.empty((n_src, T, d), dtype=src.dtype, device=src.device)
    _, _, _, dstride = _src_geometry(dsrc)
    if dqueries is None:
        dqueries = torch.empty((n_q, d), dtype=torch.float32, device=src.device)
    if dgain is None and want_dgain:
        dgain = torch.empty((d,), dtype=torch.float32, device=src.device)
    if workspace is None:
        nbytes = attnres_read_bwd_workspace_size(n_src, T, d, n_q, src.dtype)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=src.device)
    _check("attnres_block_phase1_bwd", load().attnres_block_phase1_bwd(
        _p(src), n_src, stride, T, d, _dt(src), _p(queries), n_q, _p(gain), eps, _p(d_o), _p(d_lse), _p(dsrc),
        dstride, 1 if accumulate else 0, _p(dqueries), _p(dgain), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return dsrc, dqueries, dgain


def attnres_block_phase2_bwd_workspace_size(T, d, dtype):
    import torch
    n = ctypes.c_size_t(0)
    dt = BF16 if dtype == torch.bfloat16 else F32
    _check("attnres_block_phase2_bwd_workspace_size",
           load().attnres_block_phase2_bwd_workspace_size(T, d, dt, ctypes.byref(n)))
    return n.value


def attnres_block_phase2_bwd(o, lse, partial, query, dh, gain=None, eps=1e-6, d_o=None, d_lse=None,
                             d_partial=None, accumulate=False, dquery=None, dgain=None, want_dgain=True,
                             workspace=None, stream=None):
    """Backward of the phase-2 merge: o, partial (or None), dh [T,d]; lse [T]
    -> (d_o, d_lse, d_partial (None without a partial), dquery, dgain)."""
    import torch
    T, d = o.shape
    if d_o is None:
        d_o = torch.empty_like(o)
    if d_lse is None:
        d_lse = torch.empty((T,), dtype=torch.float32, device=o.device)
    if partial is not None and d_partial is None:
        d_partial = torch.empty_like(partial)
    if dquery is None:
        dquery = torch.empty((d,), dtype=torch.float32, device=o.device)
    if dgain is None and want_dgain:
        dgain = torch.empty((d,), dtype=torch.float32, device=o.device)
    if workspace is None:
        nbytes = attnres_block_phase2_bwd_workspace_size(T, d, o.dtype)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=o.device)
    _check("attnres_block_phase2_bwd", load().attnres_block_phase2_bwd(
        _p(o), _p(lse), _p(partial), T, d, _dt(o), _p(query), _p(gain), eps, _p(dh), _p(d_o), _p(d_lse),
        _p(d_partial), 1 if accumulate else 0, _p(dquery), _p(dgain), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return d_o, d_lse, (d_partial if partial is not None else None), dquery, dgain


def mhar_read_bwd_workspace_size(n_src, T, d, H, n_q, dtype):
    import torch
    n = ctypes.c_size_t(0)
    dt = BF16 if dtype == torch.bfloat16 else F32
    _check("mhar_read_bwd_workspace_size",
           load().mhar_read_bwd_workspace_size(n_src, T, d, H, n_q, dt, ctypes.byref(n)))
    return n.value


def mhar_read_bwd(src, queries, dout, gain=None, eps=1e-6, dsrc=None, accumulate=False, dqueries=None,
                  dgain=None, want_dgain=True, workspace=None, stream=None):
    """Backward of the MHAR read of queries [n_q,H,d/H] over src [n_src,T,d]
    for output gradients dout [n_q,T,d] -> (dsrc, dqueries [n_q,H,d/H],
    dgain).  The workspace is allocated here unless given."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    n_q, H, dh = queries.shape
    if H * dh != d:
        raise ValueError("queries must be [n_q, H, d/H]")
    if dsrc is None:
        dsrc = torch.empty((n_src, T, d), dtype=src.dtype, device=src.device)
    _, _, _, dstride = _src_geometry(dsrc)
    if dqueries is None:
        dqueries = torch.empty((n_q, H, dh), dtype=torch.float32, device=src.device)
    if dgain is None and want_dgain:
        dgain = torch.empty((d,), dtype=torch.float32, device=src.device)
    if workspace is None:
        nbytes = mhar_read_bwd_workspace_size(n_src, T, d, H, n_q, src.dtype)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=src.device)
    _check("mhar_read_bwd", load().mhar_read_bwd(
        _p(src), n_src, stride, T, d, H, _dt(src), _p(queries), n_q, _p(gain), eps, _p(dout), _p(dsrc), dstride,
        1 if accumulate else 0, _p(dqueries), _p(dgain), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return dsrc, dqueries, dgain


def mhar_fwd(src, queries, gain=None, eps=1e-6, out=None, lse=None, want_lse=False, stream=None):
    """MHAR: queries [n_q,H,d/H] -> out [n_q,T,d] (lse [n_q,H,T])."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    n_q, H, _ = queries.shape
    if out is None:
        out = torch.empty((n_q, T, d), dtype=src.dtype, device=src.device)
    if lse is None and want_lse:
        lse = torch.empty((n_q, H, T), dtype=torch.float32, device=src.device)
    _check("mhar_fwd", load().mhar_fwd(
        _p(src), n_src, stride, T, d, H, _dt(src), _p(queries), n_q, _p(gain), eps, _p(out), _p(lse),
        _stream(stream)))
    return (out, lse) if want_lse else out


def msar_expand_fwd(src, ksizes, conv_w, queries, gain=None, eps=1e-6, mix_gain=None, mix_w=None,
                    mix_eps=1e-6, out=None, stream=None):
    """MSAR: src [n_src,T,d], ksizes (m-1 ints, host), conv_w packed, queries [m,d],
    mix_w [m*d,m] -> out [T,d]."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    m = queries.shape[0]
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    if out is None:
        out = torch.empty((T, d), dtype=src.dtype, device=src.device)
    _check("msar_expand_fwd", load().msar_expand_fwd(
        _p(src), n_src, stride, T, d, _dt(src), m, ctypes.cast(ks, _vp), _p(conv_w), _p(queries),
        _p(gain), eps, _p(mix_gain), _p(mix_w), mix_eps, _p(out), _stream(stream)))
    return out


def attnres_sync_status(stream=None):
    """Wait for the stream and raise if a kernel recorded a device-side timeout."""
    _check("attnres_sync_status", load().attnres_sync_status(_stream(stream)))


def attnres_debug_set_wait_timeout_ns(ns: int):
    load().attnres_debug_set_wait_timeout_ns(int(ns))


def attnres_debug_set_stall_injection(enable: bool):
    load().attnres_debug_set_stall_injection(1 if enable else 0)


def attnres_debug_set_kernel_variant(variant: int):
    """0: automatic kernel choice; 1: always the general CUDA-core depth read;
    2: the tensor-core depth reads wherever they apply; 3: the few-token kernel
    (a token per cluster of CTAs) wherever it applies."""
    load().attnres_debug_set_kernel_variant(int(variant))


def msar_expand_fwd_chunk(src, t_prev, ksizes, conv_w, queries, gain=None, eps=1e-6, mix_gain=None, mix_w=None,
                          mix_eps=1e-6, out=None, stream=None):
    """MSAR for one chunk: src [n_src, t_prev + T, d] (t_prev history rows first)
    -> out [T, d] for the last T rows."""
    import torch
    n_src, rows, d, stride = _src_geometry(src)
    T = rows - t_prev
    m = queries.shape[0]
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    if out is None:
        out = torch.empty((T, d), dtype=src.dtype, device=src.device)
    _check("msar_expand_fwd_chunk", load().msar_expand_fwd_chunk(
        _p(src), n_src, stride, t_prev, T, d, _dt(src), m, ctypes.cast(ks, _vp), _p(conv_w), _p(queries),
        _p(gain), eps, _p(mix_gain), _p(mix_w), mix_eps, _p(out), _stream(stream)))
    return out


def msar_block_phase1(src, ksizes, conv_w, queries, gain=None, eps=1e-6, o=None, lse=None, stream=None):
    """MSAR two-phase, phase 1: queries [S, m, d] of a block's layers over the
    cached sources src [n_src, T, d] -> (o [S, m, T, d], lse [S, m, T])."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    S, m, _ = queries.shape
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    if o is None:
        o = torch.empty((S, m, T, d), dtype=src.dtype, device=src.device)
    if lse is None:
        lse = torch.empty((S, m, T), dtype=torch.float32, device=src.device)
    _check("msar_block_phase1", load().msar_block_phase1(
        _p(src), n_src, stride, T, d, _dt(src), m, ctypes.cast(ks, _vp), _p(conv_w), _p(queries), S, _p(gain),
        eps, _p(o), _p(lse), _stream(stream)))
    return o, lse


def msar_block_phase2(o, lse, partial, ksizes, conv_w, query, gain=None, eps=1e-6, mix_gain=None, mix_w=None,
                      mix_eps=1e-6, out=None, stream=None):
    """MSAR two-phase, phase 2 of one layer: o [m, T, d], lse [m, T], partial
    [T, d] or None, query [m, d] -> out [T, d]."""
    import torch
    m, T, d = o.shape
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    if out is None:
        out = torch.empty((T, d), dtype=o.dtype, device=o.device)
    _check("msar_block_phase2", load().msar_block_phase2(
        _p(o), _p(lse), _p(partial), T, d, _dt(o), m, ctypes.cast(ks, _vp), _p(conv_w), _p(query), _p(gain), eps,
        _p(mix_gain), _p(mix_w), mix_eps, _p(out), _stream(stream)))
    return out


def msar_expand_fwd_ps(src, ksizes, conv_w, queries, gain=None, eps=1e-6, mix_gain=None, mix_w=None, mix_eps=1e-6,
                       out=None, stream=None):
    """MSAR with each source's own conv kernels: conv_w [n_src, d*sum(k)] (or
    any [n_src, stride >= d*sum(k)] float tensor) -> out [T, d]."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    m = queries.shape[0]
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    if out is None:
        out = torch.empty((T, d), dtype=src.dtype, device=src.device)
    _check("msar_expand_fwd_ps", load().msar_expand_fwd_ps(
        _p(src), n_src, stride, T, d, _dt(src), m, ctypes.cast(ks, _vp), _p(conv_w), conv_w.stride(0), _p(queries),
        _p(gain), eps, _p(mix_gain), _p(mix_w), mix_eps, _p(out), _stream(stream)))
    return out


def msar_expand_bwd_workspace_size(n_src, T, d, dtype, ksizes):
    import torch
    n = ctypes.c_size_t(0)
    dt = BF16 if dtype == torch.bfloat16 else F32
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    _check("msar_expand_bwd_workspace_size", load().msar_expand_bwd_workspace_size(
        n_src, T, d, dt, len(ksizes) + 1, ctypes.cast(ks, _vp), ctypes.byref(n)))
    return n.value


def msar_expand_bwd(src, ksizes, conv_w, queries, dh, gain=None, eps=1e-6, mix_gain=None, mix_w=None, mix_eps=1e-6,
                    dsrc=None, want_dgain=True, want_dmix_gain=True, grads=None, workspace=None, stream=None):
    """Backward of msar_expand_fwd for dh [T,d] -> (dsrc [n_src,T,d], dconv_w
    (packed as conv_w), dqueries [m,d], dgain [d], dmix_gain [m*d], dmix_w
    [m*d,m]).  grads: the five parameter-gradient tensors to write (else
    allocated here, as is the workspace unless given)."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    m = queries.shape[0]
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    dev = src.device
    if dsrc is None:
        dsrc = torch.empty((n_src, T, d), dtype=src.dtype, device=dev)
    _, _, _, dstride = _src_geometry(dsrc)
    if grads is not None:
        dconv_w, dqueries, dgain, dmix_gain, dmix_w = grads
    else:
        dconv_w = torch.empty_like(conv_w, dtype=torch.float32)
        dqueries = torch.empty((m, d), dtype=torch.float32, device=dev)
        dgain = torch.empty((d,), dtype=torch.float32, device=dev) if want_dgain else None
        dmix_gain = torch.empty((m * d,), dtype=torch.float32, device=dev) if want_dmix_gain else None
        dmix_w = torch.empty((m * d, m), dtype=torch.float32, device=dev)
    if workspace is None:
        nbytes = msar_expand_bwd_workspace_size(n_src, T, d, src.dtype, ksizes)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=dev)
    _check("msar_expand_bwd", load().msar_expand_bwd(
        _p(src), n_src, stride, T, d, _dt(src), m, ctypes.cast(ks, _vp), _p(conv_w), _p(queries), _p(gain), eps,
        _p(mix_gain), _p(mix_w), mix_eps, _p(dh), _p(dsrc), dstride, _p(dconv_w), _p(dqueries), _p(dgain),
        _p(dmix_gain), _p(dmix_w), _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return dsrc, dconv_w, dqueries, dgain, dmix_gain, dmix_w


def msar_expand_bwd_ps(src, ksizes, conv_w, queries, dh, gain=None, eps=1e-6, mix_gain=None, mix_w=None,
                       mix_eps=1e-6, dsrc=None, want_dgain=True, want_dmix_gain=True, grads=None, workspace=None,
                       stream=None):
    """Backward of msar_expand_fwd_ps: conv_w [n_src, stride >= d*sum(k)] ->
    (dsrc, dconv_w [n_src, stride] (each source's own; the padding past
    d*sum(k) is zero), dqueries, dgain, dmix_gain, dmix_w)."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    m = queries.shape[0]
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    dev = src.device
    if dsrc is None:
        dsrc = torch.empty((n_src, T, d), dtype=src.dtype, device=dev)
    _, _, _, dstride = _src_geometry(dsrc)
    if grads is not None:
        dconv_w, dqueries, dgain, dmix_gain, dmix_w = grads
    else:
        dconv_w = torch.zeros(conv_w.shape, dtype=torch.float32, device=dev)
        dqueries = torch.empty((m, d), dtype=torch.float32, device=dev)
        dgain = torch.empty((d,), dtype=torch.float32, device=dev) if want_dgain else None
        dmix_gain = torch.empty((m * d,), dtype=torch.float32, device=dev) if want_dmix_gain else None
        dmix_w = torch.empty((m * d, m), dtype=torch.float32, device=dev)
    if workspace is None:
        nbytes = msar_expand_bwd_workspace_size(n_src, T, d, src.dtype, ksizes)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=dev)
    _check("msar_expand_bwd_ps", load().msar_expand_bwd_ps(
        _p(src), n_src, stride, T, d, _dt(src), m, ctypes.cast(ks, _vp), _p(conv_w), conv_w.stride(0), _p(queries),
        _p(gain), eps, _p(mix_gain), _p(mix_w), mix_eps, _p(dh), _p(dsrc), dstride, _p(dconv_w), _p(dqueries),
        _p(dgain), _p(dmix_gain), _p(dmix_w), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return dsrc, dconv_w, dqueries, dgain, dmix_gain, dmix_w


def msar_expand_fwd_ws_workspace_size(n_src, T, d, dtype):
    import torch
    n = ctypes.c_size_t(0)
    dt = BF16 if dtype == torch.bfloat16 else F32
    _check("msar_expand_fwd_ws_workspace_size",
           load().msar_expand_fwd_ws_workspace_size(n_src, T, d, dt, ctypes.byref(n)))
    return n.value


def msar_expand_bwd_chunk(src, t_prev, ksizes, conv_w, queries, dh, dsrc, grads, accumulate, gain=None, eps=1e-6,
                          mix_gain=None, mix_w=None, mix_eps=1e-6, workspace=None, stream=None):
    """Backward of one chunk: src [n_src, t_prev + T, d] (t_prev history rows
    first), dh [T, d]; dsrc [n_src, t_prev + T, d] gets the chunk's rows
    written and the history rows' share added; grads = (dconv_w, dqueries,
    dgain, dmix_gain, dmix_w) are written (accumulate False) or added into."""
    import torch
    n_src, rows, d, stride = _src_geometry(src)
    T = rows - t_prev
    m = queries.shape[0]
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    _, _, _, dstride = _src_geometry(dsrc)
    dconv_w, dqueries, dgain, dmix_gain, dmix_w = grads
    if workspace is None:
        nbytes = msar_expand_bwd_workspace_size(n_src, T, d, src.dtype, ksizes)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=src.device)
    _check("msar_expand_bwd_chunk", load().msar_expand_bwd_chunk(
        _p(src), n_src, stride, t_prev, T, d, _dt(src), m, ctypes.cast(ks, _vp), _p(conv_w), _p(queries), _p(gain),
        eps, _p(mix_gain), _p(mix_w), mix_eps, _p(dh), _p(dsrc), dstride, 1 if accumulate else 0, _p(dconv_w),
        _p(dqueries), _p(dgain), _p(dmix_gain), _p(dmix_w), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return dsrc


def msar_expand_fwd_ws(src, ksizes, conv_w, queries, gain=None, eps=1e-6, mix_gain=None, mix_w=None, mix_eps=1e-6,
                       out=None, workspace=None, stream=None):
    """MSAR read through the workspace chain.  conv_w: packed 1-D (shared
    kernels) or [n_src, stride] (each source's own) -> out [T, d]."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    m = queries.shape[0]
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    if out is None:
        out = torch.empty((T, d), dtype=src.dtype, device=src.device)
    if workspace is None:
        nbytes = msar_expand_fwd_ws_workspace_size(n_src, T, d, src.dtype)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=src.device)
    cstride = conv_w.stride(0) if conv_w.dim() == 2 else 0
    _check("msar_expand_fwd_ws", load().msar_expand_fwd_ws(
        _p(src), n_src, stride, T, d, _dt(src), m, ctypes.cast(ks, _vp), _p(conv_w), cstride, _p(queries),
        _p(gain), eps, _p(mix_gain), _p(mix_w), mix_eps, _p(out), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def msar_block_phase1_ws_workspace_size(n_src, T, d, dtype, S):
    import torch
    n = ctypes.c_size_t(0)
    dt = BF16 if dtype == torch.bfloat16 else F32
    _check("msar_block_phase1_ws_workspace_size",
           load().msar_block_phase1_ws_workspace_size(n_src, T, d, dt, S, ctypes.byref(n)))
    return n.value


def msar_block_phase1_ws(src, ksizes, conv_w, queries, gain=None, eps=1e-6, o=None, lse=None, workspace=None,
                         stream=None):
    """MSAR phase 1 through the workspace chain: queries [S, m, d] ->
    (o [S, m, T, d], lse [S, m, T])."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    S, m = queries.shape[0], queries.shape[1]
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    if o is None:
        o = torch.empty((S, m, T, d), dtype=src.dtype, device=src.device)
    if lse is None:
        lse = torch.empty((S, m, T), dtype=torch.float32, device=src.device)
    if workspace is None:
        nbytes = msar_block_phase1_ws_workspace_size(n_src, T, d, src.dtype, S)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=src.device)
    _check("msar_block_phase1_ws", load().msar_block_phase1_ws(
        _p(src), n_src, stride, T, d, _dt(src), m, ctypes.cast(ks, _vp), _p(conv_w), _p(queries), S, _p(gain), eps,
        _p(o), _p(lse), _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return o, lse


def msar_block_phase2_ws_workspace_size(T, d, dtype):
    import torch
    n = ctypes.c_size_t(0)
    dt = BF16 if dtype == torch.bfloat16 else F32
    _check("msar_block_phase2_ws_workspace_size", load().msar_block_phase2_ws_workspace_size(T, d, dt, ctypes.byref(n)))
    return n.value


def msar_block_phase2_ws(o, lse, partial, ksizes, conv_w, query, gain=None, eps=1e-6, mix_gain=None, mix_w=None,
                         mix_eps=1e-6, out=None, workspace=None, stream=None):
    """MSAR phase 2 of one layer through the workspace chain: o [m, T, d],
    lse [m, T], partial [T, d] or None, query [m, d] -> out [T, d]."""
    import torch
    m, T, d = o.shape
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    if out is None:
        out = torch.empty((T, d), dtype=o.dtype, device=o.device)
    if workspace is None:
        nbytes = msar_block_phase2_ws_workspace_size(T, d, o.dtype)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=o.device)
    _check("msar_block_phase2_ws", load().msar_block_phase2_ws(
        _p(o), _p(lse), _p(partial), T, d, _dt(o), m, ctypes.cast(ks, _vp), _p(conv_w), _p(query), _p(gain), eps,
        _p(mix_gain), _p(mix_w), mix_eps, _p(out), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return out


def msar_block_phase2_bwd(o, lse, partial, ksizes, conv_w, query, dh, gain=None, eps=1e-6, mix_gain=None, mix_w=None,
                          mix_eps=1e-6, outs=None, workspace=None, stream=None):
    """Backward of msar_block_phase2 for dh [T, d] -> (d_o [m,T,d], d_lse
    [m,T], d_partial [T,d] or None, dconv_w, dquery [m,d], dgain [d],
    dmix_gain [m*d], dmix_w [m*d,m]).  outs: those eight tensors to write
    (else allocated here)."""
    import torch
    m, T, d = o.shape
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    dev, f32 = o.device, dict(dtype=torch.float32, device=o.device)
    if outs is not None:
        d_o, d_lse, d_p, dcw, dq, dg, dmg, dmw = outs
    else:
        d_o = torch.empty_like(o)
        d_lse = torch.empty((m, T), **f32)
        d_p = torch.empty_like(partial) if partial is not None else None
        dcw, dq, dg = torch.empty_like(conv_w, dtype=torch.float32), torch.empty((m, d), **f32), torch.empty((d,), **f32)
        dmg, dmw = torch.empty((m * d,), **f32), torch.empty((m * d, m), **f32)
    if workspace is None:
        n = ctypes.c_size_t(0)
        _check("msar_block_phase2_bwd_workspace_size", load().msar_block_phase2_bwd_workspace_size(
            T, d, _dt(o), m, ctypes.cast(ks, _vp), ctypes.byref(n)))
        workspace = torch.empty((max(n.value, 16) + 3) // 4, dtype=torch.float32, device=dev)
    _check("msar_block_phase2_bwd", load().msar_block_phase2_bwd(
        _p(o), _p(lse), _p(partial), T, d, _dt(o), m, ctypes.cast(ks, _vp), _p(conv_w), _p(query), _p(gain), eps,
        _p(mix_gain), _p(mix_w), mix_eps, _p(dh), _p(d_o), _p(d_lse), _p(d_p), _p(dcw), _p(dq), _p(dg), _p(dmg),
        _p(dmw), _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return d_o, d_lse, d_p, dcw, dq, dg, dmg, dmw


def msar_block_phase1_bwd(src, ksizes, conv_w, queries, d_o, d_lse, gain=None, eps=1e-6, outs=None, workspace=None,
                          stream=None):
    """Backward of msar_block_phase1 for d_o [S,m,T,d], d_lse [S,m,T] ->
    (dsrc [n_src,T,d], dconv_w, dqueries [S,m,d], dgain [d]).  outs: those
    four tensors to write (else allocated here)."""
    import torch
    n_src, T, d, stride = _src_geometry(src)
    S, m = queries.shape[0], queries.shape[1]
    ks = (ctypes.c_int32 * len(ksizes))(*[int(k) for k in ksizes])
    dev, f32 = src.device, dict(dtype=torch.float32, device=src.device)
    if outs is not None:
        dsrc, dcw, dq, dg = outs
    else:
        dsrc = torch.empty((n_src, T, d), dtype=src.dtype, device=dev)
        dcw, dq, dg = (torch.empty_like(conv_w, dtype=torch.float32), torch.empty((S, m, d), **f32),
                       torch.empty((d,), **f32))
    if workspace is None:
        n = ctypes.c_size_t(0)
        _check("msar_block_phase1_bwd_workspace_size", load().msar_block_phase1_bwd_workspace_size(
            n_src, T, d, _dt(src), m, ctypes.cast(ks, _vp), S, ctypes.byref(n)))
        workspace = torch.empty((max(n.value, 16) + 3) // 4, dtype=torch.float32, device=dev)
    _check("msar_block_phase1_bwd", load().msar_block_phase1_bwd(
        _p(src), n_src, stride, T, d, _dt(src), m, ctypes.cast(ks, _vp), _p(conv_w), _p(queries), S, _p(gain), eps,
        _p(d_o), _p(d_lse), _p(dsrc), T * d, _p(dcw), _p(dq), _p(dg), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return dsrc, dcw, dq, dg
