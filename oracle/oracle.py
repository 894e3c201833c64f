"""NumPy-facing ctypes wrapper around the C oracle (attnres_oracle.c).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The CUDA library never
imports this module and this module never imports the CUDA library.

All arrays are float64, C-contiguous; bf16 or fp32 inputs are widened exactly
by the caller before they get here.  Each function names the page passage it
follows in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attnres_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags only: it must give the same
    results on x86_64 and aarch64 hosts)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # A test may point this at a deliberately broken copy of the oracle
        # (mutation testing of the pins); normally it is the built library.
        path = os.environ.get("ATTNRES_ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        lib.oracle_full.argtypes = [_D, _I64, _I64, _I64, _D, _D, ctypes.c_double, _D, _D, _D]
        lib.oracle_weighted_sum.argtypes = [_D, _I64, _I64, _I64, _D, _D]
        lib.oracle_block_oneshot.argtypes = [_D, _I64, _D, _I64, _I64, _I64, _D, _D,
                                             ctypes.c_double, _D]
        lib.oracle_block_phase1.argtypes = [_D, _I64, _I64, _I64, _D, _I64, _D, ctypes.c_double,
                                            _D, _D]
        lib.oracle_block_phase2.argtypes = [_D, _D, _D, _I64, _I64, _D, _D, ctypes.c_double, _D]
        lib.oracle_block_phase2_update.argtypes = [_D, _D, _D, _D, _I64, _I64, _D, _D,
                                                   ctypes.c_double, _D, _D]
        lib.oracle_mhar_phase2.argtypes = [_D, _D, _D, _I64, _I64, _I64, _D, _D, ctypes.c_double, _D]
        lib.oracle_read_bwd.argtypes = [_D, _I64, _I64, _I64, _D, _I64, _D, ctypes.c_double, _D, _D, _D, _D]
        lib.oracle_read_bwd_lse.argtypes = [_D, _I64, _I64, _I64, _D, _I64, _D, ctypes.c_double, _D, _D, _D, _D,
                                            _D]
        lib.oracle_block_phase2_bwd.argtypes = [_D, _D, _D, _I64, _I64, _D, _D, ctypes.c_double, _D, _D, _D, _D,
                                                _D, _D]
        lib.oracle_mhar_bwd.argtypes = [_D, _I64, _I64, _I64, _I64, _D, _I64, _D, ctypes.c_double, _D, _D, _D,
                                        _D]
        lib.oracle_mhar.argtypes = [_D, _I64, _I64, _I64, _I64, _D, _I64, _D, ctypes.c_double,
                                    _D, _D]
        lib.oracle_msar_conv.argtypes = [_D, _I64, _I64, _I64, _D, _D]
        lib.oracle_msar.argtypes = [_D, _I64, _I64, _I64, _I64, ctypes.POINTER(ctypes.c_int32),
                                    _D, _D, _D, ctypes.c_double, _D, _D, ctypes.c_double, _D,
                                    _D, _D]
        _K = ctypes.POINTER(ctypes.c_int32)
        lib.oracle_msar_bwd.argtypes = [_D, _I64, _I64, _I64, _I64, _K, _D, _D, _D, ctypes.c_double, _D, _D,
                                        ctypes.c_double, _D, _D, _D, _D, _D, _D, _D]
        lib.oracle_msar_ps.argtypes = [_D, _I64, _I64, _I64, _I64, _K, _D, _I64, _D, _D, ctypes.c_double, _D, _D,
                                       ctypes.c_double, _D]
        lib.oracle_msar_ps_bwd.argtypes = [_D, _I64, _I64, _I64, _I64, _K, _D, _I64, _D, _D, ctypes.c_double, _D,
                                           _D, ctypes.c_double, _D, _D, _D, _D, _D, _D, _D]
        lib.oracle_msar_phase1.argtypes = [_D, _I64, _I64, _I64, _I64, _K, _D, _D, _I64, _D, ctypes.c_double,
                                           _D, _D]
        lib.oracle_msar_phase2_bwd.argtypes = [_D, _D, _D, _I64, _I64, _I64, _K, _D, _D, _D, ctypes.c_double, _D, _D,
                                               ctypes.c_double, _D, _D, _D, _D, _D, _D, _D, _D, _D]
        lib.oracle_msar_phase1_bwd.argtypes = [_D, _I64, _I64, _I64, _I64, _K, _D, _D, _I64, _D, ctypes.c_double,
                                               _D, _D, _D, _D, _D, _D]
        lib.oracle_msar_phase2.argtypes = [_D, _D, _D, _I64, _I64, _I64, _K, _D, _D, _D, ctypes.c_double, _D, _D,
                                           ctypes.c_double, _D]
        for f in ("oracle_full", "oracle_weighted_sum", "oracle_block_oneshot",
                  "oracle_block_phase1", "oracle_block_phase2", "oracle_block_phase2_update",
                  "oracle_mhar_phase2", "oracle_read_bwd", "oracle_read_bwd_lse", "oracle_block_phase2_bwd",
                  "oracle_mhar_bwd", "oracle_mhar",
                  "oracle_msar_conv", "oracle_msar", "oracle_msar_bwd", "oracle_msar_ps", "oracle_msar_ps_bwd", "oracle_msar_phase1",
                  "oracle_msar_phase2", "oracle_msar_phase2_bwd", "oracle_msar_phase1_bwd"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: invalid argument")


def full(src, query, gain=None, eps=1e-6, want_lse=False, want_alpha=False):
    """Full AttnRes read of one layer.  src [n_src,T,d] -> h [T,d]."""
    src, query, gain = _f64(src), _f64(query), _f64(gain)
    n_src, T, d = src.shape
    out = np.empty((T, d))
    lse = np.empty(T) if want_lse else None
    alpha = np.empty((T, n_src)) if want_alpha else None
    _check(_load().oracle_full(_p(src), n_src, T, d, _p(query), _p(gain), float(eps), _p(out),
                               _p(lse), _p(alpha)), "oracle_full")
    res = [out]
    if want_lse:
        res.append(lse)
    if want_alpha:
        res.append(alpha)
    return res[0] if len(res) == 1 else tuple(res)


def weighted_sum(src, alpha):
    """h[t] = sum_i alpha[t,i] src[i,t].  src [n_src,T,d], alpha [T,n_src]."""
    src, alpha = _f64(src), _f64(alpha)
    n_src, T, d = src.shape
    out = np.empty((T, d))
    _check(_load().oracle_weighted_sum(_p(src), n_src, T, d, _p(alpha), _p(out)),
           "oracle_weighted_sum")
    return out


def block_oneshot(cache, partials, queries, gain=None, eps=1e-6):
    """Block AttnRes, one block, layer by layer.  cache [N,T,d],
    partials [S,T,d] (slot 0 unused) or None when S == 1, queries [S,d]
    -> out [S,T,d]."""
    cache, queries, gain = _f64(cache), _f64(queries), _f64(gain)
    N, T, d = cache.shape
    S = queries.shape[0]
    partials = _f64(partials) if partials is not None else None
    out = np.empty((S, T, d))
    _check(_load().oracle_block_oneshot(_p(cache), N, _p(partials), S, T, d, _p(queries), _p(gain),
                                        float(eps), _p(out)), "oracle_block_oneshot")
    return out


def block_phase1(cache, queries, gain=None, eps=1e-6):
    """Phase 1: queries [n_q,d] against cache [N,T,d] -> (o [n_q,T,d], lse [n_q,T])."""
    cache, queries, gain = _f64(cache), _f64(queries), _f64(gain)
    N, T, d = cache.shape
    n_q = queries.shape[0]
    o = np.empty((n_q, T, d))
    lse = np.empty((n_q, T))
    _check(_load().oracle_block_phase1(_p(cache), N, T, d, _p(queries), n_q, _p(gain), float(eps),
                                       _p(o), _p(lse)), "oracle_block_phase1")
    return o, lse


def block_phase2(o, lse, partial, query, gain=None, eps=1e-6):
    """Phase 2 merge for one layer.  o [T,d], lse [T], partial [T,d] or None."""
    o, lse, partial, query, gain = _f64(o), _f64(lse), _f64(partial), _f64(query), _f64(gain)
    T, d = o.shape
    out = np.empty((T, d))
    _check(_load().oracle_block_phase2(_p(o), _p(lse), _p(partial), T, d, _p(query), _p(gain),
                                       float(eps), _p(out)), "oracle_block_phase2")
    return out


def block_phase2_update(p, f, o, lse, query, gain=None, eps=1e-6):
    """Partial-sum update fused with the next layer's merge: p [T,d] or None,
    f [T,d], o [T,d], lse [T] -> (p + f, merged out)."""
    f, o, lse, query, gain = _f64(f), _f64(o), _f64(lse), _f64(query), _f64(gain)
    p = _f64(p) if p is not None else None
    T, d = o.shape
    p_out = np.empty((T, d))
    out = np.empty((T, d))
    _check(_load().oracle_block_phase2_update(_p(p), _p(f), _p(o), _p(lse), T, d, _p(query), _p(gain),
                                              float(eps), _p(p_out), _p(out)), "oracle_block_phase2_update")
    return p_out, out


def mhar_phase2(o, lse, partial, query, gain=None, eps=1e-6):
    """Per-head phase-2 merge: o [T,d], lse [H,T], partial [T,d] or None,
    query [H,d/H] -> out [T,d]."""
    o, lse, query, gain = _f64(o), _f64(lse), _f64(query), _f64(gain)
    partial = _f64(partial) if partial is not None else None
    T, d = o.shape
    H = query.shape[0]
    out = np.empty((T, d))
    _check(_load().oracle_mhar_phase2(_p(o), _p(lse), _p(partial), T, d, H, _p(query), _p(gain),
                                      float(eps), _p(out)), "oracle_mhar_phase2")
    return out


def block_twophase(cache, partials, queries, gain=None, eps=1e-6):
    """The two-phase schedule of one block built from the two phases above:
    phase 1 over the cache for all S queries, then layer i >= 2 merges its
    partial (layer 1 takes the phase-1 state alone)."""
    o, lse = block_phase1(cache, queries, gain, eps)
    S = queries.shape[0]
    out = np.empty_like(o)
    out[0] = o[0]
    for i in range(1, S):
        out[i] = block_phase2(o[i], lse[i], partials[i], queries[i], gain, eps)
    return out


def read_bwd(src, queries, dout, gain=None, eps=1e-6):
    """Backward of the read of queries [n_q,d] over src [n_src,T,d] for output
    gradients dout [n_q,T,d] -> (dsrc [n_src,T,d], dq [n_q,d], dgain [d])."""
    src, queries, dout, gain = _f64(src), _f64(queries), _f64(dout), _f64(gain)
    n_src, T, d = src.shape
    n_q = queries.shape[0]
    dsrc = np.empty((n_src, T, d))
    dq = np.empty((n_q, d))
    dg = np.empty(d)
    _check(_load().oracle_read_bwd(_p(src), n_src, T, d, _p(queries), n_q, _p(gain), float(eps), _p(dout),
                                   _p(dsrc), _p(dq), _p(dg)), "oracle_read_bwd")
    return dsrc, dq, dg


def block_phase1_bwd(src, queries, d_o, dlse, gain=None, eps=1e-6):
    """Backward of Block phase 1 (the read's outputs o [n_q,T,d] and its
    log-sum-exp lse [n_q,T]) for gradients d_o and dlse (None: zero) ->
    (dsrc [n_src,T,d], dq [n_q,d], dgain [d])."""
    src, queries, d_o, dlse, gain = _f64(src), _f64(queries), _f64(d_o), _f64(dlse), _f64(gain)
    n_src, T, d = src.shape
    n_q = queries.shape[0]
    dsrc = np.empty((n_src, T, d))
    dq = np.empty((n_q, d))
    dg = np.empty(d)
    _check(_load().oracle_read_bwd_lse(_p(src), n_src, T, d, _p(queries), n_q, _p(gain), float(eps), _p(d_o),
                                       _p(dlse), _p(dsrc), _p(dq), _p(dg)), "oracle_read_bwd_lse")
    return dsrc, dq, dg


def block_phase2_bwd(o, lse, partial, query, dh, gain=None, eps=1e-6):
    """Backward of the phase-2 merge: o, partial (or None), dh [T,d]; lse [T];
    query [d] -> (d_o [T,d], dlse [T], d_partial [T,d] or None, dquery [d],
    dgain [d])."""
    o, lse, partial, query, dh, gain = _f64(o), _f64(lse), _f64(partial), _f64(query), _f64(dh), _f64(gain)
    T, d = o.shape
    d_o = np.empty((T, d))
    dlse = np.empty(T)
    dp = np.empty((T, d)) if partial is not None else None
    dq = np.empty(d)
    dg = np.empty(d)
    _check(_load().oracle_block_phase2_bwd(_p(o), _p(lse), _p(partial), T, d, _p(query), _p(gain), float(eps),
                                           _p(dh), _p(d_o), _p(dlse), _p(dp), _p(dq), _p(dg)),
           "oracle_block_phase2_bwd")
    return d_o, dlse, dp, dq, dg


def mhar_bwd(src, queries, dout, gain=None, eps=1e-6):
    """Backward of the MHAR read of queries [n_q,H,d/H] over src [n_src,T,d]
    for output gradients dout [n_q,T,d] -> (dsrc [n_src,T,d],
    dq [n_q,H,d/H], dgain [d])."""
    src, queries, dout, gain = _f64(src), _f64(queries), _f64(dout), _f64(gain)
    n_src, T, d = src.shape
    n_q, H, dh = queries.shape
    assert H * dh == d
    dsrc = np.empty((n_src, T, d))
    dq = np.empty((n_q, H, dh))
    dg = np.empty(d)
    _check(_load().oracle_mhar_bwd(_p(src), n_src, T, d, H, _p(queries), n_q, _p(gain), float(eps), _p(dout),
                                   _p(dsrc), _p(dq), _p(dg)), "oracle_mhar_bwd")
    return dsrc, dq, dg


def mhar(src, queries, gain=None, eps=1e-6, want_lse=False):
    """MHAR read.  src [n_src,T,d], queries [n_q,H,d/H] -> out [n_q,T,d]
    (and lse [n_q,H,T])."""
    src, queries, gain = _f64(src), _f64(queries), _f64(gain)
    n_src, T, d = src.shape
    n_q, H, dh = queries.shape
    assert H * dh == d
    out = np.empty((n_q, T, d))
    lse = np.empty((n_q, H, T)) if want_lse else None
    _check(_load().oracle_mhar(_p(src), n_src, T, d, H, _p(queries), n_q, _p(gain), float(eps),
                               _p(out), _p(lse)), "oracle_mhar")
    return (out, lse) if want_lse else out


def msar_conv(v, cw):
    """Causal depthwise conv of one source.  v [T,d], cw [d,k] -> u [T,d]."""
    v, cw = _f64(v), _f64(cw)
    T, d = v.shape
    k = cw.shape[1]
    u = np.empty((T, d))
    _check(_load().oracle_msar_conv(_p(v), T, d, k, _p(cw), _p(u)), "oracle_msar_conv")
    return u


def msar(src, ksizes, conv_w, queries, gain=None, eps=1e-6, mix_gain=None, mix_w=None,
         mix_eps=1e-6, want_debug=False):
    """MSAR read.  src [n_src,T,d]; ksizes (m-1 ints); conv_w packed 1-D
    (kernel r as [d,k_r], concatenated); queries [m,d]; mix_w [m*d,m]."""
    src, conv_w, queries = _f64(src), _f64(conv_w), _f64(queries)
    gain, mix_gain, mix_w = _f64(gain), _f64(mix_gain), _f64(mix_w)
    n_src, T, d = src.shape
    m = queries.shape[0]
    ks = np.ascontiguousarray(ksizes, dtype=np.int32)
    assert ks.shape == (m - 1,)
    assert conv_w.size == d * int(ks.sum())
    assert mix_w.shape == (m * d, m)
    out = np.empty((T, d))
    alpha = np.empty((T, m, n_src)) if want_debug else None
    mixc = np.empty((T, m)) if want_debug else None
    _check(_load().oracle_msar(_p(src), n_src, T, d, m,
                               ks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _p(conv_w),
                               _p(queries), _p(gain), float(eps), _p(mix_gain), _p(mix_w),
                               float(mix_eps), _p(out), _p(alpha), _p(mixc)), "oracle_msar")
    return (out, alpha, mixc) if want_debug else out


def msar_phase1(src, ksizes, conv_w, queries, gain=None, eps=1e-6):
    """MSAR two-phase, phase 1.  src [n_src,T,d]; queries [S,m,d] (every layer
    of the block, one query per stream) -> o [S,m,T,d], lse [S,m,T]."""
    src, conv_w, queries, gain = _f64(src), _f64(conv_w), _f64(queries), _f64(gain)
    n_src, T, d = src.shape
    S, m, _ = queries.shape
    ks = np.ascontiguousarray(ksizes, dtype=np.int32)
    assert ks.shape == (m - 1,) and conv_w.size == d * int(ks.sum())
    o = np.empty((S, m, T, d))
    lse = np.empty((S, m, T))
    _check(_load().oracle_msar_phase1(_p(src), n_src, T, d, m, ks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                      _p(conv_w), _p(queries), S, _p(gain), float(eps), _p(o), _p(lse)),
           "oracle_msar_phase1")
    return o, lse


def msar_phase2(o, lse, partial, ksizes, conv_w, query, gain=None, eps=1e-6, mix_gain=None, mix_w=None,
                mix_eps=1e-6):
    """MSAR two-phase, phase 2 of one layer.  o [m,T,d], lse [m,T], partial
    [T,d] or None, query [m,d], mix_w [m*d,m] -> out [T,d]."""
    o, lse, partial, conv_w = _f64(o), _f64(lse), _f64(partial), _f64(conv_w)
    query, gain, mix_gain, mix_w = _f64(query), _f64(gain), _f64(mix_gain), _f64(mix_w)
    m, T, d = o.shape
    ks = np.ascontiguousarray(ksizes, dtype=np.int32)
    assert ks.shape == (m - 1,) and conv_w.size == d * int(ks.sum()) and mix_w.shape == (m * d, m)
    out = np.empty((T, d))
    _check(_load().oracle_msar_phase2(_p(o), _p(lse), _p(partial), T, d, m,
                                      ks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _p(conv_w), _p(query),
                                      _p(gain), float(eps), _p(mix_gain), _p(mix_w), float(mix_eps), _p(out)),
           "oracle_msar_phase2")
    return out


def msar_ps(src, ksizes, conv_w, queries, gain=None, eps=1e-6, mix_gain=None, mix_w=None, mix_eps=1e-6):
    """MSAR read with each source's own conv kernels: conv_w [n_src, d*sum(k)]
    (source i's kernels packed as msar's conv_w)."""
    src, conv_w, queries = _f64(src), _f64(conv_w), _f64(queries)
    gain, mix_gain, mix_w = _f64(gain), _f64(mix_gain), _f64(mix_w)
    n_src, T, d = src.shape
    m = queries.shape[0]
    ks = np.ascontiguousarray(ksizes, dtype=np.int32)
    assert ks.shape == (m - 1,) and conv_w.shape == (n_src, d * int(ks.sum())) and mix_w.shape == (m * d, m)
    out = np.empty((T, d))
    _check(_load().oracle_msar_ps(_p(src), n_src, T, d, m, ks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                  _p(conv_w), conv_w.shape[1], _p(queries), _p(gain), float(eps), _p(mix_gain),
                                  _p(mix_w), float(mix_eps), _p(out)), "oracle_msar_ps")
    return out


def msar_ps_bwd(src, ksizes, conv_w, queries, dh, gain=None, eps=1e-6, mix_gain=None, mix_w=None, mix_eps=1e-6):
    """Backward of msar_ps for dh [T,d] -> (dsrc [n_src,T,d], dconv_w [n_src,
    d*sum(k)] (each source's own), dq [m,d], dgain [d], dmix_gain [m*d],
    dmix_w [m*d,m])."""
    src, conv_w, queries, dh = _f64(src), _f64(conv_w), _f64(queries), _f64(dh)
    gain, mix_gain, mix_w = _f64(gain), _f64(mix_gain), _f64(mix_w)
    n_src, T, d = src.shape
    m = queries.shape[0]
    ks = np.ascontiguousarray(ksizes, dtype=np.int32)
    assert ks.shape == (m - 1,) and conv_w.shape == (n_src, d * int(ks.sum())) and mix_w.shape == (m * d, m)
    dsrc = np.empty((n_src, T, d))
    dcw = np.empty(conv_w.shape)
    dq = np.empty((m, d))
    dg = np.empty(d)
    dmg = np.empty(m * d)
    dmw = np.empty((m * d, m))
    _check(_load().oracle_msar_ps_bwd(_p(src), n_src, T, d, m, ks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                      _p(conv_w), conv_w.shape[1], _p(queries), _p(gain), float(eps), _p(mix_gain),
                                      _p(mix_w), float(mix_eps), _p(dh), _p(dsrc), _p(dcw), _p(dq), _p(dg), _p(dmg),
                                      _p(dmw)), "oracle_msar_ps_bwd")
    return dsrc, dcw, dq, dg, dmg, dmw


def msar_bwd(src, ksizes, conv_w, queries, dh, gain=None, eps=1e-6, mix_gain=None, mix_w=None, mix_eps=1e-6):
    """Backward of the MSAR read for dh [T,d] -> (dsrc [n_src,T,d], dconv_w
    (packed as conv_w), dq [m,d], dgain [d], dmix_gain [m*d], dmix_w [m*d,m])."""
    src, conv_w, queries, dh = _f64(src), _f64(conv_w), _f64(queries), _f64(dh)
    gain, mix_gain, mix_w = _f64(gain), _f64(mix_gain), _f64(mix_w)
    n_src, T, d = src.shape
    m = queries.shape[0]
    ks = np.ascontiguousarray(ksizes, dtype=np.int32)
    dsrc = np.empty((n_src, T, d))
    dcw = np.empty(conv_w.shape)
    dq = np.empty((m, d))
    dg = np.empty(d)
    dmg = np.empty(m * d)
    dmw = np.empty((m * d, m))
    _check(_load().oracle_msar_bwd(_p(src), n_src, T, d, m, ks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                   _p(conv_w), _p(queries), _p(gain), float(eps), _p(mix_gain), _p(mix_w),
                                   float(mix_eps), _p(dh), _p(dsrc), _p(dcw), _p(dq), _p(dg), _p(dmg), _p(dmw)),
           "oracle_msar_bwd")
    return dsrc, dcw, dq, dg, dmg, dmw


def msar_phase2_bwd(o, lse, partial, ksizes, conv_w, query, dh, gain=None, eps=1e-6, mix_gain=None, mix_w=None,
                    mix_eps=1e-6):
    """Backward of msar_phase2 for dh [T,d] -> (d_o [m,T,d], d_lse [m,T],
    d_partial [T,d] or None, dconv_w, dquery [m,d], dgain [d], dmix_gain
    [m*d], dmix_w [m*d,m])."""
    o, lse, partial, conv_w, query, dh = _f64(o), _f64(lse), _f64(partial), _f64(conv_w), _f64(query), _f64(dh)
    gain, mix_gain, mix_w = _f64(gain), _f64(mix_gain), _f64(mix_w)
    m, T, d = o.shape
    ks = np.ascontiguousarray(ksizes, dtype=np.int32)
    d_o, d_lse = np.empty((m, T, d)), np.empty((m, T))
    d_p = np.empty((T, d)) if partial is not None else None
    dcw, dq, dg = np.empty(conv_w.shape), np.empty((m, d)), np.empty(d)
    dmg, dmw = np.empty(m * d), np.empty((m * d, m))
    _check(_load().oracle_msar_phase2_bwd(_p(o), _p(lse), _p(partial), T, d, m,
                                          ks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _p(conv_w), _p(query),
                                          _p(gain), float(eps), _p(mix_gain), _p(mix_w), float(mix_eps), _p(dh),
                                          _p(d_o), _p(d_lse), _p(d_p), _p(dcw), _p(dq), _p(dg), _p(dmg), _p(dmw)),
           "oracle_msar_phase2_bwd")
    return d_o, d_lse, d_p, dcw, dq, dg, dmg, dmw


def msar_phase1_bwd(src, ksizes, conv_w, queries, d_o, d_lse, gain=None, eps=1e-6):
    """Backward of msar_phase1 for d_o [S,m,T,d], d_lse [S,m,T] -> (dsrc
    [n_src,T,d], dconv_w, dqueries [S,m,d], dgain [d])."""
    src, conv_w, queries, d_o, d_lse, gain = _f64(src), _f64(conv_w), _f64(queries), _f64(d_o), _f64(d_lse), _f64(gain)
    n_src, T, d = src.shape
    S, m = queries.shape[0], queries.shape[1]
    ks = np.ascontiguousarray(ksizes, dtype=np.int32)
    dsrc, dcw, dq, dg = np.empty((n_src, T, d)), np.empty(conv_w.shape), np.empty((S, m, d)), np.empty(d)
    _check(_load().oracle_msar_phase1_bwd(_p(src), n_src, T, d, m, ks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                          _p(conv_w), _p(queries), S, _p(gain), float(eps), _p(d_o), _p(d_lse),
                                          _p(dsrc), _p(dcw), _p(dq), _p(dg)), "oracle_msar_phase1_bwd")
    return dsrc, dcw, dq, dg
