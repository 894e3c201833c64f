"""A second, independently written oracle in NumPy (float64), for tiny shapes.

TEST INFRASTRUCTURE ONLY.  It exists so that the C oracle can be checked by
brute force against code written a different way (vectorised NumPy instead of
scalar C loops); the two agree to round-off on tiny inputs.  It follows the
same page passages as the C oracle:

* Full AttnRes: b-lab.team summary of "Attention Residuals", section 1
  (h_l = sum_i alpha_{i->l} v_i, alpha = softmax of w_l^T RMSNorm(v_i)).
* Block AttnRes: same summary, section 2 (value matrix per layer i) and the
  ai-systems-engineering.com tutorial, Fig. 4 (first sublayer reads no
  current sum).
* MHAR: chatpaper.ai "Multi-Head Attention Residuals" abstract.
* MSAR: onedev.kr MSAR summary, section 무엇과 다른가.
"""
from __future__ import annotations

import numpy as np


def _rmsnorm(x, g, eps):
    # x [..., n]; RMS over the last axis, eps inside the square root
    ms = np.mean(x * x, axis=-1, keepdims=True)
    den = np.sqrt(ms + eps)
    y = np.divide(x, den, out=np.zeros_like(x), where=den > 0)
    return y if g is None else y * g


def _read(V, w, g, eps):
    # V [n_src, T, n] -> (h [T, n], alpha [T, n_src], lse [T])
    s = np.einsum("itc,c->ti", _rmsnorm(V, g, eps), w)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    a = e / l
    return np.einsum("ti,itc->tc", a, V), a, (m + np.log(l))[:, 0]


def full(src, query, gain=None, eps=1e-6):
    return _read(np.asarray(src, np.float64), np.asarray(query, np.float64), gain, eps)[0]


def block_oneshot(cache, partials, queries, gain=None, eps=1e-6):
    cache = np.asarray(cache, np.float64)
    S = len(queries)
    outs = []
    for li in range(S):
        V = cache if li == 0 else np.concatenate([cache, np.asarray(partials[li])[None]], 0)
        outs.append(_read(V, np.asarray(queries[li], np.float64), gain, eps)[0])
    return np.stack(outs)


def mhar(src, queries, gain=None, eps=1e-6):
    src = np.asarray(src, np.float64)
    n_src, T, d = src.shape
    n_q, H, dh = np.shape(queries)
    out = np.zeros((n_q, T, d))
    for q in range(n_q):
        for h in range(H):
            sl = slice(h * dh, (h + 1) * dh)
            out[q, :, sl] = _read(src[:, :, sl], np.asarray(queries[q][h], np.float64),
                                  None if gain is None else np.asarray(gain)[sl], eps)[0]
    return out


def msar(src, ksizes, conv_w, queries, gain=None, eps=1e-6, mix_gain=None, mix_w=None,
         mix_eps=1e-6):
    src = np.asarray(src, np.float64)
    n_src, T, d = src.shape
    m = len(queries)
    streams = [src]
    off = 0
    for k in ksizes:
        cw = np.asarray(conv_w[off:off + d * k], np.float64).reshape(d, k)
        off += d * k
        u = np.zeros_like(src)
        for j in range(k):  # u[t] += cw[:, j] * v[t - j]
            u[:, j:, :] += cw[:, j] * src[:, :T - j, :] if j < T else 0.0
        streams.append(u)
    Z = np.stack([_read(streams[r], np.asarray(queries[r], np.float64), gain, eps)[0]
                  for r in range(m)])                       # [m, T, d]
    flat = Z.transpose(1, 0, 2).reshape(T, m * d)           # stream-major per token
    z = _rmsnorm(flat, mix_gain, mix_eps)
    c = 1.0 / (1.0 + np.exp(-(z @ np.asarray(mix_w, np.float64))))   # [T, m]
    return np.einsum("tr,rtc->tc", c, Z)
