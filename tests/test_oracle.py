"""Pins for the CPU oracle (no GPU).

Each test fixes the oracle to something other than itself: the values the
tutorial page prints for its worked example, closed forms, invariants of the
method, special cases that reduce to another routine, a library routine
(np.convolve), and brute force against the independently written NumPy twin.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import numpy_twin, oracle


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "worked_example.json")) as f:
        return json.load(f)


def _example_sources(g):
    # sources [n_src=3, T=1, d=3]
    return np.asarray(g["sources"], np.float64)[:, None, :]


# --------------------------------------------------------------------------
# worked example (ai-systems-engineering.com tutorial, Figs. 2-3)
# --------------------------------------------------------------------------

def test_worked_example_alpha_and_h(golden_dir):
    g = _golden(golden_dir)
    src = _example_sources(g)
    w = np.array([0.0, math.log(2.0) / math.sqrt(3.0), 0.0])
    h, lse, alpha = oracle.full(src, w, None, eps=0.0, want_lse=True, want_alpha=True)
    assert np.allclose(alpha[0], g["alpha"], atol=1e-12, rtol=0)
    assert np.allclose(h[0], g["h"], atol=1e-12, rtol=0)
    # scores [0, ln2, 0] -> sum of exp = 1 + 2 + 1 = 4
    assert abs(lse[0] - math.log(4.0)) < 1e-12


def test_worked_example_padded_to_d8(golden_dir):
    """The same example padded with zero channels to d=8: every nonzero now
    normalises to sqrt(8); w = [0, ln2/sqrt(8), 0, ...] gives the same scores,
    weights and (padded) output.  This is the form the GPU test uses."""
    g = _golden(golden_dir)
    src = np.zeros((3, 1, 8))
    src[:, :, :3] = _example_sources(g)
    w = np.zeros(8)
    w[1] = math.log(2.0) / math.sqrt(8.0)
    h, alpha = oracle.full(src, w, None, eps=0.0, want_alpha=True)
    assert np.allclose(alpha[0], g["alpha"], atol=1e-12, rtol=0)
    assert np.allclose(h[0, :3], g["h"], atol=1e-12, rtol=0)
    assert np.all(h[0, 3:] == 0.0)


def test_worked_example_alternative_weights(golden_dir):
    g = _golden(golden_dir)
    src = _example_sources(g)
    h = oracle.weighted_sum(src, np.asarray(g["alternative_alpha"])[None, :])
    assert np.allclose(h[0], g["alternative_h"], atol=1e-12, rtol=0)


def test_equal_scores_give_mean_not_residual_sum(golden_dir):
    g = _golden(golden_dir)
    src = _example_sources(g)
    h, alpha = oracle.full(src, np.zeros(3), None, eps=0.0, want_alpha=True)
    assert np.allclose(alpha, 1.0 / 3.0, atol=1e-15)
    assert np.allclose(h[0], np.mean(src[:, 0, :], axis=0), atol=1e-15)
    assert not np.allclose(h[0], g["residual_sum"])


def test_values_are_raw_not_normalised(golden_dir):
    """A uniform read of the example gives (2/3, 4/3, 2); normalised values
    would give sqrt(3)/3 on every channel."""
    g = _golden(golden_dir)
    h = oracle.full(_example_sources(g), np.zeros(3), None, eps=0.0)
    assert np.allclose(h[0], [2.0 / 3.0, 4.0 / 3.0, 2.0], atol=1e-15)


# --------------------------------------------------------------------------
# closed forms and invariants of the read
# --------------------------------------------------------------------------

def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def test_zero_query_gives_uniform_weights():
    """Pseudo-queries start at zero (review 3-2 3), 4-2): uniform alpha, so h is
    the mean of the sources."""
    rng = np.random.default_rng(1)
    src = _rand(rng, 5, 7, 16) * np.arange(1, 6)[:, None, None]
    h, alpha = oracle.full(src, np.zeros(16), None, eps=1e-6, want_alpha=True)
    assert np.allclose(alpha, 0.2, atol=1e-15)
    assert np.allclose(h, src.mean(axis=0), atol=1e-13)


def test_weights_sum_to_one_and_are_positive():
    rng = np.random.default_rng(2)
    src = _rand(rng, 9, 11, 24, scale=3.0)
    _, alpha = oracle.full(src, _rand(rng, 24, scale=2.0), None, eps=1e-6, want_alpha=True)
    assert np.all(alpha > 0)
    assert np.allclose(alpha.sum(axis=1), 1.0, atol=1e-14)


def test_eps_sits_inside_the_square_root():
    """Constant row x on every channel: mean square x^2, so with eps inside the
    root the normalised key is x / sqrt(x^2 + eps).  x = sqrt(3), eps = 1 gives
    sqrt(3)/2 per channel; with w = e_0 * s the score is s*sqrt(3)/2.  Against a
    zero source (score 0) the weight is sigmoid(s*sqrt(3)/2)."""
    d = 4
    src = np.zeros((2, 1, d))
    src[0, 0, :] = math.sqrt(3.0)
    w = np.zeros(d)
    w[0] = 2.0
    _, alpha = oracle.full(src, w, None, eps=1.0, want_alpha=True)
    s = 2.0 * math.sqrt(3.0) / 2.0
    assert abs(alpha[0, 0] - 1.0 / (1.0 + math.exp(-s))) < 1e-14


def test_zero_source_with_zero_eps_scores_zero():
    src = np.zeros((2, 1, 8))
    src[1, 0, 3] = 5.0
    w = np.zeros(8)
    w[3] = 1.0
    h, alpha = oracle.full(src, w, None, eps=0.0, want_alpha=True)
    # zero source normalises to 0 -> score 0; the other scores sqrt(8)
    e = math.exp(math.sqrt(8.0))
    assert abs(alpha[0, 1] - e / (1.0 + e)) < 1e-14
    assert np.all(np.isfinite(h))


def test_scale_invariance_at_zero_eps():
    """RMSNorm removes the magnitude of each source from its score."""
    rng = np.random.default_rng(3)
    src = _rand(rng, 6, 5, 32)
    w = _rand(rng, 32)
    _, a1 = oracle.full(src, w, None, eps=0.0, want_alpha=True)
    scaled = src * np.array([0.1, 3.0, 7.0, 1.0, 0.5, 100.0])[:, None, None]
    _, a2 = oracle.full(scaled, w, None, eps=0.0, want_alpha=True)
    assert np.allclose(a1, a2, atol=1e-13)


def test_permutation_equivariance():
    rng = np.random.default_rng(4)
    src = _rand(rng, 7, 6, 16)
    w = _rand(rng, 16)
    h1, a1 = oracle.full(src, w, None, eps=1e-6, want_alpha=True)
    perm = rng.permutation(7)
    h2, a2 = oracle.full(src[perm], w, None, eps=1e-6, want_alpha=True)
    assert np.allclose(h1, h2, atol=1e-13)
    assert np.allclose(a1[:, perm], a2, atol=1e-14)


def test_gain_acts_on_the_key_like_a_query_scale():
    """Gain multiplies the normalised key, so gain g equals query w*g with unit
    gain; a zero gain channel drops out of the score but not out of h."""
    rng = np.random.default_rng(5)
    src = _rand(rng, 4, 3, 16)
    w = _rand(rng, 16)
    g = rng.uniform(0.5, 2.0, 16)
    h1 = oracle.full(src, w, g, eps=1e-6)
    h2 = oracle.full(src, w * g, None, eps=1e-6)
    assert np.allclose(h1, h2, atol=1e-13)
    g0 = np.ones(16)
    g0[5] = 0.0
    w2 = w.copy()
    w2[5] = 0.0
    h3 = oracle.full(src, w, g0, eps=1e-6)
    h4 = oracle.full(src, w2, None, eps=1e-6)
    assert np.allclose(h3, h4, atol=1e-13)


def test_single_source_returns_it():
    rng = np.random.default_rng(6)
    src = _rand(rng, 1, 4, 8)
    assert np.array_equal(oracle.full(src, _rand(rng, 8), None, eps=1e-6), src[0])


# --------------------------------------------------------------------------
# Block AttnRes
# --------------------------------------------------------------------------

def test_two_phase_equals_oneshot():
    """The online-softmax merge of phase 2 is exact (summary section 3; review
    3-2 4))."""
    rng = np.random.default_rng(7)
    N, S, T, d = 5, 4, 6, 24
    cache = _rand(rng, N, T, d) * (1 + np.arange(N))[:, None, None]
    partials = _rand(rng, S, T, d)
    q = _rand(rng, S, d, scale=2.0)
    g = rng.uniform(0.5, 1.5, d)
    one = oracle.block_oneshot(cache, partials, q, g, eps=1e-6)
    two = oracle.block_twophase(cache, partials, q, g, eps=1e-6)
    assert np.allclose(one, two, atol=1e-13, rtol=0)


def test_block_first_layer_reads_no_partial():
    rng = np.random.default_rng(8)
    N, S, T, d = 3, 3, 4, 16
    cache = _rand(rng, N, T, d)
    partials = _rand(rng, S, T, d)
    q = _rand(rng, S, d)
    out = oracle.block_oneshot(cache, partials, q, eps=1e-6)
    p2 = partials.copy()
    p2[0] += 100.0
    out2 = oracle.block_oneshot(cache, p2, q, eps=1e-6)
    assert np.array_equal(out[0], out2[0])
    assert np.allclose(out[0], oracle.full(cache, q[0], None, eps=1e-6), atol=1e-14)
    # later layers do read their partial
    assert not np.allclose(out[1], oracle.full(cache, q[1], None, eps=1e-6))


def test_block_size_one_is_full():
    """Block size S=1 (N=L blocks) is Full AttnRes (review 5-2 4))."""
    rng = np.random.default_rng(9)
    L, T, d = 6, 5, 16
    v = _rand(rng, L, T, d)
    w = _rand(rng, d)
    blk = oracle.block_oneshot(v, None, w[None, :], eps=1e-6)[0]
    assert np.allclose(blk, oracle.full(v, w, None, eps=1e-6), atol=1e-15)


def test_block_shares_one_weight_per_merged_source():
    """Tutorial Fig. 4: Block keeps e, f1+f2, f3; f1 and f2 share the single
    weight of their sum, which is not the sum of Full's two weights."""
    e = np.array([2.0, 0, 0, 0])
    f1 = np.array([0, 4.0, 0, 0])
    f2 = np.array([0, 0, 6.0, 0])
    f3 = np.array([0, 0, 0, 8.0])
    w = np.array([0.3, 1.2, -0.7, 0.4])
    full_h, full_a = oracle.full(np.stack([e, f1, f2, f3])[:, None, :], w, None, eps=0.0,
                                 want_alpha=True)
    cache = np.stack([e, f1 + f2])[:, None, :]
    partials = np.stack([np.zeros(4), f3])[:, None, :]
    blk = oracle.block_oneshot(cache, partials, np.stack([w, w]), None, eps=0.0)[1, 0]
    beta1 = blk[1] / 4.0
    beta2 = blk[2] / 6.0
    assert abs(beta1 - beta2) < 1e-14
    assert abs(full_h[0, 1] / 4.0 - full_h[0, 2] / 6.0) > 1e-3
    assert abs(beta1 - (full_a[0, 1] + full_a[0, 2])) > 1e-3


def test_phase2_without_partial_is_identity():
    rng = np.random.default_rng(10)
    o = _rand(rng, 3, 8)
    out = oracle.block_phase2(o, _rand(rng, 3), None, _rand(rng, 8))
    assert np.array_equal(out, o)


def test_fused_update_chain_equals_oneshot_block():
    """Summary section 2: layer i >= 2 of a block reads the partial sum of the
    block's outputs so far; Tutorial Fig. 4: each new output only changes the
    current partial.  Chaining the fused update-and-merge over a block gives the
    one-shot Block read with the cumulative partials, and the last partial is
    the block's sum of outputs."""
    rng = np.random.default_rng(21)
    N, S, T, d = 4, 5, 5, 24
    cache = _rand(rng, N, T, d) * (1 + np.arange(N))[:, None, None]
    f = _rand(rng, S, T, d)                       # outputs f_1..f_S of the block's layers
    q = _rand(rng, S, d, scale=2.0)
    g = rng.uniform(0.5, 1.5, d)
    partials = np.zeros((S, T, d))
    partials[1:] = np.cumsum(f[:-1], axis=0)       # layer i reads f_1 + ... + f_{i-1}
    ref = oracle.block_oneshot(cache, partials, q, g, eps=1e-6)
    o, lse = oracle.block_phase1(cache, q, g, eps=1e-6)
    p = None
    for i in range(1, S):
        p, out = oracle.block_phase2_update(p, f[i - 1], o[i], lse[i], q[i], g, eps=1e-6)
        assert np.allclose(out, ref[i], atol=1e-13, rtol=0)
    p, _ = oracle.block_phase2_update(p, f[S - 1], o[0], lse[0], q[0], g, eps=1e-6)
    assert np.allclose(p, f.sum(axis=0), atol=1e-13, rtol=0)


def test_fused_update_tutorial_fig4_state():
    """Tutorial Fig. 4: the block keeps e, f1+f2 and the current f3; after f4
    the current sum is f3+f4 and the next layer reads e, f1+f2, f3+f4 (a Full
    read over those three sources)."""
    e = np.array([2.0, 0, 0, 0])
    f1 = np.array([0, 4.0, 0, 0])
    f2 = np.array([0, 0, 6.0, 0])
    f3 = np.array([0, 0, 0, 8.0])
    f4 = np.array([1.0, -2.0, 0.5, 3.0])
    w = np.array([0.3, 1.2, -0.7, 0.4])
    cache = np.stack([e, f1 + f2])[:, None, :]
    o, lse = oracle.block_phase1(cache, w[None, :], None, eps=0.0)
    p, out = oracle.block_phase2_update(f3[None, :], f4[None, :], o[0], lse[0], w, None, eps=0.0)
    assert np.array_equal(p[0], f3 + f4)
    ref = oracle.full(np.stack([e, f1 + f2, f3 + f4])[:, None, :], w, None, eps=0.0)
    assert np.allclose(out, ref, atol=1e-14, rtol=0)


def test_fused_update_without_old_partial_starts_the_sum():
    rng = np.random.default_rng(22)
    T, d = 3, 16
    f, o = _rand(rng, T, d), _rand(rng, T, d)
    lse, q = _rand(rng, T), _rand(rng, d)
    p, out = oracle.block_phase2_update(None, f, o, lse, q, eps=1e-6)
    assert np.array_equal(p, f)
    assert np.allclose(out, oracle.block_phase2(o, lse, f, q, eps=1e-6), atol=0, rtol=0)


def _fd_grads(src, q, g, dout, eps, h=1e-6):
    """Central finite differences of L = sum(dout * h_out) through the forward
    oracle (Block phase 1 reads every query against every source)."""
    def loss(s_, q_, g_):
        o, _ = oracle.block_phase1(s_, q_, g_, eps)
        return float((o * dout).sum())
    out = []
    for x, put in ((src, lambda v: (v, q, g)), (q, lambda v: (src, v, g)), (g, lambda v: (src, q, v))):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            a, b = x.copy(), x.copy()
            a[idx] += h
            b[idx] -= h
            fd[idx] = (loss(*put(a)) - loss(*put(b))) / (2 * h)
        out.append(fd)
    return out


@pytest.mark.parametrize("n_src,n_q,eps,with_gain", [(3, 1, 1e-6, False), (5, 3, 1e-6, True), (2, 2, 0.1, True),
                                                     (4, 1, 0.0, True)])
def test_read_bwd_matches_finite_differences(n_src, n_q, eps, with_gain):
    """The backward of the read against central differences of the (pinned)
    forward oracle, for the sources, the queries and the gain."""
    rng = np.random.default_rng(31 + n_src * 3 + n_q)
    T, d = 2, 8
    src = _rand(rng, n_src, T, d) * (1 + np.arange(n_src))[:, None, None]
    q = _rand(rng, n_q, d, scale=1.5)
    g = rng.uniform(0.5, 1.5, d) if with_gain else np.ones(d)
    dout = _rand(rng, n_q, T, d)
    dsrc, dq, dg = oracle.read_bwd(src, q, dout, g if with_gain else None, eps)
    fs, fq, fg = _fd_grads(src, q, g, dout, eps)
    for got, ref in ((dsrc, fs), (dq, fq), (dg, fg)):
        assert np.abs(got - ref).max() <= 1e-6 * max(1.0, np.abs(ref).max())


def test_read_bwd_single_source_passes_the_gradient_straight_through():
    """One source: alpha = 1 whatever the score, so the source gets the sum of
    the output gradients and the query and the gain get nothing."""
    rng = np.random.default_rng(32)
    src = _rand(rng, 1, 4, 16)
    q, dout = _rand(rng, 3, 16), _rand(rng, 3, 4, 16)
    dsrc, dq, dg = oracle.read_bwd(src, q, dout, rng.uniform(0.5, 1.5, 16), 1e-6)
    assert np.allclose(dsrc[0], dout.sum(axis=0), atol=1e-14)
    assert np.abs(dq).max() == 0.0 and np.abs(dg).max() == 0.0


def test_read_bwd_score_path_is_orthogonal_to_the_source_at_zero_eps():
    """At eps = 0 a score does not change when its source is scaled, so the
    score path's gradient of source i (its gradient minus the value path's
    sum_q alpha_qi dout_q) is orthogonal to v_i."""
    rng = np.random.default_rng(33)
    n_src, T, d = 4, 3, 12
    src = _rand(rng, n_src, T, d) * (1 + np.arange(n_src))[:, None, None]
    q, dout = _rand(rng, 2, d, scale=2.0), _rand(rng, 2, T, d)
    dsrc, _, _ = oracle.read_bwd(src, q, dout, None, 0.0)
    _, alpha = oracle.full(src, q[0], None, eps=0.0, want_alpha=True)
    _, alpha1 = oracle.full(src, q[1], None, eps=0.0, want_alpha=True)
    value = (alpha.T[:, :, None] * dout[0][None]) + (alpha1.T[:, :, None] * dout[1][None])
    score_part = dsrc - value
    assert np.abs((score_part * src).sum(axis=2)).max() < 1e-12
    assert np.abs(score_part).max() > 1e-3


def _fd(loss, args, h=1e-6):
    """Central differences of loss(*args) with respect to every array in args
    (None entries skipped)."""
    out = []
    for n, x in enumerate(args):
        if x is None:
            out.append(None)
            continue
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            a, b = [list(args), list(args)]
            xa, xb = x.copy(), x.copy()
            xa[idx] += h
            xb[idx] -= h
            a[n], b[n] = xa, xb
            fd[idx] = (loss(*a) - loss(*b)) / (2 * h)
        out.append(fd)
    return out


@pytest.mark.parametrize("eps,with_gain", [(1e-6, True), (0.1, False), (0.0, True)])
def test_block_phase1_bwd_matches_finite_differences(eps, with_gain):
    """Block phase 1's backward for gradients of both its outputs, o and lse,
    against central differences of the (pinned) phase-1 oracle."""
    rng = np.random.default_rng(71)
    n_src, n_q, T, d = 4, 3, 2, 8
    src = _rand(rng, n_src, T, d) * (1 + np.arange(n_src))[:, None, None]
    q = _rand(rng, n_q, d, scale=1.5)
    g = rng.uniform(0.5, 1.5, d) if with_gain else np.ones(d)
    d_o, dl = _rand(rng, n_q, T, d), _rand(rng, n_q, T)

    def loss(s_, q_, g_):
        o, lse = oracle.block_phase1(s_, q_, g_, eps)
        return float((o * d_o).sum() + (lse * dl).sum())
    got = oracle.block_phase1_bwd(src, q, d_o, dl, g if with_gain else None, eps)
    ref = _fd(loss, (src, q, g))
    for x, y in zip(got, ref):
        assert np.abs(x - y).max() <= 1e-6 * max(1.0, np.abs(y).max())


def test_block_phase1_bwd_without_lse_gradient_is_the_read_backward():
    rng = np.random.default_rng(72)
    src, q, d_o = _rand(rng, 5, 3, 16), _rand(rng, 2, 16), _rand(rng, 2, 3, 16)
    a = oracle.block_phase1_bwd(src, q, d_o, None, None, 1e-6)
    b = oracle.read_bwd(src, q, d_o, None, 1e-6)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("eps,with_gain", [(1e-6, True), (0.1, False), (0.0, True)])
def test_block_phase2_bwd_matches_finite_differences(eps, with_gain):
    """The merge's backward against central differences of the (pinned)
    phase-2 oracle, for o, lse, the partial, the query and the gain."""
    rng = np.random.default_rng(73)
    T, d = 3, 8
    o, p, dh = _rand(rng, T, d), _rand(rng, T, d, scale=2.0), _rand(rng, T, d)
    lse, q = _rand(rng, T), _rand(rng, d, scale=1.5)
    g = rng.uniform(0.5, 1.5, d) if with_gain else np.ones(d)

    def loss(o_, l_, p_, q_, g_):
        return float((oracle.block_phase2(o_, l_, p_, q_, g_, eps=eps) * dh).sum())
    d_o, dl, dp, dq, dg = oracle.block_phase2_bwd(o, lse, p, q, dh, g if with_gain else None, eps)
    ref = _fd(loss, (o, lse, p, q, g))
    for x, y in zip((d_o, dl, dp, dq, dg), ref):
        assert np.abs(x - y).max() <= 1e-6 * max(1.0, np.abs(y).max())


def test_block_phase2_bwd_without_partial_passes_the_gradient_to_o():
    rng = np.random.default_rng(74)
    o, dh, lse, q = _rand(rng, 4, 8), _rand(rng, 4, 8), _rand(rng, 4), _rand(rng, 8)
    d_o, dl, dp, dq, dg = oracle.block_phase2_bwd(o, lse, None, q, dh)
    assert np.array_equal(d_o, dh) and not dl.any() and dp is None and not dq.any() and not dg.any()


@pytest.mark.parametrize("N,eps", [(4, 1e-6), (1, 0.05), (6, 0.0)])
def test_two_phase_backward_equals_one_shot_backward(N, eps):
    """The two-phase schedule computes the one-shot read of [b_0..b_{N-1}, p]
    ([Summary §3 Inference]), so its backward -- the merge's backward, then
    phase 1's backward for the merge's d_o and dlse -- gives the one-shot
    read's gradients: the cached sources', the partial's, the query's and the
    gain's."""
    rng = np.random.default_rng(75 + N)
    T, d = 3, 12
    cached = _rand(rng, N, T, d) * (1 + 0.5 * np.arange(N))[:, None, None]
    p, dh = _rand(rng, T, d, scale=1.5), _rand(rng, T, d)
    q = _rand(rng, d, scale=1.5)
    g = rng.uniform(0.5, 1.5, d)
    o, lse = oracle.block_phase1(cached, q[None], g, eps)
    d_o, dl, dp, dq2, dg2 = oracle.block_phase2_bwd(o[0], lse[0], p, q, dh, g, eps)
    ds1, dq1, dg1 = oracle.block_phase1_bwd(cached, q[None], d_o[None], dl[None], g, eps)
    ref_s, ref_q, ref_g = oracle.read_bwd(np.concatenate([cached, p[None]]), q[None], dh[None], g, eps)
    tol = lambda y: 1e-12 * max(1.0, np.abs(y).max())
    assert np.abs(ds1 - ref_s[:N]).max() <= tol(ref_s)
    assert np.abs(dp - ref_s[N]).max() <= tol(ref_s)
    assert np.abs(dq1[0] + dq2 - ref_q[0]).max() <= tol(ref_q)
    assert np.abs(dg1 + dg2 - ref_g).max() <= tol(ref_g)


def _fd_grads_mhar(src, q, g, dout, eps, h=1e-6):
    """Central finite differences of L = sum(dout * out) through the MHAR
    forward oracle; q is [n_q, H, d/H]."""
    def loss(s_, q_, g_):
        return float((oracle.mhar(s_, q_, g_, eps) * dout).sum())
    out = []
    for x, put in ((src, lambda v: (v, q, g)), (q, lambda v: (src, v, g)), (g, lambda v: (src, q, v))):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            a, b = x.copy(), x.copy()
            a[idx] += h
            b[idx] -= h
            fd[idx] = (loss(*put(a)) - loss(*put(b))) / (2 * h)
        out.append(fd)
    return out


@pytest.mark.parametrize("n_src,n_q,H,eps", [(3, 1, 2, 1e-6), (4, 2, 4, 0.05), (2, 3, 3, 0.0)])
def test_mhar_bwd_matches_finite_differences(n_src, n_q, H, eps):
    """The MHAR backward against central differences of the (pinned) MHAR
    forward oracle: per-head RMSNorm, softmax and slice of the gain."""
    rng = np.random.default_rng(41 + n_src + 7 * H)
    T, dh = 2, 4
    d = H * dh
    src = _rand(rng, n_src, T, d) * (1 + np.arange(n_src))[:, None, None]
    q = _rand(rng, n_q, H, dh, scale=1.5)
    g = rng.uniform(0.5, 1.5, d)
    dout = _rand(rng, n_q, T, d)
    dsrc, dq, dg = oracle.mhar_bwd(src, q, dout, g, eps)
    fs, fq, fg = _fd_grads_mhar(src, q, g, dout, eps)
    for got, ref in ((dsrc, fs), (dq, fq), (dg, fg)):
        assert np.abs(got - ref).max() <= 1e-6 * max(1.0, np.abs(ref).max())


def test_mhar_bwd_one_head_is_the_read_backward():
    """H = 1 recovers the single-head read ([MHAR abstract]), so its backward
    is the read's backward."""
    rng = np.random.default_rng(43)
    src, q, dout = _rand(rng, 5, 3, 16), _rand(rng, 2, 16), _rand(rng, 2, 3, 16)
    g = rng.uniform(0.5, 1.5, 16)
    a = oracle.mhar_bwd(src, q[:, None, :], dout, g, 1e-6)
    b = oracle.read_bwd(src, q, dout, g, 1e-6)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1][:, 0], b[1]) and np.array_equal(a[2], b[2])


def test_mhar_bwd_is_block_diagonal():
    """An output gradient on head h's slice alone gives gradients on that
    slice alone: the other slices of the sources, the queries and the gain get
    exactly zero."""
    rng = np.random.default_rng(44)
    n_src, T, H, dh = 4, 3, 4, 6
    d = H * dh
    src, q = _rand(rng, n_src, T, d), _rand(rng, 2, H, dh)
    dout = np.zeros((2, T, d))
    dout[:, :, 2 * dh:3 * dh] = _rand(rng, 2, T, dh)
    dsrc, dq, dg = oracle.mhar_bwd(src, q, dout, rng.uniform(0.5, 1.5, d), 1e-6)
    off = np.ones(d, dtype=bool)
    off[2 * dh:3 * dh] = False
    assert np.abs(dsrc[:, :, off]).max() == 0.0 and np.abs(dg[off]).max() == 0.0
    assert np.abs(np.delete(dq, 2, axis=1)).max() == 0.0
    assert np.abs(dsrc[:, :, ~off]).max() > 1e-3 and np.abs(dq[:, 2]).max() > 1e-3


# --------------------------------------------------------------------------
# MHAR
# --------------------------------------------------------------------------

def test_mhar_one_head_is_attnres():
    rng = np.random.default_rng(11)
    src = _rand(rng, 5, 4, 32)
    q = _rand(rng, 3, 1, 32)
    out = oracle.mhar(src, q, eps=1e-6)
    for i in range(3):
        assert np.allclose(out[i], oracle.full(src, q[i, 0], None, eps=1e-6), atol=1e-15)


def test_mhar_each_head_is_attnres_on_its_slice():
    rng = np.random.default_rng(12)
    H, dh = 4, 8
    src = _rand(rng, 6, 3, H * dh)
    q = _rand(rng, 2, H, dh, scale=2.0)
    g = rng.uniform(0.5, 1.5, H * dh)
    out, lse = oracle.mhar(src, q, g, eps=1e-6, want_lse=True)
    for i in range(2):
        for h in range(H):
            sl = slice(h * dh, (h + 1) * dh)
            ref, ref_lse = oracle.full(src[:, :, sl], q[i, h], g[sl], eps=1e-6, want_lse=True)
            assert np.allclose(out[i, :, sl], ref, atol=1e-15)
            assert np.allclose(lse[i, h], ref_lse, atol=1e-15)


def test_mhar_read_is_block_diagonal():
    rng = np.random.default_rng(13)
    H, dh = 4, 8
    src = _rand(rng, 5, 3, H * dh)
    q = _rand(rng, 1, H, dh, scale=2.0)
    base = oracle.mhar(src, q, eps=1e-6)
    src2 = src.copy()
    src2[2, :, dh:2 * dh] += _rand(rng, 3, dh, scale=5.0)   # perturb head 1 only
    pert = oracle.mhar(src2, q, eps=1e-6)
    changed = np.abs(pert - base).max(axis=(0, 1)) > 0
    assert np.all(changed[dh:2 * dh])
    assert not np.any(changed[:dh]) and not np.any(changed[2 * dh:])


def test_mhar_two_phase_equals_oneshot():
    """MHAR inside the two-phase schedule: phase 1 over the cached reps keeps
    lse per head; the per-head merge of the partial gives the one-shot MHAR
    read over the reps plus the partial."""
    rng = np.random.default_rng(23)
    H, dh, N, T = 4, 8, 5, 6
    d = H * dh
    cache = _rand(rng, N, T, d) * (1 + np.arange(N))[:, None, None]
    p = _rand(rng, T, d, scale=2.0)
    q = _rand(rng, 1, H, dh, scale=2.0)
    g = rng.uniform(0.5, 1.5, d)
    o, lse = oracle.mhar(cache, q, g, eps=1e-6, want_lse=True)
    two = oracle.mhar_phase2(o[0], lse[0], p, q[0], g, eps=1e-6)
    one = oracle.mhar(np.concatenate([cache, p[None]]), q, g, eps=1e-6)[0]
    assert np.allclose(two, one, atol=1e-13, rtol=0)


def test_mhar_phase2_one_head_is_block_phase2():
    rng = np.random.default_rng(24)
    T, d = 4, 24
    o, p = _rand(rng, T, d), _rand(rng, T, d)
    lse, q = _rand(rng, T), _rand(rng, d)
    g = rng.uniform(0.5, 1.5, d)
    a = oracle.mhar_phase2(o, lse[None], p, q[None], g, eps=1e-6)
    b = oracle.block_phase2(o, lse, p, q, g, eps=1e-6)
    assert np.allclose(a, b, atol=1e-15, rtol=0)


# --------------------------------------------------------------------------
# MSAR
# --------------------------------------------------------------------------

def test_msar_conv_matches_np_convolve():
    rng = np.random.default_rng(14)
    T, d, k = 20, 5, 8
    v = _rand(rng, T, d)
    cw = _rand(rng, d, k)
    u = oracle.msar_conv(v, cw)
    for c in range(d):
        assert np.allclose(u[:, c], np.convolve(v[:, c], cw[c])[:T], atol=1e-13)


def _delta_conv(d, ksizes):
    parts = []
    for k in ksizes:
        cw = np.zeros((d, k))
        cw[:, 0] = 1.0
        parts.append(cw.ravel())
    return np.concatenate(parts)


def test_msar_delta_conv_and_zero_mixer_is_two_attnres():
    """Delta kernels make every stream the source itself; one shared query
    makes every stream read Full AttnRes A; a zero projection gives sigmoid(0)
    = 1/2 per stream, so h = (m/2) A = 2A for m = 4."""
    rng = np.random.default_rng(15)
    N, T, d = 5, 9, 16
    ks = (4, 8, 12)
    src = _rand(rng, N, T, d)
    w = _rand(rng, d, scale=2.0)
    h = oracle.msar(src, ks, _delta_conv(d, ks), np.stack([w] * 4), None, 1e-6, None,
                    np.zeros((4 * d, 4)), 1e-6)
    assert np.allclose(h, 2.0 * oracle.full(src, w, None, eps=1e-6), atol=1e-13)


def test_msar_mixer_single_projection_entry_and_flatten_order():
    """Zero conv kernels make streams 1..3 zero, so Flatten(Z) = [A, 0, 0, 0]
    whose RMS over 4d is rms(A)/2.  A single projection entry beta at row 1
    (stream 0, channel 1), column 0 gives c_0 = sigmoid(2 A[1] beta / rms(A))
    and h = c_0 A.  The same entry at row d (stream 1, channel 0) sees a zero
    and gives h = A/2; a channel-major flatten would swap these two cases."""
    rng = np.random.default_rng(16)
    N, T, d = 4, 6, 8
    ks = (4, 8, 12)
    src = _rand(rng, N, T, d)
    q = _rand(rng, 4, d, scale=2.0)
    cw = np.zeros(d * sum(ks))
    A = oracle.full(src, q[0], None, eps=0.0)
    beta = 1.7
    P = np.zeros((4 * d, 4))
    P[1, 0] = beta
    h = oracle.msar(src, ks, cw, q, None, 0.0, None, P, 0.0)
    rmsA = np.sqrt(np.mean(A * A, axis=1))
    c0 = 1.0 / (1.0 + np.exp(-2.0 * A[:, 1] * beta / rmsA))
    assert np.allclose(h, c0[:, None] * A, atol=1e-13)
    P = np.zeros((4 * d, 4))
    P[d, 0] = beta
    h = oracle.msar(src, ks, cw, q, None, 0.0, None, P, 0.0)
    assert np.allclose(h, 0.5 * A, atol=1e-13)


def test_msar_stream_weights_sum_to_one():
    rng = np.random.default_rng(17)
    N, T, d = 6, 7, 16
    ks = (4, 8, 12)
    src = _rand(rng, N, T, d)
    _, alpha, mixc = oracle.msar(src, ks, _rand(rng, d * sum(ks), scale=0.4),
                                 _rand(rng, 4, d, scale=2.0), None, 1e-6, None,
                                 _rand(rng, 4 * d, 4, scale=0.2), 1e-6, want_debug=True)
    assert np.allclose(alpha.sum(axis=2), 1.0, atol=1e-14)
    assert np.all((mixc > 0) & (mixc < 1))


def test_msar_is_causal_with_window_twelve():
    rng = np.random.default_rng(18)
    N, T, d = 3, 30, 8
    ks = (4, 8, 12)
    src = _rand(rng, N, T, d)
    args = (ks, _rand(rng, d * sum(ks), scale=0.4), _rand(rng, 4, d, scale=2.0), None, 1e-6,
            None, _rand(rng, 4 * d, 4, scale=0.2), 1e-6)
    base = oracle.msar(src, *args)
    t = 20
    for tp, should_change in ((t + 1, False), (t - 12, False), (t - 11, True), (t, True)):
        s2 = src.copy()
        s2[1, tp] += 3.0
        h = oracle.msar(s2, *args)
        assert (np.abs(h[t] - base[t]).max() > 0) == should_change, tp


def test_msar_window_read_equals_full_sequence():
    """Tokens of a 12-row window ending at t reproduce row t of the full
    causal sequence; this is how sampled full-size checks are computed."""
    rng = np.random.default_rng(19)
    N, T, d = 3, 40, 8
    ks = (4, 8, 12)
    src = _rand(rng, N, T, d)
    args = (ks, _rand(rng, d * sum(ks), scale=0.4), _rand(rng, 4, d, scale=2.0), None, 1e-6,
            None, _rand(rng, 4 * d, 4, scale=0.2), 1e-6)
    base = oracle.msar(src, *args)
    for t in (0, 5, 11, 12, 39):
        lo = max(0, t - 11)
        win = oracle.msar(src[:, lo:t + 1], *args)
        assert np.allclose(win[-1], base[t], atol=1e-14)


def test_msar_per_source_with_equal_kernels_is_msar():
    """Every source given the same kernels is the shared-kernel read."""
    rng = np.random.default_rng(81)
    N, T, d, ks = 4, 15, 8, (4, 8, 12)
    src, q = _rand(rng, N, T, d), _rand(rng, 4, d, scale=2.0)
    cw, P = _rand(rng, d * sum(ks), scale=0.4), _rand(rng, 4 * d, 4, scale=0.2)
    a = oracle.msar_ps(src, ks, np.stack([cw] * N), q, None, 1e-6, None, P, 1e-6)
    b = oracle.msar(src, ks, cw, q, None, 1e-6, None, P, 1e-6)
    assert np.allclose(a, b, atol=1e-13, rtol=0)


def test_msar_per_source_delay_kernels_are_delayed_sources():
    """Source i's kernels all delta taps at delay j_i: its conv streams are
    the source delayed by j_i rows (zero before the sequence).  With stream
    queries that see only stream 1 and a zero mixer, the read of stream 1 is
    the Full read of the delayed sources, which the output is twice of."""
    rng = np.random.default_rng(82)
    N, T, d, ks = 3, 12, 8, (4, 4, 4)
    src = _rand(rng, N, T, d)
    delays = (0, 2, 3)
    cw = np.zeros((N, d * sum(ks)))
    for i, j in enumerate(delays):
        for r in range(3):
            k = np.zeros((d, 4))
            k[:, j] = 1.0
            cw[i, d * 4 * r: d * 4 * (r + 1)] = k.ravel()
    w = _rand(rng, d, scale=2.0)
    q = np.stack([w] * 4)
    out = oracle.msar_ps(src, ks, cw, q, None, 1e-6, None, np.zeros((4 * d, 4)), 1e-6)
    delayed = np.zeros_like(src)
    for i, j in enumerate(delays):
        delayed[i, j:] = src[i, :T - j]
    # streams 1..3 each read the delayed sources; stream 0 reads the sources
    ref = 0.5 * oracle.full(src, w, None, eps=1e-6) + 1.5 * oracle.full(delayed, w, None, eps=1e-6)
    assert np.allclose(out, ref, atol=1e-12)


def test_msar_per_source_permutation_equivariant():
    """Permuting the sources together with their kernels leaves the read
    unchanged (each stream's softmax is over a set of sources)."""
    rng = np.random.default_rng(83)
    N, T, d, ks = 5, 14, 8, (4, 8, 12)
    src, q = _rand(rng, N, T, d), _rand(rng, 4, d, scale=2.0)
    cw, P = _rand(rng, N, d * sum(ks), scale=0.4), _rand(rng, 4 * d, 4, scale=0.2)
    perm = np.array([3, 0, 4, 1, 2])
    a = oracle.msar_ps(src, ks, cw, q, None, 1e-6, None, P, 1e-6)
    b = oracle.msar_ps(src[perm], ks, cw[perm], q, None, 1e-6, None, P, 1e-6)
    assert np.allclose(a, b, atol=1e-12, rtol=0)
    c = oracle.msar_ps(src[perm], ks, cw, q, None, 1e-6, None, P, 1e-6)
    assert np.abs(a - c).max() > 1e-3        # kernels must travel with their sources


@pytest.mark.parametrize("N,T,d,ks,eps", [(3, 7, 4, (2, 3, 4), 1e-6), (2, 5, 6, (1, 4, 2), 0.05)])
def test_msar_bwd_matches_finite_differences(N, T, d, ks, eps):
    """Every gradient of the MSAR read (sources, conv kernels, stream
    queries, gain, mixer gain, mixer projection) against central differences
    of the (pinned) MSAR forward oracle."""
    rng = np.random.default_rng(91 + N + T)
    src = _rand(rng, N, T, d) * (1 + 0.5 * np.arange(N))[:, None, None]
    cw = _rand(rng, d * sum(ks), scale=0.6)
    q = _rand(rng, 4, d, scale=1.5)
    g = rng.uniform(0.5, 1.5, d)
    mg = rng.uniform(0.5, 1.5, 4 * d)
    P = _rand(rng, 4 * d, 4, scale=0.5)
    dh = _rand(rng, T, d)

    def loss(s_, cw_, q_, g_, mg_, P_):
        return float((oracle.msar(s_, ks, cw_, q_, g_, eps, mg_, P_, 1e-6) * dh).sum())
    got = oracle.msar_bwd(src, ks, cw, q, dh, g, eps, mg, P, 1e-6)
    ref = _fd(loss, (src, cw, q, g, mg, P))
    for name, x, y in zip(("dsrc", "dconv_w", "dq", "dgain", "dmix_gain", "dmix_w"), got, ref):
        assert np.abs(x - y).max() <= 2e-6 * max(1.0, np.abs(y).max()), name


def test_msar_bwd_identity_stream_only_is_read_backward():
    """Zero conv kernels make streams 1..3 zero (their reads give zero and
    send nothing back); with a zero mixer projection c_r = 1/2 and the mixer
    passes dh/2 to each stream's read minus its RMSNorm term, which a zero
    projection also zeroes (dzn = 0): stream 0's read then gets dh / 2, so the
    sources' gradient is the read backward of dh / 2."""
    rng = np.random.default_rng(92)
    N, T, d, ks = 3, 6, 8, (4, 8, 12)
    src, q, dh = _rand(rng, N, T, d), _rand(rng, 4, d, scale=1.5), _rand(rng, T, d)
    got = oracle.msar_bwd(src, ks, np.zeros(d * sum(ks)), q, dh, None, 1e-6, None, np.zeros((4 * d, 4)), 1e-6)
    ref = oracle.read_bwd(src, q[:1], 0.5 * dh[None], None, 1e-6)
    assert np.allclose(got[0], ref[0], atol=1e-12) and np.allclose(got[2][0], ref[1][0], atol=1e-12)


@pytest.mark.parametrize("N,T,d,ks", [(3, 7, 4, (2, 3, 4)), (2, 6, 4, (1, 4, 2))])
def test_msar_ps_bwd_matches_finite_differences(N, T, d, ks):
    """Every gradient of the MSAR read with per-source kernels, each source's
    kernel gradient on its own, against central differences of the (pinned)
    per-source forward oracle."""
    rng = np.random.default_rng(95 + N + T)
    src = _rand(rng, N, T, d) * (1 + 0.5 * np.arange(N))[:, None, None]
    cw = _rand(rng, N, d * sum(ks), scale=0.6)
    q = _rand(rng, 4, d, scale=1.5)
    g = rng.uniform(0.5, 1.5, d)
    mg = rng.uniform(0.5, 1.5, 4 * d)
    P = _rand(rng, 4 * d, 4, scale=0.5)
    dh = _rand(rng, T, d)

    def loss(s_, cw_, q_, g_, mg_, P_):
        return float((oracle.msar_ps(s_, ks, cw_, q_, g_, 1e-6, mg_, P_, 1e-6) * dh).sum())
    got = oracle.msar_ps_bwd(src, ks, cw, q, dh, g, 1e-6, mg, P, 1e-6)
    ref = _fd(loss, (src, cw, q, g, mg, P))
    for name, x, y in zip(("dsrc", "dconv_w", "dq", "dgain", "dmix_gain", "dmix_w"), got, ref):
        assert np.abs(x - y).max() <= 2e-6 * max(1.0, np.abs(y).max()), name


def test_msar_ps_bwd_equal_kernels_is_the_shared_backward():
    """Per-source kernels that are all equal: every gradient but the kernels'
    is the shared-kernel backward's, and the sources' kernel gradients add up
    to the shared kernel's (the shared kernel is used by every source)."""
    rng = np.random.default_rng(96)
    N, T, d, ks = 4, 9, 6, (4, 8, 12)
    src, q, dh = _rand(rng, N, T, d), _rand(rng, 4, d, scale=1.5), _rand(rng, T, d)
    cw, P = _rand(rng, d * sum(ks), scale=0.4), _rand(rng, 4 * d, 4, scale=0.3)
    shared = oracle.msar_bwd(src, ks, cw, q, dh, None, 1e-6, None, P, 1e-6)
    per = oracle.msar_ps_bwd(src, ks, np.stack([cw] * N), q, dh, None, 1e-6, None, P, 1e-6)
    for k in (0, 2, 3, 4, 5):
        assert np.allclose(per[k], shared[k], atol=1e-12, rtol=0), k
    assert np.allclose(per[1].sum(axis=0), shared[1], atol=1e-12, rtol=0)


@pytest.mark.parametrize("with_partial,ks", [(True, (2, 3, 4)), (False, (1, 4, 2)), (True, (1, 2, 3))])
def test_msar_phase2_bwd_matches_finite_differences(with_partial, ks):
    """Every gradient of MSAR phase 2 (the state o and lse, the partial, conv
    kernels, stream queries, gain, mixer gain and projection) against central
    differences of the (pinned) phase-2 forward oracle."""
    rng = np.random.default_rng(201 + with_partial + sum(ks))
    T, d = 6, 4
    o = _rand(rng, 4, T, d)
    lse = _rand(rng, 4, T, scale=0.7)
    p = _rand(rng, T, d, scale=1.3) if with_partial else None
    cw = _rand(rng, d * sum(ks), scale=0.6)
    q = _rand(rng, 4, d, scale=1.5)
    g = rng.uniform(0.5, 1.5, d)
    mg = rng.uniform(0.5, 1.5, 4 * d)
    P = _rand(rng, 4 * d, 4, scale=0.5)
    dh = _rand(rng, T, d)

    def loss(o_, l_, p_, cw_, q_, g_, mg_, P_):
        return float((oracle.msar_phase2(o_, l_, p_, ks, cw_, q_, g_, 1e-6, mg_, P_, 1e-6) * dh).sum())
    got = oracle.msar_phase2_bwd(o, lse, p, ks, cw, q, dh, g, 1e-6, mg, P, 1e-6)
    ref = _fd(loss, (o, lse, p, cw, q, g, mg, P))
    for name, x, y in zip(("d_o", "d_lse", "d_partial", "dconv_w", "dquery", "dgain", "dmix_gain", "dmix_w"),
                          got, ref):
        if y is None:
            assert x is None, name
            continue
        assert np.abs(x - y).max() <= 2e-6 * max(1.0, np.abs(y).max()), name


def test_msar_phase1_bwd_matches_finite_differences():
    """Every gradient of MSAR phase 1 (sources, conv kernels, every layer's
    stream queries, gain) for gradients of both its outputs, o and lse,
    against central differences of the (pinned) phase-1 forward oracle."""
    rng = np.random.default_rng(207)
    N, S, T, d, ks = 3, 2, 6, 4, (2, 3, 4)
    src = _rand(rng, N, T, d) * (1 + 0.5 * np.arange(N))[:, None, None]
    cw = _rand(rng, d * sum(ks), scale=0.6)
    q = _rand(rng, S, 4, d, scale=1.5)
    g = rng.uniform(0.5, 1.5, d)
    d_o = _rand(rng, S, 4, T, d)
    d_lse = _rand(rng, S, 4, T)

    def loss(s_, cw_, q_, g_):
        o, lse = oracle.msar_phase1(s_, ks, cw_, q_, g_, 1e-6)
        return float((o * d_o).sum() + (lse * d_lse).sum())
    got = oracle.msar_phase1_bwd(src, ks, cw, q, d_o, d_lse, g, 1e-6)
    ref = _fd(loss, (src, cw, q, g))
    for name, x, y in zip(("dsrc", "dconv_w", "dqueries", "dgain"), got, ref):
        assert np.abs(x - y).max() <= 2e-6 * max(1.0, np.abs(y).max()), name


@pytest.mark.parametrize("with_partial", [True, False])
def test_msar_two_phase_bwd_equals_one_shot_bwd(with_partial):
    """Phase 2's backward followed by phase 1's equals the backward of the
    one-shot MSAR read of [cached sources, partial] (first layer: the cached
    sources alone): the cached sources' and the partial's gradients, and the
    kernels', queries', gain's and mixer's as the sums of the two phases'."""
    rng = np.random.default_rng(211 + with_partial)
    N, T, d, ks = 3, 7, 6, (4, 8, 12)
    cached = _rand(rng, N, T, d) * (1 + 0.5 * np.arange(N))[:, None, None]
    p = _rand(rng, T, d, scale=1.2)
    cw = _rand(rng, d * sum(ks), scale=0.4)
    q = _rand(rng, 4, d, scale=1.5)
    g = rng.uniform(0.5, 1.5, d)
    mg = rng.uniform(0.5, 1.5, 4 * d)
    P = _rand(rng, 4 * d, 4, scale=0.4)
    dh = _rand(rng, T, d)
    o, lse = oracle.msar_phase1(cached, ks, cw, q[None], g, 1e-6)
    d_o, d_lse, d_p, dcw2, dq2, dg2, dmg, dmw = oracle.msar_phase2_bwd(o[0], lse[0], p if with_partial else None, ks,
                                                                        cw, q, dh, g, 1e-6, mg, P, 1e-6)
    dsrc, dcw1, dq1, dg1 = oracle.msar_phase1_bwd(cached, ks, cw, q[None], d_o[None], d_lse[None], g, 1e-6)
    srcs = np.concatenate([cached, p[None]]) if with_partial else cached
    r_src, r_cw, r_q, r_g, r_mg, r_mw = oracle.msar_bwd(srcs, ks, cw, q, dh, g, 1e-6, mg, P, 1e-6)
    tol = dict(atol=1e-10, rtol=0)
    assert np.allclose(dsrc, r_src[:N], **tol)
    if with_partial:
        assert np.allclose(d_p, r_src[N], **tol)
    else:
        assert d_p is None and np.count_nonzero(d_lse) == 0 and np.count_nonzero(dcw2) == 0
    assert np.allclose(dcw1 + dcw2, r_cw, **tol)
    assert np.allclose(dq1[0] + dq2, r_q, **tol)
    assert np.allclose(dg1 + dg2, r_g, **tol)
    assert np.allclose(dmg, r_mg, **tol) and np.allclose(dmw, r_mw, **tol)


def _msar_block_inputs(rng, N, S, T, d, ks=(4, 8, 12)):
    cached = _rand(rng, N, T, d) * (1 + 0.5 * np.arange(N))[:, None, None]
    parts = _rand(rng, S, T, d)
    q = _rand(rng, S, 4, d, scale=2.0)
    cw = _rand(rng, d * sum(ks), scale=0.4)
    P = _rand(rng, 4 * d, 4, scale=0.2)
    g = rng.uniform(0.5, 1.5, d)
    mg = rng.uniform(0.5, 1.5, 4 * d)
    return cached, parts, q, cw, P, g, mg


@pytest.mark.parametrize("N,S,eps", [(5, 3, 1e-6), (1, 2, 0.1), (3, 1, 0.0)])
def test_msar_two_phase_equals_one_shot(N, S, eps):
    """[MSAR §어떻게 쓰나]: two-phase MSAR (phase 1 over the cached sources for
    every layer of the block, then each layer's partial merged per stream)
    equals the one-shot MSAR read of [b_0..b_{N-1}, p_s] with that layer's
    queries; the block's first layer (no partial) equals the read of the
    cached sources alone."""
    rng = np.random.default_rng(61 + N + S)
    T, d = 14, 8
    ks = (4, 8, 12)
    cached, parts, q, cw, P, g, mg = _msar_block_inputs(rng, N, S, T, d, ks)
    o, lse = oracle.msar_phase1(cached, ks, cw, q, g, eps)
    for s_ in range(S):
        got = oracle.msar_phase2(o[s_], lse[s_], parts[s_], ks, cw, q[s_], g, eps, mg, P, 1e-6)
        ref = oracle.msar(np.concatenate([cached, parts[s_][None]]), ks, cw, q[s_], g, eps, mg, P, 1e-6)
        assert np.abs(got - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max()), s_
        first = oracle.msar_phase2(o[s_], lse[s_], None, ks, cw, q[s_], g, eps, mg, P, 1e-6)
        ref0 = oracle.msar(cached, ks, cw, q[s_], g, eps, mg, P, 1e-6)
        assert np.abs(first - ref0).max() <= 1e-12 * max(1.0, np.abs(ref0).max()), s_


def test_msar_phase1_single_source_state():
    """One cached source: every stream's weight is 1, so o_s^(r) is the
    stream itself (the source, or its causal conv, pinned against
    np.convolve) and lse_s^(r) is that stream's score."""
    rng = np.random.default_rng(62)
    T, d, ks = 9, 8, (2, 3, 5)
    src = _rand(rng, 1, T, d)
    q = _rand(rng, 2, 4, d, scale=2.0)
    cw = _rand(rng, d * sum(ks), scale=0.5)
    o, lse = oracle.msar_phase1(src, ks, cw, q, None, 0.0)
    streams = [src[0]]
    off = 0
    for k in ks:
        streams.append(oracle.msar_conv(src[0], cw[off:off + d * k].reshape(d, k)))
        off += d * k
    for s_ in range(2):
        for r in range(4):
            u = streams[r]
            assert np.allclose(o[s_, r], u, atol=1e-14)
            rms = np.sqrt(np.mean(u * u, axis=1))
            assert np.allclose(lse[s_, r], (u @ q[s_, r]) / rms, atol=1e-12)


def test_msar_phase2_is_causal_in_the_partial():
    """The partial's streams are causal convolutions of the partial: changing
    p at t' > t leaves out[t] unchanged, and at t - 11 <= t' <= t changes it."""
    rng = np.random.default_rng(63)
    N, S, T, d = 3, 1, 30, 8
    cached, parts, q, cw, P, g, mg = _msar_block_inputs(rng, N, S, T, d)
    o, lse = oracle.msar_phase1(cached, (4, 8, 12), cw, q, g, 1e-6)
    base = oracle.msar_phase2(o[0], lse[0], parts[0], (4, 8, 12), cw, q[0], g, 1e-6, mg, P, 1e-6)
    t = 20
    for tp, should_change in ((t + 1, False), (t - 12, False), (t - 11, True), (t, True)):
        p2 = parts[0].copy()
        p2[tp] += 3.0
        h = oracle.msar_phase2(o[0], lse[0], p2, (4, 8, 12), cw, q[0], g, 1e-6, mg, P, 1e-6)
        assert (np.abs(h[t] - base[t]).max() > 0) == should_change, tp


# --------------------------------------------------------------------------
# brute force: C oracle vs the NumPy twin on tiny shapes
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(4))
def test_brute_force_against_numpy_twin(seed):
    rng = np.random.default_rng(100 + seed)
    n_src, T, d = rng.integers(1, 5), rng.integers(1, 5), int(rng.choice([4, 8, 16]))
    src = _rand(rng, n_src, T, d, scale=2.0)
    w = _rand(rng, d, scale=2.0)
    g = rng.uniform(0.5, 1.5, d)
    assert np.allclose(oracle.full(src, w, g, 1e-3), numpy_twin.full(src, w, g, 1e-3),
                       atol=1e-12, rtol=0)
    N, S = rng.integers(1, 4), rng.integers(1, 4)
    cache = _rand(rng, N, T, d)
    partials = _rand(rng, S, T, d)
    q = _rand(rng, S, d, scale=2.0)
    assert np.allclose(oracle.block_oneshot(cache, partials, q, g, 1e-6),
                       numpy_twin.block_oneshot(cache, partials, q, g, 1e-6), atol=1e-12, rtol=0)
    H = int(rng.choice([1, 2, 4]))
    qh = _rand(rng, 2, H, d // H, scale=2.0)
    assert np.allclose(oracle.mhar(src, qh, g, 1e-6), numpy_twin.mhar(src, qh, g, 1e-6),
                       atol=1e-12, rtol=0)
    ks = (2, 3, 5)
    cw = _rand(rng, d * sum(ks), scale=0.5)
    qm = _rand(rng, 4, d, scale=2.0)
    P = _rand(rng, 4 * d, 4, scale=0.3)
    mg = rng.uniform(0.5, 1.5, 4 * d)
    a = oracle.msar(src, ks, cw, qm, g, 1e-6, mg, P, 1e-5)
    b = numpy_twin.msar(src, ks, cw, qm, g, 1e-6, mg, P, 1e-5)
    assert np.allclose(a, b, atol=1e-12, rtol=0)
