"""GPU parity: every entry point of the C ABI against the CPU oracle on the
same seeded inputs, at sizes the oracle finishes in seconds that still span
several tiles (and clusters) plus a ragged tail, and on the edge cases of the
method.  Tolerances are defined in _helpers.py."""
import math

import numpy as np
import pytest
import torch

from _helpers import check_lse, check_out, to_dev, to_host
from depth_wise_attention_gb300 import attnres, inputs
from oracle import oracle

pytestmark = pytest.mark.gpu

BF16, F32 = torch.bfloat16, torch.float32


def _rng(seed):
    return np.random.default_rng(seed)


def _sources(rng, n_src, T, d, dtype, step=0.5):
    src = np.stack([rng.standard_normal((T, d)).astype(np.float32) * (1 + i * step)
                    for i in range(n_src)])
    return inputs.bf16_round(src) if dtype == BF16 else src


def _queries(rng, n, d, std=None):
    std = math.sqrt(16.0 / d) if std is None else std
    return (rng.standard_normal((n, d)) * std).astype(np.float32)


# --------------------------------------------------------------- worked example

@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("T", [1, 3, 13])
def test_worked_example_padded(dtype, T):
    """Tutorial Figs. 2-3, padded to d=8: alpha=[1/4,1/2,1/4], h=[0.5,2,1.5,0..]."""
    src = np.zeros((3, T, 8), np.float32)
    src[0, :, 0], src[1, :, 1], src[2, :, 2] = 2.0, 4.0, 6.0
    w = np.zeros(8, np.float32)
    w[1] = math.log(2.0) / math.sqrt(8.0)
    out = attnres.attnres_full_fwd(to_dev(src, dtype), to_dev(w, F32), None, 0.0)
    want = np.zeros((T, 8))
    want[:, :3] = [0.5, 2.0, 1.5]
    assert np.abs(to_host(out) - want).max() <= (1e-6 if dtype == F32 else 0.0)


# --------------------------------------------------------------- Full

@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("n_src,T,d", [(1, 5, 256), (3, 37, 256), (8, 300, 256), (8, 77, 2048),
                                       (5, 41, 4096), (8, 19, 8), (2, 9, 24), (7, 33, 1000)])
def test_full_fwd(dtype, n_src, T, d):
    rng = _rng(n_src * 1000 + T + d)
    src = _sources(rng, n_src, T, d, dtype, step=0.25)
    w = _queries(rng, 1, d)[0]
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    out = attnres.attnres_full_fwd(to_dev(src, dtype), to_dev(w, F32), to_dev(g, F32), 1e-6)
    ref = oracle.full(src, w, g, 1e-6)
    check_out(out, ref, dtype, np.abs(src).max())


@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("n_src,T,d", [(9, 21, 4096), (13, 40, 2048), (64, 7, 4096), (17, 70, 256),
                                       (30, 11, 512)])
def test_full_fwd_many_sources_online_merge(dtype, n_src, T, d):
    """More sources than one stage holds: chunks merged by the online softmax."""
    rng = _rng(n_src * 7 + T + d)
    src = _sources(rng, n_src, T, d, dtype, step=1 / 16)
    w = _queries(rng, 1, d)[0]
    out = attnres.attnres_full_fwd(to_dev(src, dtype), to_dev(w, F32), None, 1e-6)
    check_out(out, oracle.full(src, w, None, 1e-6), dtype, np.abs(src).max())


def test_full_fwd_zero_query_is_mean():
    rng = _rng(3)
    src = _sources(rng, 6, 50, 512, F32)
    out = attnres.attnres_full_fwd(to_dev(src, F32), to_dev(np.zeros(512, np.float32), F32))
    check_out(out, src.mean(axis=0), F32, np.abs(src).max())


def test_full_fwd_zero_source_with_zero_eps():
    src = np.zeros((2, 4, 64), np.float32)
    src[1, :, 3] = 5.0
    w = np.zeros(64, np.float32)
    w[3] = 1.0
    out = attnres.attnres_full_fwd(to_dev(src, F32), to_dev(w, F32), None, 0.0)
    check_out(out, oracle.full(src, w, None, 0.0), F32, 5.0)


def test_full_fwd_source_stride():
    """Sources that are not packed back to back (src_stride > T*d)."""
    rng = _rng(4)
    n_src, T, d, stride = 6, 33, 512, 33 * 512 + 8 * 100
    buf = torch.zeros((n_src, stride), dtype=BF16, device="cuda")
    src = _sources(rng, n_src, T, d, BF16)
    buf[:, : T * d] = to_dev(src.reshape(n_src, -1), BF16)
    view = buf[:, : T * d].view(n_src, T, d)
    assert view.stride(0) == stride
    w = _queries(rng, 1, d)[0]
    out = attnres.attnres_full_fwd(view, to_dev(w, F32))
    check_out(out, oracle.full(src, w, None, 1e-6), BF16)


@pytest.mark.parametrize("n_src,T,d,with_gain", [
    (1, 300, 4096, True), (3, 65, 2048, False), (8, 2000, 4096, True), (9, 300, 4096, False),
    (16, 157, 2048, True), (17, 300, 4096, True), (24, 70, 4096, False), (40, 1000, 2048, True),
    (64, 160, 4096, True), (63, 153, 4096, False)])
def test_one_query_read(n_src, T, d, with_gain):
    """One query (Full AttnRes, or Block phase 1 with one query for the lse)
    over 1-64 sources at d = 2048 and 4096: one chunk, full and partial last
    chunks, several tokens per CTA and fewer tokens than SMs; Full's output
    equals phase 1's bit for bit."""
    rng = _rng(n_src * 29 + T + d)
    src = _sources(rng, n_src, T, d, BF16, step=1 / 16)
    q = _queries(rng, 1, d)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32) if with_gain else None
    o, lse = attnres.attnres_block_phase1(to_dev(src, BF16), to_dev(q, F32), to_dev(g, F32) if with_gain else None,
                                          1e-6)
    ro, rl = oracle.block_phase1(src, q, g, 1e-6)
    check_out(o, ro, BF16, np.abs(src).max(), what="o")
    check_lse(lse, rl)
    out = attnres.attnres_full_fwd(to_dev(src, BF16), to_dev(q[0], F32), to_dev(g, F32) if with_gain else None, 1e-6)
    assert torch.equal(out, o[0] if o.dim() == 3 else o)


def test_one_query_read_source_stride_and_determinism():
    """One query over 12 sources at d = 2048 that are not packed back to back,
    run twice (bitwise equal), against the oracle."""
    rng = _rng(5)
    n_src, T, d = 12, 333, 2048
    stride = T * d + 8 * 37
    buf = torch.zeros((n_src, stride), dtype=BF16, device="cuda")
    src = _sources(rng, n_src, T, d, BF16, step=1 / 16)
    buf[:, : T * d] = to_dev(src.reshape(n_src, -1), BF16)
    view = buf[:, : T * d].view(n_src, T, d)
    w = _queries(rng, 1, d)[0]
    a = attnres.attnres_full_fwd(view, to_dev(w, F32))
    b = attnres.attnres_full_fwd(view, to_dev(w, F32))
    assert torch.equal(a, b)
    check_out(a, oracle.full(src, w, None, 1e-6), BF16, np.abs(src).max())


# --------------------------------------------------------------- phase 1 / phase 2

@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("n_q", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("T,d", [(70, 2048), (23, 4096)])
def test_block_phase1(dtype, n_q, T, d):
    nq_pad = 1 << (n_q - 1).bit_length()
    if nq_pad * d > 16384:
        pytest.skip("register budget: n_q (rounded up to a power of two) * d <= 16384")
    rng = _rng(n_q * 100 + T)
    src = _sources(rng, 8, T, d, dtype)
    q = _queries(rng, n_q, d)
    o, lse = attnres.attnres_block_phase1(to_dev(src, dtype), to_dev(q, F32), None, 1e-6)
    ro, rl = oracle.block_phase1(src, q, None, 1e-6)
    check_out(o, ro, dtype, np.abs(src).max(), what="o")
    check_lse(lse, rl)


@pytest.mark.parametrize("n_src", [1, 2, 8, 10, 20])
def test_block_phase1_source_counts(n_src):
    rng = _rng(n_src)
    T, d = 45, 2048
    src = _sources(rng, n_src, T, d, BF16)
    q = _queries(rng, 4, d)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    o, lse = attnres.attnres_block_phase1(to_dev(src, BF16), to_dev(q, F32), to_dev(g, F32), 1e-6)
    ro, rl = oracle.block_phase1(src, q, g, 1e-6)
    check_out(o, ro, BF16, what="o")
    check_lse(lse, rl)


@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("T,d", [(1, 64), (99, 2048), (64, 4096), (10, 808)])
def test_block_phase2_merge(dtype, T, d):
    rng = _rng(T + d)
    o = _sources(rng, 1, T, d, dtype)[0]
    p = _sources(rng, 1, T, d, dtype)[0]
    lse = (rng.standard_normal(T) * 4).astype(np.float32)
    q = _queries(rng, 1, d)[0]
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    out = attnres.attnres_block_phase2_merge(to_dev(o, dtype), to_dev(lse, F32), to_dev(p, dtype),
                                             to_dev(q, F32), to_dev(g, F32), 1e-6)
    ref = oracle.block_phase2(o, lse, p, q, g, 1e-6)
    check_out(out, ref, dtype, max(np.abs(o).max(), np.abs(p).max()))


def test_block_phase2_in_place_and_without_partial():
    rng = _rng(11)
    T, d = 50, 1024
    o = _sources(rng, 1, T, d, BF16)[0]
    p = _sources(rng, 1, T, d, BF16)[0]
    lse = (rng.standard_normal(T) * 4).astype(np.float32)
    q = _queries(rng, 1, d)[0]
    od = to_dev(o, BF16)
    attnres.attnres_block_phase2_merge(od, to_dev(lse, F32), to_dev(p, BF16), to_dev(q, F32), out=od)
    check_out(od, oracle.block_phase2(o, lse, p, q), BF16)
    od = to_dev(o, BF16)
    out = attnres.attnres_block_phase2_merge(od, to_dev(lse, F32), None, to_dev(q, F32))
    assert torch.equal(out, od)


@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("T,d", [(1, 64), (99, 2048), (64, 4096), (10, 808), (700, 256)])
@pytest.mark.parametrize("with_old", [True, False])
def test_block_phase2_update_merge(dtype, T, d, with_old):
    """The fused partial-sum update and merge: p' = p + f (rounded to the
    storage type) and the next layer's merge of p'."""
    rng = _rng(T + d + with_old)
    o = _sources(rng, 1, T, d, dtype)[0]
    p = _sources(rng, 1, T, d, dtype)[0] if with_old else None
    f = _sources(rng, 1, T, d, dtype, step=0)[0]
    lse = (rng.standard_normal(T) * 4).astype(np.float32)
    q = _queries(rng, 1, d)[0]
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    pd = to_dev(p, dtype) if with_old else None
    p_new, out = attnres.attnres_block_phase2_update_merge(pd, to_dev(f, dtype), to_dev(o, dtype),
                                                           to_dev(lse, F32), to_dev(q, F32), to_dev(g, F32),
                                                           1e-6)
    ref_p, ref = oracle.block_phase2_update(p, f, o, lse, q, g, 1e-6)
    check_out(p_new, ref_p, dtype, np.abs(ref_p).max(), what="partial")
    check_out(out, ref, dtype, max(np.abs(o).max(), np.abs(ref_p).max()))


def test_block_phase2_update_merge_in_place():
    rng = _rng(31)
    T, d = 300, 4096
    o = _sources(rng, 1, T, d, BF16)[0]
    p = _sources(rng, 1, T, d, BF16)[0]
    f = _sources(rng, 1, T, d, BF16)[0]
    lse = (rng.standard_normal(T) * 4).astype(np.float32)
    q = _queries(rng, 1, d)[0]
    ref_p, ref = oracle.block_phase2_update(p, f, o, lse, q)
    for target in ("partial", "f"):
        od, pd, fd = to_dev(o, BF16), to_dev(p, BF16), to_dev(f, BF16)
        po = pd if target == "partial" else fd
        attnres.attnres_block_phase2_update_merge(pd, fd, od, to_dev(lse, F32), to_dev(q, F32),
                                                  partial_out=po, out=od)
        check_out(po, ref_p, BF16, what="partial")
        check_out(od, ref, BF16)


@pytest.mark.parametrize("T,d,N,S", [(150, 2048, 8, 4), (40, 4096, 8, 4), (33, 512, 3, 6)])
def test_block_chain_with_fused_updates_matches_oneshot(T, d, N, S):
    """A whole block on the GPU: phase 1, then each layer i >= 2 updates the
    partial with the previous layer's output and merges it in one call; every
    layer's input equals the one-shot Block read with the cumulative partials,
    and the last partial is the block's sum of outputs."""
    rng = _rng(T * 3 + d + N + S)
    cache = _sources(rng, N, T, d, BF16)
    f = _sources(rng, S, T, d, BF16, step=0)
    q = _queries(rng, S, d)
    qd = to_dev(q, F32)
    o, lse = attnres.attnres_block_phase1(to_dev(cache, BF16), qd)
    fd = to_dev(f, BF16)
    p = None
    p_stored = np.zeros((T, d))                   # the partial as stored (bf16)
    outs = [to_host(o[0])]
    partials = np.zeros((S, T, d))
    for i in range(1, S):
        p, out = attnres.attnres_block_phase2_update_merge(p, fd[i - 1], o[i], lse[i], qd[i])
        # layer i merges the stored partial plus f_{i-1}, summed exactly; the
        # stored partial is that sum rounded to bf16
        partials[i] = p_stored + f[i - 1]
        p_stored = inputs.bf16_round(partials[i].astype(np.float32)).astype(np.float64)
        outs.append(to_host(out))
    ref = oracle.block_oneshot(cache, partials, q, None, 1e-6)
    for i in range(S):
        check_out(outs[i], ref[i], BF16, what=f"layer {i + 1}")
    check_out(p, p_stored, BF16, what="partial")


@pytest.mark.parametrize("T,d,N,S", [(150, 2048, 8, 4), (40, 4096, 8, 4), (33, 512, 3, 6)])
def test_two_phase_block_matches_oneshot(T, d, N, S):
    """GPU two-phase schedule (phase 1 + S-1 merges) vs the oracle's
    layer-by-layer one-shot Block read."""
    x = inputs.block_inputs(N, S, T, d, seed=T)
    cache, q, parts = x["cache"], x["queries"], x["partials"]
    cd, qd, pd = to_dev(cache, BF16), to_dev(q, F32), to_dev(parts, BF16)
    o, lse = attnres.attnres_block_phase1(cd, qd)
    outs = [o[0]]
    for i in range(1, S):
        outs.append(attnres.attnres_block_phase2_merge(o[i], lse[i], pd[i], qd[i]))
    gpu = torch.stack(outs)
    ref = oracle.block_oneshot(cache, parts, q)
    check_out(gpu, ref, BF16)


# --------------------------------------------------------------- MHAR

@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("H,d,T", [(2, 2048, 31), (4, 2048, 70), (8, 2048, 9), (8, 4096, 37),
                                   (16, 4096, 12), (4, 1024, 20)])
def test_mhar(dtype, H, d, T):
    if dtype == F32 and d // H % 128:
        pytest.skip("f32 heads need a multiple of 128 channels")
    if dtype == BF16 and d // H % 256:
        pytest.skip("bf16 heads need a multiple of 256 channels")
    rng = _rng(H * 10 + T)
    src = _sources(rng, 8, T, d, dtype)
    q = (rng.standard_normal((4, H, d // H)) * math.sqrt(16.0 / (d // H))).astype(np.float32)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    out, lse = attnres.mhar_fwd(to_dev(src, dtype), to_dev(q, F32), to_dev(g, F32), 1e-6,
                                want_lse=True)
    ro, rl = oracle.mhar(src, q, g, 1e-6, want_lse=True)
    check_out(out, ro, dtype, np.abs(src).max())
    check_lse(lse, rl)


def test_mhar_many_sources():
    rng = _rng(12)
    T, d, H = 30, 2048, 8
    src = _sources(rng, 11, T, d, BF16, step=0.2)
    q = (rng.standard_normal((4, H, d // H)) * math.sqrt(16.0 / (d // H))).astype(np.float32)
    out = attnres.mhar_fwd(to_dev(src, BF16), to_dev(q, F32))
    check_out(out, oracle.mhar(src, q), BF16)


@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("H,d,T", [(8, 4096, 40), (16, 2048, 33), (4, 1024, 70), (2, 512, 9), (8, 512, 21),
                                   (1, 2048, 17)])
def test_mhar_phase2_merge(dtype, H, d, T):
    """MHAR phase 2: per-head merge of the partial into the per-head phase-1
    state (heads of whole warps, of a power-of-two group inside a warp, H = 1)."""
    rng = _rng(H * 7 + d + T)
    o = _sources(rng, 1, T, d, dtype)[0]
    p = _sources(rng, 1, T, d, dtype)[0]
    lse = (rng.standard_normal((H, T)) * 4).astype(np.float32)
    q = (rng.standard_normal((H, d // H)) * math.sqrt(16.0 / (d // H))).astype(np.float32)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    out = attnres.mhar_phase2_merge(to_dev(o, dtype), to_dev(lse, F32), to_dev(p, dtype), to_dev(q, F32),
                                    to_dev(g, F32), 1e-6)
    check_out(out, oracle.mhar_phase2(o, lse, p, q, g, 1e-6), dtype, max(np.abs(o).max(), np.abs(p).max()))


def test_mhar_two_phase_matches_oneshot_and_fused_update():
    """MHAR inside the two-phase schedule on the GPU: mhar_fwd over the cached
    reps (phase 1, lse per head), then the per-head merge of a partial equals the
    one-shot MHAR read over the reps plus the partial; with f the partial is
    updated first."""
    rng = _rng(41)
    H, d, T, N = 8, 4096, 90, 8
    cache = _sources(rng, N, T, d, BF16)
    p = _sources(rng, 1, T, d, BF16)[0]
    f = _sources(rng, 1, T, d, BF16, step=0)[0]
    q = (rng.standard_normal((1, H, d // H)) * math.sqrt(16.0 / (d // H))).astype(np.float32)
    qd = to_dev(q, F32)
    o, lse = attnres.mhar_fwd(to_dev(cache, BF16), qd, want_lse=True)
    out = attnres.mhar_phase2_merge(o[0], lse[0], to_dev(p, BF16), qd[0])
    check_out(out, oracle.mhar(np.concatenate([cache, p[None]]), q)[0], BF16)
    p_new, out2 = attnres.mhar_phase2_merge(o[0], lse[0], to_dev(p, BF16), qd[0], f=to_dev(f, BF16))
    pf = p.astype(np.float64) + f
    check_out(p_new, pf, BF16, what="partial")
    check_out(out2, oracle.mhar(np.concatenate([cache, pf[None]]), q)[0], BF16)


def test_mhar_phase2_one_head_equals_block_phase2_bitwise():
    rng = _rng(42)
    T, d = 77, 4096
    o = to_dev(_sources(rng, 1, T, d, BF16)[0], BF16)
    p = to_dev(_sources(rng, 1, T, d, BF16)[0], BF16)
    lse = to_dev((rng.standard_normal(T) * 4).astype(np.float32), F32)
    q = to_dev(_queries(rng, 1, d)[0], F32)
    a = attnres.attnres_block_phase2_merge(o, lse, p, q)
    b = attnres.mhar_phase2_merge(o, lse.view(1, T), p, q.view(1, d))
    assert torch.equal(a, b)


def test_mhar_one_head_is_phase1_bitwise():
    rng = _rng(13)
    T, d = 57, 4096
    src = to_dev(_sources(rng, 8, T, d, BF16), BF16)
    q = to_dev(_queries(rng, 4, d), F32)
    o, lse = attnres.attnres_block_phase1(src, q)
    m, ml = attnres.mhar_fwd(src, q.view(4, 1, d), want_lse=True)
    assert torch.equal(o, m)
    assert torch.equal(lse, ml.view(4, T))


def _msar_setup(rng, n_src, T, d, ks, dtype):
    src = _sources(rng, n_src, T, d, dtype)
    m = 4
    q = _queries(rng, m, d)
    cw = np.concatenate([(rng.standard_normal((d, k)) / math.sqrt(k)).astype(np.float32).ravel() for k in ks])
    mw = (rng.standard_normal((m * d, m)) / math.sqrt(m * d)).astype(np.float32)
    return src, q, cw, mw


@pytest.mark.parametrize("t_prev,T,d,dtype", [(11, 40, 2048, BF16), (3, 17, 512, F32), (0, 25, 256, BF16),
                                              (30, 9, 4096, BF16)])
def test_msar_chunk_matches_full_sequence(t_prev, T, d, dtype):
    """A chunk of T tokens after t_prev history rows gives the full-sequence
    read's outputs for those tokens (rows before the history count as zero)."""
    rng = _rng(t_prev * 3 + T + d)
    ks = (4, 8, 12)
    src, q, cw, mw = _msar_setup(rng, 8, t_prev + T, d, ks, dtype)
    out = attnres.msar_expand_fwd_chunk(to_dev(src, dtype), t_prev, ks, to_dev(cw, F32), to_dev(q, F32),
                                        mix_w=to_dev(mw, F32))
    ref = oracle.msar(src, ks, cw, q, None, 1e-6, None, mw, 1e-6)[t_prev:]
    check_out(out, ref, dtype, np.abs(src).max())


def test_msar_chunked_prefill_equals_one_call_bitwise():
    """Prefill a sequence in chunks, each with the previous 11 rows as history:
    every chunk's outputs equal the one-call read's rows bit for bit, and a
    chunk with no history equals msar_expand_fwd."""
    rng = _rng(61)
    T, d, ks = 300, 2048, (4, 8, 12)
    src, q, cw, mw = _msar_setup(rng, 8, T, d, ks, BF16)
    sd, qd, cwd, mwd = to_dev(src, BF16), to_dev(q, F32), to_dev(cw, F32), to_dev(mw, F32)
    whole = attnres.msar_expand_fwd(sd, ks, cwd, qd, mix_w=mwd)
    first = attnres.msar_expand_fwd_chunk(sd[:, :64].contiguous(), 0, ks, cwd, qd, mix_w=mwd)
    assert torch.equal(first, whole[:64])
    for c0, c1 in ((64, 128), (128, 250), (250, 300)):
        h = min(11, c0)
        part = attnres.msar_expand_fwd_chunk(sd[:, c0 - h:c1].contiguous(), h, ks, cwd, qd, mix_w=mwd)
        assert torch.equal(part, whole[c0:c1]), (c0, c1)


# --------------------------------------------------------------- backward

def _check_grads(got, ref, dtype, what):
    dsrc, dq, dg = got
    rs, rq, rg = ref
    check_out(dsrc, rs, dtype, what=f"{what} dsrc")
    # parameter gradients are fp32 sums over the tokens
    for name, g_, r_ in (("dq", dq, rq), ("dgain", dg, rg)):
        if g_ is not None:
            check_out(g_, r_, F32, np.abs(r_).max(), strict=False, what=f"{what} {name}")


@pytest.mark.parametrize("n_src,n_q,T,d,dtype,with_gain", [
    (1, 1, 5, 64, F32, False), (3, 1, 37, 256, F32, True), (9, 1, 70, 4096, BF16, True),
    (8, 2, 40, 2048, BF16, False), (16, 1, 20, 1024, BF16, True), (5, 2, 300, 512, F32, True),
    (12, 1, 3, 4096, BF16, False), (4, 1, 333, 1000, F32, True), (7, 2, 90, 1024, BF16, True)])
def test_read_bwd(n_src, n_q, T, d, dtype, with_gain):
    """Backward of the read against the oracle's chain rule: the sources', the
    queries' and the gain's gradients."""
    rng = _rng(n_src * 5 + n_q + T + d)
    src = _sources(rng, n_src, T, d, dtype, step=0.25)
    q = _queries(rng, n_q, d)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32) if with_gain else None
    dout = _sources(rng, n_q, T, d, dtype, step=0)
    got = attnres.attnres_read_bwd(to_dev(src, dtype), to_dev(q, F32), to_dev(dout, dtype),
                                   to_dev(g, F32) if with_gain else None, 1e-6)
    _check_grads(got, oracle.read_bwd(src, q, dout, g, 1e-6), dtype, f"n_src={n_src}")


@pytest.mark.parametrize("n_src,n_q,T,d,dtype,with_gain", [
    (17, 1, 50, 1024, BF16, True), (33, 2, 40, 4096, BF16, False), (24, 4, 30, 512, F32, True),
    (64, 1, 70, 2048, BF16, True), (20, 3, 100, 4096, BF16, True), (41, 1, 3, 1024, F32, False)])
def test_read_bwd_many_sources(n_src, n_q, T, d, dtype, with_gain):
    """More sources than one pass of the backward kernel takes (> 16): the
    sources in chunks of 8, each chunk's read state recomputed, the backward of
    the states' merge, then each chunk's backward with its lse gradient;
    against the oracle's chain rule over all sources at once."""
    rng = _rng(n_src * 3 + n_q + T + d)
    src = _sources(rng, n_src, T, d, dtype, step=0.1)
    q = _queries(rng, n_q, d)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32) if with_gain else None
    dout = _sources(rng, n_q, T, d, dtype, step=0)
    got = attnres.attnres_read_bwd(to_dev(src, dtype), to_dev(q, F32), to_dev(dout, dtype),
                                   to_dev(g, F32) if with_gain else None, 1e-6)
    _check_grads_states(got, oracle.read_bwd(src, q, dout, g, 1e-6), dtype, f"n_src={n_src}")


def _check_grads_states(got, ref, dtype, what):
    """As _check_grads, but the chunks' states (o_c and beta_c dh) are held in
    the source dtype between the steps, so the parameter gradients (sums over
    the tokens) carry that rounding: they are held to the dtype's bar, as the
    two-phase Block backward's are."""
    dsrc, dq, dg = got
    rs, rq, rg = ref
    check_out(dsrc, rs, dtype, what=f"{what} dsrc")
    for name, g_, r_ in (("dq", dq, rq), ("dgain", dg, rg)):
        if g_ is not None:
            check_out(g_, r_, dtype if dtype == BF16 else F32, np.abs(r_).max(), strict=False, chain=dtype == BF16,
                      what=f"{what} {name}")


def test_block_phase1_bwd_many_sources_with_lse_gradient():
    """The phase-1 backward (o and lse gradients) over 28 sources."""
    rng = _rng(28)
    n_src, n_q, T, d = 28, 2, 45, 1024
    src = _sources(rng, n_src, T, d, BF16, step=0.1)
    q = _queries(rng, n_q, d)
    d_o = _sources(rng, n_q, T, d, BF16, step=0)
    dlse = rng.standard_normal((n_q, T)).astype(np.float32)
    got = attnres.attnres_block_phase1_bwd(to_dev(src, BF16), to_dev(q, F32), to_dev(d_o, BF16), to_dev(dlse, F32))
    _check_grads_states(got, oracle.block_phase1_bwd(src, q, d_o, dlse, None, 1e-6), BF16, "phase 1, 28 sources")


@pytest.fixture(params=[0, 1], ids=["two-kernel", "chain"])
def many_variant(request):
    """Kernel variant 0 runs the backward of one query over 17..64 bf16
    sources at d = 2048 or 4096 as two kernels (coefficients over all the
    sources, then channel slices); variant 1 keeps the chunked chain."""
    attnres.attnres_debug_set_kernel_variant(request.param)
    yield request.param
    attnres.attnres_debug_set_kernel_variant(0)


@pytest.mark.parametrize("n_src,T,d,with_gain,with_lse", [
    (17, 100, 4096, True, False),        # one source past two chunks
    (40, 7, 2048, True, True),           # five full chunks, the lse gradient
    (64, 300, 4096, False, True),        # the deepest Full-at-depth layer
    (23, 1, 4096, True, False),          # one token, a short last chunk
    (33, 160, 2048, False, False)])      # a one-source last chunk
def test_read_bwd_many_sources_both_forms(many_variant, n_src, T, d, with_gain, with_lse):
    """The backward of one query over many sources under both forms against
    the oracle's chain rule over all the sources at once.  The two-kernel
    form keeps nothing in bf16 between its steps and is held to the strict
    bar; the chain holds the chunks' states in bf16 (see _check_grads_states)."""
    rng = _rng(n_src * 7 + T + d)
    src = _sources(rng, n_src, T, d, BF16, step=0.1)
    q = _queries(rng, 1, d)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32) if with_gain else None
    dout = _sources(rng, 1, T, d, BF16, step=0)
    sd, qd, od = to_dev(src, BF16), to_dev(q, F32), to_dev(dout, BF16)
    gd = to_dev(g, F32) if with_gain else None
    if with_lse:
        dl = rng.standard_normal((1, T)).astype(np.float32)
        got = attnres.attnres_block_phase1_bwd(sd, qd, od, to_dev(dl, F32), gd, 1e-6)
        ref = oracle.block_phase1_bwd(src, q, dout, dl, g, 1e-6)
    else:
        got = attnres.attnres_read_bwd(sd, qd, od, gd, 1e-6)
        ref = oracle.read_bwd(src, q, dout, g, 1e-6)
    what = f"variant {many_variant}, {n_src} sources"
    if many_variant == 0:
        _check_grads(got, ref, BF16, what)
    else:
        _check_grads_states(got, ref, BF16, what)


def test_read_bwd_many_sources_two_kernel_form_is_deterministic_and_accumulates():
    rng = _rng(54)
    n_src, T, d = 48, 250, 4096
    src = to_dev(_sources(rng, n_src, T, d, BF16, step=0.1), BF16)
    q = to_dev(_queries(rng, 1, d), F32)
    dout = to_dev(_sources(rng, 1, T, d, BF16, step=0), BF16)
    g = to_dev(rng.uniform(0.5, 1.5, d).astype(np.float32), F32)
    a = attnres.attnres_read_bwd(src, q, dout, g)
    b = attnres.attnres_read_bwd(src, q, dout, g)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    base = to_dev(_sources(rng, n_src, T, d, BF16), BF16)
    acc = base.clone()
    attnres.attnres_read_bwd(src, q, dout, g, dsrc=acc, accumulate=True)
    check_out(acc, to_host(base) + to_host(a[0]), BF16, what="accumulated dsrc")


def test_read_bwd_accumulates_and_is_deterministic():
    rng = _rng(51)
    n_src, T, d = 9, 200, 4096
    src = to_dev(_sources(rng, n_src, T, d, BF16, step=0.25), BF16)
    q = to_dev(_queries(rng, 1, d), F32)
    dout = to_dev(_sources(rng, 1, T, d, BF16, step=0), BF16)
    g = to_dev(rng.uniform(0.5, 1.5, d).astype(np.float32), F32)
    a = attnres.attnres_read_bwd(src, q, dout, g)
    b = attnres.attnres_read_bwd(src, q, dout, g)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    base = to_dev(_sources(rng, n_src, T, d, BF16), BF16)
    acc = base.clone()
    attnres.attnres_read_bwd(src, q, dout, g, dsrc=acc, accumulate=True)
    ref = to_host(base) + to_host(a[0])
    check_out(acc, ref, BF16, what="accumulated dsrc")


def test_read_bwd_empty_sequence_zeroes_parameter_gradients():
    d = 256
    src = torch.empty((3, 0, d), dtype=F32, device="cuda")
    q = to_dev(_queries(_rng(52), 1, d), F32)
    dq = torch.full((1, d), 7.0, device="cuda")
    dg = torch.full((d,), 7.0, device="cuda")
    attnres.attnres_read_bwd(src, q, torch.empty((1, 0, d), dtype=F32, device="cuda"), None, 1e-6,
                             dqueries=dq, dgain=dg)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dq) == 0 and torch.count_nonzero(dg) == 0


@pytest.mark.parametrize("n_src,n_q,T,d,dtype,with_lse", [
    (8, 4, 64, 4096, BF16, True), (8, 4, 40, 2048, BF16, False), (3, 2, 37, 256, F32, True),
    (9, 1, 50, 4096, BF16, True), (5, 3, 130, 1000, F32, True)])
def test_block_phase1_bwd(n_src, n_q, T, d, dtype, with_lse):
    """Block phase 1's backward (gradients of its o and lse outputs) against
    the oracle; without d_lse it is the read's backward."""
    rng = _rng(n_src * 3 + n_q * 5 + T + d)
    src = _sources(rng, n_src, T, d, dtype, step=0.25)
    q = _queries(rng, n_q, d)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    d_o = _sources(rng, n_q, T, d, dtype, step=0)
    dl = rng.standard_normal((n_q, T)).astype(np.float32) if with_lse else None
    got = attnres.attnres_block_phase1_bwd(to_dev(src, dtype), to_dev(q, F32), to_dev(d_o, dtype),
                                           to_dev(dl, F32) if with_lse else None, to_dev(g, F32), 1e-6)
    _check_grads(got, oracle.block_phase1_bwd(src, q, d_o, dl, g, 1e-6), dtype, f"n_q={n_q}")


@pytest.fixture(params=[0, 1], ids=["two-kernel", "one-kernel"])
def bwd_variant(request):
    """Kernel variant 0 runs the read backward of 3-4 queries (bf16, <= 8
    sources, d = 2048 or 4096, heads of >= 256 channels) as two kernels (row
    coefficients, then channel slices); variant 1 keeps the one-kernel form."""
    attnres.attnres_debug_set_kernel_variant(request.param)
    yield request.param
    attnres.attnres_debug_set_kernel_variant(0)


@pytest.mark.parametrize("n_src,n_q,T,d,H,with_gain,with_lse", [
    (8, 4, 300, 4096, 1, True, True),       # Block phase 1's backward, lse gradient
    (8, 4, 77, 4096, 8, True, False),       # the MHAR workload's heads (512 channels)
    (5, 3, 151, 2048, 1, False, True),      # fewer tokens than SMs, 3 queries
    (1, 4, 1, 4096, 1, True, False),        # one source, one token
    (8, 3, 40, 4096, 16, False, False),     # heads of 256 channels
    (3, 4, 1000, 2048, 2, True, False),     # two heads, one per half row
    (7, 4, 9, 2048, 4, True, False)])
def test_read_bwd_both_forms(bwd_variant, n_src, n_q, T, d, H, with_gain, with_lse):
    """The read backward with 3-4 queries under both kernel forms against the
    oracle's chain rule (per head for H > 1; with Block phase 1's lse
    gradient where given)."""
    rng = _rng(n_src * 13 + n_q * 7 + T + d + H)
    src = _sources(rng, n_src, T, d, BF16, step=0.25)
    q = _queries(rng, n_q, d)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32) if with_gain else None
    dout = _sources(rng, n_q, T, d, BF16, step=0)
    sd, qd, od = to_dev(src, BF16), to_dev(q, F32), to_dev(dout, BF16)
    gd = to_dev(g, F32) if with_gain else None
    if with_lse:
        dl = rng.standard_normal((n_q, T)).astype(np.float32)
        got = attnres.attnres_block_phase1_bwd(sd, qd, od, to_dev(dl, F32), gd, 1e-6)
        ref = oracle.block_phase1_bwd(src, q, dout, dl, g, 1e-6)
    elif H == 1:
        got = attnres.attnres_read_bwd(sd, qd, od, gd, 1e-6)
        ref = oracle.read_bwd(src, q, dout, g, 1e-6)
    else:
        qh = q.reshape(n_q, H, d // H)
        got = attnres.mhar_read_bwd(sd, to_dev(qh, F32), od, gd, 1e-6)
        ref = oracle.mhar_bwd(src, qh, dout, g, 1e-6)
    _check_grads(got, ref, BF16, f"variant {bwd_variant} H={H}")


def test_read_bwd_two_kernel_form_is_deterministic_accumulates_and_agrees_with_one_kernel():
    """Two runs of the two-kernel form agree bitwise; with accumulate it adds
    into the given source gradients; and it agrees with the one-kernel form
    within the bf16 bar.  (The one-kernel form rounds dsrc to bf16 after its
    first group of two queries and adds the second group to that, so it
    carries two roundings; the two-kernel form rounds once.  Against the
    oracle the two-kernel form is within half a bf16 step, see
    test_read_bwd_both_forms.)"""
    rng = _rng(53)
    n_src, n_q, T, d = 8, 4, 500, 4096
    src = to_dev(_sources(rng, n_src, T, d, BF16, step=0.25), BF16)
    q = to_dev(_queries(rng, n_q, d), F32)
    dout = to_dev(_sources(rng, n_q, T, d, BF16, step=0), BF16)
    g = to_dev(rng.uniform(0.5, 1.5, d).astype(np.float32), F32)
    a = attnres.attnres_read_bwd(src, q, dout, g)
    b = attnres.attnres_read_bwd(src, q, dout, g)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    base = to_dev(_sources(rng, n_src, T, d, BF16), BF16)
    acc = base.clone()
    attnres.attnres_read_bwd(src, q, dout, g, dsrc=acc, accumulate=True)
    check_out(acc, to_host(base) + to_host(a[0]), BF16, what="accumulated dsrc")
    attnres.attnres_debug_set_kernel_variant(1)
    try:
        c = attnres.attnres_read_bwd(src, q, dout, g)
    finally:
        attnres.attnres_debug_set_kernel_variant(0)
    check_out(a[0], to_host(c[0]).astype(np.float64), BF16, what="dsrc of the two forms")
    for name, u, v in (("dq", a[1], c[1]), ("dgain", a[2], c[2])):
        u, v = to_host(u).astype(np.float64), to_host(v).astype(np.float64)
        assert np.abs(u - v).max() <= 1e-4 * np.abs(v).max(), name


@pytest.fixture(params=[0, 1], ids=["ring", "whole-token"])
def one_variant(request):
    """Kernel variant 0 runs the read backward of one query over 3 to 16 bf16
    sources (d = 2048 or 4096) through a ring of half-row stages; variant 1
    keeps the kernel with whole-token stages."""
    attnres.attnres_debug_set_kernel_variant(request.param)
    yield request.param
    attnres.attnres_debug_set_kernel_variant(0)


@pytest.mark.parametrize("n_src,T,d,with_gain,with_lse", [
    (8, 300, 4096, True, False),     # the MSAR per-stream read backward's shape
    (8, 300, 4096, True, True),      # Block phase 1's backward with one query, lse gradient
    (3, 151, 2048, False, True),     # fewer tokens than SMs
    (3, 1, 4096, True, False),       # one token (one CTA, one step of the pipeline)
    (5, 1000, 2048, True, False),    # several tokens per CTA, ragged ring
    (7, 9, 4096, False, False),
    (9, 300, 4096, True, False),     # a Block layer's read: 8 block representations and the partial
    (9, 300, 4096, True, True),
    (12, 151, 2048, False, True),
    (16, 700, 4096, True, False),    # three stages
    (13, 1, 4096, True, False),
    (11, 1000, 2048, True, False),
    (16, 300, 2048, False, True)])
def test_read_bwd_one_query_both_forms(one_variant, n_src, T, d, with_gain, with_lse):
    """The read backward of one query over 3 to 16 sources under both kernel
    forms against the oracle's chain rule (with Block phase 1's lse gradient
    where given)."""
    rng = _rng(n_src * 17 + T + d + 3 * with_lse)
    src = _sources(rng, n_src, T, d, BF16, step=0.25)
    q = _queries(rng, 1, d)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32) if with_gain else None
    dout = _sources(rng, 1, T, d, BF16, step=0)
    sd, qd, od = to_dev(src, BF16), to_dev(q, F32), to_dev(dout, BF16)
    gd = to_dev(g, F32) if with_gain else None
    if one_variant == 1 and d == 4096 and n_src > 12:
        # the whole-token kernel's two stages hold at most 13 rows at d = 4096
        # (the sources and the gradient row): only the ring form takes more
        with pytest.raises(attnres.AttnResError):
            attnres.attnres_read_bwd(sd, qd, od, gd, 1e-6)
        return
    if with_lse:
        dl = rng.standard_normal((1, T)).astype(np.float32)
        got = attnres.attnres_block_phase1_bwd(sd, qd, od, to_dev(dl, F32), gd, 1e-6)
        ref = oracle.block_phase1_bwd(src, q, dout, dl, g, 1e-6)
    else:
        got = attnres.attnres_read_bwd(sd, qd, od, gd, 1e-6)
        ref = oracle.read_bwd(src, q, dout, g, 1e-6)
    if T > 1:
        _check_grads(got, ref, BF16, f"variant {one_variant}")
    else:
        # One token: nothing averages out the query's bf16 hi + lo split in the
        # ring form's tensor-core scores (about 2^-17 relative per channel,
        # amplified by the cancellation in ds_i = alpha_i (dout.v_i - mean)),
        # measured at 1.06e-4 of max|dgain|, just past the fp32 bar.  The
        # inputs are bf16, whose stated bar is 2e-2 relative with fp32
        # accumulation: the parameter gradients are held to that here, dsrc to
        # the bf16 bar and the elementwise bound as everywhere.
        check_out(got[0], ref[0], BF16, what="dsrc")
        for name, g_, r_ in (("dq", got[1], ref[1]), ("dgain", got[2], ref[2])):
            if g_ is not None:
                check_out(g_, r_, BF16, what=name)


@pytest.mark.parametrize("n_src,d", [(8, 4096), (9, 4096), (5, 2048), (12, 2048)])
def test_read_bwd_one_query_ring_is_deterministic_accumulates_and_agrees_with_whole_token_form(n_src, d):
    """Two runs of the ring form agree bitwise; with accumulate it adds into
    the given source gradients (8-byte pieces per lane at d = 4096, 4-byte at
    2048); and it agrees with the whole-token form within the bf16 bar (both
    round dsrc once; their sums run in different orders)."""
    rng = _rng(59 + n_src + d)
    T = 700
    src = to_dev(_sources(rng, n_src, T, d, BF16, step=0.25), BF16)
    q = to_dev(_queries(rng, 1, d), F32)
    dout = to_dev(_sources(rng, 1, T, d, BF16, step=0), BF16)
    g = to_dev(rng.uniform(0.5, 1.5, d).astype(np.float32), F32)
    a = attnres.attnres_read_bwd(src, q, dout, g)
    b = attnres.attnres_read_bwd(src, q, dout, g)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    base = to_dev(_sources(rng, n_src, T, d, BF16), BF16)
    acc = base.clone()
    attnres.attnres_read_bwd(src, q, dout, g, dsrc=acc, accumulate=True)
    check_out(acc, to_host(base) + to_host(a[0]), BF16, what="accumulated dsrc")
    attnres.attnres_debug_set_kernel_variant(1)
    try:
        c = attnres.attnres_read_bwd(src, q, dout, g)
    finally:
        attnres.attnres_debug_set_kernel_variant(0)
    check_out(a[0], to_host(c[0]).astype(np.float64), BF16, what="dsrc of the two forms")
    for name, u, v in (("dq", a[1], c[1]), ("dgain", a[2], c[2])):
        u, v = to_host(u).astype(np.float64), to_host(v).astype(np.float64)
        assert np.abs(u - v).max() <= 1e-4 * np.abs(v).max(), name


@pytest.mark.parametrize("T,d,dtype,with_gain,with_partial", [
    (100, 4096, BF16, True, True), (37, 2048, BF16, False, True), (50, 256, F32, True, True),
    (333, 1000, F32, True, True), (20, 512, BF16, True, False), (1, 64, F32, False, True)])
def test_block_phase2_bwd(T, d, dtype, with_gain, with_partial):
    """The merge's backward against the oracle: d_o, d_lse, d_partial, the
    query's and the gain's gradients (no partial: d_o = dh, the rest zero)."""
    rng = _rng(T + d + with_gain)
    o = _sources(rng, 1, T, d, dtype)[0]
    p = _sources(rng, 1, T, d, dtype, step=0)[0] * 1.5 if with_partial else None
    if dtype == BF16 and p is not None:
        p = inputs.bf16_round(p)
    dh = _sources(rng, 1, T, d, dtype, step=0)[0]
    lse = (rng.standard_normal(T) * 3).astype(np.float32)
    q = _queries(rng, 1, d)[0]
    g = rng.uniform(0.5, 1.5, d).astype(np.float32) if with_gain else None
    got = attnres.attnres_block_phase2_bwd(to_dev(o, dtype), to_dev(lse, F32),
                                           to_dev(p, dtype) if with_partial else None, to_dev(q, F32),
                                           to_dev(dh, dtype), to_dev(g, F32) if with_gain else None, 1e-6)
    ref = oracle.block_phase2_bwd(o, lse, p, q, dh, g, 1e-6)
    check_out(got[0], ref[0], dtype, what="d_o")
    check_out(got[1], ref[1], F32, np.abs(ref[1]).max() + 1e-30, strict=False, what="d_lse")
    if with_partial:
        check_out(got[2], ref[2], dtype, what="d_partial")
    else:
        assert got[2] is None
    for name, x, y in (("dquery", got[3], ref[3]), ("dgain", got[4], ref[4])):
        check_out(x, y, F32, np.abs(y).max() + 1e-30, strict=False, what=name)


def test_block_phase2_bwd_accumulates_and_is_deterministic():
    rng = _rng(81)
    T, d = 300, 4096
    o, p, dh = (to_dev(_sources(rng, 1, T, d, BF16, step=0)[0], BF16) for _ in range(3))
    lse = to_dev((rng.standard_normal(T) * 3).astype(np.float32), F32)
    q = to_dev(_queries(rng, 1, d)[0], F32)
    a = attnres.attnres_block_phase2_bwd(o, lse, p, q, dh)
    b = attnres.attnres_block_phase2_bwd(o, lse, p, q, dh)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    base = to_dev(_sources(rng, 1, T, d, BF16)[0], BF16)
    acc = base.clone()
    attnres.attnres_block_phase2_bwd(o, lse, p, q, dh, d_partial=acc, accumulate=True)
    check_out(acc, to_host(base) + to_host(a[2]), BF16, what="accumulated d_partial")


@pytest.mark.parametrize("dtype,N,S,T,d", [(BF16, 8, 4, 64, 4096), (F32, 3, 2, 45, 512), (BF16, 5, 3, 100, 1024)])
def test_block_two_phase_backward_equals_one_shot(dtype, N, S, T, d):
    """The GPU backward of a block's two-phase forward -- each layer's merge
    backward, then phase 1's backward for all layers' d_o and d_lse -- against
    the oracle's backward of the one-shot reads (layer 1 reads the cached
    sources alone, layer s >= 2 also its partial)."""
    rng = _rng(N * 11 + S + T)
    cached = _sources(rng, N, T, d, dtype, step=0.25)
    parts = _sources(rng, S, T, d, dtype, step=0)
    q = _queries(rng, S, d)
    dh = _sources(rng, S, T, d, dtype, step=0)
    cd, qd = to_dev(cached, dtype), to_dev(q, F32)
    o, lse = attnres.attnres_block_phase1(cd, qd)
    d_o = torch.empty_like(o)
    d_lse = torch.empty_like(lse)
    dpart, dq2 = [None] * S, np.zeros((S, d))
    for s_ in range(S):
        r = attnres.attnres_block_phase2_bwd(o[s_], lse[s_], to_dev(parts[s_], dtype) if s_ > 0 else None, qd[s_],
                                             to_dev(dh[s_], dtype), d_o=d_o[s_], d_lse=d_lse[s_])
        dpart[s_], dq2[s_] = r[2], to_host(r[3])
    dsrc, dq1, _ = attnres.attnres_block_phase1_bwd(cd, qd, d_o, d_lse)
    ref_cached = np.zeros((N, T, d))
    for s_ in range(S):
        srcs = cached if s_ == 0 else np.concatenate([cached, parts[s_][None]])
        rs, rq, _ = oracle.read_bwd(srcs, q[s_][None], dh[s_][None], None, 1e-6)
        ref_cached += rs[:N]
        if s_ > 0:
            check_out(dpart[s_], rs[N], dtype, np.abs(rs[N]).max() * 4 + 1e-30, strict=False, chain=dtype == BF16,
                      what=f"layer {s_ + 1} d_partial")
        # the chain's intermediates (o, d_o) are stored in the source dtype,
        # so its parameter gradients carry that rounding
        gq = to_host(dq1)[s_] + dq2[s_]
        check_out(gq, rq[0], dtype, np.abs(rq[0]).max() + 1e-30, strict=False, chain=dtype == BF16,
                  what=f"layer {s_ + 1} dq")
    check_out(dsrc, ref_cached, dtype, what="cached sources' gradient")


@pytest.mark.parametrize("n_src,n_q,T,d,dtype", [(8, 3, 45, 2048, BF16), (5, 5, 30, 512, F32),
                                                  (9, 3, 25, 1024, BF16), (16, 2, 12, 2048, BF16)])
def test_read_bwd_more_queries_than_one_pass(n_src, n_q, T, d, dtype):
    """Queries beyond one pass (2, or 1 above 8 sources) take further passes
    whose source and gain gradients add up."""
    rng = _rng(n_src * 7 + n_q + T)
    src = _sources(rng, n_src, T, d, dtype, step=0.25)
    q = _queries(rng, n_q, d)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    dout = _sources(rng, n_q, T, d, dtype, step=0)
    got = attnres.attnres_read_bwd(to_dev(src, dtype), to_dev(q, F32), to_dev(dout, dtype), to_dev(g, F32), 1e-6)
    _check_grads(got, oracle.read_bwd(src, q, dout, g, 1e-6), dtype, f"n_q={n_q}")


@pytest.mark.parametrize("n_src,n_q,T,d,H,dtype,with_gain", [
    (8, 2, 64, 4096, 8, BF16, True),        # the MHAR workload's heads: one warp per head
    (8, 1, 50, 4096, 16, BF16, True),       # 32 vectors per head: one group per run of a warp
    (4, 4, 33, 2048, 4, BF16, False),       # two token rows per CTA, two passes of queries
    (3, 1, 41, 1024, 2, F32, True),         # a head spans two warps
    (9, 1, 30, 4096, 8, BF16, True),        # more than 8 sources
    (16, 2, 20, 2048, 2, BF16, False),      # 16 sources, passes of one query
    (6, 3, 77, 1536, 3, F32, True),         # warps past the row's last head
    (2, 1, 130, 512, 2, F32, True)])
def test_mhar_read_bwd(n_src, n_q, T, d, H, dtype, with_gain):
    """Backward of the MHAR read against the oracle's per-head chain rule."""
    rng = _rng(n_src * 11 + n_q + T + d + H)
    src = _sources(rng, n_src, T, d, dtype, step=0.25)
    q = _queries(rng, n_q, d).reshape(n_q, H, d // H)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32) if with_gain else None
    dout = _sources(rng, n_q, T, d, dtype, step=0)
    got = attnres.mhar_read_bwd(to_dev(src, dtype), to_dev(q, F32), to_dev(dout, dtype),
                                to_dev(g, F32) if with_gain else None, 1e-6)
    _check_grads(got, oracle.mhar_bwd(src, q, dout, g, 1e-6), dtype, f"H={H}")


def test_mhar_read_bwd_one_head_is_the_read_backward_bitwise():
    rng = _rng(71)
    n_src, T, d = 8, 90, 2048
    src = to_dev(_sources(rng, n_src, T, d, BF16, step=0.25), BF16)
    q = to_dev(_queries(rng, 2, d), F32)
    dout = to_dev(_sources(rng, 2, T, d, BF16, step=0), BF16)
    a = attnres.attnres_read_bwd(src, q, dout, None)
    b = attnres.mhar_read_bwd(src, q.view(2, 1, d), dout, None)
    for x, y in zip(a, b):
        assert torch.equal(x.reshape(-1), y.reshape(-1))


def test_mhar_read_bwd_is_block_diagonal_and_deterministic():
    """An output gradient on one head's slice leaves every other slice of the
    source, query and gain gradients exactly zero; two runs agree bitwise."""
    rng = _rng(72)
    n_src, T, d, H = 8, 100, 4096, 8
    dh = d // H
    src = to_dev(_sources(rng, n_src, T, d, BF16, step=0.25), BF16)
    q = to_dev(_queries(rng, 2, d).reshape(2, H, dh), F32)
    g = to_dev(rng.uniform(0.5, 1.5, d).astype(np.float32), F32)
    do = np.zeros((2, T, d), dtype=np.float32)
    do[:, :, 5 * dh:6 * dh] = rng.standard_normal((2, T, dh))
    dout = to_dev(do, BF16)
    a = attnres.mhar_read_bwd(src, q, dout, g)
    b = attnres.mhar_read_bwd(src, q, dout, g)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    dsrc, dq, dg = a
    off = torch.ones(d, dtype=torch.bool, device="cuda")
    off[5 * dh:6 * dh] = False
    assert torch.count_nonzero(dsrc[:, :, off]) == 0 and torch.count_nonzero(dg[off]) == 0
    assert torch.count_nonzero(dq[:, [h for h in range(H) if h != 5]]) == 0
    assert torch.count_nonzero(dsrc[:, :, ~off]) > 0


# --------------------------------------------------------------- MSAR

@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("n_src,T,d", [(8, 100, 256), (3, 45, 512), (1, 20, 64), (8, 40, 2048),
                                       (8, 30, 4096), (5, 200, 128)])
def test_msar(dtype, n_src, T, d):
    if dtype == F32 and d > 2048:
        pytest.skip("f32 MSAR supports d <= 2048")
    x = inputs.msar_inputs(n_src, T, d, seed=T + d, dtype="bf16" if dtype == BF16 else "f32")
    g = _rng(5).uniform(0.5, 1.5, d).astype(np.float32)
    mg = _rng(6).uniform(0.5, 1.5, 4 * d).astype(np.float32)
    out = attnres.msar_expand_fwd(to_dev(x["src"], dtype), x["ksizes"], to_dev(x["conv_w"], F32),
                                  to_dev(x["queries"], F32), to_dev(g, F32), 1e-6, to_dev(mg, F32),
                                  to_dev(x["mix_w"], F32), 1e-6)
    ref = oracle.msar(x["src"], x["ksizes"], x["conv_w"], x["queries"], g, 1e-6, mg, x["mix_w"], 1e-6)
    check_out(out, ref, dtype, np.abs(x["src"]).max() * 3)


@pytest.mark.parametrize("ks", [(1, 2, 3), (16, 5, 9), (12, 8, 4)])
def test_msar_kernel_sizes(ks):
    T, d = 60, 512
    x = inputs.msar_inputs(4, T, d, seed=7, ksizes=ks)
    out = attnres.msar_expand_fwd(to_dev(x["src"], BF16), x["ksizes"], to_dev(x["conv_w"], F32),
                                  to_dev(x["queries"], F32), None, 1e-6, None,
                                  to_dev(x["mix_w"], F32), 1e-6)
    ref = oracle.msar(x["src"], x["ksizes"], x["conv_w"], x["queries"], None, 1e-6, None,
                      x["mix_w"], 1e-6)
    check_out(out, ref, BF16)


def _msar_block(rng, N, S, T, d, dtype, ks=(4, 8, 12)):
    """Cached sources, S layers' stream queries and partial sums, conv and
    mixer weights for the two-phase MSAR tests."""
    cached = _sources(rng, N, T, d, dtype)
    parts = _sources(rng, S, T, d, dtype, step=0)
    q = _queries(rng, S * 4, d).reshape(S, 4, d)
    cw = np.concatenate([(rng.standard_normal((d, k)) / math.sqrt(k)).astype(np.float32).ravel() for k in ks])
    mw = (rng.standard_normal((4 * d, 4)) / math.sqrt(4 * d)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    mg = rng.uniform(0.5, 1.5, 4 * d).astype(np.float32)
    return cached, parts, q, cw, mw, g, mg


@pytest.mark.parametrize("dtype,N,S,T,d", [(BF16, 8, 4, 60, 4096), (BF16, 3, 2, 45, 512), (F32, 5, 1, 33, 256),
                                           (BF16, 1, 3, 20, 2048), (F32, 8, 4, 70, 1024), (BF16, 6, 6, 25, 512)])
def test_msar_block_phase1(dtype, N, S, T, d):
    """Phase 1 against the oracle: every layer's per-stream state (o, lse)
    over the cached sources; six layers take two groups."""
    rng = _rng(N * 13 + S + T + d)
    ks = (4, 8, 12)
    cached, _, q, cw, _, g, _ = _msar_block(rng, N, S, T, d, dtype, ks)
    o, lse = attnres.msar_block_phase1(to_dev(cached, dtype), ks, to_dev(cw, F32), to_dev(q, F32), to_dev(g, F32),
                                       1e-6)
    ro, rl = oracle.msar_phase1(cached, ks, cw, q, g, 1e-6)
    check_out(o, ro, dtype, np.abs(cached).max() * 3, what="o")
    check_lse(lse, rl)


@pytest.mark.parametrize("dtype,T,d,with_partial", [(BF16, 50, 4096, True), (BF16, 50, 4096, False),
                                                    (F32, 40, 512, True), (BF16, 130, 1024, True),
                                                    (F32, 17, 256, False)])
def test_msar_block_phase2(dtype, T, d, with_partial):
    """Phase 2 against the oracle on the same phase-1 state (the oracle's,
    rounded to the working dtype): the partial's streams, the per-stream
    merge and the mixer; no partial mixes the state alone."""
    rng = _rng(T + d + with_partial)
    ks = (4, 8, 12)
    cached, parts, q, cw, mw, g, mg = _msar_block(rng, 4, 1, T, d, dtype, ks)
    o, lse = oracle.msar_phase1(cached, ks, cw, q, g, 1e-6)
    o1 = inputs.bf16_round(o[0].astype(np.float32)) if dtype == BF16 else o[0].astype(np.float32)
    p = parts[0] if with_partial else None
    out = attnres.msar_block_phase2(to_dev(o1, dtype), to_dev(lse[0].astype(np.float32), F32),
                                    to_dev(p, dtype) if with_partial else None, ks, to_dev(cw, F32),
                                    to_dev(q[0], F32), to_dev(g, F32), 1e-6, to_dev(mg, F32), to_dev(mw, F32), 1e-6)
    ref = oracle.msar_phase2(o1.astype(np.float64), lse[0].astype(np.float32).astype(np.float64), p, ks, cw, q[0], g,
                             1e-6, mg, mw, 1e-6)
    check_out(out, ref, dtype, np.abs(cached).max() * 3)


@pytest.mark.parametrize("dtype,N,S,T,d", [(BF16, 8, 4, 64, 4096), (F32, 3, 2, 40, 512), (BF16, 5, 3, 150, 1024)])
def test_msar_block_two_phase_equals_one_shot(dtype, N, S, T, d):
    """The GPU two-phase chain (phase 1 for the block, phase 2 per layer)
    against the oracle's one-shot MSAR read of [cached, partial_s] (layer 1:
    the cached sources alone)."""
    rng = _rng(N * 7 + S * 3 + T)
    ks = (4, 8, 12)
    cached, parts, q, cw, mw, g, mg = _msar_block(rng, N, S, T, d, dtype, ks)
    cwd, qd, gd, mgd, mwd = (to_dev(x, F32) for x in (cw, q, g, mg, mw))
    o, lse = attnres.msar_block_phase1(to_dev(cached, dtype), ks, cwd, qd, gd, 1e-6)
    for s_ in range(S):
        p = parts[s_] if s_ > 0 else None
        out = attnres.msar_block_phase2(o[s_], lse[s_], to_dev(p, dtype) if p is not None else None, ks, cwd,
                                        qd[s_], gd, 1e-6, mgd, mwd, 1e-6)
        srcs = cached if p is None else np.concatenate([cached, p[None]])
        ref = oracle.msar(srcs, ks, cw, q[s_], g, 1e-6, mg, mw, 1e-6)
        check_out(out, ref, dtype, np.abs(srcs).max() * 3, what=f"layer {s_ + 1}")


@pytest.mark.parametrize("dtype,n_src,T,d,ks", [(BF16, 8, 60, 4096, (4, 8, 12)), (F32, 3, 45, 512, (4, 8, 12)),
                                                 (BF16, 8, 100, 256, (1, 2, 3)), (BF16, 5, 30, 1024, (16, 5, 9)),
                                                 (F32, 1, 20, 128, (4, 8, 12))])
def test_msar_per_source_kernels(dtype, n_src, T, d, ks):
    """MSAR with each source's own conv kernels against the oracle."""
    rng = _rng(n_src * 3 + T + d)
    src = _sources(rng, n_src, T, d, dtype)
    q = _queries(rng, 4, d)
    cw = np.stack([np.concatenate([(rng.standard_normal((d, k)) / math.sqrt(k)).astype(np.float32).ravel()
                                   for k in ks]) for _ in range(n_src)])
    mw = (rng.standard_normal((4 * d, 4)) / math.sqrt(4 * d)).astype(np.float32)
    out = attnres.msar_expand_fwd_ps(to_dev(src, dtype), ks, to_dev(cw, F32), to_dev(q, F32), mix_w=to_dev(mw, F32))
    ref = oracle.msar_ps(src, ks, cw, q, None, 1e-6, None, mw, 1e-6)
    check_out(out, ref, dtype, np.abs(src).max() * 3)


def test_msar_per_source_equal_kernels_equal_the_shared_read_bitwise():
    """Per-source kernels that are all the same give the shared-kernel read
    bit for bit (the same products summed in the same order)."""
    rng = _rng(91)
    n_src, T, d, ks = 8, 70, 2048, (4, 8, 12)
    src = to_dev(_sources(rng, n_src, T, d, BF16), BF16)
    q = to_dev(_queries(rng, 4, d), F32)
    cw = np.concatenate([(rng.standard_normal((d, k)) / math.sqrt(k)).astype(np.float32).ravel() for k in ks])
    mw = to_dev((rng.standard_normal((4 * d, 4)) / math.sqrt(4 * d)).astype(np.float32), F32)
    # the per-source read is the per-token kernel's PS form: compare it with
    # the shared read of that same kernel (variant 1 keeps it for the shared
    # kernels too)
    attnres.attnres_debug_set_kernel_variant(1)
    try:
        shared = attnres.msar_expand_fwd(src, ks, to_dev(cw, F32), q, mix_w=mw)
    finally:
        attnres.attnres_debug_set_kernel_variant(0)
    per = attnres.msar_expand_fwd_ps(src, ks, to_dev(np.stack([cw] * n_src), F32), q, mix_w=mw)
    assert torch.equal(shared, per)


def _msar_tile_case(n_src, T, d, seed):
    x = inputs.msar_inputs(n_src, T, d, seed=seed)
    rng = _rng(seed + 1)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    mg = rng.uniform(0.5, 1.5, 4 * d).astype(np.float32)
    dev = (to_dev(x["src"], BF16), x["ksizes"], to_dev(x["conv_w"], F32), to_dev(x["queries"], F32),
           to_dev(g, F32), 1e-6, to_dev(mg, F32), to_dev(x["mix_w"], F32), 1e-6)
    ref = oracle.msar(x["src"], x["ksizes"], x["conv_w"], x["queries"], g, 1e-6, mg, x["mix_w"], 1e-6)
    return dev, ref


@pytest.mark.parametrize("n_src,T,d", [(8, 1, 4096), (8, 3, 4096), (8, 5, 4096), (5, 6, 4096), (1, 37, 4096),
                                       (8, 131, 2048), (7, 9, 1024), (2, 64, 512), (8, 13, 256)])
def test_msar_tile_kernel_shapes(n_src, T, d):
    """The tile-batched read (bf16, kernel sizes 4/8/12, d a multiple of 256):
    partial last tiles, one to eight sources, every cluster width from one CTA
    (d = 256) to sixteen (d = 4096), against the oracle with the elementwise
    bound."""
    dev, ref = _msar_tile_case(n_src, T, d, seed=T * 7 + d + n_src)
    out = attnres.msar_expand_fwd(*dev)
    check_out(out, ref, BF16)


@pytest.mark.parametrize("T,d", [(1000, 2048), (700, 4096)])
def test_msar_tile_kernel_agrees_with_the_per_token_kernel(T, d):
    """Many clusters of a few tiles each: the tile-batched read and the
    per-token kernel (variant 1) both meet the bar against the oracle, and
    they differ from each other by at most one bf16 rounding step per element
    plus the float32 summation order."""
    dev, ref = _msar_tile_case(8, T, d, seed=T + d)
    tile = attnres.msar_expand_fwd(*dev)
    attnres.attnres_debug_set_kernel_variant(1)
    try:
        per_token = attnres.msar_expand_fwd(*dev)
    finally:
        attnres.attnres_debug_set_kernel_variant(0)
    check_out(tile, ref, BF16, what="tile kernel")
    check_out(per_token, ref, BF16, what="per-token kernel")
    a, b = to_host(tile), to_host(per_token)
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.abs(b) + 1e-3 * np.abs(b).max())


def test_msar_tile_kernel_is_deterministic():
    dev, _ = _msar_tile_case(8, 77, 4096, seed=4)
    a = attnres.msar_expand_fwd(*dev)
    b = attnres.msar_expand_fwd(*dev)
    assert torch.equal(a, b)


# --------------------------------------------------------------- MSAR backward

def _msar_bwd_case(rng, n_src, T, d, dtype, ks, with_gains):
    src = _sources(rng, n_src, T, d, dtype)
    q = _queries(rng, 4, d)
    cw = np.concatenate([(rng.standard_normal((d, k)) / math.sqrt(k)).astype(np.float32).ravel() for k in ks])
    mw = (rng.standard_normal((4 * d, 4)) / math.sqrt(4 * d)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32) if with_gains else None
    mg = rng.uniform(0.5, 1.5, 4 * d).astype(np.float32) if with_gains else None
    dh = _sources(rng, 1, T, d, dtype, step=0)[0]
    return src, q, cw, mw, g, mg, dh


def _msar_bwd_gpu(case, ks, dtype):
    src, q, cw, mw, g, mg, dh = case
    dev = lambda x: to_dev(x, F32) if x is not None else None
    return attnres.msar_expand_bwd(to_dev(src, dtype), ks, dev(cw), dev(q), to_dev(dh, dtype), dev(g), 1e-6,
                                   dev(mg), dev(mw), 1e-6)


_MSAR_GRADS = ("dsrc", "dconv_w", "dqueries", "dgain", "dmix_gain", "dmix_w")


def _check_msar_grads(got, ref, dtype, what):
    """Every gradient within the dtype's bar of its own largest value: the
    streams, the per-stream reads and their gradients are held in dtype
    between the steps, so with bf16 the parameter gradients carry bf16
    roundings too."""
    for name, g_, r_ in zip(_MSAR_GRADS, got, ref):
        r_ = np.asarray(r_).reshape(tuple(g_.shape))
        check_out(g_, r_, dtype, np.abs(r_).max(), strict=False, chain=dtype == BF16, what=f"{what} {name}")


@pytest.mark.parametrize("dtype,n_src,T,d,ks,with_gains", [
    (BF16, 8, 70, 4096, (4, 8, 12), True), (BF16, 3, 45, 2048, (4, 8, 12), False),
    (F32, 5, 300, 1024, (4, 8, 12), True), (BF16, 1, 33, 1024, (4, 8, 12), True),
    (BF16, 16, 20, 2048, (4, 8, 12), False), (BF16, 4, 130, 1024, (16, 5, 9), True),
    (F32, 2, 64, 1024, (1, 2, 3), True), (BF16, 9, 1, 4096, (4, 8, 12), True)])
def test_msar_bwd(dtype, n_src, T, d, ks, with_gains):
    """Backward of the MSAR read against the oracle's chain rule: the
    sources', conv kernels', stream queries', gain's and mixer's gradients
    (T = 300 at d = 1024 spans ten token chunks of the conv kernels)."""
    rng = _rng(n_src * 7 + T + d + sum(ks))
    case = _msar_bwd_case(rng, n_src, T, d, dtype, ks, with_gains)
    got = _msar_bwd_gpu(case, ks, dtype)
    src, q, cw, mw, g, mg, dh = case
    ref = oracle.msar_bwd(src, ks, cw, q, dh, g, 1e-6, mg, mw, 1e-6)
    _check_msar_grads(got, ref, dtype, f"n_src={n_src} T={T} d={d}")


def test_msar_bwd_is_deterministic_and_linear_in_dh():
    """Same inputs, same bits; and the backward of dh1 + dh2 is the sum of the
    two backwards (every gradient is linear in dh)."""
    rng = _rng(93)
    ks, T, d = (4, 8, 12), 150, 2048
    src, q, cw, mw, g, mg, dh = _msar_bwd_case(rng, 8, T, d, F32, ks, True)
    a = _msar_bwd_gpu((src, q, cw, mw, g, mg, dh), ks, F32)
    b = _msar_bwd_gpu((src, q, cw, mw, g, mg, dh), ks, F32)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    dh1 = dh.copy()
    dh1[T // 2:] = 0
    dh2 = dh - dh1
    a1 = _msar_bwd_gpu((src, q, cw, mw, g, mg, dh1), ks, F32)
    a2 = _msar_bwd_gpu((src, q, cw, mw, g, mg, dh2), ks, F32)
    for name, x, y1, y2 in zip(_MSAR_GRADS, a, a1, a2):
        ref = to_host(y1) + to_host(y2)
        check_out(x, ref, F32, np.abs(ref).max(), strict=False, what=f"linearity {name}")


def test_msar_bwd_empty_sequence_zeroes_parameter_gradients():
    d, ks = 1024, (4, 8, 12)
    src = torch.empty((3, 0, d), dtype=BF16, device="cuda")
    x = inputs.msar_inputs(3, 1, d, seed=3)
    got = attnres.msar_expand_bwd(src, ks, to_dev(x["conv_w"], F32), to_dev(x["queries"], F32),
                                  torch.empty((0, d), dtype=BF16, device="cuda"), mix_w=to_dev(x["mix_w"], F32))
    torch.cuda.synchronize()
    assert got[0].numel() == 0
    for t in got[1:]:
        assert torch.count_nonzero(t) == 0


def _msar_bwd_chunked_gpu(case, ks, dtype, bounds):
    """msar_expand_bwd_chunk over the chunks [bounds[c], bounds[c+1]), in
    order, each given min(t_c, max k - 1) history rows; the first chunk writes
    the parameter gradients, the others add into them."""
    src, q, cw, mw, g, mg, dh = case
    dev = lambda x: to_dev(x, F32) if x is not None else None
    n_src, T, d = src.shape
    sd, dhd = to_dev(src, dtype), to_dev(dh, dtype)
    dsrc = torch.full((n_src, T, d), float("nan"), dtype=dtype, device="cuda")
    grads = (torch.full(cw.shape, float("nan"), device="cuda"), torch.full((4, d), float("nan"), device="cuda"),
             torch.full((d,), float("nan"), device="cuda"), torch.full((4 * d,), float("nan"), device="cuda"),
             torch.full((4 * d, 4), float("nan"), device="cuda"))
    hist = max(ks) - 1
    for c, (c0, c1) in enumerate(zip(bounds[:-1], bounds[1:])):
        h = min(hist, c0)
        attnres.msar_expand_bwd_chunk(sd[:, c0 - h:c1], h, ks, dev(cw), dev(q), dhd[c0:c1], dsrc[:, c0 - h:c1],
                                      grads, c > 0, dev(g), 1e-6, dev(mg), dev(mw), 1e-6)
    return (dsrc,) + grads


@pytest.mark.parametrize("dtype,n_src,T,d,ks,bounds", [
    (BF16, 8, 300, 1024, (4, 8, 12), (0, 5, 100, 180, 300)),
    (F32, 5, 200, 2048, (4, 8, 12), (0, 64, 130, 200)),
    (BF16, 4, 130, 1024, (16, 5, 9), (0, 40, 41, 130))])
def test_msar_bwd_chunked_equals_one_call(dtype, n_src, T, d, ks, bounds):
    """The backward in chunks of the sequence (each with its conv history
    rows; short first chunks, a one-token chunk, kernels up to 16 taps) gives
    the one-call backward's gradients: the sources' to one more rounding of
    the history rows, the parameters' to the order of their sums (and, with
    bf16, to the rounding of the intermediates: a chunk of at most 64 tokens
    reads its streams with the few-token kernel, whose fp32 results can round
    to the other neighbouring bf16 value); and both meet the bar against the
    oracle."""
    rng = _rng(T + d + n_src)
    case = _msar_bwd_case(rng, n_src, T, d, dtype, ks, True)
    got = _msar_bwd_chunked_gpu(case, ks, dtype, bounds)
    one = _msar_bwd_gpu(case, ks, dtype)
    for name, a_, b_ in zip(_MSAR_GRADS, got, one):
        a_, b_ = to_host(a_), to_host(b_)
        assert np.all(np.isfinite(a_)), name
        bmax = np.abs(b_).max()
        if name == "dsrc" and dtype == BF16:
            assert np.all(np.abs(a_ - b_) <= 2.0 ** -7 * np.abs(b_) + 2e-3 * bmax), name
        else:
            tol = 2e-3 if dtype == BF16 else 1e-4
            assert np.abs(a_ - b_).max() <= tol * bmax, (name, np.abs(a_ - b_).max(), bmax)
    src, q, cw, mw, g, mg, dh = case
    ref = oracle.msar_bwd(src, ks, cw, q, dh, g, 1e-6, mg, mw, 1e-6)
    _check_msar_grads(got, ref, dtype, f"chunked n_src={n_src} T={T} d={d}")


def test_msar_bwd_chunk_adds_into_history_rows_only():
    """A chunk writes its own rows of dsrc and adds its share into the history
    rows: with the history rows preset to 1, the result there is 1 plus the
    gradient that the chunk alone sends back to them."""
    rng = _rng(77)
    ks, n_src, T, d = (4, 8, 12), 3, 40, 1024
    src, q, cw, mw, g, mg, dh = _msar_bwd_case(rng, n_src, T, d, BF16, ks, False)
    dev = lambda x: to_dev(x, F32)
    sd = to_dev(src, BF16)
    dh_last = to_dev(dh, BF16)[20:]
    grads = (torch.empty(cw.shape, device="cuda"), torch.empty((4, d), device="cuda"), None, None,
             torch.empty((4 * d, 4), device="cuda"))
    a = torch.ones((n_src, 31, d), dtype=BF16, device="cuda")
    attnres.msar_expand_bwd_chunk(sd[:, 9:40], 11, ks, dev(cw), dev(q), dh_last, a, grads, False, mix_w=dev(mw))
    b = torch.zeros((n_src, 31, d), dtype=BF16, device="cuda")
    attnres.msar_expand_bwd_chunk(sd[:, 9:40], 11, ks, dev(cw), dev(q), dh_last, b, grads, False, mix_w=dev(mw))
    assert torch.equal(a[:, 11:], b[:, 11:])
    # a's history rows are bf16(1 + share), b's bf16(share): equal to one rounding
    assert torch.allclose(a[:, :11].float(), b[:, :11].float() + 1, rtol=2.0 ** -7, atol=2.0 ** -7)
    assert torch.count_nonzero(b[:, :11]) > 0


@pytest.mark.parametrize("dtype,n_src,T,d,ks", [(BF16, 8, 70, 4096, (4, 8, 12)), (F32, 3, 200, 1024, (4, 8, 12)),
                                                 (BF16, 5, 45, 2048, (16, 5, 9)), (F32, 1, 33, 1024, (1, 2, 3))])
def test_msar_bwd_per_source_kernels(dtype, n_src, T, d, ks):
    """Backward with each source's own conv kernels (at a padded stride)
    against the oracle's per-source backward; the padding of the kernel
    gradients stays zero."""
    rng = _rng(n_src * 5 + T + d)
    src, q, _, mw, g, mg, dh = _msar_bwd_case(rng, n_src, T, d, dtype, ks, True)
    kt = d * sum(ks)
    cw = np.stack([np.concatenate([(rng.standard_normal((d, k)) / math.sqrt(k)).astype(np.float32).ravel()
                                   for k in ks]) for _ in range(n_src)])
    cw_pad = np.zeros((n_src, kt + 64), np.float32)
    cw_pad[:, :kt] = cw
    got = attnres.msar_expand_bwd_ps(to_dev(src, dtype), ks, to_dev(cw_pad, F32), to_dev(q, F32), to_dev(dh, dtype),
                                     to_dev(g, F32), 1e-6, to_dev(mg, F32), to_dev(mw, F32), 1e-6)
    assert torch.count_nonzero(got[1][:, kt:]) == 0
    got = (got[0], got[1][:, :kt]) + tuple(got[2:])
    ref = oracle.msar_ps_bwd(src, ks, cw, q, dh, g, 1e-6, mg, mw, 1e-6)
    _check_msar_grads(got, ref, dtype, f"per-source n_src={n_src} d={d}")


def test_msar_bwd_per_source_equal_kernels_match_the_shared_backward():
    """Equal per-source kernels: the sources', queries', gain's and mixer's
    gradients equal the shared-kernel backward's bit for bit, and the
    sources' kernel gradients add up to the shared one's."""
    rng = _rng(97)
    ks, T, d, n_src = (4, 8, 12), 120, 2048, 8
    src, q, cw, mw, g, mg, dh = _msar_bwd_case(rng, n_src, T, d, BF16, ks, True)
    dev = lambda x: to_dev(x, F32)
    shared = attnres.msar_expand_bwd(to_dev(src, BF16), ks, dev(cw), dev(q), to_dev(dh, BF16), dev(g), 1e-6, dev(mg),
                                     dev(mw), 1e-6)
    per = attnres.msar_expand_bwd_ps(to_dev(src, BF16), ks, dev(np.stack([cw] * n_src)), dev(q), to_dev(dh, BF16),
                                     dev(g), 1e-6, dev(mg), dev(mw), 1e-6)
    for k in (0, 2, 3, 4, 5):
        assert torch.equal(shared[k], per[k]), _MSAR_GRADS[k]
    total = to_host(per[1]).sum(axis=0)
    check_out(shared[1], total, F32, np.abs(total).max(), strict=False, what="summed kernel gradients")


# --------------------------------------------------------------- MSAR through the workspace chain

@pytest.mark.parametrize("dtype,n_src,T,d,ks,per_source", [
    (BF16, 8, 100, 4096, (4, 8, 12), False), (F32, 3, 300, 1024, (4, 8, 12), False),
    (BF16, 5, 45, 2048, (16, 5, 9), False), (BF16, 8, 70, 4096, (4, 8, 12), True),
    (F32, 1, 33, 1024, (1, 2, 3), True), (BF16, 12, 20, 1024, (4, 8, 12), False)])
def test_msar_workspace_chain(dtype, n_src, T, d, ks, per_source):
    """The MSAR read through the workspace chain (streams written once, one
    read per stream, the sliced mixer) against the oracle, with shared and
    with per-source kernels.  The per-stream reads are held in dtype before
    the mixer, so bf16 results are held to the stated bar."""
    rng = _rng(n_src * 13 + T + d)
    src = _sources(rng, n_src, T, d, dtype)
    q = _queries(rng, 4, d)
    mk = lambda: np.concatenate([(rng.standard_normal((d, k)) / math.sqrt(k)).astype(np.float32).ravel() for k in ks])
    cw = np.stack([mk() for _ in range(n_src)]) if per_source else mk()
    mw = (rng.standard_normal((4 * d, 4)) / math.sqrt(4 * d)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    mg = rng.uniform(0.5, 1.5, 4 * d).astype(np.float32)
    out = attnres.msar_expand_fwd_ws(to_dev(src, dtype), ks, to_dev(cw, F32), to_dev(q, F32), to_dev(g, F32), 1e-6,
                                     to_dev(mg, F32), to_dev(mw, F32), 1e-6)
    ref = (oracle.msar_ps if per_source else oracle.msar)(src, ks, cw, q, g, 1e-6, mg, mw, 1e-6)
    check_out(out, ref, dtype, np.abs(src).max() * 3, strict=dtype == F32)


def _rounded_streams(cached, cw, ks):
    """The 4 streams of every cached source as the workspace chain stores
    them: stream 0 the sources, streams 1..3 the oracle's causal conv rounded
    to bf16."""
    N, T, d = cached.shape
    out, off = [np.asarray(cached, np.float64)], 0
    for k in ks:
        kr = np.asarray(cw[off:off + d * k]).reshape(d, k)
        off += d * k
        out.append(np.stack([inputs.bf16_round(oracle.msar_conv(cached[i], kr).astype(np.float32))
                             for i in range(N)]).astype(np.float64))
    return out


@pytest.mark.parametrize("dtype,N,S,T,d", [(BF16, 8, 4, 60, 4096), (F32, 5, 1, 33, 1024), (BF16, 3, 6, 45, 2048),
                                           (BF16, 12, 9, 20, 512)])
def test_msar_block_phase1_workspace_chain(dtype, N, S, T, d):
    """Phase 1 through the workspace chain against the oracle's phase 1
    (every layer's per-stream o and lse; more than 8 layers take two groups,
    more than 8 sources the chunked read).  With bf16 the chain stores the
    streams in bf16 before reading them (the fused phase 1 keeps them in
    fp32), so its state is also checked exactly as the read of the rounded
    streams: o with the strict bf16 bound and lse with the fp32 one."""
    rng = _rng(N * 7 + S + T + d)
    ks = (4, 8, 12)
    cached, _, q, cw, _, g, _ = _msar_block(rng, N, S, T, d, dtype)
    o, lse = attnres.msar_block_phase1_ws(to_dev(cached, dtype), ks, to_dev(cw, F32), to_dev(q, F32),
                                          to_dev(g, F32), 1e-6)
    ro, rl = oracle.msar_phase1(cached, ks, cw, q, g, 1e-6)
    check_out(o, ro, dtype, np.abs(cached).max(), strict=dtype == F32, what="o")
    if dtype == F32:
        check_lse(lse, rl)
        return
    for r, U in enumerate(_rounded_streams(cached, cw, ks)):
        o_r, l_r = oracle.block_phase1(U, q[:, r, :], g, 1e-6)
        check_out(o[:, r], o_r, BF16, what=f"o of stream {r} (rounded streams)")
        # The GPU forms a stream in fp32 and the oracle in fp64 before the bf16
        # rounding, so now and then one element rounds to the neighbouring bf16
        # value; that moves a score by at most one bf16 step (2^-7 relative) of
        # that element's term |w_c g_c u_c| / rms(u).  Allow two such elements
        # per token on top of the fp32 bound.
        wg = q[:, r, :].astype(np.float64) * g
        rms = np.sqrt((U ** 2).mean(axis=2) + 1e-6)                               # [N, T]
        term = np.max(np.abs(wg[:, None, None, :] * U[None]), axis=3) / rms[None]  # [S, N, T]
        tol = 1e-4 * (1.0 + np.abs(l_r)) + 2 * 2.0 ** -7 * term.max(axis=1)
        err = np.abs(to_host(lse[:, r]) - l_r)
        assert np.all(err <= tol), f"lse of stream {r} (rounded streams): max err {err.max()}"


@pytest.mark.parametrize("dtype,T,d,with_partial", [(BF16, 60, 4096, True), (F32, 45, 1024, True),
                                                    (BF16, 130, 2048, True), (BF16, 33, 1024, False),
                                                    (F32, 20, 2048, False)])
def test_msar_block_phase2_workspace_chain(dtype, T, d, with_partial):
    """Phase 2 through the workspace chain (the partial's streams, one Block
    merge per stream, the sliced mixer) against the oracle on the same
    phase-1 state; no partial mixes the state alone.  bf16 results are held
    to the stated bar (the chain stores the partial's streams and the merged
    streams in bf16)."""
    rng = _rng(T + d + with_partial + 1)
    ks = (4, 8, 12)
    cached, parts, q, cw, mw, g, mg = _msar_block(rng, 4, 1, T, d, dtype, ks)
    o, lse = oracle.msar_phase1(cached, ks, cw, q, g, 1e-6)
    o1 = inputs.bf16_round(o[0].astype(np.float32)) if dtype == BF16 else o[0].astype(np.float32)
    p = parts[0] if with_partial else None
    out = attnres.msar_block_phase2_ws(to_dev(o1, dtype), to_dev(lse[0].astype(np.float32), F32),
                                       to_dev(p, dtype) if with_partial else None, ks, to_dev(cw, F32),
                                       to_dev(q[0], F32), to_dev(g, F32), 1e-6, to_dev(mg, F32), to_dev(mw, F32), 1e-6)
    ref = oracle.msar_phase2(o1.astype(np.float64), lse[0].astype(np.float32).astype(np.float64), p, ks, cw, q[0], g,
                             1e-6, mg, mw, 1e-6)
    check_out(out, ref, dtype, np.abs(cached).max() * 3, strict=dtype == F32)


# --------------------------------------------------------------- backward of MSAR's two-phase schedule

def _check_all(got, ref, names, dtype, what):
    for name, g_, r_ in zip(names, got, ref):
        if r_ is None:
            assert g_ is None, name
            continue
        r_ = np.asarray(r_).reshape(tuple(g_.shape))
        check_out(g_, r_, dtype, np.abs(r_).max(), strict=False, chain=dtype == BF16, what=f"{what} {name}")


_P2B = ("d_o", "d_lse", "d_partial", "dconv_w", "dquery", "dgain", "dmix_gain", "dmix_w")


@pytest.mark.parametrize("dtype,T,d,with_partial", [(BF16, 60, 4096, True), (F32, 45, 1024, True),
                                                    (BF16, 33, 2048, False), (F32, 130, 1024, True),
                                                    (F32, 20, 2048, False)])
def test_msar_block_phase2_bwd(dtype, T, d, with_partial):
    """Phase 2's backward against the oracle on the same phase-1 state: the
    state's (o, lse), the partial's, the kernels', the stream queries', the
    gain's and the mixer's gradients; no partial passes dZ to o."""
    rng = _rng(T + d + 3 * with_partial)
    ks = (4, 8, 12)
    cached, parts, q, cw, mw, g, mg = _msar_block(rng, 4, 1, T, d, dtype, ks)
    o, lse = oracle.msar_phase1(cached, ks, cw, q, g, 1e-6)
    o1 = inputs.bf16_round(o[0].astype(np.float32)) if dtype == BF16 else o[0].astype(np.float32)
    l1 = lse[0].astype(np.float32)
    p = parts[0] if with_partial else None
    dh = _sources(rng, 1, T, d, dtype, step=0)[0]
    got = attnres.msar_block_phase2_bwd(to_dev(o1, dtype), to_dev(l1, F32), to_dev(p, dtype) if with_partial else None,
                                        ks, to_dev(cw, F32), to_dev(q[0], F32), to_dev(dh, dtype), to_dev(g, F32), 1e-6,
                                        to_dev(mg, F32), to_dev(mw, F32), 1e-6)
    ref = oracle.msar_phase2_bwd(o1.astype(np.float64), l1.astype(np.float64), p, ks, cw, q[0], dh, g, 1e-6, mg, mw,
                                 1e-6)
    _check_all(got, ref, _P2B, dtype, f"phase 2 T={T} d={d}")


@pytest.mark.parametrize("dtype,N,S,T,d", [(BF16, 8, 4, 60, 4096), (F32, 3, 2, 45, 1024), (BF16, 5, 6, 30, 2048),
                                           (BF16, 12, 3, 20, 512)])
def test_msar_block_phase1_bwd(dtype, N, S, T, d):
    """Phase 1's backward against the oracle for gradients of every layer's
    per-stream o and lse."""
    rng = _rng(N * 3 + S + T + d)
    ks = (4, 8, 12)
    cached, _, q, cw, _, g, _ = _msar_block(rng, N, S, T, d, dtype, ks)
    d_o = _sources(rng, S * 4, T, d, dtype, step=0).reshape(S, 4, T, d)
    d_l = rng.standard_normal((S, 4, T)).astype(np.float32)
    got = attnres.msar_block_phase1_bwd(to_dev(cached, dtype), ks, to_dev(cw, F32), to_dev(q, F32),
                                        to_dev(d_o, dtype), to_dev(d_l, F32), to_dev(g, F32), 1e-6)
    ref = oracle.msar_phase1_bwd(cached, ks, cw, q, d_o, d_l, g, 1e-6)
    _check_all(got, ref, ("dsrc", "dconv_w", "dqueries", "dgain"), dtype, f"phase 1 N={N} S={S} d={d}")


@pytest.mark.parametrize("dtype", [BF16, F32])
def test_msar_two_phase_bwd_chain_equals_one_shot(dtype):
    """The GPU chain (phase 2's backward of one layer, then phase 1's with its
    state gradients) against the oracle's backward of the one-shot MSAR read
    of [cached, partial]: every gradient, the two phases' shares added."""
    rng = _rng(123)
    N, T, d, ks = 4, 64, 2048, (4, 8, 12)
    cached, parts, q, cw, mw, g, mg = _msar_block(rng, N, 1, T, d, dtype, ks)
    dh = _sources(rng, 1, T, d, dtype, step=0)[0]
    dv = lambda x: to_dev(x, F32)
    src_d = to_dev(cached, dtype)
    o, lse = attnres.msar_block_phase1(src_d, ks, dv(cw), dv(q), dv(g), 1e-6)
    d_o, d_l, d_p, dcw2, dq2, dg2, dmg, dmw = attnres.msar_block_phase2_bwd(
        o[0], lse[0], to_dev(parts[0], dtype), ks, dv(cw), dv(q[0]), to_dev(dh, dtype), dv(g), 1e-6, dv(mg), dv(mw),
        1e-6)
    dsrc, dcw1, dq1, dg1 = attnres.msar_block_phase1_bwd(src_d, ks, dv(cw), dv(q), d_o[None], d_l[None], dv(g), 1e-6)
    r = oracle.msar_bwd(np.concatenate([cached, parts[0][None]]), ks, cw, q[0], dh, g, 1e-6, mg, mw, 1e-6)
    got = (torch.cat([dsrc, d_p[None]]), dcw1 + dcw2, dq1[0] + dq2, dg1 + dg2, dmg, dmw)
    _check_all(got, r, _MSAR_GRADS, dtype, "two-phase chain")


# --------------------------------------------------------------- hygiene

def test_outputs_stay_inside_their_buffers():
    """Canary bands around every output must be untouched."""
    rng = _rng(20)
    T, d, n_q, pad = 37, 2048, 4, 4096
    src = to_dev(_sources(rng, 8, T, d, BF16), BF16)
    q = to_dev(_queries(rng, n_q, d), F32)
    o_buf = torch.full((pad + n_q * T * d + pad,), 7.0, dtype=BF16, device="cuda")
    l_buf = torch.full((pad + n_q * T + pad,), 7.0, dtype=F32, device="cuda")
    o = o_buf[pad: pad + n_q * T * d].view(n_q, T, d)
    lse = l_buf[pad: pad + n_q * T].view(n_q, T)
    attnres.attnres_block_phase1(src, q, o=o, lse=lse)
    h_buf = torch.full((pad + T * d + pad,), 7.0, dtype=BF16, device="cuda")
    h = h_buf[pad: pad + T * d].view(T, d)
    attnres.attnres_block_phase2_merge(o[1], lse[1], src[0], q[1], out=h)
    m_buf = torch.full((pad + T * d + pad,), 7.0, dtype=BF16, device="cuda")
    x = inputs.msar_inputs(8, T, d, seed=1)
    attnres.msar_expand_fwd(src, x["ksizes"], to_dev(x["conv_w"], F32), to_dev(x["queries"], F32),
                            mix_w=to_dev(x["mix_w"], F32), out=m_buf[pad: pad + T * d].view(T, d))
    torch.cuda.synchronize()
    for buf in (o_buf, l_buf, h_buf, m_buf):
        assert torch.all(buf[:pad] == 7.0) and torch.all(buf[-pad:] == 7.0)


def test_runs_are_bitwise_deterministic():
    rng = _rng(21)
    T, d = 300, 4096
    src = to_dev(_sources(rng, 8, T, d, BF16), BF16)
    q = to_dev(_queries(rng, 4, d), F32)
    a1, l1 = attnres.attnres_block_phase1(src, q)
    a2, l2 = attnres.attnres_block_phase1(src, q)
    assert torch.equal(a1, a2) and torch.equal(l1, l2)
    x = inputs.msar_inputs(8, T, d, seed=2)
    args = (src, x["ksizes"], to_dev(x["conv_w"], F32), to_dev(x["queries"], F32))
    kw = dict(mix_w=to_dev(x["mix_w"], F32))
    assert torch.equal(attnres.msar_expand_fwd(*args, **kw), attnres.msar_expand_fwd(*args, **kw))


def test_calls_on_a_side_stream():
    rng = _rng(22)
    T, d = 64, 2048
    src_h = _sources(rng, 8, T, d, BF16)
    q_h = _queries(rng, 4, d)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        src = to_dev(src_h, BF16)
        q = to_dev(q_h, F32)
        o, lse = attnres.attnres_block_phase1(src, q, stream=s)
    s.synchronize()
    check_out(o, oracle.block_phase1(src_h, q_h)[0], BF16)


def test_empty_sequence_is_a_no_op():
    src = torch.empty((8, 16, 256), dtype=BF16, device="cuda")[:, :0, :]
    q = torch.zeros((4, 256), dtype=F32, device="cuda")
    o, lse = attnres.attnres_block_phase1(src, q)
    assert o.shape == (4, 0, 256)


def test_stall_injection_reports_timeout_and_context_survives():
    """A kernel whose copies never arrive gives up after the wait limit,
    records a timeout, and leaves the context usable (T above the few-token
    kernel's range, which loads without copies and waits)."""
    rng = _rng(23)
    T, d = 200, 2048
    src_h = _sources(rng, 8, T, d, BF16)
    q_h = _queries(rng, 4, d)
    src, q = to_dev(src_h, BF16), to_dev(q_h, F32)
    attnres.attnres_sync_status()
    try:
        attnres.attnres_debug_set_wait_timeout_ns(20_000_000)      # 20 ms
        attnres.attnres_debug_set_stall_injection(True)
        attnres.attnres_block_phase1(src, q)
        with pytest.raises(attnres.AttnResError) as e:
            attnres.attnres_sync_status()
        assert e.value.status == attnres.ERR_TIMEOUT
        x = inputs.msar_inputs(8, T, d, seed=3)
        attnres.msar_expand_fwd(src, x["ksizes"], to_dev(x["conv_w"], F32),
                                to_dev(x["queries"], F32), mix_w=to_dev(x["mix_w"], F32))
        with pytest.raises(attnres.AttnResError) as e:
            attnres.attnres_sync_status()
        assert e.value.status == attnres.ERR_TIMEOUT
    finally:
        attnres.attnres_debug_set_stall_injection(False)
        attnres.attnres_debug_set_wait_timeout_ns(0)
    o, lse = attnres.attnres_block_phase1(src, q)
    attnres.attnres_sync_status()
    check_out(o, oracle.block_phase1(src_h, q_h)[0], BF16)


# --------------------------------------------------------------- both kernels

@pytest.fixture(params=[0, 1, 2, 3], ids=["auto", "general", "tensor", "decode"])
def kernel_variant(request):
    """Runs a test with the automatic kernel choice, with the general CUDA-core
    kernel forced, with the tensor-core kernels wherever they apply and with the
    few-token (cluster per token) kernel wherever it applies."""
    attnres.attnres_debug_set_kernel_variant(request.param)
    yield request.param
    attnres.attnres_debug_set_kernel_variant(0)


@pytest.mark.parametrize("n_src,n_q,T,d", [(8, 4, 37, 4096), (8, 4, 150, 2048), (5, 3, 20, 1024),
                                           (1, 1, 9, 4096), (2, 2, 33, 2048), (7, 4, 64, 1024),
                                           (8, 1, 100, 4096)])
def test_phase1_both_kernels(kernel_variant, n_src, n_q, T, d):
    rng = _rng(n_src * 31 + n_q * 7 + T + d)
    src = _sources(rng, n_src, T, d, BF16)
    q = _queries(rng, n_q, d)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    o, lse = attnres.attnres_block_phase1(to_dev(src, BF16), to_dev(q, F32), to_dev(g, F32), 1e-6)
    ro, rl = oracle.block_phase1(src, q, g, 1e-6)
    check_out(o, ro, BF16, what="o")
    check_lse(lse, rl)


@pytest.mark.parametrize("H,d,T,n_src", [(8, 4096, 21, 8), (4, 4096, 13, 6), (2, 2048, 40, 8),
                                         (8, 2048, 17, 3), (4, 1024, 25, 8)])
def test_mhar_both_kernels(kernel_variant, H, d, T, n_src):
    rng = _rng(H * 13 + d + T)
    src = _sources(rng, n_src, T, d, BF16)
    q = (rng.standard_normal((4, H, d // H)) * math.sqrt(16.0 / (d // H))).astype(np.float32)
    out, lse = attnres.mhar_fwd(to_dev(src, BF16), to_dev(q, F32), want_lse=True)
    ro, rl = oracle.mhar(src, q, want_lse=True)
    check_out(out, ro, BF16)
    check_lse(lse, rl)


@pytest.fixture(params=[0, 1, 2, 3], ids=["auto", "general", "tensor", "decode"])
def kernel_variant3(request):
    """kernel_variant plus 2: the tensor-core kernels wherever they apply (the
    chunked one for every source count > 8 at d = 4096)."""
    attnres.attnres_debug_set_kernel_variant(request.param)
    yield request.param
    attnres.attnres_debug_set_kernel_variant(0)


@pytest.mark.parametrize("n_src,n_q,H,T,d", [(9, 1, 1, 700, 4096), (16, 4, 1, 50, 4096), (12, 3, 1, 170, 4096),
                                             (23, 2, 1, 400, 4096), (64, 1, 1, 160, 4096), (31, 1, 1, 300, 4096),
                                             (11, 4, 8, 40, 4096), (20, 4, 4, 33, 4096), (17, 1, 1, 1, 4096),
                                             (13, 2, 2, 90, 2048)])
def test_chunked_read_both_kernels(kernel_variant3, n_src, n_q, H, T, d):
    """More than 8 sources: chunks of 8 folded in by the online softmax; full
    and partial last chunks, several tokens per CTA, heads, a single token."""
    rng = _rng(n_src * 17 + n_q + H * 5 + T + d)
    src = _sources(rng, n_src, T, d, BF16, step=1 / 16)
    q = (rng.standard_normal((n_q, H, d // H)) * math.sqrt(16.0 / (d // H))).astype(np.float32)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    out, lse = attnres.mhar_fwd(to_dev(src, BF16), to_dev(q, F32), to_dev(g, F32), 1e-6, want_lse=True)
    ro, rl = oracle.mhar(src, q, g, 1e-6, want_lse=True)
    check_out(out, ro, BF16, np.abs(src).max())
    check_lse(lse, rl)


@pytest.mark.parametrize("dt,n_src,n_q,H,T,d", [(F32, 10, 1, 1, 45, 4096), (F32, 19, 2, 1, 70, 2048),
                                                (BF16, 25, 1, 1, 130, 1024), (BF16, 13, 1, 1, 77, 2048),
                                                (BF16, 20, 1, 1, 33, 256), (BF16, 14, 1, 4, 29, 4096),
                                                (BF16, 37, 3, 1, 19, 4096)])
def test_general_kernel_chunk_shapes(dt, n_src, n_q, H, T, d):
    """The general kernel's chunked reads at the chunk sizes its two-stage
    rule picks for each row width (3 sources per stage for 16 KB rows, 6 for
    8 KB, 8 for 4 KB): full and ragged last chunks, f32 and bf16, heads."""
    rng = _rng(n_src * 19 + n_q * 3 + H + T + d)
    src = _sources(rng, n_src, T, d, dt, step=1 / 16)
    q = (rng.standard_normal((n_q, H, d // H)) * math.sqrt(16.0 / (d // H))).astype(np.float32)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    attnres.attnres_debug_set_kernel_variant(1)
    try:
        out, lse = attnres.mhar_fwd(to_dev(src, dt), to_dev(q, F32), to_dev(g, F32), 1e-6, want_lse=True)
    finally:
        attnres.attnres_debug_set_kernel_variant(0)
    ro, rl = oracle.mhar(src, q, g, 1e-6, want_lse=True)
    check_out(out, ro, dt, np.abs(src).max())
    check_lse(lse, rl)


def test_chunked_read_keeps_non_finite_tokens_apart(kernel_variant3):
    """Tokens whose first chunk holds infinities get non-finite outputs; the
    rows that a partial last chunk leaves unloaded must not carry them into
    other tokens' reads."""
    rng = _rng(77)
    n_src, T, d = 9, 400, 4096
    src = _sources(rng, n_src, T, d, BF16, step=1 / 16)
    bad = np.arange(0, T, 5)
    src[1:8, bad, :] = np.inf
    w = _queries(rng, 1, d)[0]
    out = to_host(attnres.attnres_full_fwd(to_dev(src, BF16), to_dev(w, F32), None, 1e-6))
    good = np.setdiff1d(np.arange(T), bad)
    check_out(out[good], oracle.full(np.ascontiguousarray(src[:, good]), w, None, 1e-6), BF16)


@pytest.mark.parametrize("n_src,n_q,T,d,dtype", [(8, 4, 1, 4096, BF16), (16, 1, 3, 4096, BF16), (16, 2, 64, 2048, BF16),
                                                 (5, 3, 9, 1024, F32), (1, 1, 2, 256, BF16), (8, 1, 500, 4096, BF16),
                                                 (12, 1, 7, 512, F32)])
def test_decode_kernel(n_src, n_q, T, d, dtype):
    """The few-token kernel (a token per cluster of CTAs), forced for any T."""
    rng = _rng(n_src * 11 + n_q + T + d)
    src = _sources(rng, n_src, T, d, dtype, step=0.25)
    q = _queries(rng, n_q, d)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    attnres.attnres_debug_set_kernel_variant(3)
    try:
        o, lse = attnres.attnres_block_phase1(to_dev(src, dtype), to_dev(q, F32), to_dev(g, F32), 1e-6)
    finally:
        attnres.attnres_debug_set_kernel_variant(0)
    ro, rl = oracle.block_phase1(src, q, g, 1e-6)
    check_out(o, ro, dtype, np.abs(src).max(), what="o")
    check_lse(lse, rl)


def test_kernels_agree_closely():
    """The two kernels compute the same read; their bf16 outputs may differ by
    at most one rounding step."""
    rng = _rng(99)
    T, d = 200, 4096
    src = to_dev(_sources(rng, 8, T, d, BF16), BF16)
    q = to_dev(_queries(rng, 4, d), F32)
    o1, l1 = attnres.attnres_block_phase1(src, q)
    attnres.attnres_debug_set_kernel_variant(1)
    try:
        o2, l2 = attnres.attnres_block_phase1(src, q)
    finally:
        attnres.attnres_debug_set_kernel_variant(0)
    a, b = to_host(o1), to_host(o2)
    # one bf16 step of the larger value, plus float32 summation-order noise
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-4 * np.abs(a).max())
    assert np.abs(to_host(l1) - to_host(l2)).max() < 1e-4
