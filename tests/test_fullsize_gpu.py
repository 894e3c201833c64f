"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times.  Outputs are checked against the oracle on sampled tokens:
t = 0, t = T-1, t = 1..12 (the causal-convolution edge) and 300 tokens drawn
with seed 1.  Tokens are independent in every read except MSAR, whose oracle
is given the 12-row causal window that ends at each sampled token."""
import numpy as np
import pytest
import torch

from _helpers import check_lse, check_out, to_dev, to_host
from depth_wise_attention_gb300 import attnres, inputs
from oracle import oracle

pytestmark = pytest.mark.gpu
BF16, F32 = torch.bfloat16, torch.float32


def sampled_tokens(T, n=300):
    rng = np.random.default_rng(1)
    extra = rng.choice(T, size=min(n, T), replace=False)
    return np.unique(np.concatenate([[0, T - 1], np.arange(1, min(13, T)), extra]))


def rows(t, idx):
    """t [..., T, d] -> float64 numpy rows at token indices idx."""
    it = torch.from_numpy(idx).to(t.device)
    return t.index_select(t.dim() - 2, it).float().cpu().numpy().astype(np.float64)


def test_full_fp32_T256_d256_L8():
    x = inputs.full_inputs(8, 256, 256, seed=0, std_step=0.25)
    out = attnres.attnres_full_fwd(to_dev(x["src"], F32), to_dev(x["query"], F32),
                                   to_dev(x["gain"], F32), x["eps"])
    ref = oracle.full(x["src"], x["query"], x["gain"], x["eps"])
    check_out(out, ref, F32, np.abs(x["src"]).max())


@pytest.mark.parametrize("all_partials", [False, True])
def test_block_two_phase_T8192_d2048(all_partials):
    """Default: layer 1 reads no partial (summary section 2; tutorial Fig. 4);
    all_partials=True covers the other reading of 'per-layer partial sums'."""
    N, S, T, d = 8, 4, 8192, 2048
    x = inputs.block_inputs(N, S, T, d, seed=0)
    cache, q, parts = to_dev(x["cache"], BF16), to_dev(x["queries"], F32), to_dev(x["partials"], BF16)
    o, lse = attnres.attnres_block_phase1(cache, q)
    first = 0 if all_partials else 1
    for i in range(first, S):
        attnres.attnres_block_phase2_merge(o[i], lse[i], parts[i], q[i], out=o[i])
    attnres.attnres_sync_status()
    idx = sampled_tokens(T)
    c = x["cache"][:, idx, :].astype(np.float64)
    p = x["partials"][:, idx, :].astype(np.float64)
    if all_partials:
        ref = np.stack([oracle.full(np.concatenate([c, p[i:i + 1]]), x["queries"][i])
                        for i in range(S)])
    else:
        ref = oracle.block_oneshot(c, p, x["queries"])
    check_out(rows(o, idx), ref, BF16)


def _device_block(T, d, N=8, S=4, seed=0):
    cache, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=seed)
    cache = cache.view(N, T, d)
    q = inputs.device_normal((S, d), (16.0 / d) ** 0.5, g)
    parts = torch.empty((S, T, d), dtype=BF16, device="cuda")
    for i in range(S):
        parts[i].copy_(torch.randn((T, d), generator=g, device="cuda"))
    return cache, q, parts


def test_block_two_phase_T32768_d4096_bench_workload():
    T, d, N, S = 32768, 4096, 8, 4
    cache, q, parts = _device_block(T, d, N, S)
    o = torch.empty((S, T, d), dtype=BF16, device="cuda")
    lse = torch.empty((S, T), dtype=F32, device="cuda")
    attnres.attnres_block_phase1(cache, q, o=o, lse=lse)
    idx = sampled_tokens(T)
    lse_ph1 = lse[:, torch.from_numpy(idx).cuda()].cpu().numpy()
    for i in range(1, S):
        attnres.attnres_block_phase2_merge(o[i], lse[i], parts[i], q[i], out=o[i])
    attnres.attnres_sync_status()
    c, p = rows(cache, idx), rows(parts, idx)
    qh = q.cpu().numpy().astype(np.float64)
    check_out(rows(o, idx), oracle.block_oneshot(c, p, qh), BF16)
    check_lse(lse_ph1, oracle.block_phase1(c, qh)[1])


def test_block_fused_update_T32768_d4096_bench_workload():
    """The bench's fused schedule: phase 1, then layers 2..4 each add the
    previous layer's output to the partial and merge it in one call.  Layer i
    merges the stored partial plus f_{i-1} summed exactly; the stored partial is
    that sum rounded to bf16."""
    T, d, N, S = 32768, 4096, 8, 4
    cache, q, f = _device_block(T, d, N, S)
    o = torch.empty((S, T, d), dtype=BF16, device="cuda")
    lse = torch.empty((S, T), dtype=F32, device="cuda")
    p = torch.empty((T, d), dtype=BF16, device="cuda")
    attnres.attnres_block_phase1(cache, q, o=o, lse=lse)
    idx = sampled_tokens(T)
    c, fh = rows(cache, idx), rows(f, idx)
    stored = np.zeros_like(fh[0])
    partials = np.zeros_like(fh)
    for i in range(1, S):
        attnres.attnres_block_phase2_update_merge(p if i > 1 else None, f[i - 1], o[i], lse[i], q[i],
                                                  partial_out=p, out=o[i])
        partials[i] = stored + fh[i - 1]
        stored = inputs.bf16_round(partials[i].astype(np.float32)).astype(np.float64)
    attnres.attnres_sync_status()
    qh = q.cpu().numpy().astype(np.float64)
    check_out(rows(o, idx), oracle.block_oneshot(c, partials, qh), BF16)
    check_out(rows(p, idx), stored, BF16, what="partial")


def test_full_at_depth_T16384_d4096_L64():
    """Layer l = 1..64 reads sources 0..l-1, one call per layer in order."""
    T, d, L = 16384, 4096, 64
    src, g = inputs.device_sources(L, T, d, lambda i: 1.0 + i / 16.0, seed=0)
    src = src.view(L, T, d)
    q = inputs.device_normal((L, d), (16.0 / d) ** 0.5, g)
    out = torch.empty((T, d), dtype=BF16, device="cuda")
    idx = sampled_tokens(T, n=24)
    s_h = rows(src, idx)
    q_h = q.cpu().numpy().astype(np.float64)
    for l in range(1, L + 1):
        attnres.attnres_full_fwd(src[:l], q[l - 1], None, 1e-6, out=out)
        if l in (1, 2, 7, 8, 9, 16, 17, 24, 29, 33, 45, 63, 64):
            check_out(rows(out, idx), oracle.full(s_h[:l], q_h[l - 1]), BF16, what=f"layer {l}")
    attnres.attnres_sync_status()


def test_mhar_T131072_d4096_H8():
    T, d, N, S, H = 131072, 4096, 8, 4, 8
    src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=0)
    src = src.view(N, T, d)
    q = inputs.device_normal((S, H, d // H), (16.0 / (d // H)) ** 0.5, g)
    out, lse = attnres.mhar_fwd(src, q, want_lse=True)
    idx = sampled_tokens(T)
    ro, rl = oracle.mhar(rows(src, idx), q.cpu().numpy().astype(np.float64), want_lse=True)
    check_out(rows(out, idx), ro, BF16)
    check_lse(lse[:, :, torch.from_numpy(idx).cuda()].cpu().numpy(), rl)
    # H = 1 is AttnRes exactly: the same kernel as phase 1, bit for bit
    del out, lse
    q1 = inputs.device_normal((S, 1, d), (16.0 / d) ** 0.5, g)
    m1 = attnres.mhar_fwd(src, q1)
    o1, _ = attnres.attnres_block_phase1(src, q1.view(S, d), want_lse=False)
    assert torch.equal(m1, o1)


def test_mhar_two_phase_T131072_d4096_H8():
    """MHAR inside the two-phase schedule at the MHAR size: mhar_fwd (phase 1,
    lse per head) and the per-head merge of a partial per query equal the
    one-shot MHAR read over the reps plus the partial."""
    T, d, N, S, H = 131072, 4096, 8, 4, 8
    src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=0)
    src = src.view(N, T, d)
    q = inputs.device_normal((S, H, d // H), (16.0 / (d // H)) ** 0.5, g)
    part = torch.randn((T, d), generator=g, device="cuda").to(BF16)
    out, lse = attnres.mhar_fwd(src, q, want_lse=True)
    for i in range(1, S):
        attnres.mhar_phase2_merge(out[i], lse[i], part, q[i], out=out[i])
    attnres.attnres_sync_status()
    idx = sampled_tokens(T)
    s_h, p_h = rows(src, idx), rows(part, idx)
    q_h = q.cpu().numpy().astype(np.float64)
    got = rows(out, idx)
    check_out(got[0], oracle.mhar(s_h, q_h[:1])[0], BF16, what="layer 1")
    ref = oracle.mhar(np.concatenate([s_h, p_h[None]]), q_h[1:])
    check_out(got[1:], ref, BF16)


def test_mhar_read_bwd_T131072_d4096_H8_bench_workload():
    """The MHAR backward at the MHAR size (4 queries, two passes): source
    gradients on sampled tokens against the oracle; the query and gain
    gradients (sums over all tokens) equal the sums of the two halves'."""
    T, d, N, S, H = 131072, 4096, 8, 4, 8
    src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=0)
    src = src.view(N, T, d)
    q = inputs.device_normal((S, H, d // H), (16.0 / (d // H)) ** 0.5, g)
    gain = torch.ones((d,), dtype=F32, device="cuda")
    dout = torch.randn((S, T, d), generator=g, device="cuda").to(BF16)
    dsrc, dq, dg = attnres.mhar_read_bwd(src, q, dout, gain)
    attnres.attnres_sync_status()
    idx = sampled_tokens(T)
    ref = oracle.mhar_bwd(rows(src, idx), q.cpu().numpy().astype(np.float64), rows(dout, idx), None, 1e-6)
    check_out(rows(dsrc, idx), ref[0], BF16, what="dsrc")
    del dsrc
    h = T // 2
    parts = [attnres.mhar_read_bwd(src[:, a:b].contiguous(), q, dout[:, a:b].contiguous(), gain, dsrc=None)[1:]
             for a, b in ((0, h), (h, T))]
    for name, whole, (x, y) in (("dq", dq, (parts[0][0], parts[1][0])), ("dgain", dg, (parts[0][1], parts[1][1]))):
        w, s_ = to_host(whole), to_host(x) + to_host(y)
        assert np.abs(w - s_).max() <= 1e-4 * np.abs(w).max(), name


def test_msar_T32768_d4096():
    T, d, N = 32768, 4096, 8
    ks = (4, 8, 12)
    src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=0)
    src = src.view(N, T, d)
    q = inputs.device_normal((4, d), (16.0 / d) ** 0.5, g)
    cw = torch.cat([inputs.device_normal((d * k,), (1.0 / k) ** 0.5, g) for k in ks])
    mw = inputs.device_normal((4 * d, 4), (1.0 / (4 * d)) ** 0.5, g)
    out = attnres.msar_expand_fwd(src, ks, cw, q, None, 1e-6, None, mw, 1e-6)
    attnres.attnres_sync_status()
    idx = sampled_tokens(T, n=150)
    cw_h, q_h, mw_h = (t.cpu().numpy().astype(np.float64) for t in (cw, q, mw))
    got = rows(out, idx)
    ref = np.empty_like(got)
    for j, t in enumerate(idx):
        lo = max(0, int(t) - 11)
        win = src[:, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64)
        ref[j] = oracle.msar(win, ks, cw_h, q_h, None, 1e-6, None, mw_h, 1e-6)[-1]
    check_out(got, ref, BF16)


def test_msar_two_phase_T32768_d4096_bench_workload():
    """MSAR in the two-phase Block schedule at the MSAR size (N=8 cached
    sources, S=4 layers): phase 1 for the block, phase 2 per layer with its
    partial (layer 1 without), each layer's output against the oracle's
    one-shot MSAR read of the 12-row causal window of [cached, partial]."""
    T, d, N, S = 32768, 4096, 8, 4
    ks = (4, 8, 12)
    src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=0)
    src = src.view(N, T, d)
    q = inputs.device_normal((S, 4, d), (16.0 / d) ** 0.5, g)
    cw = torch.cat([inputs.device_normal((d * k,), (1.0 / k) ** 0.5, g) for k in ks])
    mw = inputs.device_normal((4 * d, 4), (1.0 / (4 * d)) ** 0.5, g)
    parts = torch.randn((S, T, d), generator=g, device="cuda").to(BF16)
    o, lse = attnres.msar_block_phase1(src, ks, cw, q)
    outs = [attnres.msar_block_phase2(o[s_], lse[s_], parts[s_] if s_ > 0 else None, ks, cw, q[s_], None, 1e-6,
                                      None, mw, 1e-6) for s_ in range(S)]
    attnres.attnres_sync_status()
    idx = sampled_tokens(T, n=60)
    cw_h, q_h, mw_h = (t.cpu().numpy().astype(np.float64) for t in (cw, q, mw))
    for s_ in range(S):
        got = rows(outs[s_], idx)
        ref = np.empty_like(got)
        for j, t in enumerate(idx):
            lo = max(0, int(t) - 11)
            win = src[:, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64)
            if s_ > 0:
                pw = parts[s_, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64)
                win = np.concatenate([win, pw[None]])
            ref[j] = oracle.msar(win, ks, cw_h, q_h[s_], None, 1e-6, None, mw_h, 1e-6)[-1]
        # The phase-1 state is stored in bf16 and the mixer adds up to 4
        # rounded streams with weights that need not sum to 1, so where the
        # streams cancel, an element's relative error can exceed the
        # elementwise bound of one rounding; the bf16 tolerance on the
        # output's scale (2e-2 of max |ref|) is the bar here.
        check_out(got, ref, BF16, chain=True, what=f"layer {s_ + 1}")


def test_block_two_phase_backward_T32768_d4096():
    """The backward of the headline Block step at full size: each layer's
    merge backward (layers 2..4 with their partials, layer 1 without), then
    phase 1's backward for all four layers' d_o and d_lse.  Sampled tokens'
    source and partial gradients against the oracle's backward of the
    one-shot reads."""
    T, d, N, S = 32768, 4096, 8, 4
    cache, q, parts = _device_block(T, d, N, S)
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    dh = torch.randn((S, T, d), generator=g, device="cuda").to(BF16)
    o, lse = attnres.attnres_block_phase1(cache, q)
    d_o, d_lse = torch.empty_like(o), torch.empty_like(lse)
    dparts = []
    for s_ in range(S):
        r = attnres.attnres_block_phase2_bwd(o[s_], lse[s_], parts[s_] if s_ > 0 else None, q[s_], dh[s_],
                                             d_o=d_o[s_], d_lse=d_lse[s_])
        dparts.append(r[2])
    dsrc, _, _ = attnres.attnres_block_phase1_bwd(cache, q, d_o, d_lse)
    attnres.attnres_sync_status()
    idx = sampled_tokens(T)
    c, p, h = rows(cache, idx), rows(parts, idx), rows(dh, idx)
    qh = q.cpu().numpy().astype(np.float64)
    ref_cached = np.zeros_like(c)
    for s_ in range(S):
        srcs = c if s_ == 0 else np.concatenate([c, p[s_][None]])
        rs, _, _ = oracle.read_bwd(srcs, qh[s_][None], h[s_][None], None, 1e-6)
        ref_cached += rs[:N]
        if s_ > 0:
            check_out(rows(dparts[s_], idx), rs[N], BF16, chain=True, what=f"layer {s_ + 1} d_partial")
    check_out(rows(dsrc, idx), ref_cached, BF16, chain=True, what="cached sources' gradient")


def test_msar_per_source_and_chunked_T32768_d4096():
    """MSAR at the MSAR size with each source's own kernels (sampled tokens
    against the oracle on causal windows), and the chunked prefill of the
    shared-kernel read (8 chunks of 4096 with 11 history rows) equal to the
    one-call read bit for bit."""
    T, d, N = 32768, 4096, 8
    ks = (4, 8, 12)
    src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=0)
    src = src.view(N, T, d)
    q = inputs.device_normal((4, d), (16.0 / d) ** 0.5, g)
    mw = inputs.device_normal((4 * d, 4), (1.0 / (4 * d)) ** 0.5, g)
    cw = torch.stack([torch.cat([inputs.device_normal((d * k,), (1.0 / k) ** 0.5, g) for k in ks]) for _ in range(N)])
    out = attnres.msar_expand_fwd_ps(src, ks, cw, q, None, 1e-6, None, mw, 1e-6)
    attnres.attnres_sync_status()
    idx = sampled_tokens(T, n=60)
    cw_h, q_h, mw_h = (t.cpu().numpy().astype(np.float64) for t in (cw, q, mw))
    got = rows(out, idx)
    ref = np.empty_like(got)
    for j, t in enumerate(idx):
        lo = max(0, int(t) - 11)
        win = src[:, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64)
        ref[j] = oracle.msar_ps(win, ks, cw_h, q_h, None, 1e-6, None, mw_h, 1e-6)[-1]
    check_out(got, ref, BF16, what="per-source kernels")
    del out
    shared_cw = cw[0].contiguous()
    whole = attnres.msar_expand_fwd(src, ks, shared_cw, q, None, 1e-6, None, mw, 1e-6)
    chunked = torch.empty_like(whole)
    for c0 in range(0, T, 4096):
        h = min(11, c0)
        attnres.msar_expand_fwd_chunk(src[:, c0 - h:c0 + 4096], h, ks, shared_cw, q, None, 1e-6, None, mw, 1e-6,
                                      out=chunked[c0:c0 + 4096])
    assert torch.equal(whole, chunked)


def test_read_bwd_T32768_d4096_bench_workload():
    """The backward of a Block layer's read at the bench size (9 sources, 1
    query): sampled source gradients against the oracle; the query and gain
    gradients equal the sums of the two halves' runs."""
    T, d, N = 32768, 4096, 8
    src, g = inputs.device_sources(N + 1, T, d, lambda n: 1.0 + n / 2.0 if n < N else 1.0, seed=0)
    src = src.view(N + 1, T, d)
    q = inputs.device_normal((1, d), (16.0 / d) ** 0.5, g)
    gain = torch.ones((d,), dtype=F32, device="cuda")
    dout = torch.randn((1, T, d), generator=g, device="cuda").to(BF16)
    dsrc, dq, dg = attnres.attnres_read_bwd(src, q, dout, gain)
    attnres.attnres_sync_status()
    idx = sampled_tokens(T)
    ref = oracle.read_bwd(rows(src, idx), q.cpu().numpy().astype(np.float64), rows(dout, idx), None, 1e-6)
    check_out(rows(dsrc, idx), ref[0], BF16, what="dsrc")
    del dsrc
    h = T // 2
    parts = [attnres.attnres_read_bwd(src[:, a:b].contiguous(), q, dout[:, a:b].contiguous(), gain)[1:]
             for a, b in ((0, h), (h, T))]
    for name, whole, (x, y) in (("dq", dq, (parts[0][0], parts[1][0])), ("dgain", dg, (parts[0][1], parts[1][1]))):
        w, s_ = to_host(whole), to_host(x) + to_host(y)
        assert np.abs(w - s_).max() <= 1e-4 * np.abs(w).max(), name


def test_read_bwd_64_sources_T16384_d4096():
    """The backward of the deepest layer of Full AttnRes at depth (64 sources,
    T = 16384, d = 4096, bf16), past one pass of the backward kernel: sampled
    source gradients against the oracle; the query and gain gradients equal
    the sums of the two halves' runs."""
    T, d, L = 16384, 4096, 64
    src, g = inputs.device_sources(L, T, d, lambda n: 1.0 + n / 16.0, seed=4)
    src = src.view(L, T, d)
    q = inputs.device_normal((1, d), (16.0 / d) ** 0.5, g)
    gain = torch.ones((d,), dtype=F32, device="cuda")
    dout = torch.randn((1, T, d), generator=g, device="cuda").to(BF16)
    dsrc, dq, dg = attnres.attnres_read_bwd(src, q, dout, gain)
    attnres.attnres_sync_status()
    idx = sampled_tokens(T, n=100)
    ref = oracle.read_bwd(rows(src, idx), q.cpu().numpy().astype(np.float64), rows(dout, idx), None, 1e-6)
    check_out(rows(dsrc, idx), ref[0], BF16, what="dsrc")
    del dsrc
    h = T // 2
    parts = [attnres.attnres_read_bwd(src[:, a:b].contiguous(), q, dout[:, a:b].contiguous(), gain)[1:]
             for a, b in ((0, h), (h, T))]
    for name, whole, (x, y) in (("dq", dq, (parts[0][0], parts[1][0])), ("dgain", dg, (parts[0][1], parts[1][1]))):
        w, s_ = to_host(whole), to_host(x) + to_host(y)
        assert np.abs(w - s_).max() <= 1e-4 * np.abs(w).max(), name


def test_msar_bwd_T32768_d4096():
    """Backward of the MSAR read at the MSAR size.  Every gradient is linear
    in dh and the read of token t sees source rows t-11..t only, so with dh
    nonzero on a few clusters of 4 tokens each gradient is the sum of the
    oracle's backward over the clusters' 15-row causal windows, and dsrc is
    exactly zero outside them.  Clusters at the start, across a boundary of
    the conv kernels' token chunks, in the middle and at the end.  Then a
    dense dh: two calls agree bit for bit."""
    T, d, N = 32768, 4096, 8
    ks = (4, 8, 12)
    src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=0)
    src = src.view(N, T, d)
    q = inputs.device_normal((4, d), (16.0 / d) ** 0.5, g)
    cw = torch.cat([inputs.device_normal((d * k,), (1.0 / k) ** 0.5, g) for k in ks])
    mw = inputs.device_normal((4 * d, 4), (1.0 / (4 * d)) ** 0.5, g)
    starts = [0, 3275, 17001, T - 4]
    dh = torch.zeros((T, d), dtype=BF16, device="cuda")
    for c in starts:
        dh[c:c + 4] = torch.randn((4, d), generator=g, device="cuda").to(BF16)
    got = attnres.msar_expand_bwd(src, ks, cw, q, dh, None, 1e-6, None, mw, 1e-6)
    attnres.attnres_sync_status()
    cw_h, q_h, mw_h = (t.cpu().numpy().astype(np.float64) for t in (cw, q, mw))
    ref_par = None
    inside = torch.zeros(T, dtype=torch.bool, device="cuda")
    for c in starts:
        lo = max(0, c - 11)
        win = src[:, lo:c + 4, :].float().cpu().numpy().astype(np.float64)
        dwin = dh[lo:c + 4].float().cpu().numpy().astype(np.float64)
        r = oracle.msar_bwd(win, ks, cw_h, q_h, dwin, None, 1e-6, None, mw_h, 1e-6)
        check_out(got[0][:, lo:c + 4], r[0], BF16, chain=True, what=f"dsrc rows {lo}..{c + 3}")
        inside[lo:c + 4] = True
        ref_par = list(r[1:]) if ref_par is None else [a + b for a, b in zip(ref_par, r[1:])]
    assert torch.count_nonzero(got[0][:, ~inside]) == 0
    for name, g_, r_ in zip(("dconv_w", "dqueries", "dgain", "dmix_gain", "dmix_w"), got[1:], ref_par):
        check_out(g_, np.asarray(r_).reshape(tuple(g_.shape)), BF16, chain=True, what=name)
    del got
    dense = torch.randn((T, d), generator=g, device="cuda").to(BF16)
    a = attnres.msar_expand_bwd(src, ks, cw, q, dense, None, 1e-6, None, mw, 1e-6)
    b = attnres.msar_expand_bwd(src, ks, cw, q, dense, None, 1e-6, None, mw, 1e-6)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_msar_bwd_chunked_T32768_d4096():
    """The MSAR backward at the MSAR size in 8 chunks of 4096 tokens, each
    with its 11 history rows, against the one-call backward: dsrc within the
    bf16 elementwise bound (one more rounding of each chunk's history rows),
    the parameter gradients within 2e-3 of their largest value; the chunk
    workspace is an eighth of the one-call workspace (plus fixed parts)."""
    T, d, N, chunk = 32768, 4096, 8, 4096
    ks = (4, 8, 12)
    src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=2)
    src = src.view(N, T, d)
    q = inputs.device_normal((4, d), (16.0 / d) ** 0.5, g)
    cw = torch.cat([inputs.device_normal((d * k,), (1.0 / k) ** 0.5, g) for k in ks])
    mw = inputs.device_normal((4 * d, 4), (1.0 / (4 * d)) ** 0.5, g)
    dh = torch.randn((T, d), generator=g, device="cuda").to(BF16)
    one = attnres.msar_expand_bwd(src, ks, cw, q, dh, None, 1e-6, None, mw, 1e-6)
    ws_one = attnres.msar_expand_bwd_workspace_size(N, T, d, BF16, ks)
    ws_chunk = attnres.msar_expand_bwd_workspace_size(N, chunk, d, BF16, ks)
    assert ws_chunk * 6 < ws_one
    dsrc = torch.empty_like(src)
    grads = (torch.empty_like(cw), torch.empty((4, d), device="cuda"), torch.empty((d,), device="cuda"),
             torch.empty((4 * d,), device="cuda"), torch.empty((4 * d, 4), device="cuda"))
    ws = torch.empty((ws_chunk + 3) // 4, dtype=torch.float32, device="cuda")
    for c0 in range(0, T, chunk):
        h = min(11, c0)
        attnres.msar_expand_bwd_chunk(src[:, c0 - h:c0 + chunk], h, ks, cw, q, dh[c0:c0 + chunk],
                                      dsrc[:, c0 - h:c0 + chunk], grads, c0 > 0, None, 1e-6, None, mw, 1e-6,
                                      workspace=ws)
    attnres.attnres_sync_status()
    a, b = dsrc.float(), one[0].float()
    bmax = b.abs().max()
    assert bool(((a - b).abs() <= 2.0 ** -7 * b.abs() + 2e-3 * bmax).all())
    for name, x, y in zip(("dconv_w", "dqueries", "dgain", "dmix_gain", "dmix_w"), grads, one[1:]):
        assert float((x - y).abs().max()) <= 2e-3 * float(y.abs().max()), name


def test_msar_bwd_per_source_T32768_d4096():
    """The backward with each source's own kernels at the MSAR size, by the
    same construction as the shared-kernel test: dh on a few clusters of 4
    tokens, every gradient (each source's kernel gradient on its own) against
    the oracle's per-source backward over the clusters' causal windows."""
    T, d, N = 32768, 4096, 8
    ks = (4, 8, 12)
    src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=0)
    src = src.view(N, T, d)
    q = inputs.device_normal((4, d), (16.0 / d) ** 0.5, g)
    cw = torch.stack([torch.cat([inputs.device_normal((d * k,), (1.0 / k) ** 0.5, g) for k in ks]) for _ in range(N)])
    mw = inputs.device_normal((4 * d, 4), (1.0 / (4 * d)) ** 0.5, g)
    starts = [0, 9000, T - 4]
    dh = torch.zeros((T, d), dtype=BF16, device="cuda")
    for c in starts:
        dh[c:c + 4] = torch.randn((4, d), generator=g, device="cuda").to(BF16)
    got = attnres.msar_expand_bwd_ps(src, ks, cw, q, dh, None, 1e-6, None, mw, 1e-6)
    attnres.attnres_sync_status()
    cw_h, q_h, mw_h = (t.cpu().numpy().astype(np.float64) for t in (cw, q, mw))
    ref_par = None
    inside = torch.zeros(T, dtype=torch.bool, device="cuda")
    for c in starts:
        lo = max(0, c - 11)
        win = src[:, lo:c + 4, :].float().cpu().numpy().astype(np.float64)
        dwin = dh[lo:c + 4].float().cpu().numpy().astype(np.float64)
        r = oracle.msar_ps_bwd(win, ks, cw_h, q_h, dwin, None, 1e-6, None, mw_h, 1e-6)
        check_out(got[0][:, lo:c + 4], r[0], BF16, chain=True, what=f"dsrc rows {lo}..{c + 3}")
        inside[lo:c + 4] = True
        ref_par = list(r[1:]) if ref_par is None else [a + b for a, b in zip(ref_par, r[1:])]
    assert torch.count_nonzero(got[0][:, ~inside]) == 0
    for name, g_, r_ in zip(("dconv_w", "dqueries", "dgain", "dmix_gain", "dmix_w"), got[1:], ref_par):
        check_out(g_, np.asarray(r_).reshape(tuple(g_.shape)), BF16, chain=True, what=name)


def test_msar_workspace_chain_T32768_d4096():
    """The MSAR read and the MSAR two-phase block through the workspace chains
    at the MSAR size: sampled tokens of the read against the oracle on causal
    windows, and the chains' phase 1 followed by each layer's phase 2 against
    the one-shot oracle read of the cached sources plus the layer's
    partial."""
    T, d, N, S = 32768, 4096, 8, 4
    ks = (4, 8, 12)
    src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=0)
    src = src.view(N, T, d)
    q = inputs.device_normal((4, d), (16.0 / d) ** 0.5, g)
    cw = torch.cat([inputs.device_normal((d * k,), (1.0 / k) ** 0.5, g) for k in ks])
    mw = inputs.device_normal((4 * d, 4), (1.0 / (4 * d)) ** 0.5, g)
    out = attnres.msar_expand_fwd_ws(src, ks, cw, q, None, 1e-6, None, mw, 1e-6)
    attnres.attnres_sync_status()
    idx = sampled_tokens(T, n=100)
    cw_h, q_h, mw_h = (t.cpu().numpy().astype(np.float64) for t in (cw, q, mw))
    got = rows(out, idx)
    ref = np.empty_like(got)
    for j, t in enumerate(idx):
        lo = max(0, int(t) - 11)
        win = src[:, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64)
        ref[j] = oracle.msar(win, ks, cw_h, q_h, None, 1e-6, None, mw_h, 1e-6)[-1]
    check_out(got, ref, BF16, chain=True, what="workspace-chain read")
    del out
    qs = inputs.device_normal((S, 4, d), (16.0 / d) ** 0.5, g)
    parts = torch.randn((S, T, d), generator=g, device="cuda").to(BF16)
    o, lse = attnres.msar_block_phase1_ws(src, ks, cw, qs)
    outs = [attnres.msar_block_phase2_ws(o[s_], lse[s_], parts[s_] if s_ > 0 else None, ks, cw, qs[s_], None, 1e-6,
                                         None, mw, 1e-6) for s_ in range(S)]
    attnres.attnres_sync_status()
    idx = sampled_tokens(T, n=40)
    qs_h = qs.cpu().numpy().astype(np.float64)
    for s_ in range(S):
        got = rows(outs[s_], idx)
        ref = np.empty_like(got)
        for j, t in enumerate(idx):
            lo = max(0, int(t) - 11)
            win = src[:, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64)
            if s_ > 0:
                pw = parts[s_, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64)
                win = np.concatenate([win, pw[None]])
            ref[j] = oracle.msar(win, ks, cw_h, qs_h[s_], None, 1e-6, None, mw_h, 1e-6)[-1]
        check_out(got, ref, BF16, chain=True, what=f"layer {s_ + 1} through the workspace chains")


def test_msar_two_phase_bwd_T32768_d4096():
    """The backward of one MSAR two-phase layer at the MSAR size (N=8 cached
    sources, T=32768), phase 2 then phase 1, with dh on three clusters of 4
    tokens: every gradient against the oracle's one-shot backward of
    [cached, partial] over the clusters' 15-row causal windows (the backward
    is linear in dh and a token's read sees rows t-11..t), and the sources'
    and the partial's gradients exactly zero elsewhere."""
    T, d, N = 32768, 4096, 8
    ks = (4, 8, 12)
    src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=0)
    src = src.view(N, T, d)
    q = inputs.device_normal((1, 4, d), (16.0 / d) ** 0.5, g)
    cw = torch.cat([inputs.device_normal((d * k,), (1.0 / k) ** 0.5, g) for k in ks])
    mw = inputs.device_normal((4 * d, 4), (1.0 / (4 * d)) ** 0.5, g)
    part = torch.randn((T, d), generator=g, device="cuda").to(BF16)
    starts = [0, 12345, T - 4]
    dh = torch.zeros((T, d), dtype=BF16, device="cuda")
    for c in starts:
        dh[c:c + 4] = torch.randn((4, d), generator=g, device="cuda").to(BF16)
    o, lse = attnres.msar_block_phase1(src, ks, cw, q)
    d_o, d_l, d_p, dcw2, dq2, dg2, dmg, dmw = attnres.msar_block_phase2_bwd(o[0], lse[0], part, ks, cw, q[0], dh,
                                                                            None, 1e-6, None, mw, 1e-6)
    del o, lse
    dsrc, dcw1, dq1, dg1 = attnres.msar_block_phase1_bwd(src, ks, cw, q, d_o[None], d_l[None])
    attnres.attnres_sync_status()
    cw_h, q_h, mw_h = (t.cpu().numpy().astype(np.float64) for t in (cw, q[0], mw))
    ref_par = None
    inside = torch.zeros(T, dtype=torch.bool, device="cuda")
    for c in starts:
        lo = max(0, c - 11)
        win = torch.cat([src[:, lo:c + 4], part[None, lo:c + 4]]).float().cpu().numpy().astype(np.float64)
        dwin = dh[lo:c + 4].float().cpu().numpy().astype(np.float64)
        r = oracle.msar_bwd(win, ks, cw_h, q_h, dwin, None, 1e-6, None, mw_h, 1e-6)
        check_out(dsrc[:, lo:c + 4], r[0][:N], BF16, chain=True, what=f"dsrc rows {lo}..{c + 3}")
        check_out(d_p[lo:c + 4], r[0][N], BF16, chain=True, what=f"d_partial rows {lo}..{c + 3}")
        inside[lo:c + 4] = True
        ref_par = list(r[1:]) if ref_par is None else [a + b for a, b in zip(ref_par, r[1:])]
    assert torch.count_nonzero(dsrc[:, ~inside]) == 0 and torch.count_nonzero(d_p[~inside]) == 0
    got = (dcw1 + dcw2, dq1[0] + dq2, dg1 + dg2, dmg, dmw)
    for name, g_, r_ in zip(("dconv_w", "dqueries", "dgain", "dmix_gain", "dmix_w"), got, ref_par):
        check_out(g_, np.asarray(r_).reshape(tuple(g_.shape)), BF16, chain=True, what=name)
