"""The no-allocation backward entry point (built-in scratch instead of a
caller workspace), for callers that cannot give the library device memory.

It is checked against the workspace entry point, which runs the same kernels,
so the results must agree bit for bit, on two consecutive calls (the second
reuses the scratch the first left behind).  The outputs are allocated before
the call, so the device's free memory must not change across it.  This file
is collected last, so a run that stops at the first failure has run every
other test first."""
import numpy as np
import pytest
import torch

from depth_wise_attention_gb300 import attnres

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


def _outputs(n_src, n_q, T, d, dtype):
    return (torch.empty((n_src, T, d), dtype=dtype, device="cuda"),
            torch.empty((n_q, d), dtype=torch.float32, device="cuda"),
            torch.empty((d,), dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("n_src,n_q,T,d,dtype", [(9, 1, 300, 4096, torch.bfloat16), (5, 2, 77, 512, torch.float32)])
def test_noalloc_backward_matches_workspace_backward_on_two_calls(n_src, n_q, T, d, dtype):
    g = torch.Generator(device="cuda").manual_seed(n_src + T)
    for call in range(2):
        src = (torch.randn((n_src, T, d), generator=g, device="cuda") * (1 + call)).to(dtype)
        q = torch.randn((n_q, d), generator=g, device="cuda") * (16.0 / d) ** 0.5
        gain = torch.rand((d,), generator=g, device="cuda") + 0.5
        dout = torch.randn((n_q, T, d), generator=g, device="cuda").to(dtype)
        ref = attnres.attnres_read_bwd(src, q, dout, gain, 1e-6)
        dsrc, dq, dg = _outputs(n_src, n_q, T, d, dtype)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        got = attnres.attnres_read_bwd_noalloc(src, q, dout, gain, 1e-6, dsrc=dsrc, dqueries=dq, dgain=dg)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        for a, b in zip(got, ref):
            assert torch.equal(a, b), f"call {call}"
        # nothing was allocated by the call (the driver's own bookkeeping moves
        # free memory in steps of 2 MB at most; the scratch array is 8 MB)
        assert free_after >= free_before - (2 << 20), f"call {call}: {free_before - free_after} bytes taken"


def test_noalloc_backward_falls_back_to_passes_of_one_query():
    """Two queries at d = 8192 need more workspace than the scratch holds in
    one pass; the entry point then runs one query per pass and its gradients
    agree with the oracle."""
    from _helpers import check_out, to_host
    from oracle import oracle
    n_src, n_q, T, d = 3, 2, 21, 8192
    need2 = attnres.attnres_read_bwd_workspace_size(n_src, T, d, n_q, torch.bfloat16)
    need1 = attnres.attnres_read_bwd_workspace_size(n_src, T, d, 1, torch.bfloat16)
    if not (need1 <= SCRATCH_BYTES < need2):
        pytest.skip(f"workspace {need1} / {need2} bytes: this device needs no fallback to one query at this size")
    g = torch.Generator(device="cuda").manual_seed(11)
    src = torch.randn((n_src, T, d), generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn((n_q, d), generator=g, device="cuda") * (16.0 / d) ** 0.5
    dout = torch.randn((n_q, T, d), generator=g, device="cuda").to(torch.bfloat16)
    dsrc, dq, dg = attnres.attnres_read_bwd_noalloc(src, q, dout)
    ref = oracle.read_bwd(to_host(src).astype(np.float64), to_host(q).astype(np.float64),
                          to_host(dout).astype(np.float64), None, 1e-6)
    check_out(dsrc, ref[0], torch.bfloat16, what="dsrc")
    check_out(dq, ref[1], torch.float32, np.abs(ref[1]).max(), strict=False, what="dq")


def test_noalloc_backward_rejects_sizes_beyond_its_scratch():
    """Only a device with enough SMs makes even a one-query pass outgrow the
    scratch; there the call must fail with an error rather than run."""
    n_src, T, d = 1, 1, 8192
    need1 = attnres.attnres_read_bwd_workspace_size(n_src, T, d, 1, torch.bfloat16)
    if need1 <= SCRATCH_BYTES:
        pytest.skip(f"one query at d={d} needs {need1} bytes, within the scratch on this device")
    src = torch.zeros((n_src, T, d), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((1, d), device="cuda")
    dout = torch.zeros((1, T, d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(attnres.AttnResError):
        attnres.attnres_read_bwd_noalloc(src, q, dout)


def test_noalloc_backward_with_four_queries_at_d4096():
    """Four queries at d = 4096: the no-allocation backward takes the
    two-kernel form when its workspace (which grows with T) fits the 8 MB
    scratch, else passes of two; its gradients agree with the oracle."""
    from _helpers import check_out, to_host
    from oracle import oracle
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    n_src, n_q, T, d = 8, 4, 40, 4096
    src = (torch.randn((n_src, T, d), generator=g, device="cuda") *
           (1 + 0.25 * torch.arange(n_src, device="cuda"))[:, None, None]).to(torch.bfloat16)
    q = torch.randn((n_q, d), generator=g, device="cuda") * (16.0 / d) ** 0.5
    dout = torch.randn((n_q, T, d), generator=g, device="cuda").to(torch.bfloat16)
    dsrc, dq, dg = attnres.attnres_read_bwd_noalloc(src, q, dout)
    ref = oracle.read_bwd(to_host(src).astype(np.float64), to_host(q).astype(np.float64),
                          to_host(dout).astype(np.float64), None, 1e-6)
    check_out(dsrc, ref[0], torch.bfloat16, what="dsrc")
    check_out(dq, ref[1], torch.float32, np.abs(ref[1]).max(), strict=False, what="dq")
