"""The no-allocation backward entry point (built-in scratch instead of a
caller workspace) against the workspace entry point: the same kernels, so the
results must agree bit for bit, on two consecutive calls (the second reuses
the scratch the first left behind)."""
import numpy as np
import pytest
import torch

from depth_wise_attention_gb300 import attnres

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_src,n_q,T,d,dtype", [(9, 1, 300, 4096, torch.bfloat16), (5, 2, 77, 512, torch.float32)])
def test_noalloc_backward_matches_workspace_backward_on_two_calls(n_src, n_q, T, d, dtype):
    g = torch.Generator(device="cuda").manual_seed(n_src + T)
    for call in range(2):
        src = (torch.randn((n_src, T, d), generator=g, device="cuda") * (1 + call)).to(dtype)
        q = torch.randn((n_q, d), generator=g, device="cuda") * (16.0 / d) ** 0.5
        gain = torch.rand((d,), generator=g, device="cuda") + 0.5
        dout = torch.randn((n_q, T, d), generator=g, device="cuda").to(dtype)
        ref = attnres.attnres_read_bwd(src, q, dout, gain, 1e-6)
        free_before = torch.cuda.mem_get_info()[0]
        got = attnres.attnres_read_bwd_noalloc(src, q, dout, gain, 1e-6)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b), f"call {call}"
        # the library allocated nothing (only torch's outputs, above, are new)
        assert torch.cuda.mem_get_info()[0] >= free_before - (64 << 20)


def test_noalloc_backward_rejects_sizes_beyond_its_scratch():
    d = 8192
    src = torch.zeros((1, 1, d), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((2, d), device="cuda")
    dout = torch.zeros((2, 1, d), dtype=torch.bfloat16, device="cuda")
    need = attnres.attnres_read_bwd_workspace_size(1, 1, d, 2, torch.bfloat16)
    if need <= (8 << 20):
        pytest.skip("this device's largest backward fits the built-in scratch")
    with pytest.raises(attnres.AttnResError):
        attnres.attnres_read_bwd_noalloc(src, q, dout)


def test_noalloc_backward_with_four_queries_at_d4096():
    """Four queries at d = 4096 would need a 10 MB workspace in one pass; the
    no-allocation backward then takes passes of two within its 8 MB scratch,
    and its gradients agree with the oracle."""
    import numpy as np
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
