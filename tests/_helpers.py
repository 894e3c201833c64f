"""Shared test helpers: dtype conversion and the tolerance checks.

Tolerances (written here once, used by every GPU parity test):
* bf16 storage: max|gpu - ref| <= 2e-2 * max|ref| per output tensor (the
  stated bar), and elementwise |gpu - ref| <= 2^-7 |ref| + 2e-3 max|ref|
  (bf16 keeps 8 significant bits, so one round-to-nearest of the float32
  result is at most 2^-8 relative; the bound leaves room for the float32
  arithmetic before it, or for the two-phase path's second rounding of its
  phase-1 state where the two errors do not line up).
* bf16 chains (chain=True): paths that hold intermediates in bf16 between
  their steps (the MSAR workspace chains and backwards, the two-phase
  backwards, the read backward's chunk states) round up to about seven more
  times before the output, each rounding at most 2^-8 relative to what it
  rounds.  Elementwise they are held to 4x the bound above (measured worst
  3.34x, on under 4% of the elements of a tensor), and per tensor to the
  stated bar.  Their fp32 parameter gradients (sums over the tokens of those
  intermediates) are held to the same pair of bounds.
* f32 storage: max|gpu - ref| <= 1e-4 * max|v| over the sources (the stated
  bar), and elementwise <= 1e-5 * max|v|.
* lse (float32): |gpu - ref| <= 1e-4 * (1 + |ref|).
"""
import numpy as np
import torch

BF16_REL = 2e-2
F32_REL = 1e-4


def to_dev(a, dtype):
    """float32/float64 numpy (already rounded to dtype's grid) -> CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda").to(dtype)


def to_host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_out(gpu, ref, dtype, src_absmax=None, strict=True, what="out", chain=False):
    gpu = to_host(gpu) if isinstance(gpu, torch.Tensor) else gpu
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    err = np.abs(gpu - ref)
    rmax = float(np.abs(ref).max()) if ref.size else 0.0
    if dtype == torch.bfloat16:
        assert err.max(initial=0.0) <= BF16_REL * rmax + 1e-30, \
            f"{what}: max err {err.max()} > {BF16_REL} * {rmax}"
        if strict or chain:
            bound = (4.0 if chain else 1.0) * (2.0 ** -7 * np.abs(ref) + 2e-3 * rmax)
            bad = err > bound
            assert not bad.any(), f"{what}: {bad.sum()} elements beyond the elementwise bound, " \
                                  f"worst {err.max()}"
    else:
        vmax = src_absmax if src_absmax is not None else rmax
        assert err.max(initial=0.0) <= F32_REL * vmax, f"{what}: max err {err.max()} > 1e-4 * {vmax}"
        if strict:
            assert err.max(initial=0.0) <= 1e-5 * vmax, f"{what}: max err {err.max()} > 1e-5 * {vmax}"
    return float(err.max(initial=0.0))


def check_lse(gpu, ref, what="lse"):
    gpu = to_host(gpu) if isinstance(gpu, torch.Tensor) else gpu
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    assert np.all(err <= 1e-4 * (1.0 + np.abs(ref))), f"{what}: max err {err.max()}"
    return float(err.max(initial=0.0))
