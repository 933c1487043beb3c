"""Shared helpers for the parity tests: run the CUDA path through the C ABI
binding and compare it with the fp64 oracle on the same seeded inputs.

Tolerances (the fp32 and bf16 bounds of the attention workloads):
  fp32 path:  |O - O_ref| <= 1e-5 and |LSE - LSE_ref| <= 1e-5.
  bf16 path:  |O - O_ref| <= 1e-2 + ulp_bf16(O_ref) / 2   (the second term is
              the rounding of the bf16 output format itself, which alone can
              exceed 1e-2 once |O| >= 4), and |LSE - LSE_ref| <= 1e-3, with the
              oracle run on the bf16-rounded inputs.
"""

from __future__ import annotations

import numpy as np

F32_TOL = 1e-5
BF16_O_TOL = 1e-2
BF16_LSE_TOL = 1e-3


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values around |x| (8 significant bits)."""
    ax = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def check_bf16(o, lse, o_ref, lse_ref, what=""):
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    bound = BF16_O_TOL + 0.5 * ulp_bf16(o_ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} O elements out of tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: LSE finiteness differs"
    if fin.any():
        lerr = np.abs(lse[fin] - lse_ref[fin])
        assert lerr.max() <= BF16_LSE_TOL, f"{what}: LSE max err {lerr.max():.3e}"
    if (~fin).any():
        assert np.all(np.isneginf(lse[~fin])), f"{what}: rows without keys must have LSE = -inf"
    return float(err.max()), float(np.abs(lse[fin] - lse_ref[fin]).max()) if fin.any() else 0.0


def check_f32(o, lse, o_ref, lse_ref, what=""):
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    err = np.abs(o - o_ref).max() if o.size else 0.0
    assert err <= F32_TOL, f"{what}: O max err {err:.3e}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin)
    if fin.any():
        lerr = np.abs(lse[fin] - lse_ref[fin]).max()
        assert lerr <= F32_TOL, f"{what}: LSE max err {lerr:.3e}"
    return float(err)


def to_device_bf16(x: np.ndarray, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device).to(torch.bfloat16).contiguous()


def run_bf16(q, k, v, scale, causal, device="cuda"):
    """q [B,H,M,D], k/v [B,H,N,D] float32 (bf16-exact) arrays -> (O, LSE) numpy."""
    import torch

    import flashattention_fa_fwd_gb300 as fa

    tq, tk, tv = (to_device_bf16(x, device) for x in (q, k, v))
    o = torch.empty_like(tq)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=device)
    fa.fa_fwd(tq, tk, tv, o, lse, scale, causal)
    assert fa.fa_get_device_status() == fa.FA_OK
    return o.float().cpu().numpy(), lse.cpu().numpy()


def run_f32(q, k, v, scale, causal, device="cuda"):
    import torch

    import flashattention_fa_fwd_gb300 as fa

    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device) for x in (q, k, v))
    o = torch.empty_like(tq)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=device)
    fa.fa_fwd_f32(tq, tk, tv, o, lse, scale, causal)
    assert fa.fa_get_device_status() == fa.FA_OK
    return o.cpu().numpy(), lse.cpu().numpy()
