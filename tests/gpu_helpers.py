"""Shared helpers for the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import torch

import oracle
import flexible_mask_attention_gb300 as ffa

OUT_TOL = 2e-2      # max-abs on out
LSE_TOL = 1e-3      # max-abs on finite lse
GRAD_REL = 5e-2     # max-abs relative to max |grad|


def bf16(*shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def run_fwd(q, k, v, qr, kr, ty, split_below=0, scale=None):
    dev = torch.device("cuda", 0)
    plan = ffa.ffa_plan_create(qr, kr, ty, q.shape[0], k.shape[0], q.shape[1], k.shape[1],
                               q.shape[2], split_below=split_below)
    out, lse = ffa.ffa_fwd(plan, q.to(dev), k.to(dev), v.to(dev), softmax_scale=scale)
    torch.cuda.synchronize()
    err = ffa.ffa_get_last_device_error(plan)
    assert err == (0, 0), f"device error {err}"
    return plan, out.float().cpu().numpy(), lse.cpu().numpy()


def check_fwd(out, lse, ref_out, ref_lse, rows=None):
    if rows is not None:
        out, lse = out[rows], lse[:, rows]
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), "-inf pattern of lse differs"
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    d_out = np.abs(out - ref_out).max()
    d_lse = np.abs(lse[fin] - ref_lse[fin]).max(initial=0.0)
    assert d_out <= OUT_TOL, f"out max-abs {d_out}"
    assert d_lse <= LSE_TOL, f"lse max-abs {d_lse}"
    return d_out, d_lse


def check_grad(g, r, name):
    scale = max(np.abs(r).max(), 1e-6)
    d = np.abs(g - r).max()
    assert d <= GRAD_REL * scale, f"{name}: max-abs {d} vs bound {GRAD_REL * scale}"
    return d / scale
