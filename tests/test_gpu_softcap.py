"""Softcap: forward and backward of the CUDA path against the fp64 oracle
with scores capped to c * tanh(score / c) (scores made large, so that the
cap changes the result), with and without split items and with a sink."""
import numpy as np
import pytest
import torch

import oracle
import flexible_mask_attention_gb300 as ffa
from flexible_mask_attention_gb300 import workloads as W
from gpu_helpers import check_fwd, check_grad

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def bf16(*shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (scale * torch.randn(*shape, generator=g)).to(torch.bfloat16)


CASES = [
    # (Tq, Tk, Hq, Hkv, D, n_segments, seed, cap)
    (1000, 1000, 4, 2, 128, 5, 61, 5.0),
    (777, 777, 2, 2, 128, 4, 62, 20.0),
    (640, 900, 3, 1, 64, 6, 63, 8.0),
]


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}_D{c[4]}_cap{c[7]:g}" for c in CASES])
@pytest.mark.parametrize("split_below", [0, -1])
def test_softcap_fwd_bwd(case, split_below):
    Tq, Tk, Hq, Hkv, D, nseg, seed, cap = case
    qr, kr, ty = W.random_slices(Tq, Tk, nseg, seed=seed)
    q, k = bf16(Tq, Hq, D, seed=seed, scale=2.5), bf16(Tk, Hkv, D, seed=seed + 1, scale=2.5)
    v, do = bf16(Tk, Hkv, D, seed=seed + 2), bf16(Tq, Hq, D, seed=seed + 3)
    plan = ffa.ffa_plan_create(qr, kr, ty, Tq, Tk, Hq, Hkv, D, split_below=split_below)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = ffa.ffa_fwd_ex(plan, qd, kd, vd, softcap=cap)
    dq, dk, dv, _ = ffa.ffa_bwd_ex(plan, qd, kd, vd, out, dod, lse, softcap=cap)
    torch.cuda.synchronize()
    assert ffa.ffa_get_last_device_error(plan) == (0, 0)
    ro, rl = oracle.fwd(q, k, v, qr, kr, ty, softcap=cap)
    check_fwd(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl)
    rq, rk, rv = oracle.bwd(q, k, v, do, qr, kr, ty, softcap=cap)
    check_grad(dq.float().cpu().numpy(), rq, "dq")
    check_grad(dk.float().cpu().numpy(), rk, "dk")
    check_grad(dv.float().cpu().numpy(), rv, "dv")


def test_softcap_with_sink():
    T, H, D, cap = 900, 2, 128, 6.0
    qr, kr, ty = W.random_slices(T, T, 5, seed=71)
    q, k = bf16(T, H, D, seed=71, scale=2.5), bf16(T, H, D, seed=72, scale=2.5)
    v, do = bf16(T, H, D, seed=73), bf16(T, H, D, seed=74)
    sink = (2.0 * torch.randn(2, H, generator=torch.Generator().manual_seed(75))).float()
    plan = ffa.ffa_plan_create(qr, kr, ty, T, T, H, H, D)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = ffa.ffa_fwd_ex(plan, qd, kd, vd, sink=sink.to(DEV), softcap=cap)
    dq, dk, dv, ds = ffa.ffa_bwd_ex(plan, qd, kd, vd, out, dod, lse, sink=sink.to(DEV), softcap=cap)
    torch.cuda.synchronize()
    assert ffa.ffa_get_last_device_error(plan) == (0, 0)
    ro, rl = oracle.fwd(q, k, v, qr, kr, ty, sink=sink, softcap=cap)
    check_fwd(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl)
    rq, rk, rv = oracle.bwd(q, k, v, do, qr, kr, ty, sink=sink, softcap=cap)
    check_grad(dq.float().cpu().numpy(), rq, "dq")
    check_grad(dk.float().cpu().numpy(), rk, "dk")
    check_grad(dv.float().cpu().numpy(), rv, "dv")
    rs = oracle.dsink(q, k, v, do, qr, kr, ty, sink, "sh", softcap=cap)
    check_grad(ds.cpu().numpy(), rs, "dsink")


# Scores of unit-scale inputs stay well inside the tanh polynomial's range
# (|score / c| <= 0.75) for these caps, so the warps take the polynomial path;
# in the mixed case a few query rows are scaled up so that the warps holding
# them fall back to the exponential form inside the same launch.
POLY_CASES = [
    # (Tq, Tk, Hq, Hkv, D, n_segments, seed, cap, rows scaled up)
    (1000, 1000, 4, 2, 128, 5, 81, 30.0, 0),
    (640, 900, 3, 1, 64, 6, 82, 8.0, 0),
    (1100, 1100, 2, 2, 128, 5, 83, 8.0, 12),
    (700, 700, 2, 1, 128, 4, 84, 1.0e6, 0),
]


@pytest.mark.parametrize("case", POLY_CASES,
                         ids=[f"T{c[0]}_D{c[4]}_cap{c[7]:g}_big{c[8]}" for c in POLY_CASES])
def test_softcap_polynomial_path(case):
    Tq, Tk, Hq, Hkv, D, nseg, seed, cap, n_big = case
    qr, kr, ty = W.random_slices(Tq, Tk, nseg, seed=seed)
    q, k = bf16(Tq, Hq, D, seed=seed), bf16(Tk, Hkv, D, seed=seed + 1)
    v, do = bf16(Tk, Hkv, D, seed=seed + 2), bf16(Tq, Hq, D, seed=seed + 3)
    if n_big:
        rows = np.random.default_rng(seed).choice(Tq, n_big, replace=False)
        q[rows] = (q[rows].float() * 6.0).to(torch.bfloat16)
    plan = ffa.ffa_plan_create(qr, kr, ty, Tq, Tk, Hq, Hkv, D)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = ffa.ffa_fwd_ex(plan, qd, kd, vd, softcap=cap)
    dq, dk, dv, _ = ffa.ffa_bwd_ex(plan, qd, kd, vd, out, dod, lse, softcap=cap)
    torch.cuda.synchronize()
    assert ffa.ffa_get_last_device_error(plan) == (0, 0)
    ro, rl = oracle.fwd(q, k, v, qr, kr, ty, softcap=cap)
    check_fwd(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl)
    rq, rk, rv = oracle.bwd(q, k, v, do, qr, kr, ty, softcap=cap)
    check_grad(dq.float().cpu().numpy(), rq, "dq")
    check_grad(dk.float().cpu().numpy(), rk, "dk")
    check_grad(dv.float().cpu().numpy(), rv, "dv")
