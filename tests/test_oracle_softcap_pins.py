"""Pins for the oracle's softcap, each against something other than the
oracle itself: the uncapped limit, a closed form on the diagonal mask, torch
fp64 autograd through torch.tanh, and planted mistakes.

Reading (the pages show `softcap=0` as an argument of flex_flash_attn_func,
no formula): for c > 0 every score becomes x = c * tanh(scale * q.k / c)."""
import math
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle import dense
from flexible_mask_attention_gb300 import workloads as W


def _bf16(*shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (scale * torch.randn(*shape, generator=g)).to(torch.bfloat16)


def torch_dense_capped(q, k, v, mask, scale, cap):
    """fp64 reference: masked scores capped by cap * tanh(s / cap), then the
    masked softmax; lse by torch.logsumexp (rows without keys: -inf, out 0)."""
    Hq, Hkv = q.shape[1], k.shape[1]
    kk = k.repeat_interleave(Hq // Hkv, dim=1)
    vv = v.repeat_interleave(Hq // Hkv, dim=1)
    s = torch.einsum("qhd,khd->hqk", q, kk) * scale
    s = cap * torch.tanh(s / cap)
    s = s.masked_fill(~mask[None], float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    p = torch.exp(s - torch.where(torch.isfinite(lse), lse, torch.zeros_like(lse))[..., None])
    return torch.einsum("hqk,khd->qhd", p, vv), lse


def _case(seed, Hq=4, Hkv=2, D=8):
    rng = np.random.default_rng(900 + seed)
    Tq, Tk = int(rng.integers(40, 110)), int(rng.integers(40, 110))
    qr, kr, ty = W.random_slices(Tq, Tk, 4, seed=seed + 90)
    # large scores, so that the cap matters
    q = _bf16(Tq, Hq, D, seed=seed, scale=3.0)
    k, v = _bf16(Tk, Hkv, D, seed=seed + 1, scale=3.0), _bf16(Tk, Hkv, D, seed=seed + 2)
    do = _bf16(Tq, Hq, D, seed=seed + 3)
    return Tq, Tk, qr, kr, ty, q, k, v, do


def _check_vs_torch(seed, cap, lib=None):
    Tq, Tk, qr, kr, ty, q, k, v, do = _case(seed)
    mask = torch.from_numpy(dense.dense_mask(Tq, Tk, qr, kr, ty))
    qq, kk, vv = (t.to(torch.float64).requires_grad_() for t in (q, k, v))
    ref_o, ref_l = torch_dense_capped(qq, kk, vv, mask, 1.0 / math.sqrt(q.shape[-1]), cap)
    ref_o.backward(do.to(torch.float64))
    o, l = oracle.fwd(q, k, v, qr, kr, ty, lib=lib, softcap=cap)
    fin = np.isfinite(ref_l.detach().numpy())
    assert np.array_equal(np.isfinite(l), fin)
    assert np.abs(o - ref_o.detach().numpy()).max() < 1e-12
    assert np.abs(l[fin] - ref_l.detach().numpy()[fin]).max() < 1e-12
    dq, dk, dv = oracle.bwd(q, k, v, do, qr, kr, ty, lib=lib, softcap=cap)
    assert np.abs(dq - qq.grad.numpy()).max() < 1e-10
    assert np.abs(dk - kk.grad.numpy()).max() < 1e-10
    assert np.abs(dv - vv.grad.numpy()).max() < 1e-10


@pytest.mark.parametrize("cap", [5.0, 20.0])
@pytest.mark.parametrize("seed", range(2))
def test_softcap_matches_torch_autograd(seed, cap):
    _check_vs_torch(seed, cap)


def test_huge_cap_is_no_cap():
    """c * tanh(x / c) = x - x^3 / (3 c^2) + ...: with c = 1e7 the results
    equal the uncapped oracle to rounding."""
    Tq, Tk, qr, kr, ty, q, k, v, do = _case(4)
    o0, l0 = oracle.fwd(q, k, v, qr, kr, ty)
    o1, l1 = oracle.fwd(q, k, v, qr, kr, ty, softcap=1e7)
    fin = np.isfinite(l0)
    assert np.array_equal(np.isfinite(l1), fin)
    assert np.abs(o1 - o0).max() < 1e-9 and np.abs(l1[fin] - l0[fin]).max() < 1e-9
    g0 = oracle.bwd(q, k, v, do, qr, kr, ty)
    g1 = oracle.bwd(q, k, v, do, qr, kr, ty, softcap=1e7)
    assert all(np.abs(a - b).max() < 1e-8 for a, b in zip(g0, g1))


def test_diagonal_closed_form():
    """On the diagonal mask each row sees one key: lse_i = c tanh(scale q_i.k_i / c),
    out_i = v_i."""
    T, H, D, c = 60, 2, 16, 3.0
    q, k, v = _bf16(T, H, D, seed=1, scale=2.0), _bf16(T, H, D, seed=2, scale=2.0), _bf16(T, H, D, seed=3)
    o, l = oracle.fwd(q, k, v, [[0, T]], [[0, T]], [3], softcap=c)
    qf, kf, vf = (t.to(torch.float64).numpy() for t in (q, k, v))
    for h in range(H):
        x = (qf[:, h] * kf[:, h]).sum(-1) / math.sqrt(D)
        assert np.abs(l[h] - c * np.tanh(x / c)).max() < 1e-13
        assert np.abs(o[:, h] - vf[:, h]).max() < 1e-13


# --- planted mistakes in the softcap code: each must fail a pin ------------------

MUTANTS = {
    "cap_outside_scale": (r"const double x = P->scale \* dot;\n  return P->softcap > 0.0 \? P->softcap \* tanh\(x / P->softcap\) : x;",
                          "const double x = P->scale * dot;\n  return P->softcap > 0.0 ? P->scale * P->softcap * tanh(dot / P->softcap) : x;"),
    "grad_factor_dropped": (r"return 1.0 - t \* t;", "return 1.0;"),
    "grad_factor_sign": (r"return 1.0 - t \* t;", "return 1.0 + t * t;"),
}


def _cap_pins_fail(lib):
    try:
        _check_vs_torch(0, 5.0, lib=lib)
    except AssertionError:
        return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_softcap_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "ffa_oracle.c")).read()
    pat, rep = MUTANTS[name]
    mutated, n = re.subn(pat, rep, src)
    assert n >= 1, f"mutation {name} did not apply"
    c = tmp_path / "m.c"
    c.write_text(mutated)
    so = tmp_path / "libm.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o", str(so), str(c), "-lm"])
    assert _cap_pins_fail(oracle.load_library(str(so))), f"mutant {name} passed every pin"


def test_unmutated_oracle_passes_softcap_pins():
    assert not _cap_pins_fail(None)
