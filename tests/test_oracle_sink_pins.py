"""Pins for the oracle's attention-sink support, each against something other
than the oracle itself: exact special cases, a closed form, torch fp64
autograd through a logsumexp over the row with the sink logits appended, and
finite differences.

Reading (the pages show the `sink` argument, layouts "sh" [n_sink, Hq] and
"ssh" [Tq, n_sink, Hq] in fp32, but not its formula): sink logits, not
multiplied by the softmax scale, join only the row normaliser."""
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


def _bf16(*shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def _sink(shape, seed, scale=1.5):
    g = torch.Generator().manual_seed(seed)
    return (scale * torch.randn(*shape, generator=g)).to(torch.float32)


def torch_dense_sink(q, k, v, mask, scale, sink, layout):
    """fp64 reference: masked scores with the sink logits appended to every
    row; lse by torch.logsumexp over the augmented row, out over the keys."""
    Hq, Hkv = q.shape[1], k.shape[1]
    kk = k.repeat_interleave(Hq // Hkv, dim=1)
    vv = v.repeat_interleave(Hq // Hkv, dim=1)
    s = torch.einsum("qhd,khd->hqk", q, kk) * scale
    s = s.masked_fill(~mask[None], float("-inf"))
    Tq = q.shape[0]
    if layout == "sh":
        sk = sink.t()[:, None, :].expand(Hq, Tq, sink.shape[0])
    else:
        sk = sink.permute(2, 0, 1)
    lse = torch.logsumexp(torch.cat([s, sk], dim=-1), dim=-1)
    p = torch.exp(s - lse[..., None])
    return torch.einsum("hqk,khd->qhd", p, vv), lse


def _case(seed, Hq=4, Hkv=2, D=8):
    rng = np.random.default_rng(700 + seed)
    Tq, Tk = int(rng.integers(40, 110)), int(rng.integers(40, 110))
    qr, kr, ty = W.random_slices(Tq, Tk, 4, seed=seed + 80)
    q, k, v = _bf16(Tq, Hq, D, seed=seed), _bf16(Tk, Hkv, D, seed=seed + 1), _bf16(Tk, Hkv, D, seed=seed + 2)
    do = _bf16(Tq, Hq, D, seed=seed + 3)
    return Tq, Tk, qr, kr, ty, q, k, v, do


def _check_vs_torch(seed, layout, n_sink, lib=None):
    Tq, Tk, qr, kr, ty, q, k, v, do = _case(seed)
    Hq = q.shape[1]
    sink = _sink((n_sink, Hq) if layout == "sh" else (Tq, n_sink, Hq), seed=seed + 9)
    mask = torch.from_numpy(dense.dense_mask(Tq, Tk, qr, kr, ty))
    qq, kk, vv = (t.to(torch.float64).requires_grad_() for t in (q, k, v))
    ss = sink.to(torch.float64).requires_grad_()
    ref_o, ref_l = torch_dense_sink(qq, kk, vv, mask, 1.0 / math.sqrt(q.shape[-1]), ss, layout)
    ref_o.backward(do.to(torch.float64))
    o, l = oracle.fwd(q, k, v, qr, kr, ty, lib=lib, sink=sink, sink_layout=layout)
    assert np.abs(o - ref_o.detach().numpy()).max() < 1e-12
    assert np.abs(l - ref_l.detach().numpy()).max() < 1e-12
    dq, dk, dv = oracle.bwd(q, k, v, do, qr, kr, ty, lib=lib, sink=sink, sink_layout=layout)
    assert np.abs(dq - qq.grad.numpy()).max() < 1e-10
    assert np.abs(dk - kk.grad.numpy()).max() < 1e-10
    assert np.abs(dv - vv.grad.numpy()).max() < 1e-10
    ds = oracle.dsink(q, k, v, do, qr, kr, ty, sink, layout, lib=lib)
    assert np.abs(ds - ss.grad.numpy()).max() < 1e-10


@pytest.mark.parametrize("layout,n_sink", [("sh", 1), ("sh", 4), ("ssh", 2)])
@pytest.mark.parametrize("seed", range(2))
def test_sink_matches_torch_autograd(seed, layout, n_sink):
    _check_vs_torch(seed, layout, n_sink)


def test_minus_inf_sink_is_no_sink():
    """exp(-inf) adds exactly nothing: results equal the no-sink oracle bit for bit."""
    Tq, Tk, qr, kr, ty, q, k, v, do = _case(5)
    sink = torch.full((3, q.shape[1]), float("-inf"))
    o0, l0 = oracle.fwd(q, k, v, qr, kr, ty)
    o1, l1 = oracle.fwd(q, k, v, qr, kr, ty, sink=sink)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    g0 = oracle.bwd(q, k, v, do, qr, kr, ty)
    g1 = oracle.bwd(q, k, v, do, qr, kr, ty, sink=sink)
    assert all(np.array_equal(a, b) for a, b in zip(g0, g1))


@pytest.mark.parametrize("layout", ["sh", "ssh"])
def test_diagonal_closed_form(layout):
    """A square bi-causal slice is the diagonal: row i sees only key i, so
    lse_i = log(e^x_ii + sum_s e^sigma_s) and out_i = v_i e^(x_ii - lse_i)."""
    T, H, D = 50, 2, 16
    q, k, v = _bf16(T, H, D, seed=1), _bf16(T, H, D, seed=2), _bf16(T, H, D, seed=3)
    sink = _sink((2, H) if layout == "sh" else (T, 2, H), seed=4)
    o, l = oracle.fwd(q, k, v, [[0, T]], [[0, T]], [3], sink=sink, sink_layout=layout)
    qf, kf, vf = (t.to(torch.float64).numpy() for t in (q, k, v))
    sf = sink.to(torch.float64).numpy()
    for h in range(H):
        x = (qf[:, h] * kf[:, h]).sum(-1) / math.sqrt(D)
        sig = np.broadcast_to(sf[:, h], (T, 2)) if layout == "sh" else sf[:, :, h]
        lse = np.log(np.exp(x) + np.exp(sig).sum(-1))
        assert np.abs(l[h] - lse).max() < 1e-13
        assert np.abs(o[:, h] - vf[:, h] * np.exp(x - lse)[:, None]).max() < 1e-13


def _check_empty_rows(lib=None):
    T, H, D = 40, 2, 8
    q, k, v = _bf16(T, H, D, seed=1), _bf16(T, H, D, seed=2), _bf16(T, H, D, seed=3)
    sink = _sink((3, H), seed=6)
    o, l = oracle.fwd(q, k, v, [[10, 20]], [[0, 30]], [0], lib=lib, sink=sink)
    empty = [i for i in range(T) if not 10 <= i < 20]
    sf = sink.to(torch.float64).numpy()
    ref = np.log(np.exp(sf).sum(0))
    assert (o[empty] == 0).all()
    for h in range(H):
        assert np.abs(l[h, empty] - ref[h]).max() < 1e-15


def test_empty_rows_with_sink():
    """A row that sees no key: out = 0, lse = log sum_s exp(sigma_s)."""
    _check_empty_rows()


def test_dsink_finite_difference():
    """dsink against central differences of L = <dO, out(sigma)>."""
    Tq, Tk, qr, kr, ty, q, k, v, do = _case(3)
    Hq = q.shape[1]
    sink = _sink((2, Hq), seed=12).to(torch.float64)
    dof = do.to(torch.float64).numpy()
    ds = oracle.dsink(q, k, v, do, qr, kr, ty, sink, "sh")
    eps = 1e-5
    for s in range(2):
        for h in range(Hq):
            sp, sm = sink.clone(), sink.clone()
            sp[s, h] += eps
            sm[s, h] -= eps
            lp = (oracle.fwd(q, k, v, qr, kr, ty, sink=sp)[0] * dof).sum()
            lm = (oracle.fwd(q, k, v, qr, kr, ty, sink=sm)[0] * dof).sum()
            assert abs((lp - lm) / (2 * eps) - ds[s, h]) < 1e-7 * max(1.0, abs(ds[s, h]))


def test_ssh_broadcast_equals_sh():
    """Per-row sinks that repeat the per-head values give the same forward,
    and the per-row gradients sum to the per-head one."""
    Tq, Tk, qr, kr, ty, q, k, v, do = _case(7)
    Hq = q.shape[1]
    sh = _sink((3, Hq), seed=21)
    ssh = sh[None].expand(Tq, 3, Hq).contiguous()
    o1, l1 = oracle.fwd(q, k, v, qr, kr, ty, sink=sh)
    o2, l2 = oracle.fwd(q, k, v, qr, kr, ty, sink=ssh, sink_layout="ssh")
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    d1 = oracle.dsink(q, k, v, do, qr, kr, ty, sh, "sh")
    d2 = oracle.dsink(q, k, v, do, qr, kr, ty, ssh, "ssh")
    assert np.abs(d2.sum(0) - d1).max() < 1e-12
    rows = [0, Tq // 2, Tq - 1]
    d3 = oracle.dsink(q, k, v, do, qr, kr, ty, ssh, "ssh", rows=rows)
    assert np.abs(d3 - d2[rows]).max() < 1e-15


# --- planted mistakes in the sink code: each must fail a pin ---------------------

MUTANTS = {
    "sink_scaled": (r"sum \+= exp\(sink_value\(P, h, i, s\) - m\);",
                    "sum += exp(P->scale * sink_value(P, h, i, s) - m);"),
    "sink_not_in_sum": (r"for \(int s = 0; s < ns; \+\+s\) sum \+= exp\(sink_value\(P, h, i, s\) - m\);", ""),
    "ssh_index": (r"return P->sink\[\(\(size_t\)i \* P->n_sink \+ s\) \* P->Hq \+ h\];",
                  "return P->sink[((size_t)s * P->Tq + i) * P->Hq + h];"),
    "dsink_sign": (r"= -exp\(sink_value\(&P, h, i, s\) - lse\) \* delta;",
                   "= exp(sink_value(&P, h, i, s) - lse) * delta;"),
    "dsink_no_delta": (r"= -exp\(sink_value\(&P, h, i, s\) - lse\) \* delta;",
                       "= -exp(sink_value(&P, h, i, s) - lse);"),
    "empty_row_drops_sink": (r"if \(cnt == 0\) return lse;", "if (cnt == 0) return -INFINITY;"),
}


def _sink_pins_fail(lib):
    failures = []
    for layout, n in (("sh", 2), ("ssh", 2)):
        try:
            _check_vs_torch(0, layout, n, lib=lib)
        except (AssertionError, ValueError):
            failures.append(layout)
    try:
        _check_empty_rows(lib)
    except AssertionError:
        failures.append("empty rows")
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_sink_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "ffa_oracle.c")).read()
    pat, rep = MUTANTS[name]
    mutated, n = re.subn(pat, rep, src)
    assert n >= 1, f"mutation {name} did not apply"
    c = tmp_path / "m.c"
    c.write_text(mutated)
    so = tmp_path / "libm.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o", str(so), str(c), "-lm"])
    assert _sink_pins_fail(oracle.load_library(str(so))), f"mutant {name} passed every pin"


def test_unmutated_oracle_passes_sink_pins():
    assert _sink_pins_fail(None) == []
