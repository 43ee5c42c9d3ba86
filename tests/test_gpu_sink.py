"""Attention sink: forward (out, lse) and backward (dq, dk, dv, dsink) of the
CUDA path against the fp64 oracle, for both sink layouts, with split items
(whose sink term is added by the merge kernel) and without."""
import numpy as np
import pytest
import torch

import oracle
import flexible_mask_attention_gb300 as ffa
from flexible_mask_attention_gb300 import workloads as W
from gpu_helpers import bf16, check_fwd, check_grad

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def sink_tensor(layout, n, Tq, Hq, seed, scale=2.0):
    g = torch.Generator().manual_seed(seed)
    shape = (n, Hq) if layout == "sh" else (Tq, n, Hq)
    return (scale * torch.randn(*shape, generator=g)).to(torch.float32)


def run(q, k, v, do, qr, kr, ty, sink, layout, split_below=0):
    plan = ffa.ffa_plan_create(qr, kr, ty, q.shape[0], k.shape[0], q.shape[1], k.shape[1],
                               q.shape[2], split_below=split_below)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    sd = sink.to(DEV)
    out, lse = ffa.ffa_fwd_ex(plan, qd, kd, vd, sink=sd, sink_layout=layout)
    res = [out.float().cpu().numpy(), lse.cpu().numpy()]
    if do is not None:
        dq, dk, dv, ds = ffa.ffa_bwd_ex(plan, qd, kd, vd, out, do.to(DEV), lse, sink=sd,
                                        sink_layout=layout)
        res += [t.float().cpu().numpy() for t in (dq, dk, dv, ds)]
    torch.cuda.synchronize()
    assert ffa.ffa_get_last_device_error(plan) == (0, 0)
    return res


CASES = [
    # (Tq, Tk, Hq, Hkv, D, n_segments, seed, layout, n_sink)
    (1000, 1000, 4, 2, 128, 5, 31, "sh", 1),
    (777, 777, 2, 2, 128, 4, 32, "sh", 4),
    (640, 900, 3, 1, 128, 6, 33, "ssh", 2),
    (1000, 1000, 4, 2, 64, 5, 34, "ssh", 1),
    (515, 515, 1, 1, 64, 3, 35, "sh", 3),
]


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}x{c[1]}_H{c[2]}/{c[3]}_D{c[4]}_{c[7]}{c[8]}" for c in CASES])
@pytest.mark.parametrize("split_below", [0, -1])
def test_sink_fwd(case, split_below):
    Tq, Tk, Hq, Hkv, D, nseg, seed, layout, n = case
    qr, kr, ty = W.random_slices(Tq, Tk, nseg, seed=seed)
    q, k, v = bf16(Tq, Hq, D, seed=seed), bf16(Tk, Hkv, D, seed=seed + 1), bf16(Tk, Hkv, D, seed=seed + 2)
    sink = sink_tensor(layout, n, Tq, Hq, seed + 3)
    out, lse = run(q, k, v, None, qr, kr, ty, sink, layout, split_below)
    ro, rl = oracle.fwd(q, k, v, qr, kr, ty, sink=sink, sink_layout=layout)
    check_fwd(out, lse, ro, rl)


@pytest.mark.parametrize("case", CASES[:4], ids=[f"T{c[0]}_D{c[4]}_{c[7]}{c[8]}" for c in CASES[:4]])
def test_sink_bwd(case):
    Tq, Tk, Hq, Hkv, D, nseg, seed, layout, n = case
    qr, kr, ty = W.random_slices(Tq, Tk, nseg, seed=seed)
    q, k, v = bf16(Tq, Hq, D, seed=seed), bf16(Tk, Hkv, D, seed=seed + 1), bf16(Tk, Hkv, D, seed=seed + 2)
    do = bf16(Tq, Hq, D, seed=seed + 4)
    sink = sink_tensor(layout, n, Tq, Hq, seed + 3)
    out, lse, dq, dk, dv, ds = run(q, k, v, do, qr, kr, ty, sink, layout)
    ro, rl = oracle.fwd(q, k, v, qr, kr, ty, sink=sink, sink_layout=layout)
    check_fwd(out, lse, ro, rl)
    rq, rk, rv = oracle.bwd(q, k, v, do, qr, kr, ty, sink=sink, sink_layout=layout)
    check_grad(dq, rq, "dq"); check_grad(dk, rk, "dk"); check_grad(dv, rv, "dv")
    rs = oracle.dsink(q, k, v, do, qr, kr, ty, sink, layout)
    check_grad(ds, rs, "dsink")


def test_sink_empty_rows():
    """No slice at all: every row has out = 0 and lse = logsumexp(sink)."""
    T, H, D = 300, 2, 128
    q, k, v = bf16(T, H, D, seed=1), bf16(T, H, D, seed=2), bf16(T, H, D, seed=3)
    sink = sink_tensor("sh", 3, T, H, 4)
    out, lse = run(q, k, v, None, np.zeros((0, 2)), np.zeros((0, 2)), np.zeros((0,)), sink, "sh")
    assert (out == 0).all()
    ref = torch.logsumexp(sink.double(), dim=0).numpy()
    assert np.abs(lse - ref[:, None]).max() < 1e-5


def test_minus_inf_sink_matches_plain():
    """A sink of -inf adds nothing: identical bits to ffa_fwd / ffa_bwd."""
    T, H, D = 700, 2, 128
    qr, kr, ty = W.random_slices(T, T, 4, seed=41)
    q, k, v, do = (bf16(T, H, D, seed=41 + i).to(DEV) for i in range(4))
    plan = ffa.ffa_plan_create(qr, kr, ty, T, T, H, H, D)
    o0, l0 = ffa.ffa_fwd(plan, q, k, v)
    sink = torch.full((2, H), float("-inf"), device=DEV)
    o1, l1 = ffa.ffa_fwd_ex(plan, q, k, v, sink=sink)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    g0 = ffa.ffa_bwd(plan, q, k, v, o0, do, l0)
    g1 = ffa.ffa_bwd_ex(plan, q, k, v, o1, do, l1, sink=sink)
    assert all(torch.equal(a, b) for a, b in zip(g0, g1[:3]))
    assert (g1[3] == 0).all()


def test_dsink_repeatable():
    """The per-head dsink sums run in a fixed order: two calls agree bit for bit."""
    T, H, D = 2048, 4, 128
    qr, kr, ty = W.random_slices(T, T, 6, seed=51)
    q, k, v, do = (bf16(T, H, D, seed=51 + i).to(DEV) for i in range(4))
    sink = sink_tensor("sh", 2, T, H, 55).to(DEV)
    plan = ffa.ffa_plan_create(qr, kr, ty, T, T, H, H, D)
    o, l = ffa.ffa_fwd_ex(plan, q, k, v, sink=sink)
    d1 = ffa.ffa_bwd_ex(plan, q, k, v, o, do, l, sink=sink)[3].clone()
    d2 = ffa.ffa_bwd_ex(plan, q, k, v, o, do, l, sink=sink)[3]
    assert torch.equal(d1, d2)


def test_sink_argument_checks():
    T, H, D = 256, 2, 64
    q, k, v = (bf16(T, H, D, seed=i).to(DEV) for i in range(3))
    plan = ffa.ffa_plan_create([[0, T]], [[0, T]], [1], T, T, H, H, D, split_below=-1)
    lib = ffa.load_library()
    out, lse = torch.empty_like(q), torch.empty(H, T, device=DEV)
    big = torch.zeros(ffa.FFA_MAX_SINK + 1, H, device=DEV)
    P = ffa._ptr
    args = lambda sink, n, lay, cap=0.0: (plan.handle, P(q), P(k), P(v), sink, n, lay, 0.0, cap,
                                          P(out), P(lse), None, 0, None)
    assert lib.ffa_fwd_ex(*args(P(big), ffa.FFA_MAX_SINK + 1, 0)) == 1
    assert lib.ffa_fwd_ex(*args(None, 2, 0)) == 1
    assert lib.ffa_fwd_ex(*args(P(big), 2, 7)) == 1
    assert lib.ffa_fwd_ex(*args(P(big), -1, 0)) == 1
    assert lib.ffa_fwd_ex(*args(None, 0, 0, -1.0)) == 1
    assert lib.ffa_fwd_ex(*args(None, 0, 0, float("nan"))) == 1
    assert lib.ffa_fwd_ex(*args(None, 0, 0)) == 0
    torch.cuda.synchronize()
