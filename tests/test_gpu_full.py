"""Parity at the full workload sizes, in the launch configuration the
benchmark times, on outputs the oracle can compute one by one: query rows
(every slice boundary plus seeded random rows) for out, lse and dq, and keys
whose gradient the oracle can afford (few rows see them) for dk and dv."""
import numpy as np
import pytest
import torch

import oracle
from oracle import planner
import flexible_mask_attention_gb300 as ffa
from flexible_mask_attention_gb300 import workloads as W
from gpu_helpers import check_fwd, check_grad

pytestmark = pytest.mark.gpu


def sample_rows(wl, n_random, seed):
    rng = np.random.default_rng(seed)
    rows = set()
    for qs, qe in wl.q_ranges:
        for r in (qs, qs + 1, qe - 2, qe - 1):
            if 0 <= r < wl.total_q:
                rows.add(int(r))
    rows |= {int(x) for x in rng.choice(wl.total_q, n_random, replace=False)}
    return np.array(sorted(rows), dtype=np.int64)


def cheap_keys(wl, n, budget, seed):
    """Keys whose dK/dV the oracle computes quickly: the visible entries of
    the rows that see the key sum to at most `budget`.  Within one slice the
    window [lo(r), hi(r)) of every mask type is non-decreasing in the row r,
    so the rows that see key j are the contiguous range hi(r) > j >= lo(r),
    found by binary search, and prefix sums of the rows' costs give its cost."""
    rng = np.random.default_rng(seed)
    counts = np.zeros(wl.total_q, dtype=np.int64)
    ivs = []
    for (qs, qe), (ks, ke), t in zip(wl.q_ranges, wl.k_ranges, wl.mask_types):
        if qe > qs and ke > ks:
            rows, lo, hi = planner.row_intervals(int(qs), int(qe), int(ks), int(ke), int(t))
            counts[rows] += np.clip(hi - lo, 0, None)
            ivs.append((rows, lo, hi))
    cand = rng.choice(wl.total_k, min(wl.total_k, 4000), replace=False)
    # always consider the ends of the key ranges (seen by few rows under causal masks)
    ends = {int(ke) - 1 for _, (ks, ke) in zip(wl.q_ranges, wl.k_ranges) if ke > ks}
    cand = np.unique(np.concatenate([cand, np.array(sorted(ends), dtype=np.int64)]))
    cost = np.zeros(cand.shape[0], dtype=np.int64)
    for rows, lo, hi in ivs:
        assert (np.diff(lo) >= 0).all() and (np.diff(hi) >= 0).all()
        pre = np.concatenate([[0], np.cumsum(counts[rows])])
        first = np.searchsorted(hi, cand, side="right")  # first row with hi > j
        stop = np.searchsorted(lo, cand, side="right")   # first row with lo > j
        cost += np.where(stop > first, pre[np.maximum(stop, first)] - pre[first], 0)
    ok = cand[(cost > 0) & (cost <= budget)]
    pick = rng.choice(ok, min(n, ok.shape[0]), replace=False)
    return np.sort(pick)


def run(wl, with_bwd):
    dev = torch.device("cuda", 0)
    tensors = W.make_tensors(wl, with_dout=with_bwd)
    d = [t.to(dev) for t in tensors]
    plan = ffa.ffa_plan_create(wl.q_ranges, wl.k_ranges, wl.mask_types, wl.total_q, wl.total_k,
                               wl.num_heads_q, wl.num_heads_kv, wl.head_dim)
    out, lse = ffa.ffa_fwd(plan, d[0], d[1], d[2])
    grads = None
    if with_bwd:
        grads = ffa.ffa_bwd(plan, d[0], d[1], d[2], out, d[3], lse)
    torch.cuda.synchronize()
    assert ffa.ffa_get_last_device_error(plan) == (0, 0)
    return tensors, out, lse, grads


@pytest.mark.parametrize("name,n_random", [("packed_causal", 64), ("heterogeneous", 64),
                                           ("long_context", 32)])
def test_forward_full_size(name, n_random):
    wl = W.CONFIGS[name]()
    (q, k, v), out, lse, _ = run(wl, with_bwd=False)
    rows = sample_rows(wl, n_random, seed=7)
    ro, rl = oracle.fwd(q, k, v, wl.q_ranges, wl.k_ranges, wl.mask_types, rows=rows)
    check_fwd(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, rows=rows)


@pytest.mark.parametrize("name", ["packed_causal", "heterogeneous", "long_context"])
def test_backward_full_size(name):
    wl = W.CONFIGS[name]()
    (q, k, v, do), out, lse, (dq, dk, dv) = run(wl, with_bwd=True)
    rows = sample_rows(wl, 16, seed=11)
    keys = cheap_keys(wl, 24, budget=3_000_000, seed=12)
    assert keys.shape[0] >= 8
    rq, rk, rv = oracle.bwd(q, k, v, do, wl.q_ranges, wl.k_ranges, wl.mask_types,
                            dq_rows=rows, dkv_keys=keys)
    check_grad(dq.float().cpu().numpy()[rows], rq, "dq")
    check_grad(dk.float().cpu().numpy()[keys], rk, "dk")
    check_grad(dv.float().cpu().numpy()[keys], rv, "dv")
    # properties that hold at any size: every gradient is finite and the rows
    # / keys nothing reaches are exactly zero
    for g in (dq, dk, dv):
        assert torch.isfinite(g.float()).all()
