"""Uniform block-sparse masks (many tiny full slices): forward and backward of
the CUDA path against the fp64 oracle, on small cases in full and on the
benchmark-size tables on sampled rows and keys."""
import numpy as np
import pytest
import torch

import oracle
import flexible_mask_attention_gb300 as ffa
from flexible_mask_attention_gb300 import workloads as W
from gpu_helpers import bf16, check_fwd, check_grad

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
BLOCKS = [(64, 64), (128, 128), (32, 64), (16, 64), (8, 64), (64, 32), (64, 16), (64, 8), (64, 1)]


def run(wl, q, k, v, do=None):
    plan = ffa.ffa_plan_create(wl.q_ranges, wl.k_ranges, wl.mask_types, wl.total_q, wl.total_k,
                               wl.num_heads_q, wl.num_heads_kv, wl.head_dim)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    out, lse = ffa.ffa_fwd(plan, qd, kd, vd)
    res = [out, lse]
    if do is not None:
        res += list(ffa.ffa_bwd(plan, qd, kd, vd, out, do.to(DEV), lse))
    torch.cuda.synchronize()
    assert ffa.ffa_get_last_device_error(plan) == (0, 0)
    return [t.float().cpu().numpy() for t in res]


@pytest.mark.parametrize("blocks", BLOCKS, ids=[f"q{a}_k{b}" for a, b in BLOCKS])
def test_block_sparse_small(blocks):
    wl = W.block_sparse(total=2048, hq=4, hkv=2, d=128, q_block=blocks[0], k_block=blocks[1],
                        seed=17)
    q, k, v, do = W.make_tensors(wl, with_dout=True)
    out, lse, dq, dk, dv = run(wl, q, k, v, do)
    ro, rl = oracle.fwd(q, k, v, wl.q_ranges, wl.k_ranges, wl.mask_types)
    check_fwd(out, lse, ro, rl)
    rq, rk, rv = oracle.bwd(q, k, v, do, wl.q_ranges, wl.k_ranges, wl.mask_types)
    check_grad(dq, rq, "dq"); check_grad(dk, rk, "dk"); check_grad(dv, rv, "dv")


def test_block_sparse_d64_gqa():
    wl = W.block_sparse(total=1500, hq=6, hkv=2, d=64, q_block=64, k_block=16, seed=23)
    q, k, v, do = W.make_tensors(wl, with_dout=True)
    out, lse, dq, dk, dv = run(wl, q, k, v, do)
    ro, rl = oracle.fwd(q, k, v, wl.q_ranges, wl.k_ranges, wl.mask_types)
    check_fwd(out, lse, ro, rl)
    rq, rk, rv = oracle.bwd(q, k, v, do, wl.q_ranges, wl.k_ranges, wl.mask_types)
    check_grad(dq, rq, "dq"); check_grad(dk, rk, "dk"); check_grad(dv, rv, "dv")


@pytest.mark.parametrize("name,with_dkv", [("block_sparse_64x64", True), ("block_sparse_16x64", True),
                                           ("block_sparse_64x1", False)])
def test_block_sparse_full_size_sampled(name, with_dkv):
    """Benchmark-size tables: forward on a sample of rows, dq on fewer rows,
    dk/dv on a few keys (skipped for the half-million-slice table, where the
    oracle's per-key pass alone takes half a minute)."""
    wl = W.CONFIGS[name]()
    q, k, v, do = W.make_tensors(wl, with_dout=True)
    out, lse, dq, dk, dv = run(wl, q, k, v, do)
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(wl.total_q, 48, replace=False))
    ro, rl = oracle.fwd(q, k, v, wl.q_ranges, wl.k_ranges, wl.mask_types, rows=rows)
    check_fwd(out, lse, ro, rl, rows=rows)
    keys = np.sort(rng.choice(wl.total_k, 4, replace=False)) if with_dkv else np.zeros(0, np.int64)
    rq, rk, rv = oracle.bwd(q, k, v, do, wl.q_ranges, wl.k_ranges, wl.mask_types,
                            dq_rows=rows[:12], dkv_keys=keys)
    check_grad(dq[rows[:12]], rq, "dq")
    if with_dkv:
        check_grad(dk[keys], rk, "dk"); check_grad(dv[keys], rv, "dv")


# Gathered steps in the capped kernels and with sink logits: the tables gather
# in both directions (every forward unit and every k-tile; the T = 1500 one
# with a ragged last query block, GQA g = 3, D = 64).  Scale 2.5 and cap 5
# push scores outside the tanh polynomial's range (exponential form); scale 1
# and cap 30 keep them inside it.
GATHERED_EXT = [
    # (total, hq, hkv, d, q_block, k_block, seed, input scale, cap)
    (2048, 4, 2, 128, 32, 64, 31, 2.5, 5.0),
    (2048, 4, 2, 128, 64, 64, 32, 1.0, 30.0),
    (1500, 6, 2, 64, 64, 16, 33, 2.5, 5.0),
]


@pytest.mark.parametrize("case", GATHERED_EXT,
                         ids=[f"T{c[0]}_D{c[3]}_q{c[4]}_k{c[5]}_cap{c[8]:g}" for c in GATHERED_EXT])
def test_block_sparse_gathered_softcap_sink(case):
    total, hq, hkv, d, qb, kb, seed, scale, cap = case
    wl = W.block_sparse(total=total, hq=hq, hkv=hkv, d=d, q_block=qb, k_block=kb, seed=seed)
    q, k, v, do = W.make_tensors(wl, with_dout=True)
    q = (q.float() * scale).to(torch.bfloat16)
    k = (k.float() * scale).to(torch.bfloat16)
    sink = (2.0 * torch.randn(2, hq, generator=torch.Generator().manual_seed(seed))).float()
    plan = ffa.ffa_plan_create(wl.q_ranges, wl.k_ranges, wl.mask_types, wl.total_q, wl.total_k,
                               hq, hkv, d)
    info = ffa.ffa_plan_info(plan)
    assert info["gathers"] > 0 and info["bgathers"] > 0
    qd, kd, vd, dod, sd = (t.to(DEV) for t in (q, k, v, do, sink))
    out, lse = ffa.ffa_fwd_ex(plan, qd, kd, vd, sink=sd, softcap=cap)
    dq, dk, dv, ds = ffa.ffa_bwd_ex(plan, qd, kd, vd, out, dod, lse, sink=sd, softcap=cap)
    torch.cuda.synchronize()
    assert ffa.ffa_get_last_device_error(plan) == (0, 0)
    a = (wl.q_ranges, wl.k_ranges, wl.mask_types)
    ro, rl = oracle.fwd(q, k, v, *a, sink=sink, softcap=cap)
    check_fwd(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl)
    rq, rk, rv = oracle.bwd(q, k, v, do, *a, sink=sink, softcap=cap)
    check_grad(dq.float().cpu().numpy(), rq, "dq")
    check_grad(dk.float().cpu().numpy(), rk, "dk")
    check_grad(dv.float().cpu().numpy(), rv, "dv")
    rs = oracle.dsink(q, k, v, do, *a, sink, "sh", softcap=cap)
    check_grad(ds.cpu().numpy(), rs, "dsink")



# Head-stacked forward units (a 128-row tile holds one 64-row slab of two
# query heads, or one 32-row slab of four): Hq / Hkv = 4, 6 or 8, ragged T,
# D = 128 and 64, with and without sink logits and softcap.
STACKED = [
    # (total, hq, hkv, d, q_block, k_block, seed, sink, cap)
    (2000, 8, 2, 128, 64, 64, 51, False, 0.0),
    (2000, 8, 2, 128, 16, 64, 52, True, 0.0),
    (1500, 12, 2, 64, 32, 64, 53, False, 0.0),
    (1000, 4, 1, 128, 64, 8, 54, True, 5.0),
    (2000, 8, 2, 128, 16, 64, 55, False, 30.0),   # 32-row slabs of four heads
    (1000, 16, 2, 64, 16, 64, 56, True, 0.0),     # 32-row slabs, both halves busy
]


@pytest.mark.parametrize("case", STACKED,
                         ids=[f"T{c[0]}_H{c[1]}x{c[2]}_D{c[3]}_q{c[4]}_k{c[5]}" for c in STACKED])
def test_block_sparse_stacked(case):
    total, hq, hkv, d, qb, kb, seed, with_sink, cap = case
    wl = W.block_sparse(total=total, hq=hq, hkv=hkv, d=d, q_block=qb, k_block=kb, seed=seed)
    q, k, v, do = W.make_tensors(wl, with_dout=True)
    if cap > 0:
        q = (q.float() * 2.5).to(torch.bfloat16)
        k = (k.float() * 2.5).to(torch.bfloat16)
    sink = (2.0 * torch.randn(2, hq, generator=torch.Generator().manual_seed(seed))).float() \
        if with_sink else None
    plan = ffa.ffa_plan_create(wl.q_ranges, wl.k_ranges, wl.mask_types, wl.total_q, wl.total_k,
                               hq, hkv, d)
    assert ffa.ffa_plan_info(plan)["stacked"] in (32, 64)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    sd = sink.to(DEV) if sink is not None else None
    out, lse = ffa.ffa_fwd_ex(plan, qd, kd, vd, sink=sd, softcap=cap)
    dq, dk, dv, ds = ffa.ffa_bwd_ex(plan, qd, kd, vd, out, dod, lse, sink=sd, softcap=cap)
    torch.cuda.synchronize()
    assert ffa.ffa_get_last_device_error(plan) == (0, 0)
    a = (wl.q_ranges, wl.k_ranges, wl.mask_types)
    ro, rl = oracle.fwd(q, k, v, *a, sink=sink, softcap=cap)
    check_fwd(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl)
    rq, rk, rv = oracle.bwd(q, k, v, do, *a, sink=sink, softcap=cap)
    check_grad(dq.float().cpu().numpy(), rq, "dq")
    check_grad(dk.float().cpu().numpy(), rk, "dk")
    check_grad(dv.float().cpu().numpy(), rv, "dv")
    if sink is not None:
        rs = oracle.dsink(q, k, v, do, *a, sink, "sh", softcap=cap)
        check_grad(ds.cpu().numpy(), rs, "dsink")
