"""Parity of the longest dK/dV accumulations against the oracle.

A shared prefix visible to every later document (MagiAttention pages, card
"Initialize MagiAttention Meta Configs": block-causal masks where every
later block sees the first) gives the prefix k-tiles the most (q-tile, head)
steps of any dK/dV work item: 128 per item on the 16K-token case below, 512
on the 64K-token benchmark mask.  These tests compare exactly those
gradients with the fp64 oracle:

  * the 16K-token version of the benchmark mask (4096-token prefix, 11
    documents of all four mask types, 2 heads) in full: every element of
    out, lse, dq, dk and dv;
  * the 32K-token packed-causal mask (its documents, one kv head of 4 query
    heads) in full;
  * the 64K-token benchmark mask and the packed-causal mask at full size, in
    the launch configuration the benchmark times, on the keys seen by the
    most rows (prefix keys, the first keys of the longest causal documents,
    the last keys of the longest inverse-causal ones) and on random prefix
    keys.  Heads are independent, so the oracle runs on two kv-head groups
    only, which keeps its all-rows lse pass to seconds."""
import numpy as np
import pytest
import torch

import oracle
import flexible_mask_attention_gb300 as ffa
from flexible_mask_attention_gb300 import workloads as W
from gpu_helpers import check_fwd, check_grad
from heavy_keys import heaviest_keys

pytestmark = pytest.mark.gpu


def run_path(wl):
    dev = torch.device("cuda", 0)
    q, k, v, do = W.make_tensors(wl, with_dout=True)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    plan = ffa.ffa_plan_create(wl.q_ranges, wl.k_ranges, wl.mask_types, wl.total_q, wl.total_k,
                               wl.num_heads_q, wl.num_heads_kv, wl.head_dim)
    out, lse = ffa.ffa_fwd(plan, qd, kd, vd)
    dq, dk, dv = ffa.ffa_bwd(plan, qd, kd, vd, out, dod, lse)
    torch.cuda.synchronize()
    assert ffa.ffa_get_last_device_error(plan) == (0, 0)
    plan.destroy()
    return (q, k, v, do), out, lse, (dq, dk, dv)


def test_mid_size_prefix_mask_every_element():
    wl = W.CONFIGS["heterogeneous_mid"]()
    assert set(wl.meta["doc_types"]) == {0, 1, 2, 3}
    (q, k, v, do), out, lse, (dq, dk, dv) = run_path(wl)
    ro, rl = oracle.fwd(q, k, v, wl.q_ranges, wl.k_ranges, wl.mask_types)
    check_fwd(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl)
    rq, rk, rv = oracle.bwd(q, k, v, do, wl.q_ranges, wl.k_ranges, wl.mask_types)
    check_grad(dq.float().cpu().numpy(), rq, "dq")
    check_grad(dk.float().cpu().numpy(), rk, "dk")
    check_grad(dv.float().cpu().numpy(), rv, "dv")
    # the prefix keys are the heaviest items: each is seen by every row
    prefix = wl.meta["bounds"][0]
    for g, r, n in ((dk, rk, "dk prefix"), (dv, rv, "dv prefix")):
        check_grad(g.float().cpu().numpy()[:prefix], r[:prefix], n)


def _head_subset(wl, tensors, kv_heads):
    g = wl.num_heads_q // wl.num_heads_kv
    qh = [h for hk in kv_heads for h in range(hk * g, (hk + 1) * g)]
    q, k, v, do = tensors
    return qh, (q[:, qh].contiguous(), k[:, kv_heads].contiguous(), v[:, kv_heads].contiguous(),
                do[:, qh].contiguous())


@pytest.mark.parametrize("name", ["heterogeneous", "packed_causal"])
def test_full_size_heaviest_keys(name):
    wl = W.CONFIGS[name]()
    tensors, out, lse, (dq, dk, dv) = run_path(wl)
    prefix = wl.meta["bounds"][0] if "bounds" in wl.meta else None
    keys, seen = heaviest_keys(wl, n_top=8, n_random_prefix=4 if prefix else 0, prefix=prefix,
                               seed=21)
    # the chosen keys include ones every row sees (prefix) or a whole long
    # document sees
    assert seen[keys].max() >= (wl.total_q if prefix else max(wl.meta["doc_lens"]))
    kv_heads = [0, wl.num_heads_kv - 1]
    qh, sub = _head_subset(wl, tensors, kv_heads)
    _, rk, rv = oracle.bwd(*sub, wl.q_ranges, wl.k_ranges, wl.mask_types, dq_rows=[],
                           dkv_keys=keys)
    gk = dk.float().cpu().numpy()[keys][:, kv_heads]
    gv = dv.float().cpu().numpy()[keys][:, kv_heads]
    check_grad(gk, rk, "dk")
    check_grad(gv, rv, "dv")


def test_packed_causal_every_element():
    """The packed-document causal mask (32768 tokens, lognormal document
    lengths up to 16K, the backward workload of the benchmark tables) with
    one kv head of 4 query heads: every element of out, lse, dq, dk and dv
    against the oracle.  Its longest document (12386 tokens) gives dK/dV
    items of up to 97 q-tile steps per head."""
    wl = W.CONFIGS["packed_causal_h4"]()
    assert wl.total_q == 32768 and wl.num_heads_q == 4 * wl.num_heads_kv
    (q, k, v, do), out, lse, (dq, dk, dv) = run_path(wl)
    a = (wl.q_ranges, wl.k_ranges, wl.mask_types)
    ro, rl = oracle.fwd(q, k, v, *a)
    check_fwd(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl)
    rq, rk, rv = oracle.bwd(q, k, v, do, *a)
    check_grad(dq.float().cpu().numpy(), rq, "dq")
    check_grad(dk.float().cpu().numpy(), rk, "dk")
    check_grad(dv.float().cpu().numpy(), rv, "dv")
