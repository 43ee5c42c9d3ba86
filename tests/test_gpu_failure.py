"""Failure detection without a GPU fault: a wait limit far below any real
wait makes the kernels' bounded waits run out; they must stop, report a
timeout through the error word, and leave the context usable."""
import pytest
import torch

import flexible_mask_attention_gb300 as ffa
from flexible_mask_attention_gb300 import workloads as W
from gpu_helpers import bf16

pytestmark = pytest.mark.gpu


def _causal():
    T = 2048
    return [[0, T]], [[0, T]], [1]


def _block_sparse():
    # gathered steps in every pass: their producers split over three warps
    wl = W.block_sparse(total=2048, hq=4, hkv=4, d=128, q_block=32, k_block=64, seed=41)
    return wl.q_ranges, wl.k_ranges, wl.mask_types


@pytest.mark.parametrize("mask", [_causal, _block_sparse], ids=["causal", "block_sparse_gathered"])
def test_timeout_is_reported_and_context_survives(mask):
    T, H, D = 2048, 4, 128
    dev = torch.device("cuda", 0)
    q, k, v, do = (bf16(T, H, D, seed=s).to(dev) for s in range(4))
    qr, kr, ty = mask()
    ref = ffa.ffa_plan_create(qr, kr, ty, T, T, H, H, D)
    out_ref, lse_ref = ffa.ffa_fwd(ref, q, k, v)
    dq_ref, dk_ref, dv_ref = ffa.ffa_bwd(ref, q, k, v, out_ref, do, lse_ref)
    torch.cuda.synchronize()
    assert ffa.ffa_get_last_device_error(ref) == (0, 0)
    if mask is _block_sparse:
        info = ffa.ffa_plan_info(ref)
        assert info["gathers"] > 0 and info["bgathers"] > 0

    plan = ffa.ffa_plan_create(qr, kr, ty, T, T, H, H, D)
    ffa.ffa_plan_set_wait_limit(plan, 1)  # 1 ns: the first wait that must block gives up
    ffa.ffa_fwd(plan, q, k, v)
    torch.cuda.synchronize()
    code, where = ffa.ffa_get_last_device_error(plan)
    assert code == 1 and where != 0
    ffa.ffa_bwd(plan, q, k, v, out_ref, do, lse_ref)
    torch.cuda.synchronize()
    code, where = ffa.ffa_get_last_device_error(plan)
    assert code == 1 and where != 0

    # the same plan with a normal limit runs correctly afterwards
    ffa.ffa_plan_set_wait_limit(plan, 2_000_000_000)
    out, lse = ffa.ffa_fwd(plan, q, k, v)
    dq, dk, dv = ffa.ffa_bwd(plan, q, k, v, out, do, lse)
    torch.cuda.synchronize()
    assert ffa.ffa_get_last_device_error(plan) == (0, 0)
    assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref)
    assert torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref)
    assert (dq.float() - dq_ref.float()).abs().max() <= 1e-2 * dq_ref.float().abs().max()
