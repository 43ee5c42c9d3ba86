"""The allocation-free backward entry point (ffa_bwd_noalloc), called through
the C ABI, gives the same gradients as ffa_bwd with a caller workspace, on two
calls in a row (the second call reuses the shared scratch array, so whatever
must start at zero has to be cleared again).  Collected last on purpose."""
import ctypes

import pytest
import torch

import flexible_mask_attention_gb300 as ffa
from gpu_helpers import GRAD_REL, bf16

pytestmark = pytest.mark.gpu


def _c_noalloc(lib, plan, q, k, v, out, do, lse, dq, dk, dv):
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.ffa_bwd_noalloc(plan.handle, P(q), P(k), P(v), P(out), P(do), P(lse),
                               ctypes.c_float(0.0), P(dq), P(dk), P(dv), st)


def test_noalloc_matches_workspace_backward_twice():
    lib = ffa.load_library()
    dev = torch.device("cuda", 0)
    Tq, Tk, Hq, Hkv, D = 1500, 1300, 4, 2, 128
    qr = [[0, 700], [700, 1500], [200, 600]]
    kr = [[0, 650], [500, 1300], [1000, 1300]]
    ty = [1, 3, 0]
    q, do = bf16(Tq, Hq, D, seed=1).to(dev), bf16(Tq, Hq, D, seed=2).to(dev)
    k, v = bf16(Tk, Hkv, D, seed=3).to(dev), bf16(Tk, Hkv, D, seed=4).to(dev)
    plan = ffa.ffa_plan_create(qr, kr, ty, Tq, Tk, Hq, Hkv, D)
    assert ffa.ffa_bwd_workspace_size(plan) <= lib.ffa_bwd_noalloc_max_workspace()
    out, lse = ffa.ffa_fwd(plan, q, k, v)
    ref = ffa.ffa_bwd(plan, q, k, v, out, do, lse)
    torch.cuda.synchronize()
    for _ in range(2):
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in ref)
        assert _c_noalloc(lib, plan, q, k, v, out, do, lse, dq, dk, dv) == 0
        torch.cuda.synchronize()
        assert ffa.ffa_get_last_device_error(plan) == (0, 0)
        for g, r in zip((dq, dk, dv), ref):
            gf, rf = g.float(), r.float()
            assert torch.isfinite(gf).all()
            assert (gf - rf).abs().max().item() <= GRAD_REL * max(rf.abs().max().item(), 1e-6)


def test_noalloc_rejects_plans_beyond_the_scratch_size():
    lib = ffa.load_library()
    dev = torch.device("cuda", 0)
    # 262144 rows x 64 heads: the lse/delta scratch alone is 128 MiB
    T, H, D = 262144, 64, 128
    plan = ffa.ffa_plan_create([[0, 256]], [[0, 256]], [0], T, T, H, H, D)
    assert ffa.ffa_bwd_workspace_size(plan) > lib.ffa_bwd_noalloc_max_workspace()
    # the size check comes before any use of the tensors, so small stand-ins do
    x = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(16, dtype=torch.float32, device=dev)
    assert _c_noalloc(lib, plan, x, x, x, x, x, lse, x, x, x) == 5  # FFA_ERR_WORKSPACE
