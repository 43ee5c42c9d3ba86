"""Forward parity: CUDA path vs the fp64 oracle on the same seeded bf16 inputs."""
import numpy as np
import pytest

import oracle
from flexible_mask_attention_gb300 import workloads as W
from gpu_helpers import bf16, check_fwd, run_fwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("split_below", [0, -1])
def test_tiny_causal_docs(split_below):
    wl = W.tiny_causal_docs()
    q, k, v = W.make_tensors(wl)
    _, out, lse = run_fwd(q, k, v, wl.q_ranges, wl.k_ranges, wl.mask_types, split_below=split_below)
    ro, rl = oracle.fwd(q, k, v, wl.q_ranges, wl.k_ranges, wl.mask_types)
    check_fwd(out, lse, ro, rl)


CASES = [
    # (Tq, Tk, Hq, Hkv, D, n_segments, seed)
    (1000, 1000, 4, 2, 128, 5, 1),   # grouped heads -> head pairs, ragged tail
    (777, 777, 2, 2, 128, 4, 2),     # one head per kv head -> q-tile pairs
    (640, 900, 3, 1, 128, 6, 3),     # odd group size, Tq != Tk
    (1000, 1000, 4, 2, 64, 5, 4),
    (515, 515, 1, 1, 64, 3, 5),
]


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}x{c[1]}_H{c[2]}/{c[3]}_D{c[4]}" for c in CASES])
@pytest.mark.parametrize("split_below", [-1, 0])
def test_random_slices(case, split_below):
    Tq, Tk, Hq, Hkv, D, nseg, seed = case
    qr, kr, ty = W.random_slices(Tq, Tk, nseg, seed=seed)
    q, k, v = bf16(Tq, Hq, D, seed=seed), bf16(Tk, Hkv, D, seed=seed + 1), bf16(Tk, Hkv, D, seed=seed + 2)
    _, out, lse = run_fwd(q, k, v, qr, kr, ty, split_below=split_below)
    ro, rl = oracle.fwd(q, k, v, qr, kr, ty)
    check_fwd(out, lse, ro, rl)


@pytest.mark.parametrize("t", [0, 1, 2, 3])
def test_single_type_aligned_and_unaligned(t):
    T, H, D = 1024, 2, 128
    qr = [[0, 300], [300, 700], [700, 1024], [128, 256]]
    kr = [[0, 512], [300, 701], [650, 1024], [900, 1000]]
    # slice 3's rectangle is disjoint from the others only for keys >= 900 rows 128..256:
    # rows 128..256 are also in slice 0 (keys 0..512), so keys 900..1000 do not overlap.
    q, k, v = bf16(T, H, D, seed=10 + t), bf16(T, H, D, seed=20 + t), bf16(T, H, D, seed=30 + t)
    ty = [t, t, t, (t + 1) % 4]
    _, out, lse = run_fwd(q, k, v, qr, kr, ty)
    ro, rl = oracle.fwd(q, k, v, qr, kr, ty)
    check_fwd(out, lse, ro, rl)


def test_no_slices_all_rows_empty():
    T, H, D = 300, 2, 128
    q, k, v = bf16(T, H, D, seed=1), bf16(T, H, D, seed=2), bf16(T, H, D, seed=3)
    _, out, lse = run_fwd(q, k, v, np.zeros((0, 2)), np.zeros((0, 2)), np.zeros((0,)))
    assert (out == 0).all() and np.isneginf(lse).all()


def test_large_scores_rescale():
    """Inputs with a large spread of scores exercise the lazy max-rescale path."""
    T, H, D = 1024, 2, 128
    q = bf16(T, H, D, seed=7) * 4
    k = bf16(T, H, D, seed=8) * 4
    v = bf16(T, H, D, seed=9)
    q, k = q.to(q.dtype), k.to(k.dtype)
    qr, kr, ty = [[0, T]], [[0, T]], [1]
    _, out, lse = run_fwd(q, k, v, qr, kr, ty)
    ro, rl = oracle.fwd(q, k, v, qr, kr, ty)
    check_fwd(out, lse, ro, rl)


def test_scores_far_below_zero():
    """Every visible score lies far below 0 (q ~ +1, k ~ -1): the running
    maximum starts far under the scale of the first tile's values, and the
    result must not underflow to an empty row."""
    import torch
    T, H, D = 700, 2, 128
    g = torch.Generator().manual_seed(11)
    q = (1.0 + 0.1 * torch.randn(T, H, D, generator=g)).to(torch.bfloat16)
    k = (-1.0 + 0.1 * torch.randn(T, H, D, generator=g)).to(torch.bfloat16)
    v = bf16(T, H, D, seed=12)
    qr, kr, ty = [[0, 400], [400, T]], [[0, 400], [0, T]], [1, 0]
    _, out, lse = run_fwd(q, k, v, qr, kr, ty)
    ro, rl = oracle.fwd(q, k, v, qr, kr, ty)
    assert np.isfinite(lse).all() and (lse < -3).all()
    check_fwd(out, lse, ro, rl)
