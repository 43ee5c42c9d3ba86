"""The device planner's work lists equal the CPU re-derivation bit for bit."""
import numpy as np
import pytest
import torch

import flexible_mask_attention_gb300 as ffa
from flexible_mask_attention_gb300 import workloads as W
from oracle import planner

pytestmark = pytest.mark.gpu

NAMES = ["fwd_steps", "fwd_items", "fwd_order", "bwd_steps", "bwd_items", "bwd_order", "merges",
         "fwd_masks", "bwd_masks", "gathers", "bgathers"]


def compare(qr, kr, ty, Tq, Tk, Hq, Hkv, D, split_below=0):
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    plan = ffa.ffa_plan_create(qr, kr, ty, Tq, Tk, Hq, Hkv, D, split_below=split_below)
    ref = planner.plan(Tq, Tk, Hq, Hkv, qr, kr, ty, num_sms=nsm, split_below=split_below)
    for which, name in enumerate(NAMES):
        got = ffa.ffa_plan_export(plan, which)
        exp = ref[name].reshape(got.shape) if ref[name].size == got.size else ref[name]
        assert got.shape == exp.shape and np.array_equal(got, exp), f"{name} differs"
    info = ffa.ffa_plan_info(plan)
    assert info["area"] == ref["area"]
    assert info["grid_fwd"] == ref["grid_fwd"] and info["grid_bwd"] == ref["grid_bwd"]
    assert info["stacked"] == ref["stacked"]
    plan.destroy()
    return ref


@pytest.mark.parametrize("name", ["tiny", "packed_causal", "heterogeneous", "long_context"])
def test_configs(name):
    wl = W.CONFIGS[name]()
    compare(wl.q_ranges, wl.k_ranges, wl.mask_types, wl.total_q, wl.total_k, wl.num_heads_q,
            wl.num_heads_kv, wl.head_dim)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("heads", [(4, 2), (2, 2), (3, 1)])
def test_random(seed, heads):
    rng = np.random.default_rng(seed)
    Tq, Tk = int(rng.integers(100, 3000)), int(rng.integers(100, 3000))
    qr, kr, ty = W.random_slices(Tq, Tk, int(rng.integers(1, 12)), seed=seed)
    compare(qr, kr, ty, Tq, Tk, heads[0], heads[1], 128, split_below=[0, -1, 400][seed % 3])


def test_rejects_bad_slices():
    with pytest.raises(ffa.FFAError) as e:
        ffa.ffa_plan_create([[0, 10], [5, 20]], [[0, 10], [5, 20]], [0, 0], 32, 32, 1, 1, 128)
    assert e.value.status == 3
    with pytest.raises(ffa.FFAError) as e:
        ffa.ffa_plan_create([[0, 40]], [[0, 10]], [0], 32, 32, 1, 1, 128)
    assert e.value.status == 2
    with pytest.raises(ffa.FFAError) as e:
        ffa.ffa_plan_create([[0, 10]], [[0, 10]], [5], 32, 32, 1, 1, 128)
    assert e.value.status == 2
    with pytest.raises(ffa.FFAError) as e:
        ffa.ffa_plan_create([[0, 10]], [[0, 10]], [0], 32, 32, 1, 1, 96)
    assert e.value.status == 4


@pytest.mark.parametrize("blocks", [(64, 64), (128, 128), (16, 64), (8, 64), (64, 8), (64, 1)])
def test_block_sparse(blocks):
    """Many tiny slices (uniform block-sparse masks): same lists as the CPU derivation."""
    wl = W.block_sparse(total=4096, hq=4, hkv=2, q_block=blocks[0], k_block=blocks[1], seed=9)
    compare(wl.q_ranges, wl.k_ranges, wl.mask_types, wl.total_q, wl.total_k, wl.num_heads_q,
            wl.num_heads_kv, wl.head_dim)


def test_overlap_found_between_tiny_slices():
    """The tile-local overlap check still sees an overlap hidden among many slices."""
    wl = W.block_sparse(total=4096, hq=2, hkv=2, q_block=64, k_block=8, seed=3)
    qr, kr = wl.q_ranges.copy(), wl.k_ranges.copy()
    qr[-1] = [qr[5][0] + 3, qr[5][0] + 9]   # rows inside q block 0
    kr[-1] = [kr[5][0] + 1, kr[5][0] + 2]   # a key of slice 5
    with pytest.raises(ffa.FFAError) as e:
        ffa.ffa_plan_create(qr, kr, wl.mask_types, 4096, 4096, 2, 2, 128)
    assert e.value.status == 3


@pytest.mark.parametrize("blocks,heads,T", [((64, 64), (8, 2), 4096), ((16, 64), (8, 2), 4096),
                                            ((64, 8), (4, 1), 4096), ((32, 64), (12, 2), 1000),
                                            ((16, 64), (16, 2), 1000)])
def test_block_sparse_stacked(blocks, heads, T):
    """Head-stacked forward units (4, 6 or 8 query heads per kv head; 64- and
    32-row slabs): the same lists and the same choice as the CPU derivation."""
    wl = W.block_sparse(total=T, hq=heads[0], hkv=heads[1], q_block=blocks[0],
                        k_block=blocks[1], seed=11)
    ref = compare(wl.q_ranges, wl.k_ranges, wl.mask_types, T, T, heads[0], heads[1],
                  wl.head_dim)
    assert ref["stacked"]
