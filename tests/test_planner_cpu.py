"""CPU checks of the planner pieces that do not need a GPU:

* the oracle's counting planner against a dense brute force,
* the device planner's closed-form tile classification (compiled for the
  host from the product header) against the counting planner,
* the seeded workload generators against fixed values (document lengths,
  boundaries, mask types) computed independently with numpy's PCG64 when
  the workloads were specified.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from oracle import dense, planner
from flexible_mask_attention_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SEG_HEADER = os.path.join(ROOT, "flexible_mask_attention_gb300", "csrc", "ffa_segments.cuh")


@pytest.mark.parametrize("seed", range(8))
def test_counts_match_dense(seed):
    rng = np.random.default_rng(seed)
    Tq, Tk = int(rng.integers(100, 700)), int(rng.integers(100, 700))
    qr, kr, ty = W.random_slices(Tq, Tk, int(rng.integers(2, 8)), seed=seed)
    counts = planner.tile_counts(qr, kr, ty)
    for s in range(len(ty)):
        m = dense.dense_mask(Tq, Tk, qr[s:s + 1], kr[s:s + 1], ty[s:s + 1])
        nq, nk = -(-Tq // 128), -(-Tk // 128)
        pad = np.zeros((nq * 128, nk * 128), dtype=np.int64)
        pad[:Tq, :Tk] = m
        blocks = pad.reshape(nq, 128, nk, 128).sum(axis=(1, 3))
        got = np.zeros_like(blocks)
        for (qt, kt), c in counts[s].items():
            got[qt, kt] = c
        assert (got == blocks).all()
    assert planner.visible_area(qr, kr, ty) == dense.dense_mask(Tq, Tk, qr, kr, ty).sum()


@pytest.fixture(scope="module")
def seg_lib(tmp_path_factory):
    d = tmp_path_factory.mktemp("seg")
    src = d / "harness.cpp"
    src.write_text(f"""
#define __host__
#define __device__
#include "{SEG_HEADER}"
using namespace ffa;
extern "C" int fwd_run(int qs, int qe, int ks, int ke, int t, int qt, int* o) {{
  SliceDesc s{{qs, qe, ks, ke, t}}; TileRun r;
  if (!fwd_tile_run(s, qt, r)) return 0;
  o[0] = r.b; o[1] = r.fb; o[2] = r.fe; o[3] = r.e; return 1;
}}
extern "C" int bwd_run(int qs, int qe, int ks, int ke, int t, int kt, int* o) {{
  SliceDesc s{{qs, qe, ks, ke, t}}; TileRun r;
  if (!bwd_tile_run(s, kt, r)) return 0;
  o[0] = r.b; o[1] = r.fb; o[2] = r.fe; o[3] = r.e; return 1;
}}
extern "C" long long area(int qs, int qe, int ks, int ke, int t) {{
  return slice_area(SliceDesc{{qs, qe, ks, ke, t}});
}}
""")
    so = d / "libseg.so"
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-o", str(so), str(src)])
    lib = ctypes.CDLL(str(so))
    lib.area.restype = ctypes.c_longlong
    return lib


def _closed_form_counts(lib, s, Tq, Tk):
    """{(qt, kt): 'F'|'P'} from the closed forms, forward and backward views."""
    o = (ctypes.c_int * 4)()
    fwd, bwd = {}, {}
    for qt in range(-(-Tq // 128)):
        if lib.fwd_run(*s, qt, o):
            b, fb, fe, e = list(o)
            for kt in range(b, e):
                fwd[(qt, kt)] = "F" if fb <= kt < fe else "P"
    for kt in range(-(-Tk // 128)):
        if lib.bwd_run(*s, kt, o):
            b, fb, fe, e = list(o)
            for qt in range(b, e):
                bwd[(qt, kt)] = "F" if fb <= qt < fe else "P"
    return fwd, bwd


def _check_slices(lib, qr, kr, ty, Tq, Tk):
    counts = planner.tile_counts(qr, kr, ty)
    for s in range(len(ty)):
        sl = (int(qr[s][0]), int(qr[s][1]), int(kr[s][0]), int(kr[s][1]), int(ty[s]))
        ref = {key: ("F" if c == 128 * 128 else "P") for key, c in counts[s].items()}
        fwd, bwd = _closed_form_counts(lib, sl, Tq, Tk)
        assert fwd == ref, f"forward classification differs for slice {sl}"
        assert bwd == ref, f"backward classification differs for slice {sl}"
        assert lib.area(*sl) == planner.visible_area(qr[s:s + 1], kr[s:s + 1], ty[s:s + 1])


@pytest.mark.parametrize("seed", range(20))
def test_closed_forms_random(seg_lib, seed):
    rng = np.random.default_rng(1000 + seed)
    Tq, Tk = int(rng.integers(50, 1500)), int(rng.integers(50, 1500))
    qr, kr, ty = W.random_slices(Tq, Tk, int(rng.integers(1, 9)), seed=seed,
                                 aligned=bool(seed % 3 == 0))
    _check_slices(seg_lib, qr, kr, ty, Tq, Tk)


def test_closed_forms_edge_shapes(seg_lib):
    cases = []
    for t in range(4):
        for qlen, klen in [(1, 1), (1, 300), (300, 1), (128, 128), (129, 127), (127, 129),
                           (256, 384), (384, 256), (500, 500)]:
            for qs, ks in [(0, 0), (5, 130), (128, 0), (77, 255)]:
                cases.append((qs, qs + qlen, ks, ks + klen, t))
    for c in cases:
        qr, kr, ty = np.array([[c[0], c[1]]]), np.array([[c[2], c[3]]]), np.array([c[4]])
        _check_slices(seg_lib, qr, kr, ty, c[1] + 3, c[3] + 3)


def test_workload_generators_match_recorded_values():
    assert W.packed_doc_lengths(32768, 2) == [2474, 1214, 1355, 277, 12386, 6430, 1479, 4440, 2713]
    wl = W.heterogeneous_prefix_docs()
    assert wl.meta["bounds"] == [4096, 6140, 12656, 14098, 18967, 20502, 21601, 23129, 27005, 29038,
                                 29636, 31385, 31699, 34519, 35807, 37712, 38846, 47227, 49095,
                                 50973, 52109, 56750, 64494, 65536]
    assert wl.meta["doc_types"] == [1, 2, 1, 3, 0, 0, 2, 2, 3, 0, 2, 0, 1, 3, 0, 1, 1, 2, 3, 2, 0, 1, 3]
    assert wl.num_slices == 47
    assert W.long_context_docs().num_slices == 64


@pytest.mark.parametrize("name,area,full,partial", [
    ("packed_causal", 1.1678e8, 6773, 727),
    ("heterogeneous", 4.0434e8, 23296, 2740),
    ("long_context", 2.8858e9, 175104, 2048),
])
def test_config_areas_and_tile_mix(name, area, full, partial):
    wl = W.CONFIGS[name]()
    counts = planner.tile_counts(wl.q_ranges, wl.k_ranges, wl.mask_types)
    nf = sum(1 for d in counts.values() for c in d.values() if c == 128 * 128)
    npart = sum(1 for d in counts.values() for c in d.values() if c < 128 * 128)
    a = planner.visible_area(wl.q_ranges, wl.k_ranges, wl.mask_types)
    assert abs(a - area) / area < 1e-4
    assert (nf, npart) == (full, partial)


def test_plan_split_and_order_rules():
    wl = W.tiny_causal_docs()
    p = planner.plan(256, 256, 1, 1, wl.q_ranges, wl.k_ranges, wl.mask_types, num_sms=152)
    # one unit (q-tiles 0, 1), two steps, split into two single-step chunks
    # info = (slice << 2) | partial
    assert p["fwd_steps"].tolist() == [[0, 1, -1, 0], [1, -1, 5, 0]]
    assert p["fwd_items"].tolist() == [[0, 1, 0, 0, 0, 1, 0, 5], [0, 1, 0, 0, 1, 2, 1, 5]]
    assert p["merges"].tolist() == [[0, 1, 0, 0, 0, 2, 0, 0]]
    q = planner.plan(256, 256, 1, 1, wl.q_ranges, wl.k_ranges, wl.mask_types, num_sms=152,
                     split_below=-1)
    assert q["fwd_items"].tolist() == [[0, 1, 0, 0, 0, 2, -1, 10]]
    assert q["bwd_items"].tolist() == [[0, 0, 0, 1, 5, 0, 0, 0], [1, 0, 1, 2, 5, 0, 0, 0]]


# (q block, k block, seed, heads) of tables the planner gathers for
FWD_GATHER_CASES = [((64, 64), 1, (4, 2)), ((64, 64), 1, (2, 2)), ((64, 8), 2, (4, 2)),
                    ((64, 8), 2, (2, 2)), ((16, 64), 3, (4, 2)), ((64, 16), 5, (2, 2))]
BWD_GATHER_CASES = [((64, 64), 1, (4, 2)), ((16, 64), 3, (2, 2)), ((8, 64), 4, (4, 2)),
                    ((64, 16), 5, (2, 2))]


def _block_sparse_plan(blocks, seed, heads, T=1000):
    """A ragged block-sparse table (T not a multiple of the tile or of the
    blocks), its dense mask and the CPU planner's lists."""
    wl = W.block_sparse(total=T, hq=heads[0], hkv=heads[1], q_block=blocks[0],
                        k_block=blocks[1], seed=seed)
    m = dense.dense_mask(T, T, wl.q_ranges, wl.k_ranges, wl.mask_types).astype(bool)
    p = planner.plan(T, T, heads[0], heads[1], wl.q_ranges, wl.k_ranges, wl.mask_types,
                     num_sms=152)
    return m, p


def test_tile_aligned_blocks_do_not_gather():
    m, p = _block_sparse_plan((128, 128), 6, (4, 2), T=1024)
    assert p["gathers"].shape[0] == 0 and p["bgathers"].shape[0] == 0


@pytest.mark.parametrize("blocks,seed,heads", FWD_GATHER_CASES)
def test_gathered_steps_cover_the_mask_exactly(blocks, seed, heads):
    """Gathered forward steps (the planner specification for units of full,
    8-key aligned slices): for every item half, the (row, key) pairs its
    steps' slot row bits mark are exactly the visible pairs of its q-tile's
    rows in the dense mask, each once; keys past Tk are never marked, unused
    slots (start -8) carry no bits, slot starts ascend within a step."""
    m, p = _block_sparse_plan(blocks, seed, heads)
    T = m.shape[1]
    steps, rec = p["fwd_steps"], p["gathers"]
    assert rec.shape[0] > 0
    # a (q-tile, head) may be cut into several items (split): sum over them
    marked_by = {}
    for it in p["fwd_items"]:
        for h in range(2):
            qt, head = it[h], it[2 + h]
            if qt < 0 or head < 0:
                continue
            marked, gathered = marked_by.setdefault((qt, head), [np.zeros((128, T), np.int64), False])
            for st in steps[it[4]:it[5]]:
                if st[3] <= 0:
                    continue
                r = rec[st[3] - 1]
                starts = r[:16]
                assert (np.diff(starts[starts >= 0]) > 0).all() and (starts[starts < 0] == -8).all()
                words = r[16 + 64 * h: 16 + 64 * (h + 1)].view(np.uint32).reshape(16, 4)
                assert (st[1 + h] >= 0) == bool(words.any())
                for slot, y in enumerate(starts):
                    if y < 0:
                        assert not words[slot].any()
                        continue
                    bits = (words[slot][np.arange(128) >> 5] >> (np.arange(128) & 31)) & 1
                    for rr in np.nonzero(bits)[0]:
                        marked[rr, y:min(y + 8, T)] += 1
                marked_by[(qt, head)][1] = True
    n_halves = 0
    for (qt, head), (marked, gathered) in marked_by.items():
        if not gathered:
            continue
        n_halves += 1
        ref = m[128 * qt: min(128 * qt + 128, T)]
        got = marked[: ref.shape[0]]
        assert (got[ref] == 1).all(), "a visible pair is missed or listed twice"
        assert (got[~ref] == 0).all(), "an invisible pair is marked visible"
    assert n_halves > 0


@pytest.mark.parametrize("blocks,seed,heads", BWD_GATHER_CASES)
def test_gathered_backward_steps_cover_the_mask_exactly(blocks, seed, heads):
    """Gathered backward steps (the transpose: k-tiles of full slices with
    8-row aligned query ranges): over a k-tile's steps, the (row, key) pairs
    the slots' key bits mark are exactly the visible pairs of its keys in the
    dense mask, each once; rows past Tq are never marked; every kv head's
    item of the k-tile has the same steps."""
    m, p = _block_sparse_plan(blocks, seed, heads)
    Tq, Tk = m.shape
    steps, rec = p["bwd_steps"], p["bgathers"]
    assert rec.shape[0] > 0
    seen_tiles = 0
    for it in p["bwd_items"]:
        kt = it[0]
        st = steps[it[2]:it[3]]
        if not (st[:, 3] > 0).any():
            continue
        assert (st[:, 3] > 0).all() and (st[:, 1] == 1).all()
        seen_tiles += 1
        marked = np.zeros((Tq, 128), dtype=np.int64)
        for s_ in st:
            r = rec[s_[3] - 1]
            starts = r[:16]
            assert (np.diff(starts[starts >= 0]) > 0).all() and (starts[starts < 0] == -8).all()
            words = r[16:].view(np.uint32).reshape(16, 4)
            for slot, y in enumerate(starts):
                if y < 0:
                    assert not words[slot].any()
                    continue
                bits = (words[slot][np.arange(128) >> 5] >> (np.arange(128) & 31)) & 1
                for kk in np.nonzero(bits)[0]:
                    marked[y:min(y + 8, Tq), kk] += 1
        ref = m[:, 128 * kt: min(128 * kt + 128, Tk)]
        got = marked[:, : ref.shape[1]]
        assert (got[ref] == 1).all(), "a visible pair is missed or listed twice"
        assert (got[~ref] == 0).all(), "an invisible pair is marked visible"
    assert seen_tiles > 0


# (q block, k block, seed, heads) of tables whose forward units are stacked:
# Hq / Hkv = 4 or 6, T = 1000 (the last 64-row slab is ragged)
STACK_CASES = [((64, 64), 1, (8, 2)), ((16, 64), 3, (8, 2)), ((64, 8), 2, (4, 1)),
               ((32, 64), 7, (12, 2)), ((16, 64), 5, (16, 2)), ((16, 32), 8, (12, 2))]


@pytest.mark.parametrize("blocks,seed,heads", STACK_CASES)
def test_stacked_units_cover_the_mask_exactly(blocks, seed, heads):
    """Head-stacked forward units (the planner specification for g even and
    >= 4): with slabs of R rows and m = 128 / R heads per half, every (slab,
    query head) is tile rows [R j, R j + R) of one half of exactly one item;
    the (row, key) pairs its steps' row bits mark are exactly the visible
    pairs of the slab's rows, each once; the m row groups of a half carry
    the same bits; the plan is not split."""
    m_, p = _block_sparse_plan(blocks, seed, heads)
    R = p["stacked"]
    assert R in (32, 64) and p["merges"].shape[0] == 0
    T, Hq, g = m_.shape[1], heads[0], heads[0] // heads[1]
    m = 128 // R
    n_slabs = -(-T // R)
    steps, rec = p["fwd_steps"], p["gathers"]
    assert (steps[:, 3] > 0).all(), "every step of a stacked plan is gathered"
    marked, seen = {}, {}
    for it in p["fwd_items"]:
        assert it[6] == -1
        # with alternating halves both halves are the same (slab, heads): the
        # item covers them once, each half with its own steps
        covers = {(it[h], it[2 + h]) for h in range(2) if it[h] >= 0 and it[2 + h] >= 0}
        assert p["alternate"] == (len(covers) == 1 and it[1] >= 0)
        for u, h0 in covers:
            for j in range(m):
                seen[(u, h0 + j)] = seen.get((u, h0 + j), 0) + 1
                marked.setdefault((u, h0 + j), np.zeros((R, T), np.int64))
        for h in range(2):
            u, h0 = it[h], it[2 + h]
            if u < 0 or h0 < 0:
                continue
            assert h0 % m == 0 and h0 // g == (h0 + m - 1) // g
            for st in steps[it[4]:it[5]]:
                r = rec[st[3] - 1]
                starts = r[:16]
                words = r[16 + 64 * h: 16 + 64 * (h + 1)].view(np.uint32).reshape(16, 4)
                if p["alternate"] and st[1 + h] < 0:
                    continue  # the other half's step
                assert (st[1 + h] >= 0) == bool(words.any())
                for slot, y in enumerate(starts):
                    if y < 0:
                        assert not words[slot].any()
                        continue
                    bits = (words[slot][np.arange(128) >> 5] >> (np.arange(128) & 31)) & 1
                    for j in range(m):
                        assert (bits[R * j: R * j + R] == bits[:R]).all()
                        for rr in np.nonzero(bits[R * j: R * j + R])[0]:
                            marked[(u, h0 + j)][rr, y:min(y + 8, T)] += 1
    assert set(seen) == {(u, hq) for u in range(n_slabs) for hq in range(Hq)}
    assert all(c == 1 for c in seen.values())
    for (u, _), got in marked.items():
        ref = m_[R * u: min(R * u + R, T)]
        got = got[: ref.shape[0]]
        assert (got[ref] == 1).all(), "a visible pair is missed or listed twice"
        assert (got[~ref] == 0).all(), "an invisible pair is marked visible"


def test_stacking_needs_four_heads_and_every_slab_eligible():
    """Two heads per kv head do not stack; one causal slice among the blocks
    keeps the tile units."""
    _, p = _block_sparse_plan((64, 64), 1, (4, 2))
    assert not p["stacked"]
    wl = W.block_sparse(total=1000, hq=8, hkv=2, q_block=64, k_block=64, seed=1)
    ty = wl.mask_types.copy()
    ty[0] = 1
    p = planner.plan(1000, 1000, 8, 2, wl.q_ranges, wl.k_ranges, ty, num_sms=152)
    assert not p["stacked"]
