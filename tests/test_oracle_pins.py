"""Pins for the CPU oracle: everything here checks it against something other
than itself (page fixtures, library routines, brute force, invariants)."""
import math
import os
import re
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

import oracle
from oracle import dense
from flexible_mask_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(*shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def _f64(t):
    return t.to(torch.float64)


def read_mask_fixture(name):
    meta, rows = {}, []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tok = line.split()
        if tok[0] in ("*", "0"):
            rows.append([c == "*" for c in tok])
        else:
            meta[tok[0]] = [int(x) for x in tok[1:]]
    return meta, np.array(rows, dtype=bool)


def visible_counts_from_oracle(total, qr, kr, ty, lib=None):
    """|V(i)| read back from the oracle: with q = 0 every visible score is 0,
    so lse_i = log |V(i)| (and -inf for an empty row)."""
    q = torch.zeros(total, 1, 8, dtype=torch.bfloat16)
    k = _bf16(total, 1, 8, seed=5)
    v = _bf16(total, 1, 8, seed=6)
    _, lse = oracle.fwd(q, k, v, qr, kr, ty, lib=lib)
    with np.errstate(over="ignore"):
        return np.where(np.isfinite(lse[0]), np.rint(np.exp(lse[0])), 0).astype(np.int64)


@pytest.mark.parametrize("fixture", ["quickstart_mask_blocks.txt", "block_causal_ranges.txt"])
def test_page_mask_pictures(fixture):
    meta, picture = read_mask_fixture(fixture)
    total, blk = meta["total"][0], meta["block"][0]
    qr = np.array(meta["q_ranges"]).reshape(-1, 2)
    kr = np.array(meta["k_ranges"]).reshape(-1, 2)
    ty = np.array(meta["types"])
    if total > 4096:
        # full slices only: shrinking every coordinate by f keeps the block picture
        assert (ty == 0).all()
        f = total // 2048
        assert total % f == 0 and blk % f == 0 and (qr % f == 0).all() and (kr % f == 0).all()
        total, blk, qr, kr = total // f, blk // f, qr // f, kr // f
    mask = dense.dense_mask(total, total, qr, kr, ty)
    nb = total // blk
    blocks = mask.reshape(nb, blk, nb, blk).any(axis=(1, 3))
    assert (blocks == picture).all()
    if total <= 4096:
        counts = visible_counts_from_oracle(total, qr, kr, ty)
        assert (counts == mask.sum(axis=1)).all()


def test_quickstart_row_alignment():
    """Bottom-right alignment of the 1024 x 2048 causal slice: the first row of
    the slice (token 1024) sees keys [0, 1025), the last sees all 2048."""
    qr, kr, ty = [[0, 1024], [1024, 2048]], [[0, 1024], [0, 2048]], [0, 1]
    counts = visible_counts_from_oracle(2048, qr, kr, ty)
    assert counts[0] == 1024 and counts[1023] == 1024
    assert counts[1024] == 1025 and counts[2047] == 2048


def _check_vs_dense(Tq, Tk, Hq, Hkv, D, qr, kr, ty, seed, lib=None, tol=1e-12):
    q, k, v = _bf16(Tq, Hq, D, seed=seed), _bf16(Tk, Hkv, D, seed=seed + 1), _bf16(Tk, Hkv, D, seed=seed + 2)
    mask, count = dense.dense_mask(Tq, Tk, qr, kr, ty, return_count=True)
    assert count.max() <= 1, "slices overlap"
    ref_o, ref_l = dense.attention(dense.to_f64(q), dense.to_f64(k), dense.to_f64(v), mask)
    o, l = oracle.fwd(q, k, v, qr, kr, ty, lib=lib)
    fin = np.isfinite(ref_l)
    assert (np.isfinite(l) == fin).all()
    assert np.abs(l[fin] - ref_l[fin]).max(initial=0) < tol
    assert np.abs(o - ref_o).max() < tol
    return mask


@pytest.mark.parametrize("seed", range(6))
def test_oracle_matches_dense_random_slices(seed):
    rng = np.random.default_rng(100 + seed)
    Tq = int(rng.integers(40, 260))
    Tk = Tq if seed % 2 == 0 else int(rng.integers(40, 260))
    qr, kr, ty = W.random_slices(Tq, Tk, int(rng.integers(2, 7)), seed=seed)
    _check_vs_dense(Tq, Tk, 4, 2, 16, qr, kr, ty, seed)


def test_oracle_all_types_square_and_rect():
    # one slice of each type per block, with rectangles both wide and tall
    qr = [[0, 30], [30, 50], [50, 90], [90, 100], [100, 140], [140, 150], [150, 170], [170, 200]]
    kr = [[0, 30], [30, 80], [80, 100], [100, 140], [140, 150], [150, 190], [190, 195], [195, 200]]
    for t in range(4):
        _check_vs_dense(200, 200, 2, 1, 8, qr, kr, [t] * len(qr), seed=40 + t)


def test_single_full_slice_equals_sdpa_gqa():
    Tq, Tk, Hq, Hkv, D = 70, 90, 8, 2, 32
    q, k, v = _bf16(Tq, Hq, D, seed=1), _bf16(Tk, Hkv, D, seed=2), _bf16(Tk, Hkv, D, seed=3)
    o, l = oracle.fwd(q, k, v, [[0, Tq]], [[0, Tk]], [0])
    ref = F.scaled_dot_product_attention(_f64(q).permute(1, 0, 2)[None], _f64(k).permute(1, 0, 2)[None],
                                         _f64(v).permute(1, 0, 2)[None], enable_gqa=True)[0]
    assert np.abs(o - ref.permute(1, 0, 2).numpy()).max() < 1e-12
    # lse against torch.logsumexp of the scaled scores (library routine)
    kk = _f64(k).repeat_interleave(Hq // Hkv, dim=1)
    s = torch.einsum("qhd,khd->hqk", _f64(q), kk) / math.sqrt(D)
    assert np.abs(l - torch.logsumexp(s, -1).numpy()).max() < 1e-12


def test_square_causal_equals_sdpa_is_causal():
    T, H, D = 96, 3, 16
    q, k, v = _bf16(T, H, D, seed=7), _bf16(T, H, D, seed=8), _bf16(T, H, D, seed=9)
    o, _ = oracle.fwd(q, k, v, [[0, T]], [[0, T]], [1])
    ref = F.scaled_dot_product_attention(_f64(q).transpose(0, 1), _f64(k).transpose(0, 1),
                                         _f64(v).transpose(0, 1), is_causal=True).transpose(0, 1)
    assert np.abs(o - ref.numpy()).max() < 1e-12


@pytest.mark.parametrize("qlen,klen", [(40, 100), (100, 40), (64, 64)])
def test_rect_causal_equals_causal_lower_right(qlen, klen):
    H, D = 2, 16
    q, k, v = _bf16(qlen, H, D, seed=11), _bf16(klen, H, D, seed=12), _bf16(klen, H, D, seed=13)
    o, l = oracle.fwd(q, k, v, [[0, qlen]], [[0, klen]], [1])
    bias = causal_lower_right(qlen, klen)
    keep = bias._materialize(device="cpu").numpy()
    ok_rows = keep.any(axis=1)
    ref = F.scaled_dot_product_attention(_f64(q).transpose(0, 1), _f64(k).transpose(0, 1),
                                         _f64(v).transpose(0, 1), attn_mask=bias).transpose(0, 1).numpy()
    assert np.abs(o[ok_rows] - ref[ok_rows]).max() < 1e-12
    # rows that the clamp leaves empty: exactly zero output and -inf lse
    assert (o[~ok_rows] == 0).all() and np.isneginf(l[:, ~ok_rows]).all()
    # the dense characterisation agrees with the library's bottom-right mask
    assert (dense.slice_block(qlen, klen, 1) == keep).all()


@pytest.mark.parametrize("qlen,klen", [(40, 100), (100, 40), (50, 50)])
def test_inverse_causal_is_reversed_causal(qlen, klen):
    H, D = 2, 16
    q, k, v = _bf16(qlen, H, D, seed=21), _bf16(klen, H, D, seed=22), _bf16(klen, H, D, seed=23)
    o_inv, l_inv = oracle.fwd(q, k, v, [[0, qlen]], [[0, klen]], [2])
    o_c, l_c = oracle.fwd(q.flip(0), k.flip(0), v.flip(0), [[0, qlen]], [[0, klen]], [1])
    assert np.array_equal(np.isfinite(l_inv), np.isfinite(l_c[:, ::-1]))
    fin = np.isfinite(l_inv)
    assert np.abs(l_inv[fin] - l_c[:, ::-1][fin]).max(initial=0) < 1e-12
    assert np.abs(o_inv - o_c[::-1]).max() < 1e-12


@pytest.mark.parametrize("qlen,klen", [(40, 100), (30, 30), (60, 45)])
def test_bi_causal_is_both_clamps(qlen, klen):
    H, D = 1, 8
    q, k, v = _bf16(qlen, H, D, seed=31), _bf16(klen, H, D, seed=32), _bf16(klen, H, D, seed=33)
    causal = causal_lower_right(qlen, klen)._materialize(device="cpu").numpy()
    inverse = causal_lower_right(qlen, klen)._materialize(device="cpu").numpy()[::-1, ::-1]
    both = causal & inverse
    o, l = oracle.fwd(q, k, v, [[0, qlen]], [[0, klen]], [3])
    ref_o, ref_l = dense.attention(dense.to_f64(q), dense.to_f64(k), dense.to_f64(v), both)
    assert np.array_equal(np.isfinite(l), np.isfinite(ref_l))
    assert np.abs(o - ref_o).max() < 1e-12
    if qlen == klen:  # square bi-causal keeps the diagonal only: out_i = v_i
        qf, kf = dense.to_f64(q), dense.to_f64(k)
        assert np.abs(o - dense.to_f64(v)).max() < 1e-12
        assert np.abs(l[0] - (qf[:, 0] * kf[:, 0]).sum(-1) / math.sqrt(D)).max() < 1e-12


def test_empty_rows_exact():
    T, H, D = 64, 2, 8
    q, k, v = _bf16(T, H, D, seed=41), _bf16(T, H, D, seed=42), _bf16(T, H, D, seed=43)
    # rows 0..9 in no slice; rows 10..19 causal with klen < qlen (first rows empty)
    qr, kr, ty = [[10, 30], [30, 64]], [[0, 5], [5, 64]], [1, 0]
    o, l = oracle.fwd(q, k, v, qr, kr, ty)
    assert (o[:10] == 0).all() and np.isneginf(l[:, :10]).all()
    empty = np.arange(10, 25)  # causal [10,30)x[0,5): rows 10..24 see nothing
    assert (o[empty] == 0).all() and np.isneginf(l[:, empty]).all()
    assert np.isfinite(l[:, 25:]).all()


def _split_case():
    T, H, D = 160, 2, 16
    q, k, v = _bf16(T, H, D, seed=51), _bf16(T, H, D, seed=52), _bf16(T, H, D, seed=53)
    return q, k, v


def test_split_k_range_full_merge():
    q, k, v = _split_case()
    o, l = oracle.fwd(q, k, v, [[20, 150]], [[10, 140]], [0])
    oa, la = oracle.fwd(q, k, v, [[20, 150]], [[10, 77]], [0])
    ob, lb = oracle.fwd(q, k, v, [[20, 150]], [[77, 140]], [0])
    lm, om = oracle.lse_merge(np.stack([la, lb]), np.stack([oa.transpose(1, 0, 2), ob.transpose(1, 0, 2)]))
    fin = np.isfinite(l)
    assert np.array_equal(fin, np.isfinite(lm))
    assert np.abs(lm[fin] - l[fin]).max() < 1e-12
    assert np.abs(om.transpose(1, 0, 2) - o).max() < 1e-12


def test_split_k_range_causal_merge():
    """A causal slice cut at key km: keys >= km stay one causal slice (same
    bottom-right corner); keys < km become a causal slice over the first rows
    plus a full block under it."""
    q, k, v = _split_case()
    qs, qe, ks, ke, km = 20, 150, 10, 140, 90
    r = qe - (ke - km)
    o, l = oracle.fwd(q, k, v, [[qs, qe]], [[ks, ke]], [1])
    oa, la = oracle.fwd(q, k, v, [[qs, r], [r, qe]], [[ks, km], [ks, km]], [1, 0])
    ob, lb = oracle.fwd(q, k, v, [[qs, qe]], [[km, ke]], [1])
    lm, om = oracle.lse_merge(np.stack([la, lb]), np.stack([oa.transpose(1, 0, 2), ob.transpose(1, 0, 2)]))
    fin = np.isfinite(l)
    assert np.array_equal(fin, np.isfinite(lm))
    assert np.abs(lm[fin] - l[fin]).max() < 1e-12
    assert np.abs(om.transpose(1, 0, 2) - o).max() < 1e-12


def test_lse_merge_all_empty_parts():
    lm, om = oracle.lse_merge(np.full((3, 4), -np.inf), np.zeros((3, 4, 2)))
    assert np.isneginf(lm).all() and (om == 0).all()


def torch_dense_reference(q, k, v, mask, scale):
    """fp64 autograd reference: dense masked softmax attention in torch."""
    Hq, Hkv = q.shape[1], k.shape[1]
    kk = k.repeat_interleave(Hq // Hkv, dim=1)
    vv = v.repeat_interleave(Hq // Hkv, dim=1)
    s = torch.einsum("qhd,khd->hqk", q, kk) * scale
    s = s.masked_fill(~mask[None], float("-inf"))
    rowok = mask.any(dim=1)
    p = torch.softmax(torch.where(rowok[None, :, None], s, torch.zeros_like(s)), dim=-1)
    p = torch.where(mask[None], p, torch.zeros_like(p))
    return torch.einsum("hqk,khd->qhd", p, vv)


def _bwd_case(seed):
    rng = np.random.default_rng(300 + seed)
    Tq = int(rng.integers(30, 120))
    Tk = int(rng.integers(30, 120))
    qr, kr, ty = W.random_slices(Tq, Tk, 4, seed=seed + 50)
    Hq, Hkv, D = 4, 2, 8
    q, k, v = _bf16(Tq, Hq, D, seed=seed), _bf16(Tk, Hkv, D, seed=seed + 1), _bf16(Tk, Hkv, D, seed=seed + 2)
    do = _bf16(Tq, Hq, D, seed=seed + 3)
    return Tq, Tk, qr, kr, ty, q, k, v, do


def _autograd_grads(Tq, Tk, qr, kr, ty, q, k, v, do):
    mask = torch.from_numpy(dense.dense_mask(Tq, Tk, qr, kr, ty))
    qq, kk, vv = (_f64(t).requires_grad_() for t in (q, k, v))
    out = torch_dense_reference(qq, kk, vv, mask, 1.0 / math.sqrt(q.shape[-1]))
    out.backward(_f64(do))
    return qq.grad.numpy(), kk.grad.numpy(), vv.grad.numpy()


@pytest.mark.parametrize("seed", range(4))
def test_oracle_bwd_matches_autograd(seed):
    Tq, Tk, qr, kr, ty, q, k, v, do = _bwd_case(seed)
    gq, gk, gv = _autograd_grads(Tq, Tk, qr, kr, ty, q, k, v, do)
    dq, dk, dv = oracle.bwd(q, k, v, do, qr, kr, ty)
    assert np.abs(dq - gq).max() < 1e-10
    assert np.abs(dk - gk).max() < 1e-10
    assert np.abs(dv - gv).max() < 1e-10


def test_oracle_bwd_subsets_match_full():
    Tq, Tk, qr, kr, ty, q, k, v, do = _bwd_case(9)
    dq, dk, dv = oracle.bwd(q, k, v, do, qr, kr, ty)
    rows = [0, 3, Tq - 1, Tq // 2]
    keys = [1, Tk - 1, Tk // 3]
    sq, sk, sv = oracle.bwd(q, k, v, do, qr, kr, ty, dq_rows=rows, dkv_keys=keys)
    assert np.abs(sq - dq[rows]).max() < 1e-13
    assert np.abs(sk - dk[keys]).max() < 1e-13 and np.abs(sv - dv[keys]).max() < 1e-13
    o, l = oracle.fwd(q, k, v, qr, kr, ty)
    so, sl = oracle.fwd(q, k, v, qr, kr, ty, rows=rows)
    assert np.abs(so - o[rows]).max() < 1e-13 and np.array_equal(sl, l[:, rows])


def test_dense_reference_gradcheck():
    """Finite differences pin the autograd reference used above."""
    T, H, D = 12, 2, 4
    qr, kr, ty = [[0, 5], [5, 12], [2, 9]], [[0, 6], [6, 12], [0, 0]], [1, 2, 0]
    mask = torch.from_numpy(dense.dense_mask(T, T, qr, kr, ty))
    g = torch.Generator().manual_seed(3)
    q, k, v = (torch.randn(T, H, D, generator=g, dtype=torch.float64, requires_grad=True) for _ in range(3))
    assert torch.autograd.gradcheck(lambda a, b, c: torch_dense_reference(a, b, c, mask, 0.5), (q, k, v))


def test_delta_identity():
    """sum_j P_ij dP_ij = <dO_i, O_i> (row-wise), in fp64."""
    Tq, Tk, qr, kr, ty, q, k, v, do = _bwd_case(2)
    mask = dense.dense_mask(Tq, Tk, qr, kr, ty)
    qf, kf, vf, df = (dense.to_f64(t) for t in (q, k, v, do))
    o, l = dense.attention(qf, kf, vf, mask)
    g = qf.shape[1] // kf.shape[1]
    for h in range(qf.shape[1]):
        s = (qf[:, h] @ kf[:, h // g].T) / math.sqrt(qf.shape[-1])
        p = np.where(mask, np.exp(s - np.where(np.isfinite(l[h]), l[h], 0)[:, None]), 0.0)
        dp = df[:, h] @ vf[:, h // g].T
        assert np.abs((p * dp).sum(1) - (df[:, h] * o[:, h]).sum(1)).max() < 1e-12


# --- planted mistakes: each mutant of the C oracle must fail a pin --------------

MUTANTS = {
    "swapped_type_bits": (r"if \(s->type & 2\) start", "if (s->type & 1) start"),
    "causal_off_by_one": (r"end -= s->qe - 1 - i;", "end -= s->qe - i;"),
    "gqa_mapping": (r"const int hk = h / \(P->Hq / P->Hkv\);", "const int hk = h % P->Hkv;"),
    "dropped_max": (r"const double lse = m \+ log\(sum\);", "const double lse = log(sum);"),
    "dq_dropped_scale": (r"dqi\[t\] \+= scale \* ds", "dqi[t] += ds"),
    "dropped_delta": (r"const double ds = p \* \(dp - delta\) \* score_grad\(&P, xbuf\[j\]\);",
                      "const double ds = p * dp * score_grad(&P, xbuf[j]);"),
    "dk_transposed_operand": (r"dkj\[t\] \+= scale \* ds \* bf16_to_double\(qi\[t\]\)",
                              "dkj[t] += scale * ds * bf16_to_double(kj[t])"),
}


def _fast_pins(lib):
    """A small subset of the pins above, run against an alternate library."""
    failures = []
    checks = [
        lambda: _check_vs_dense(150, 150, 4, 2, 16, *W.random_slices(150, 150, 4, seed=1), seed=1, lib=lib),
        lambda: _check_vs_dense(120, 90, 2, 1, 8, [[0, 60], [60, 120]], [[0, 50], [40, 90]], [1, 2], seed=2, lib=lib),
    ]
    for c in checks:
        try:
            c()
        except AssertionError:
            failures.append(c)
    Tq, Tk, qr, kr, ty, q, k, v, do = _bwd_case(0)
    gq, gk, gv = _autograd_grads(Tq, Tk, qr, kr, ty, q, k, v, do)
    dq, dk, dv = oracle.bwd(q, k, v, do, qr, kr, ty, lib=lib)
    if max(np.abs(dq - gq).max(), np.abs(dk - gk).max(), np.abs(dv - gv).max()) > 1e-10:
        failures.append("bwd")
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "ffa_oracle.c")).read()
    pat, rep = MUTANTS[name]
    mutated, n = re.subn(pat, rep, src)
    assert n >= 1, f"mutation {name} did not apply"
    c = tmp_path / "m.c"
    c.write_text(mutated)
    so = tmp_path / "libm.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o", str(so), str(c), "-lm"])
    lib = oracle.load_library(str(so))
    assert _fast_pins(lib), f"mutant {name} passed every pin"


def test_unmutated_oracle_passes_fast_pins():
    assert _fast_pins(None) == []
