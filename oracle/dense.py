"""Dense brute-force reference on an explicit Tq x Tk mask (small sizes only).

Test infrastructure.  The mask is built here from a characterisation of the
mask types that does not use the per-row interval formula of the C oracle:

  * full: every (q, k) pair of the slice rectangle;
  * causal: lower triangle of the rectangle aligned to its bottom-right corner
    (FlagAttention user guide, "Rectangular causal attention is bottom-right
    aligned"; MagiAttention quickstart mask picture, whose second slice is a
    1024 x 2048 causal block ending on the diagonal of the full mask);
  * inverse causal: upper triangle aligned to the top-left corner, i.e. the
    causal mask of the rectangle read with both axes reversed;
  * bidirectional causal: the entries both of the above keep.

Attention is then plain fp64 softmax over each row of scale * Q K^T with the
masked entries removed.
"""
from __future__ import annotations

import math

import numpy as np


def slice_block(qlen: int, klen: int, mask_type: int) -> np.ndarray:
    """Boolean [qlen, klen] pattern of one slice in its own coordinates."""
    ones = np.ones((qlen, klen), dtype=bool)
    causal = np.tril(ones, k=klen - qlen)          # ends on the bottom-right corner
    inverse = np.tril(ones[::-1, ::-1], k=klen - qlen)[::-1, ::-1]  # reversed causal
    if mask_type == 0:
        return ones
    if mask_type == 1:
        return causal
    if mask_type == 2:
        return inverse
    if mask_type == 3:
        return causal & inverse
    raise ValueError(mask_type)


def dense_mask(total_q: int, total_k: int, q_ranges, k_ranges, mask_types,
               return_count: bool = False):
    """Union over slices of their patterns placed in the global grid."""
    count = np.zeros((total_q, total_k), dtype=np.int32)
    for (qs, qe), (ks, ke), t in zip(np.asarray(q_ranges).reshape(-1, 2),
                                     np.asarray(k_ranges).reshape(-1, 2),
                                     np.asarray(mask_types).reshape(-1)):
        if qe <= qs or ke <= ks:
            continue
        count[qs:qe, ks:ke] += slice_block(int(qe - qs), int(ke - ks), int(t))
    mask = count > 0
    return (mask, count) if return_count else mask


def to_f64(t) -> np.ndarray:
    """bf16 torch tensor -> float64 numpy (exact)."""
    import torch
    return t.detach().cpu().to(torch.float64).numpy()


def attention(q, k, v, mask, softmax_scale=None):
    """fp64 masked softmax attention. q [Tq,Hq,D], k/v [Tk,Hkv,D] (float64
    arrays), mask [Tq,Tk] bool. Returns out [Tq,Hq,D], lse [Hq,Tq]."""
    Tq, Hq, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else softmax_scale
    out = np.zeros((Tq, Hq, D))
    lse = np.full((Hq, Tq), -np.inf)
    for h in range(Hq):
        s = scale * (q[:, h, :] @ k[:, h // g, :].T)
        s = np.where(mask, s, -np.inf)
        m = s.max(axis=1)
        ok = np.isfinite(m)
        e = np.where(mask, np.exp(s - np.where(ok, m, 0.0)[:, None]), 0.0)
        z = e.sum(axis=1)
        lse[h] = np.where(ok, np.where(ok, m, 0.0) + np.log(np.where(ok, z, 1.0)), -np.inf)
        p = e / np.where(ok, z, 1.0)[:, None]
        out[:, h, :] = p @ v[:, h // g, :]
    return out, lse
