"""Seeded synthetic workloads for flexible-mask attention.

This module only builds inputs: slice tables (q_range, k_range, mask_type) and
bf16 tensors drawn from N(0, 1).  It holds none of the attention arithmetic, so
both the CUDA path and the CPU oracle can be fed from it.

The document structures follow the workloads the MagiAttention pages show:
packed variable-length documents with one causal slice each (varlen key,
"magi_attn_varlen_key" card), a shared prefix visible to later documents
(quickstart "Single-GPU Flex-Flash-Attention" mask picture and the block-causal
example), and long-context block sliding windows built from consecutive
causal/full slices, and uniform block-sparse masks given by a (q block,
k block) size pair ("Configure ... Block Sizes for Sparse Attention" cards:
64/128 square blocks, q blocks of 32..8 against k blocks of 64, k blocks of
32..1 against q blocks of 64).  No dataset is involved; every value is
synthetic.

Mask-type codes: 0 = full, 1 = causal (bottom-right aligned), 2 = inverse
causal (top-left aligned), 3 = bidirectional causal (both clamps).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

FULL, CAUSAL, INV_CAUSAL, BI_CAUSAL = 0, 1, 2, 3


@dataclass
class Workload:
    name: str
    total_q: int
    total_k: int
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    q_ranges: np.ndarray  # [S, 2] int32, half-open
    k_ranges: np.ndarray  # [S, 2] int32, half-open
    mask_types: np.ndarray  # [S] int32
    seed: int
    dout_seed: int | None = None
    meta: dict = field(default_factory=dict)

    @property
    def num_slices(self) -> int:
        return int(self.mask_types.shape[0])


def _pack(name, tq, tk, hq, hkv, d, qr, kr, ty, seed, dout_seed=None, **meta):
    return Workload(
        name=name, total_q=tq, total_k=tk, num_heads_q=hq, num_heads_kv=hkv,
        head_dim=d,
        q_ranges=np.asarray(qr, dtype=np.int32).reshape(-1, 2),
        k_ranges=np.asarray(kr, dtype=np.int32).reshape(-1, 2),
        mask_types=np.asarray(ty, dtype=np.int32).reshape(-1),
        seed=seed, dout_seed=dout_seed, meta=dict(meta))


def packed_doc_lengths(total: int, seed: int, median: int = 2048, sigma: float = 1.0,
                       lo: int = 128, hi: int = 16384) -> list[int]:
    """Lognormal document lengths summing to ``total``.

    Lengths are ``clip(round(median * exp(sigma * z)), lo, hi)`` with z drawn
    one at a time from ``numpy.random.default_rng(seed).standard_normal``
    until the sum reaches ``total``.  The last document takes the remainder;
    a remainder shorter than ``lo`` is folded into the shortest earlier one.
    """
    rng = np.random.default_rng(seed)
    lens: list[int] = []
    while sum(lens) < total:
        z = rng.standard_normal()
        lens.append(int(np.clip(round(median * np.exp(sigma * z)), lo, hi)))
    lens[-1] = total - sum(lens[:-1])
    if lens[-1] < lo and len(lens) > 1:
        rem = lens.pop()
        i = int(np.argmin(lens))
        lens[i] += rem
    return lens


def tiny_causal_docs() -> Workload:
    """256 tokens, one head, head_dim 64: two 128-token causal documents."""
    qr = [[0, 128], [128, 256]]
    return _pack("tiny_causal_docs_T256_H1_D64", 256, 256, 1, 1, 64, qr, qr,
                 [CAUSAL, CAUSAL], seed=1, dout_seed=101)


def packed_causal_docs(total: int = 32768, hq: int = 32, hkv: int = 8, d: int = 128,
                       seed: int = 2, dout_seed: int = 5) -> Workload:
    """Packed documents with lognormal lengths, one causal self-slice each."""
    lens = packed_doc_lengths(total, seed)
    b = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    qr = np.stack([b[:-1], b[1:]], axis=1)
    return _pack(f"packed_causal_T{total}_Hq{hq}_Hkv{hkv}_D{d}", total, total, hq, hkv, d,
                 qr, qr, [CAUSAL] * len(lens), seed=seed, dout_seed=dout_seed,
                 doc_lens=lens)


def heterogeneous_prefix_docs(total: int = 65536, h: int = 16, d: int = 128,
                              prefix: int = 4096, n_docs: int = 23, min_doc: int = 256,
                              seed: int = 3, dout_seed: int = 7) -> Workload:
    """A shared full prefix block plus documents of mixed mask types.

    ``default_rng(seed)``: ``n_docs - 1`` distinct cut points drawn with
    ``choice(arange(prefix + 256, total - 256), n_docs - 1, replace=False)``,
    redrawn until every document has at least ``min_doc`` tokens.  The
    documents' self-slice types are then ``permutation`` of a multiset that
    splits ``n_docs`` as evenly as possible over {full, causal,
    inverse-causal, bi-causal}, the first types taking the remainder (23
    documents: full x6, causal x6, inverse-causal x6, bi-causal x5) from the
    same generator.  Slices: the prefix's own full block, one self-slice per
    document, and one full slice per document over the prefix keys.
    """
    rng = np.random.default_rng(seed)
    lo, hi = prefix + 256, total - 256
    while True:
        cuts = rng.choice(np.arange(lo, hi), n_docs - 1, replace=False)
        bounds = [prefix] + sorted(int(c) for c in cuts) + [total]
        if len(set(bounds)) == len(bounds) and min(np.diff(bounds)) >= min_doc:
            break
    per = [n_docs // 4 + (1 if i < n_docs % 4 else 0) for i in range(4)]
    base = [FULL] * per[0] + [CAUSAL] * per[1] + [INV_CAUSAL] * per[2] + [BI_CAUSAL] * per[3]
    assert len(base) == n_docs
    types = [int(t) for t in rng.permutation(base)]
    qr, kr, ty = [[0, prefix]], [[0, prefix]], [FULL]
    for i in range(n_docs):
        a, b = bounds[i], bounds[i + 1]
        qr.append([a, b]); kr.append([a, b]); ty.append(types[i])
    for i in range(n_docs):
        a, b = bounds[i], bounds[i + 1]
        qr.append([a, b]); kr.append([0, prefix]); ty.append(FULL)
    return _pack(f"heterogeneous_prefix_T{total}_H{h}_D{d}", total, total, h, h, d,
                 qr, kr, ty, seed=seed, dout_seed=dout_seed, bounds=bounds,
                 doc_types=types)


def short_causal_docs(total: int = 32768, h: int = 8, d: int = 128, lo: int = 128,
                      hi: int = 512, seed: int = 8) -> Workload:
    """Packed short documents (the memory-bound regime): lengths drawn one at a
    time from ``default_rng(seed).integers(lo, hi + 1)`` until they reach
    ``total`` (the last one takes the remainder, folded into the previous
    document when shorter than ``lo``), one causal self-slice each."""
    rng = np.random.default_rng(seed)
    lens: list[int] = []
    while sum(lens) < total:
        lens.append(int(rng.integers(lo, hi + 1)))
    lens[-1] = total - sum(lens[:-1])
    if lens[-1] < lo and len(lens) > 1:
        rem = lens.pop()
        lens[-1] += rem
    b = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    qr = np.stack([b[:-1], b[1:]], axis=1)
    return _pack(f"short_causal_T{total}_H{h}_D{d}_L{lo}-{hi}", total, total, h, h, d, qr, qr,
                 [CAUSAL] * len(lens), seed=seed, doc_lens=lens)


def long_context_docs(total: int = 262144, hq: int = 16, hkv: int = 4, d: int = 128,
                      n_docs: int = 8, chunk: int = 4096, seed: int = 4) -> Workload:
    """Eight equal documents: even ones one causal slice, odd ones a block
    sliding window made of consecutive ``chunk``-wide slices (causal chunk x
    chunk on the diagonal, full chunk x previous-chunk below it)."""
    doc = total // n_docs
    qr, kr, ty = [], [], []
    for di in range(n_docs):
        s = di * doc
        if di % 2 == 0:
            qr.append([s, s + doc]); kr.append([s, s + doc]); ty.append(CAUSAL)
        else:
            for c in range(doc // chunk):
                a = s + c * chunk
                qr.append([a, a + chunk]); kr.append([a, a + chunk]); ty.append(CAUSAL)
                if c >= 1:
                    qr.append([a, a + chunk]); kr.append([a - chunk, a]); ty.append(FULL)
    return _pack(f"long_context_T{total}_Hq{hq}_Hkv{hkv}_D{d}", total, total, hq, hkv, d,
                 qr, kr, ty, seed=seed)


def random_slices(total_q: int, total_k: int, n: int, seed: int,
                  aligned: bool = False, n_empty: int = 1, p_uncovered: float = 0.15
                  ) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Random slices whose (q x k) rectangles are pairwise disjoint.

    Cuts the q and k axes into ``n`` segments each, then pairs every q
    segment (except a random ``p_uncovered`` share, whose rows stay fully
    masked) with one or two distinct k segments and a random mask type.
    ``n_empty`` zero-length slices are appended.  Used for small parity cases
    with ragged, non tile-aligned boundaries.
    """
    rng = np.random.default_rng(seed)
    def cuts(total):
        c = np.sort(rng.choice(np.arange(1, total), min(n - 1, total - 1), replace=False))
        if aligned:
            c = np.unique((c // 128) * 128)
            c = c[(c > 0) & (c < total)]
        return np.concatenate([[0], c, [total]]).astype(np.int64)
    qb, kb = cuts(total_q), cuts(total_k)
    qr, kr, ty = [], [], []
    for qi in range(len(qb) - 1):
        if rng.random() < p_uncovered:
            continue
        picks = rng.choice(len(kb) - 1, min(int(rng.integers(1, 3)), len(kb) - 1), replace=False)
        for ki in sorted(int(x) for x in picks):
            qr.append([qb[qi], qb[qi + 1]]); kr.append([kb[ki], kb[ki + 1]])
            ty.append(int(rng.integers(0, 4)))
    for _ in range(n_empty):
        a = int(rng.integers(0, total_q + 1)); b = int(rng.integers(0, total_k + 1))
        qr.append([a, a]); kr.append([b, min(total_k, b + 5)]); ty.append(int(rng.integers(0, 4)))
    return (np.asarray(qr, np.int32).reshape(-1, 2), np.asarray(kr, np.int32).reshape(-1, 2),
            np.asarray(ty, np.int32))


def block_sparse(total: int = 16384, hq: int = 16, hkv: int = 4, d: int = 128,
                 q_block: int = 64, k_block: int = 64, density: float = 0.125,
                 seed: int = 6) -> Workload:
    """Uniform block-sparse attention: the sequence is cut into q blocks of
    ``q_block`` rows and k blocks of ``k_block`` keys; every q block attends
    to ``round(density * n_k_blocks)`` (at least one) k blocks drawn without
    replacement, and every selected (q block, k block) pair is one full
    slice.  Slices are listed q block by q block, k blocks ascending, so the
    table holds many tiny slices (the density is this module's choice: the
    pages give the block sizes only).
    """
    rng = np.random.default_rng(seed)
    nq, nk = -(-total // q_block), -(-total // k_block)
    per = max(1, int(round(density * nk)))
    qr, kr = [], []
    for qb in range(nq):
        q0, q1 = qb * q_block, min(total, (qb + 1) * q_block)
        for kb in np.sort(rng.choice(nk, per, replace=False)):
            k0, k1 = int(kb) * k_block, min(total, (int(kb) + 1) * k_block)
            qr.append([q0, q1]); kr.append([k0, k1])
    ty = [FULL] * len(qr)
    return _pack(f"block_sparse_T{total}_Hq{hq}_Hkv{hkv}_D{d}_q{q_block}_k{k_block}", total,
                 total, hq, hkv, d, qr, kr, ty, seed=seed, q_block=q_block, k_block=k_block,
                 density=density)


def make_tensors(wl: Workload, with_dout: bool = False):
    """bf16 q, k, v (and dout) ~ N(0, 1) from a seeded CPU torch generator."""
    import torch
    g = torch.Generator(device="cpu").manual_seed(wl.seed)
    q = torch.randn(wl.total_q, wl.num_heads_q, wl.head_dim, generator=g).to(torch.bfloat16)
    k = torch.randn(wl.total_k, wl.num_heads_kv, wl.head_dim, generator=g).to(torch.bfloat16)
    v = torch.randn(wl.total_k, wl.num_heads_kv, wl.head_dim, generator=g).to(torch.bfloat16)
    if not with_dout:
        return q, k, v
    gd = torch.Generator(device="cpu").manual_seed(wl.dout_seed if wl.dout_seed is not None
                                                   else wl.seed + 1000)
    do = torch.randn(wl.total_q, wl.num_heads_q, wl.head_dim, generator=gd).to(torch.bfloat16)
    return q, k, v, do


CONFIGS = {
    "tiny": tiny_causal_docs,
    "packed_causal": packed_causal_docs,
    "heterogeneous": heterogeneous_prefix_docs,
    # the same structure at a quarter of the length (4096-token prefix, 11
    # documents of all four types), small enough for a full oracle backward
    "heterogeneous_mid": lambda: heterogeneous_prefix_docs(total=16384, h=2, n_docs=11, seed=13,
                                                           dout_seed=17),
    # the 64K mask with 2 heads (inputs 134 MB, larger than L2): the
    # single-kernel profiling case
    "heterogeneous_h2": lambda: heterogeneous_prefix_docs(h=2),
    # packed causal documents with 8 query / 2 kv heads (inputs 168 MB)
    "packed_causal_h8": lambda: packed_causal_docs(hq=8, hkv=2),
    # the same documents with one kv head of 4 query heads (the GQA ratio of
    # the 32 / 8 head table), small enough for a full oracle backward
    "packed_causal_h4": lambda: packed_causal_docs(hq=4, hkv=1),
    "long_context": long_context_docs,
    "short_docs": short_causal_docs,
    "block_sparse_64x64": lambda: block_sparse(q_block=64, k_block=64),
    "block_sparse_128x128": lambda: block_sparse(q_block=128, k_block=128),
    "block_sparse_16x64": lambda: block_sparse(q_block=16, k_block=64),
    "block_sparse_64x8": lambda: block_sparse(q_block=64, k_block=8),
    "block_sparse_64x1": lambda: block_sparse(q_block=64, k_block=1),
}
