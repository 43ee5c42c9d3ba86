"""CPU oracle for flexible-mask attention (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product path never does, and nothing here imports
the product package: the two share only the seeded input generators.

Contents
  * ``fwd`` / ``bwd``: the fp64 C oracle (``ffa_oracle.c``), the
    masked-softmax definition written out, on all rows/keys or a subset,
    optionally with attention-sink logits in the normaliser; ``dsink`` their
    gradient.
  * ``lse_merge``: combination of partial (out, lse) pairs with a global
    logsumexp (FlagAttention user guide, "Split-KV and paged attention").
  * ``dense``: a numpy brute force over an explicit Tq x Tk mask built from a
    different characterisation of the mask types, used to pin the C oracle.
  * ``planner``: a CPU re-derivation of the tile work list by counting
    visible elements per tile.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libffa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, OpenMP, portable flags) into oracle/_build."""
    src = os.path.join(_HERE, "ffa_oracle.c")
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(src)):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp",
                           "-shared", "-fPIC", "-o", tmp, src, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def load_library(path: str):
    """Open an oracle shared library and declare its entry points."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    L = ctypes.c_long
    I = ctypes.c_int
    D = ctypes.c_double
    lib.ffa_oracle_fwd.argtypes = [P, P, P, L, L, I, I, I, P, P, P, I, D, D, P, I, I, P, L, P, P]
    lib.ffa_oracle_fwd.restype = I
    lib.ffa_oracle_bwd.argtypes = [P, P, P, P, L, L, I, I, I, P, P, P, I, D, D, P, I, I,
                                   P, L, P, P, L, P, P]
    lib.ffa_oracle_bwd.restype = I
    lib.ffa_oracle_dsink.argtypes = [P, P, P, P, L, L, I, I, I, P, P, P, I, D, D, P, I, I, P, L, P]
    lib.ffa_oracle_dsink.restype = I
    lib.ffa_oracle_num_threads.restype = I
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = load_library(_SO)
    return _lib


def num_threads() -> int:
    return int(_load().ffa_oracle_num_threads())


def _u16(t) -> np.ndarray:
    """bf16 torch tensor or uint16 numpy array -> contiguous uint16 numpy."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


_LAYOUTS = {"sh": 0, "ssh": 1}


def _sink(sink, sink_layout, Tq, Hq):
    """(fp64 array or None, n_sink, layout code) for an optional sink tensor."""
    if sink is None:
        return None, 0, 0
    code = _LAYOUTS[sink_layout]
    a = np.ascontiguousarray(np.asarray(sink.detach().cpu() if hasattr(sink, "detach") else sink,
                                        dtype=np.float64))
    if code == 0 and (a.ndim != 2 or a.shape[1] != Hq):
        raise ValueError("sink layout 'sh' wants [n_sink, Hq]")
    if code == 1 and (a.ndim != 3 or a.shape[0] != Tq or a.shape[2] != Hq):
        raise ValueError("sink layout 'ssh' wants [Tq, n_sink, Hq]")
    return a, a.shape[-2], code


def fwd(q, k, v, q_ranges, k_ranges, mask_types, softmax_scale=None, rows=None, lib=None, *,
        sink=None, sink_layout="sh", softcap=0.0):
    """fp64 forward. Returns (out[n, Hq, D], lse[Hq, n]) for ``rows`` (all by default).
    ``sink``: optional fp32 sink logits, [n_sink, Hq] ("sh") or [Tq, n_sink, Hq] ("ssh").
    ``softcap`` c > 0 caps every score to c * tanh(score / c)."""
    qn, kn, vn = _u16(q), _u16(k), _u16(v)
    Tq, Hq, D = qn.shape
    Tk, Hkv, _ = kn.shape
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    qr, kr, ty = _i32(q_ranges).reshape(-1, 2), _i32(k_ranges).reshape(-1, 2), _i32(mask_types)
    rows_a = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = Tq if rows_a is None else rows_a.shape[0]
    sk, ns, lay = _sink(sink, sink_layout, Tq, Hq)
    out = np.zeros((n, Hq, D), np.float64)
    lse = np.zeros((Hq, n), np.float64)
    rc = (lib or _load()).ffa_oracle_fwd(_ptr(qn), _ptr(kn), _ptr(vn), Tq, Tk, Hq, Hkv, D, _ptr(qr),
                                _ptr(kr), _ptr(ty), ty.shape[0], scale, float(softcap),
                                None if sk is None else _ptr(sk), ns, lay,
                                None if rows_a is None else _ptr(rows_a), n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle: bad arguments")
    return out, lse


def bwd(q, k, v, dout, q_ranges, k_ranges, mask_types, softmax_scale=None,
        dq_rows=None, dkv_keys=None, lib=None, *, sink=None, sink_layout="sh", softcap=0.0):
    """fp64 backward. Returns (dq[nq, Hq, D], dk[nk, Hkv, D], dv[nk, Hkv, D])."""
    qn, kn, vn, dn = _u16(q), _u16(k), _u16(v), _u16(dout)
    Tq, Hq, D = qn.shape
    Tk, Hkv, _ = kn.shape
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    qr, kr, ty = _i32(q_ranges).reshape(-1, 2), _i32(k_ranges).reshape(-1, 2), _i32(mask_types)
    rq = None if dq_rows is None else np.ascontiguousarray(np.asarray(dq_rows, np.int64))
    rk = None if dkv_keys is None else np.ascontiguousarray(np.asarray(dkv_keys, np.int64))
    nq = Tq if rq is None else rq.shape[0]
    nk = Tk if rk is None else rk.shape[0]
    dq = np.zeros((nq, Hq, D), np.float64)
    dk = np.zeros((nk, Hkv, D), np.float64)
    dv = np.zeros((nk, Hkv, D), np.float64)
    sk, ns, lay = _sink(sink, sink_layout, Tq, Hq)
    rc = (lib or _load()).ffa_oracle_bwd(_ptr(qn), _ptr(kn), _ptr(vn), _ptr(dn), Tq, Tk, Hq, Hkv, D,
                                _ptr(qr), _ptr(kr), _ptr(ty), ty.shape[0], scale, float(softcap),
                                None if sk is None else _ptr(sk), ns, lay,
                                None if rq is None else _ptr(rq), nq, _ptr(dq),
                                None if rk is None else _ptr(rk), nk, _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError("oracle: bad arguments")
    return dq, dk, dv


def dsink(q, k, v, dout, q_ranges, k_ranges, mask_types, sink, sink_layout="sh",
          softmax_scale=None, rows=None, lib=None, softcap=0.0):
    """fp64 gradient of the sink logits: [n_sink, Hq] ("sh", summed over all
    rows) or [n, n_sink, Hq] for ``rows`` ("ssh", all rows by default)."""
    qn, kn, vn, dn = _u16(q), _u16(k), _u16(v), _u16(dout)
    Tq, Hq, D = qn.shape
    Tk, Hkv, _ = kn.shape
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    qr, kr, ty = _i32(q_ranges).reshape(-1, 2), _i32(k_ranges).reshape(-1, 2), _i32(mask_types)
    sk, ns, lay = _sink(sink, sink_layout, Tq, Hq)
    rows_a = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = Tq if rows_a is None else rows_a.shape[0]
    out = np.zeros((ns, Hq) if lay == 0 else (n, ns, Hq), np.float64)
    rc = (lib or _load()).ffa_oracle_dsink(_ptr(qn), _ptr(kn), _ptr(vn), _ptr(dn), Tq, Tk, Hq, Hkv,
                                  D, _ptr(qr), _ptr(kr), _ptr(ty), ty.shape[0], scale,
                                  float(softcap), _ptr(sk),
                                  ns, lay, None if rows_a is None else _ptr(rows_a), n, _ptr(out))
    if rc != 0:
        raise ValueError("oracle: bad arguments")
    return out


def lse_merge(lse_parts, out_parts):
    """Combine partial results computed over disjoint key sets.

    Each part i holds a row log-normalizer lse_i and the output o_i
    normalised over its own keys.  The merged row is lse = log sum_i
    exp(lse_i) and out = sum_i exp(lse_i - lse) o_i; rows where every part
    is -inf give lse = -inf and out = 0 (FlagAttention user guide,
    "Split-KV and paged attention": partial outputs and log-normalizers
    combined with a global logsumexp).
    lse_parts: [n, ...rows], out_parts: [n, ...rows, D].
    """
    lse_parts = np.asarray(lse_parts, np.float64)
    out_parts = np.asarray(out_parts, np.float64)
    m = np.max(lse_parts, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.exp(lse_parts - m_safe[None])
    s = np.sum(w, axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, s, 1.0)), -np.inf)
    coef = np.where(finite[None], np.exp(lse_parts - np.where(finite, lse, 0.0)[None]), 0.0)
    out = np.sum(coef[..., None] * out_parts, axis=0)
    return lse, out
