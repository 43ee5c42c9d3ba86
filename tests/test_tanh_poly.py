"""The softcap kernels' tanh polynomial: the table compiled into the CUDA
sources is the one the committed generator produces, and its error against
numpy's tanh stays within the bound the kernels rely on (1.4e-6 relative
to tanh, so that a capped score is accurate relative to the score for any
cap)."""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_table():
    text = open(os.path.join(ROOT, "flexible_mask_attention_gb300", "csrc",
                             "ffa_internal.cuh")).read()
    body = re.search(r"kTanhPoly\[kTanhPolyTerms\]\s*=\s*\{([^}]*)\}", text).group(1)
    rng = float(re.search(r"kTanhPolyRange\s*=\s*([0-9.eE+-]+);", text).group(1))
    return np.array([float(x) for x in body.split(",")]), rng


def test_table_matches_generator():
    pytest.importorskip("scipy")
    from flexible_mask_attention_gb300 import tanh_poly
    q, rng = header_table()
    assert rng == tanh_poly.U
    fit = tanh_poly.fit()
    assert np.allclose(q, fit, rtol=1e-9, atol=1e-12)


def test_error_bound():
    from flexible_mask_attention_gb300 import tanh_poly
    q, rng = header_table()
    # relative to tanh(u): the capped score c tanh(x / c) is then accurate
    # relative to the score for every cap c
    assert tanh_poly.max_error(q, rng) < 1.4e-6
    assert tanh_poly.max_error(q, rng, fp32=True) < 1.5e-6
    # odd and close to the identity near zero
    u = np.linspace(1e-4, 1e-2, 50)
    p = u * np.polyval(q[::-1], u * u)
    assert (np.abs(p - np.tanh(u)) / np.tanh(u)).max() < 1.4e-6
