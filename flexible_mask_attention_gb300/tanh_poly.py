"""Coefficients of the odd polynomial the softcap kernels use for tanh.

The kernels cap a score x to c * tanh(x / c).  Where every argument
u = x / c of a tile lies in [-U, U] they evaluate tanh(u) as
u * Q(u^2) with Q(w) = q_0 + q_1 w + ... + q_4 w^4 (an odd polynomial of
degree 9), on the FMA pipe; elsewhere they fall back to the exponential
identity tanh(u) = 1 - 2 / (exp(2u) + 1).

Q is the minimax approximation of tanh on [-U, U] in relative error: the
polynomial whose largest error relative to tanh(u) is smallest, i.e. the one
whose weighted error equioscillates (Chebyshev's alternation theorem).
Relative error keeps the capped score c * tanh(x / c) accurate relative to
the score itself for every cap c (an absolute bound would be multiplied by
c).  It is found here as a linear program over a dense grid (minimise t
subject to |p(u_i) - tanh(u_i)| <= t * tanh(u_i)), with p written in the odd
Chebyshev polynomials T_1, T_3, ..., T_9 of u / U so that the program is
well conditioned, and then converted to the monomial coefficients q_k.

    python -m flexible_mask_attention_gb300.tanh_poly   # prints the C table

The printed table is pasted into csrc/ffa_internal.cuh (kTanhPoly).
"""
from __future__ import annotations

import numpy as np

U = 0.75       # range of the polynomial: |u| <= U
N_TERMS = 5    # q_0 .. q_4 (degree 9)


def fit(U: float = U, n_terms: int = N_TERMS, n_grid: int = 20001):
    from numpy.polynomial import chebyshev as C
    from scipy.optimize import linprog

    t = np.linspace(0.0, 1.0, n_grid)[1:]      # u / U on (0, 1]; the error is odd
    y = np.tanh(U * t)
    basis = np.stack([C.chebval(t, [0] * (2 * k + 1) + [1]) for k in range(n_terms)], axis=1)
    nv = n_terms + 1
    cost = np.zeros(nv)
    cost[-1] = 1.0
    wt = y[:, None]  # relative error: the bound scales with tanh(u)
    a_ub = np.vstack([np.hstack([basis, -wt]), np.hstack([-basis, -wt])])
    b_ub = np.concatenate([y, -y])
    res = linprog(cost, A_ub=a_ub, b_ub=b_ub, bounds=[(None, None)] * nv, method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    cheb = np.zeros(2 * n_terms)
    cheb[1::2] = res.x[:n_terms]
    mono_t = C.cheb2poly(cheb)                  # coefficients of t^0 .. t^(2n-1)
    # p(u) = sum_j m_j (u / U)^j, odd j only  ->  q_k = m_(2k+1) / U^(2k+1)
    q = np.array([mono_t[2 * k + 1] / U ** (2 * k + 1) for k in range(n_terms)])
    return q


def max_error(q, U: float = U, fp32: bool = False, n: int = 400001) -> float:
    """Largest error relative to tanh(u) over 0 < |u| <= U."""
    u = np.linspace(-U, U, n)
    u = u[u != 0.0]
    if fp32:
        u = u.astype(np.float32)
        w = u * u
        p = np.float32(q[-1])
        for c in q[-2::-1]:
            p = (p * w + np.float32(c)).astype(np.float32)
        approx = (u * p).astype(np.float64)
        ref = np.tanh(u.astype(np.float64))
    else:
        w = u * u
        p = np.zeros_like(u) + q[-1]
        for c in q[-2::-1]:
            p = p * w + c
        approx, ref = u * p, np.tanh(u)
    return float(np.abs((approx - ref) / ref).max())


def main():
    q = fit()
    print(f"// tanh(u) ~ u * sum_k kTanhPoly[k] * u^(2k) on |u| <= {U}: max relative error "
          f"{max_error(q):.2e} (fp64), {max_error(q, fp32=True):.2e} (fp32 Horner)")
    print("constexpr double kTanhPoly[%d] = {" % len(q))
    print(",\n".join(f"    {c:.17e}" for c in q) + "};")


if __name__ == "__main__":
    main()
