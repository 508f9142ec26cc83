"""50-digit decimal brute force of the GDN recurrence -- TEST INFRASTRUCTURE ONLY.

An implementation independent of ``gdn_oracle.c``: it writes the per-token update of the
logicaffeine ``codegen_cuda::gdn`` page (module description) in closed matrix form.
Substituting u = S k^ into S_new = alpha S + beta (v - alpha u) k^T gives

    S_new = alpha * S @ (I - beta k^ k^T)  +  beta * v k^T

which is evaluated here with explicit full matrix products (an n^3 brute force), never with
the row-wise u / coef shortcut the C oracle and the CUDA kernels use.  Then o = S_new q^, and
the gated norm o <- rmsnorm(o * silu(z)) * GN (gate first).  Every scalar is a
``decimal.Decimal`` with 50 significant digits; exp and sqrt are Decimal's own.

Readings shared with the C oracle (the pages leave them open): k^ = k / sqrt(sum k^2 + eps),
q^ = q / sqrt(sum q^2 + eps) / sqrt(Dk), alpha = exp(log_decay), beta as given, key head
hk = hv // (Hv // Hk), state row = value index, rmsnorm eps added to the mean square.

Tiny shapes only (B*Hv*S * Dk^2 * Dv multiplications).
"""
from __future__ import annotations

from decimal import Decimal, localcontext

import numpy as np

PREC = 50


def _dec(x) -> Decimal:
    return Decimal(float(x))  # exact: every double is a finite decimal


def _sqrt(x: Decimal) -> Decimal:
    return x.sqrt()


def run(q, k, v, log_decay, beta, *, z=None, gn=None, s0=None, head_major=False,
        qk_eps=1e-6, norm_eps=1e-6):
    """Return ``(y, state)`` as float64 numpy arrays rounded from 50-digit results.

    Arguments are float64-convertible arrays in the same layouts as :func:`oracle.run`.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    g = np.asarray(log_decay, dtype=np.float64)
    bt = np.asarray(beta, dtype=np.float64)
    if head_major:  # bring everything to [B,S,H,W] views for indexing
        q = q.transpose(0, 2, 1, 3)
        k = k.transpose(0, 2, 1, 3)
        v = v.transpose(0, 2, 1, 3)
        g = g.transpose(0, 2, 1)
        bt = bt.transpose(0, 2, 1)
        if z is not None:
            z = np.asarray(z, dtype=np.float64).transpose(0, 2, 1, 3)
    B, S, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    group = Hv // Hk
    y = np.zeros((B, S, Hv, Dv))
    state = np.zeros((B, Hv, Dv, Dk))

    with localcontext() as ctx:
        ctx.prec = PREC
        one = Decimal(1)
        qeps, neps = _dec(qk_eps), _dec(norm_eps)
        inv_sqrt_dk = one / _sqrt(Decimal(Dk))
        gn_d = None if gn is None else [_dec(x) for x in np.asarray(gn, dtype=np.float64)]
        for b in range(B):
            for hv in range(Hv):
                hk = hv // group
                if s0 is None:
                    Sm = [[Decimal(0)] * Dk for _ in range(Dv)]
                else:
                    s0a = np.asarray(s0, dtype=np.float64)
                    Sm = [[_dec(s0a[b, hv, a, j]) for j in range(Dk)] for a in range(Dv)]
                for t in range(S):
                    kk = [_dec(x) for x in k[b, t, hk]]
                    qq = [_dec(x) for x in q[b, t, hk]]
                    nk = _sqrt(sum(x * x for x in kk) + qeps)
                    nq = _sqrt(sum(x * x for x in qq) + qeps)
                    kh = [x / nk for x in kk]
                    qh = [x / nq * inv_sqrt_dk for x in qq]
                    alpha = _dec(g[b, t, hv]).exp()
                    be = _dec(bt[b, t, hv])
                    vv = [_dec(x) for x in v[b, t, hv]]
                    # M = I - beta k^ k^T  (Dk x Dk)
                    M = [[(one if i == j else Decimal(0)) - be * kh[i] * kh[j]
                          for j in range(Dk)] for i in range(Dk)]
                    # S_new = alpha * (S @ M) + beta * v k^T
                    Sn = []
                    for a in range(Dv):
                        row = Sm[a]
                        Sn.append([alpha * sum(row[m] * M[m][j] for m in range(Dk))
                                   + be * vv[a] * kh[j] for j in range(Dk)])
                    Sm = Sn
                    o = [sum(Sm[a][j] * qh[j] for j in range(Dk)) for a in range(Dv)]
                    if z is not None:
                        zz = [_dec(x) for x in np.asarray(z)[b, t, hv]]
                        x = [o[a] * zz[a] / (one + (-zz[a]).exp()) for a in range(Dv)]
                        ms = sum(xi * xi for xi in x) / Decimal(Dv)
                        r = one / _sqrt(ms + neps)
                        o = [x[a] * r * gn_d[a] for a in range(Dv)]
                    for a in range(Dv):
                        y[b, t, hv, a] = float(o[a])
                for a in range(Dv):
                    for j in range(Dk):
                        state[b, hv, a, j] = float(Sm[a][j])
    if head_major:
        y = np.ascontiguousarray(y.transpose(0, 2, 1, 3))
    return y, state
