"""The chunked (WY) form of the recurrence equals the page's per-token recurrence.

The update of logicaffeine codegen_cuda::gdn (module description) is affine in the memory:
S_t = alpha_t S_{t-1} + d_t k^_t^T with d_t = beta_t (v_t - alpha_t S_{t-1} k^_t), and its
"The fusion" section writes o_t from the old memory plus the token's own correction.
Unrolled over a chunk of C tokens from a start memory S (G_t = prod_{r<=t} alpha_r):
    S_t = G_t S + sum_{s<=t} (G_t / G_s) d_s k^_s^T,
    (I + A) D = diag(beta) V - diag(beta G) K^ S^T,   A[t][s] = beta_t (G_t/G_s) k^_t.k^_s (s < t),
so with T = (I + A)^-1:  D = U - W S^T,  U = T diag(beta) V,  W = T diag(beta G) K^, and
    o_t = G_t S q^_t + sum_{s<=t} (G_t/G_s) (k^_s.q^_t) d_s,
    S_end = G_{C-1} S + sum_s (G_{C-1}/G_s) d_s k^_s^T.
This file evaluates exactly those steps in float64 numpy, with the scalings the tensor-core
kernel uses (raw k, q with the l2 norms as per-token scalars rk, rq; every decay factor an exp
of a non-positive sum), on shapes with several chunks and a ragged last chunk, and checks y
and the final state against the fp64 oracle.  It pins the algebra the chunked kernel relies
on; the kernel itself is checked against the oracle on the GPU.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_gdn_gb300.workloads import TINY, make_inputs


def chunked_scan(q, k, v, g, beta, s0, z, gn, C, qk_eps=1e-6, norm_eps=1e-6, mutate=None):
    """One sequence and one value head: q, k [S, Dk]; v, z [S, Dv]; g, beta [S]; s0 [Dv, Dk]."""
    S_len, Dk = k.shape
    Dv = v.shape[1]
    S = s0.copy()
    ys = np.zeros((S_len, Dv))
    for c0 in range(0, S_len, C):
        n = min(C, S_len - c0)
        K, Q, V = np.zeros((C, Dk)), np.zeros((C, Dk)), np.zeros((C, Dv))
        K[:n], Q[:n], V[:n] = k[c0:c0 + n], q[c0:c0 + n], v[c0:c0 + n]
        gc = np.zeros(C)
        bc = np.zeros(C)
        gc[:n] = np.maximum(g[c0:c0 + n], -80.0)     # padded tokens: alpha = 1, beta = 0
        bc[:n] = beta[c0:c0 + n]
        cum = np.cumsum(gc)
        rk = 1.0 / np.sqrt((K * K).sum(1) + qk_eps)
        rq = 1.0 / np.sqrt((Q * Q).sum(1) + qk_eps) / np.sqrt(Dk)
        KK, QK = K @ K.T, Q @ K.T
        decay = np.exp(np.minimum(cum[:, None] - cum[None, :], 0.0))   # G_t / G_s, s <= t
        A = np.tril(bc[:, None] * decay * rk[:, None] * rk[None, :] * KK, -1)
        T = np.linalg.inv(np.eye(C) + A)
        Bu = T * bc[None, :]
        Bw = -T * (bc * np.exp(cum) * rk)[None, :]
        X = V.T @ Bu.T + S @ (K.T @ Bw.T)            # [Dv, C]: d_t as columns (U - W S^T)^T
        Y = S @ Q.T                                   # raw S q_t
        P = np.tril(decay * rk[None, :] * rq[:, None] * QK)
        O = (np.exp(cum) * rq)[None, :] * Y + X @ P.T
        cvec = rk * np.exp(cum[-1] - cum)
        if mutate == "update_factor_from_chunk_start":
            cvec = rk * np.exp(cum - cum[0])
        if mutate == "o_inter_without_decay":
            O = rq[None, :] * Y + X @ P.T

        S = np.exp(cum[-1]) * S + (X * cvec[None, :]) @ K
        o = O.T[:n]
        if z is not None:
            x = o * (z[c0:c0 + n] / (1.0 + np.exp(-z[c0:c0 + n])))
            o = x / np.sqrt((x * x).mean(1, keepdims=True) + norm_eps) * gn[None, :]
        ys[c0:c0 + n] = o
    return ys, S


def run_both(inp, C, gated):
    f = lambda t: t.double().numpy()
    q, k, v, g, b = f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["log_decay"]), f(inp["beta"])
    z = f(inp["z"]) if gated else None
    gn = f(inp["gn"]) if gated else None
    B, S_len, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    s0 = f(inp["s0"]) if inp["s0"] is not None else np.zeros((B, Hv, Dv, Dk))
    y = np.zeros((B, S_len, Hv, Dv))
    st = np.zeros((B, Hv, Dv, Dk))
    for bi in range(B):
        for hv in range(Hv):
            hk = hv // (Hv // Hk)
            y[bi, :, hv], st[bi, hv] = chunked_scan(
                q[bi, :, hk], k[bi, :, hk], v[bi, :, hv], g[bi, :, hv], b[bi, :, hv],
                s0[bi, hv], None if z is None else z[bi, :, hv], gn, C)
    yr, sr = oracle.run(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"],
                        z=inp["z"] if gated else None, gn=inp["gn"] if gated else None,
                        s0=inp["s0"])
    return y, st, yr, sr


@pytest.mark.parametrize("gated", [True, False])
@pytest.mark.parametrize("shape", [
    # B, S, Hk, Hv, D, C, log_decay range
    (1, 8, 2, 2, 16, 4, (-3.0, 0.0)),
    (1, 150, 1, 2, 16, 64, (-4.0, 0.0)),       # 3 chunks, ragged last
    (2, 70, 1, 2, 8, 16, (-8.0, -3.0)),        # slow decay
    (1, 64, 1, 1, 8, 64, (2.0, 3.0)),          # log_decay down to -20 per token (clamped at -80)
])
def test_chunked_form_equals_sequential_oracle(shape, gated):
    B, S, Hk, Hv, D, C, ldr = shape
    w = TINY.replace(name="chunk", B=B, S=S, Hk=Hk, Hv=Hv, Dk=D, Dv=D, act="f32",
                     log_decay_range=ldr, s0_std=0.1, seed=77 + S)
    inp = make_inputs(w)
    y, st, yr, sr = run_both(inp, C, gated)
    assert np.max(np.abs(y - yr)) <= 1e-9 * (1 + np.max(np.abs(yr)))
    assert np.max(np.abs(st - sr)) <= 1e-9 * (1 + np.max(np.abs(sr)))


@pytest.mark.parametrize("mutate", ["update_factor_from_chunk_start", "o_inter_without_decay"])
def test_chunked_form_detects_a_wrong_decay_reference(mutate):
    # the same evaluation with a decay factor taken against the wrong reference must fail the
    # comparison: the pin resolves the decay bookkeeping, not just the shapes
    w = TINY.replace(name="chunk", B=1, S=40, Hk=1, Hv=1, Dk=8, Dv=8, act="f32",
                     log_decay_range=(-3.0, 0.0), s0_std=0.1, seed=5)
    inp = make_inputs(w)
    f = lambda t: t.double().numpy()
    q, k, v, g, b = (f(inp[n])[0, :, 0] for n in ("q", "k", "v", "log_decay", "beta"))
    s0 = f(inp["s0"])[0, 0]
    yr, sr = oracle.run(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"],
                        s0=inp["s0"])
    y_ok, s_ok = chunked_scan(q, k, v, g, b, s0, None, None, 16)
    y_bad, s_bad = chunked_scan(q, k, v, g, b, s0, None, None, 16, mutate=mutate)
    assert np.max(np.abs(y_ok - yr[0, :, 0])) <= 1e-9
    assert max(np.max(np.abs(y_bad - yr[0, :, 0])), np.max(np.abs(s_bad - sr[0, 0]))) > 1e-3
