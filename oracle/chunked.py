"""Chunked (WY / UT-transform) evaluation of the gated delta rule, FP64 numpy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  This is a second,
independent derivation of the same recurrence in the blocked form that the
"[CUDA] Add compact GatedDeltaNet operator" page names for its tensor-core
chunked prefill (Description).  The tests use it to show that chunked and
sequential evaluation agree, which pins the chunk algebra a tensor-core kernel
relies on.  It never feeds an expected value to a GPU test.

Per chunk of C tokens (positions r = 0..C-1), with S0 the state entering the
chunk, gamma_r = g_0 g_1 ... g_r the within-chunk cumulative decay and
Gamma_r = log gamma_r:

    A[r, s] = beta_r * gamma_r / gamma_s * (k_r . k_s)   for s < r, else 0
    Tm      = (I + A)^-1                                  (unit lower triangular)
    Wm      = Tm diag(beta * gamma) K
    U       = Tm diag(beta) V - Wm S0^T                   (rows are the deltas u_r)
    O       = scale * (diag(gamma) Q S0^T + (tril(Q K^T) o D) U),  D[r,s] = gamma_r/gamma_s
    S1      = gamma_{C-1} S0 + (diag(gamma_{C-1} / gamma) U)^T K

Derivation: S_r = gamma_r S0 + sum_{s<=r} (gamma_r/gamma_s) u_s k_s^T, and the
delta u_r = beta_r (v_r - g_r S_{r-1} k_r) expands into the unit lower
triangular system (I + A) U = diag(beta) V - diag(beta gamma) K S0^T.
Requires g > 0 (log-space decays).
"""
from __future__ import annotations

import numpy as np


def _unit(x, eps=1e-6):
    n = np.linalg.norm(x, axis=-1, keepdims=True)
    return x / np.maximum(n, eps)


def _forward_substitution_inverse(L):
    """Inverse of a unit lower triangular matrix by forward substitution."""
    n = L.shape[0]
    X = np.zeros_like(L)
    for i in range(n):
        X[i, i] = 1.0
        for j in range(i):
            X[i, j] = -np.dot(L[i, j:i], X[j:i, j])
    return X


def chunked_chain(q, k, v, g, beta, S0, scale, chunk):
    """One (sequence, value head) chain.

    q, k: [L, dk] (unnormalised); v: [L, dv]; g, beta: [L]; S0: [dv, dk].
    Returns (o [L, dv], S [dv, dk], u [L, dv]).
    """
    q = _unit(np.asarray(q, np.float64))
    k = _unit(np.asarray(k, np.float64))
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    S = np.array(S0, np.float64, copy=True)
    L = g.shape[0]
    o = np.zeros((L, v.shape[1]))
    u = np.zeros((L, v.shape[1]))
    for c0 in range(0, L, chunk):
        c1 = min(c0 + chunk, L)
        Q, K, V = q[c0:c1], k[c0:c1], v[c0:c1]
        bt = beta[c0:c1]
        Gam = np.cumsum(np.log(g[c0:c1]))
        D = np.tril(np.exp(Gam[:, None] - Gam[None, :]))
        A = np.tril(bt[:, None] * D * (K @ K.T), -1)
        Tm = _forward_substitution_inverse(np.eye(c1 - c0) + A)
        Wm = Tm @ ((bt * np.exp(Gam))[:, None] * K)
        U = Tm @ (bt[:, None] * V) - Wm @ S.T
        o[c0:c1] = scale * (np.exp(Gam)[:, None] * (Q @ S.T) + (np.tril(Q @ K.T) * D) @ U)
        u[c0:c1] = U
        S = np.exp(Gam[-1]) * S + (U * np.exp(Gam[-1] - Gam)[:, None]).T @ K
    return o, S, u


def raw_gates(a, b, A_log, dt_bias):
    """Effective decay and beta from the raw gate inputs (FP64)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    x = a + np.asarray(dt_bias, np.float64)
    sp = np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))
    g = np.exp(-np.exp(np.asarray(A_log, np.float64)) * sp)
    return g, 1.0 / (1.0 + np.exp(-b))


def chunked_forward(q, k, v, a, b, cu_seqlens, *, A_log=None, dt_bias=None, gate_mode="raw",
                    scale=None, initial_state=None, chunk=64):
    """Chunked evaluation over a packed batch (identity slots).

    Returns (output [T,Hv,dv], final_state [B,Hv,dv,dk], u [T,Hv,dv]).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    r = Hv // Hk
    B = len(cu_seqlens) - 1
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(dk)
    if gate_mode == "raw":
        g, beta = raw_gates(a, b, A_log, dt_bias)
    else:
        g, beta = np.asarray(a, np.float64), np.asarray(b, np.float64)
    out = np.zeros((T, Hv, dv))
    uu = np.zeros((T, Hv, dv))
    final = np.zeros((B, Hv, dv, dk))
    for s in range(B):
        t0, t1 = int(cu_seqlens[s]), int(cu_seqlens[s + 1])
        for h in range(Hv):
            kh = h // r
            S0 = np.zeros((dv, dk)) if initial_state is None else initial_state[s, h]
            o, S, u = chunked_chain(q[t0:t1, kh], k[t0:t1, kh], v[t0:t1, h], g[t0:t1, h], beta[t0:t1, h],
                                    S0, scale, chunk)
            out[t0:t1, h] = o
            uu[t0:t1, h] = u
            final[s, h] = S
    return out, final, uu
