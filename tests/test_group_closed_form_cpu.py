"""The four-token closed form that the tensor-core short-span path evaluates,
checked in FP64 against the token-by-token oracle (CPU only).

Within a group of tokens t = 0 .. n-1 entering with state S0 (V-major, rows
are value channels), with G_t = g_0 ... g_t and r(t, s) = g_{s+1} ... g_t:
    P_t = S0 k_t,  Q_t = S0 q_t
    u_t = beta_t v_t - beta_t G_t P_t - sum_{s<t} beta_t r(t,s) (k_s . k_t) u_s
    o_t = scale (G_t Q_t + sum_{s<=t} r(t,s) (k_s . q_t) u_s)
    S   = G_{n-1} S0 + sum_s r(n-1,s) u_s k_s^T
Groups hold at most four tokens; a group with fewer tokens is padded with
zero vectors, g = 1 and beta = 0, which must leave every result unchanged.
The decay ratios are formed as products (never G_t / G_s), so gates of 0 and
of 1e-30 stay exact.  Written from the recurrence, independently of the CUDA
code; the oracle is the reference.
"""
import numpy as np
import pytest

import oracle
from gated_delta_rule_gateddeltanet_gb300 import workloads as wl


TB = 4


def _unit(x):
    n = np.sqrt((x * x).sum(-1, keepdims=True))
    return x / np.maximum(n, 1e-6)


def _group(S0, k, q, v, g, beta, n, scale):
    """One padded group of TB tokens (n live) for one head: returns o [n, dv], u [n, dv], S."""
    live = np.arange(TB) < n
    gp = np.where(live, g, 1.0)
    bp = np.where(live, beta, 0.0)
    kp = np.where(live[:, None], k, 0.0)
    qp = np.where(live[:, None], q, 0.0)
    vp = np.where(live[:, None], v, 0.0)
    r = lambda t, s: np.prod(gp[s + 1:t + 1])  # empty product = 1
    G = [r(t, 0) * gp[0] for t in range(TB)]
    P = S0 @ kp.T  # [dv, TB]
    Q = S0 @ qp.T
    u = np.zeros((S0.shape[0], TB))
    for t in range(TB):
        x = bp[t] * vp[t] - bp[t] * G[t] * P[:, t]
        for s in range(t):
            x = x - bp[t] * r(t, s) * (kp[s] @ kp[t]) * u[:, s]
        u[:, t] = x
    o = np.zeros((S0.shape[0], TB))
    for t in range(TB):
        acc = G[t] * Q[:, t] if live[t] else 0.0 * Q[:, t]
        for s in range(t + 1):
            if live[t]:
                acc = acc + r(t, s) * (kp[s] @ qp[t]) * u[:, s]
        o[:, t] = scale * acc
    e = np.array([r(n - 1, s) if live[s] else 0.0 for s in range(TB)])
    S = G[n - 1] * S0 + (u * e) @ kp
    return o[:, :n].T, u[:, :n].T, S


def _grouped_forward(inp, g_all, beta_all):
    """The whole batch through the grouped closed form (precomputed gates)."""
    Hk, Hv, dk, dv = inp.dims
    rep = Hv // Hk
    scale = 1.0 / np.sqrt(dk)
    q = _unit(inp.q.astype(np.float64))
    k = _unit(inp.k.astype(np.float64))
    v = inp.v.astype(np.float64)
    out = np.zeros((inp.T, Hv, dv))
    final = inp.initial_state.astype(np.float64).copy()
    deltas = np.zeros((inp.T, Hv, dv))
    cu = inp.cu_seqlens
    for b in range(inp.B):
        for h in range(Hv):
            S = final[b, h]
            for t0 in range(cu[b], cu[b + 1], TB):
                n = min(TB, cu[b + 1] - t0)
                sl = slice(t0, t0 + TB)
                pad = lambda x: np.concatenate([x[sl], np.zeros((TB - len(x[sl]),) + x.shape[1:])])
                o, u, S = _group(S, pad(k[:, h // rep]), pad(q[:, h // rep]), pad(v[:, h]),
                                 pad(g_all[:, h].astype(np.float64)), pad(beta_all[:, h].astype(np.float64)), n, scale)
                out[t0:t0 + n, h] = o
                deltas[t0:t0 + n, h] = u
            final[b, h] = S
    return out, final, deltas


@pytest.mark.parametrize("lengths", [[4, 3, 9, 1, 0, 7], [32, 2, 5]])
def test_grouped_closed_form_equals_recurrence(lengths):
    inp = wl.make_inputs(700 + len(lengths), lengths, Hk=2, Hv=4, dk=16, dv=8, io_dtype=np.float32, state_std=0.3,
                         capacity=max(lengths))
    rng = np.random.default_rng(701)
    g = rng.choice(np.array([0.0, 1e-30, 0.3, 0.9, 1.0]), size=inp.a.shape)
    beta = rng.choice(np.array([0.0, 0.5, 1.0]), size=inp.b.shape)
    o_ref, f_ref, caps = oracle.gdn_forward(inp.q, inp.k, inp.v, g, beta, inp.cu_seqlens, gate_mode="precomputed",
                                            initial_state=inp.initial_state, capacity=max(lengths))
    out, final, deltas = _grouped_forward(inp, g, beta)
    assert np.abs(out - o_ref).max() <= 1e-12 * max(1.0, np.abs(o_ref).max())
    assert np.abs(final - f_ref).max() <= 1e-12 * max(1.0, np.abs(f_ref).max())
    # the capsule deltas (u per token) are the grouped form's u
    Hk, Hv, dk, dv = inp.dims
    ubase = Hv + Hk * dk
    cu = inp.cu_seqlens
    for b in range(inp.B):
        for i in range(cu[b + 1] - cu[b]):
            u_ref = caps[b, i, ubase:ubase + Hv * dv].reshape(Hv, dv)
            assert np.abs(deltas[cu[b] + i] - u_ref).max() <= 1e-12 * max(1.0, np.abs(u_ref).max())


def test_padding_tokens_change_nothing():
    """A lone token in a padded group equals the recurrence's single step."""
    rng = np.random.default_rng(702)
    dk, dv = 8, 5
    S0 = rng.normal(size=(dv, dk))
    k = _unit(rng.normal(size=(TB, dk)))
    q = _unit(rng.normal(size=(TB, dk)))
    v = rng.normal(size=(TB, dv))
    g = np.array([0.7, 0.2, 0.3, 0.4])
    beta = np.array([0.6, 0.1, 0.2, 0.3])
    o, u, S = _group(S0, k, q, v, g, beta, 1, 0.5)
    S1 = g[0] * S0
    u_ref = beta[0] * (v[0] - S1 @ k[0])
    S1 = S1 + np.outer(u_ref, k[0])
    assert np.allclose(u[0], u_ref, rtol=0, atol=1e-14)
    assert np.allclose(o[0], 0.5 * S1 @ q[0], rtol=0, atol=1e-14)
    assert np.allclose(S, S1, rtol=0, atol=1e-14)
