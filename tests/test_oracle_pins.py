"""Pins for the FP64 oracle, independent of the oracle's own loop.

* an exact rational brute force of the unrolled transition
  S_t = g_t S_{t-1} (I - beta_t k k^T) + beta_t v_t k^T  (unit k), with the
  delta read back from the transition as u_t = (S_t - g_t S_{t-1}) k_t and the
  read-out o_t = scale S_t q_t;
* raw gate inputs whose gates are exact dyadic numbers (softplus(0) = ln 2);
* the invariants of the gated delta rule (identity gates, orthonormal-key
  recall, pack vs. one-by-one, chunked vs. sequential, replay vs. the
  sequential state, pure decay, GQA vs. repeated heads);
* the pages' closed-form footprint of dense checkpoints.

Each plausible slip in the oracle (dropped decay, wrong sign of the delta,
read-out before the update, transposed state, wrong key head) breaks at least
one of these.
"""
import json
import math
import os
from fractions import Fraction as Fr

import numpy as np
import pytest

import oracle
from oracle import chunked
from helpers import max_rel

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- brute force

def _int_vectors_with_int_norm(rng, dim, count, lim):
    out = []
    while len(out) < count:
        x = rng.integers(-lim, lim + 1, dim)
        ss = int(np.sum(x * x))
        r = math.isqrt(ss)
        if ss > 0 and r * r == ss:
            out.append((x.astype(int).tolist(), r))
    return out


def _brute(qs, ks, vs, gs, bs, S0, scale):
    """Exact rational evaluation of one chain via the unrolled transition."""
    dv, dk = len(S0), len(S0[0])
    S = [row[:] for row in S0]
    outs, us = [], []
    for (q, nq), (k, nk), v, g, beta in zip(qs, ks, vs, gs, bs):
        kn = [Fr(x, nk) for x in k]
        qn = [Fr(x, nq) for x in q]
        P = [[(1 if i == j else 0) - beta * kn[i] * kn[j] for j in range(dk)] for i in range(dk)]
        Snew = [[g * sum(S[a][m] * P[m][j] for m in range(dk)) + beta * v[a] * kn[j] for j in range(dk)]
                for a in range(dv)]
        u = [sum((Snew[a][j] - g * S[a][j]) * kn[j] for j in range(dk)) for a in range(dv)]
        o = [scale * sum(Snew[a][j] * qn[j] for j in range(dk)) for a in range(dv)]
        S = Snew
        outs.append(o)
        us.append(u)
    return outs, S, us


def _case(seed, lengths, Hk, Hv, dk, dv, gate_choices, beta_choices, lim):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    qv = _int_vectors_with_int_norm(rng, dk, T * Hk, lim)
    kv = _int_vectors_with_int_norm(rng, dk, T * Hk, lim)
    v = rng.integers(-4, 5, (T, Hv, dv)) / 2.0
    g = rng.choice(gate_choices, (T, Hv))
    beta = rng.choice(beta_choices, (T, Hv))
    S0 = rng.integers(-3, 4, (len(lengths), Hv, dv, dk)) / 4.0
    q = np.array([x for x, _ in qv], dtype=np.float64).reshape(T, Hk, dk)
    k = np.array([x for x, _ in kv], dtype=np.float64).reshape(T, Hk, dk)
    return q, k, v, g, beta, S0, qv, kv


@pytest.mark.parametrize("seed,lengths,Hk,Hv,dk,dv", [
    (1, [5], 1, 1, 4, 3),
    (2, [3, 0, 4], 1, 2, 4, 2),
    (3, [2, 6], 2, 4, 4, 4),
    (4, [4], 1, 1, 16, 2),
])
def test_oracle_matches_exact_brute_force(seed, lengths, Hk, Hv, dk, dv):
    gate_choices = [1.0, 0.75, 0.5, 0.875, 0.0]
    beta_choices = [0.5, 0.25, 1.0, 0.0, 0.375]
    q, k, v, g, beta, S0, qv, kv = _case(seed, lengths, Hk, Hv, dk, dv, gate_choices, beta_choices,
                                         lim=6 if dk == 4 else 3)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    cap = max(lengths)
    out, final, caps = oracle.gdn_forward(q, k, v, g, beta, cu, gate_mode="precomputed",
                                          initial_state=S0, capacity=cap)
    scale = Fr(1, int(math.isqrt(dk)))
    r = Hv // Hk
    W = oracle.capsule_width(Hk, Hv, dk, dv)
    assert caps.shape == (len(lengths), cap, W)
    for s in range(len(lengths)):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        for h in range(Hv):
            kh = h // r
            S0f = [[Fr(x) for x in row] for row in S0[s, h]]
            outs, Sx, us = _brute([qv[t * Hk + kh] for t in range(t0, t1)],
                                  [kv[t * Hk + kh] for t in range(t0, t1)],
                                  [[Fr(x) for x in v[t, h]] for t in range(t0, t1)],
                                  [Fr(g[t, h]) for t in range(t0, t1)],
                                  [Fr(beta[t, h]) for t in range(t0, t1)], S0f, scale)
            ex_final = np.array([[float(x) for x in row] for row in Sx])
            assert max_rel(final[s, h], ex_final) <= 1e-13
            for i, t in enumerate(range(t0, t1)):
                ex_o = np.array([float(x) for x in outs[i]])
                ex_u = np.array([float(x) for x in us[i]])
                assert np.max(np.abs(out[t, h] - ex_o)) <= 1e-13 * max(1.0, np.max(np.abs(ex_o)))
                row = caps[s, i]
                assert row[h] == g[t, h]
                assert np.max(np.abs(row[Hv + Hk * dk + h * dv: Hv + Hk * dk + (h + 1) * dv] - ex_u)) <= 1e-13
                kx, nk = kv[t * Hk + kh]
                assert np.allclose(row[Hv + kh * dk: Hv + (kh + 1) * dk], np.array(kx) / nk, rtol=0, atol=1e-15)
            # rows past the sequence stay untouched
            assert np.all(np.isnan(caps[s, t1 - t0:]))


def test_raw_gates_exact_dyadic_cases():
    """softplus(0) = ln 2, so A_log in {0, ln 2, ln 3} gives g = 1/2, 1/4, 1/8;
    b in {0, ln 3, -ln 3, ln 7} gives beta = 1/2, 3/4, 1/4, 7/8.  Checked against
    the exact brute force with those rational gates."""
    rng = np.random.default_rng(7)
    Hk, Hv, dk, dv, T = 1, 3, 4, 3, 6
    A_log = np.log(np.array([1.0, 2.0, 3.0]))
    gmap = [Fr(1, 2), Fr(1, 4), Fr(1, 8)]
    dt_bias = np.array([0.375, -1.25, 2.5])
    a = np.tile(-dt_bias, (T, 1))  # a + dt_bias == 0 exactly
    bvals = np.log(np.array([1.0, 3.0, 1.0 / 3.0, 7.0]))
    bmap = [Fr(1, 2), Fr(3, 4), Fr(1, 4), Fr(7, 8)]
    bidx = rng.integers(0, 4, (T, Hv))
    b = bvals[bidx]
    qv = _int_vectors_with_int_norm(rng, dk, T, 6)
    kv = _int_vectors_with_int_norm(rng, dk, T, 6)
    q = np.array([x for x, _ in qv], float).reshape(T, Hk, dk)
    k = np.array([x for x, _ in kv], float).reshape(T, Hk, dk)
    v = rng.integers(-4, 5, (T, Hv, dv)) / 2.0
    S0 = rng.integers(-3, 4, (1, Hv, dv, dk)) / 4.0
    cu = np.array([0, T], np.int32)
    out, final, caps = oracle.gdn_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias,
                                          initial_state=S0, capacity=T)
    for h in range(Hv):
        outs, Sx, us = _brute(qv, kv, [[Fr(x) for x in v[t, h]] for t in range(T)], [gmap[h]] * T,
                              [bmap[bidx[t, h]] for t in range(T)],
                              [[Fr(x) for x in row] for row in S0[0, h]], Fr(1, 2))
        assert max_rel(final[0, h], np.array([[float(x) for x in r] for r in Sx])) <= 1e-13
        assert max_rel(out[:, h], np.array([[float(x) for x in o] for o in outs])) <= 1e-13
        assert np.allclose(caps[0, :, h], float(gmap[h]), rtol=1e-15, atol=0)


def test_raw_gates_stable_at_extremes():
    """softplus must not overflow: a + dt_bias = -800 gives g = 1 exactly, +800
    gives g = 0; b = +-800 gives beta = 1 and 0."""
    Hk, Hv, dk, dv = 1, 2, 4, 2
    q = np.ones((2, Hk, dk))
    k = np.ones((2, Hk, dk))
    v = np.ones((2, Hv, dv))
    a = np.array([[-800.0, 800.0], [-800.0, 800.0]])
    b = np.array([[800.0, -800.0], [-800.0, 800.0]])
    out, final, caps = oracle.gdn_forward(q, k, v, a, b, np.array([0, 2]), A_log=np.zeros(Hv),
                                          dt_bias=np.zeros(Hv), capacity=2)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(final))
    assert caps[0, 0, 0] == 1.0 and caps[0, 0, 1] == 0.0


# ------------------------------------------------------- L2-norm clamp (eps)
#
# The pages fuse the Qwen q/k normalisation into the operator ("[CUDA] Add
# compact GatedDeltaNet operator", Description) without printing it; the
# reading taken is x / max(|x|, 1e-6).  These cases fix that reading by hand:
# a zero key gives kn = 0, so u = beta v and the state is only decayed; a zero
# query gives a zero output; a vector shorter than eps is divided by eps (a
# non-unit direction, exact in rationals up to the one rounding of the
# division); a vector just longer than eps is normalised as usual.  A missing
# clamp (NaN), eps added to the norm, eps on the squared norm, or another eps
# each change one of the expected values below.

EPS = Fr(1e-6)  # the double nearest 1e-6, exactly


def _exact_unit(x):
    """x / max(|x|, eps) in rationals for integer-times-power-of-two vectors
    whose norm is rational (so sqrt is exact)."""
    xs = [Fr(float(e)) for e in x]
    ss = sum(e * e for e in xs)
    if ss == 0:
        return [Fr(0)] * len(xs)
    n_num, n_den = math.isqrt(ss.numerator), math.isqrt(ss.denominator)
    assert Fr(n_num, n_den) ** 2 == ss, "test vector must have a rational norm"
    nrm = Fr(n_num, n_den)
    return [e / max(nrm, EPS) for e in xs]


def _brute_units(qns, kns, vs, gs, bs, S0, scale):
    """The unrolled transition S_t = g S (I - beta kn kn^T) + beta v kn^T with
    the normalised vectors given (any length), read-out o = scale S_t qn."""
    dv, dk = len(S0), len(S0[0])
    S = [row[:] for row in S0]
    outs, us = [], []
    for qn, kn, v, g, beta in zip(qns, kns, vs, gs, bs):
        P = [[(1 if i == j else 0) - beta * kn[i] * kn[j] for j in range(dk)] for i in range(dk)]
        Snew = [[g * sum(S[a][m] * P[m][j] for m in range(dk)) + beta * v[a] * kn[j] for j in range(dk)]
                for a in range(dv)]
        u = [beta * (v[a] - g * sum(S[a][j] * kn[j] for j in range(dk))) for a in range(dv)]
        outs.append([scale * sum(Snew[a][j] * qn[j] for j in range(dk)) for a in range(dv)])
        us.append(u)
        S = Snew
    return outs, S, us


def test_l2_norm_clamp_zero_and_tiny_vectors():
    Hk, Hv, dk, dv = 1, 2, 4, 3
    e23, e22 = 2.0 ** -23, 2.0 ** -22
    normal_q, normal_k = [1, 2, 2, 4], [2, 4, 1, 2]           # norms 5 and 5
    rows = [  # (q, k) per token
        (normal_q, normal_k),
        (normal_q, [0, 0, 0, 0]),                               # zero key
        ([0, 0, 0, 0], normal_k),                               # zero query
        (normal_q, [3 * e23, 4 * e23, 0, 0]),                   # |k| = 5.96e-7 < eps
        ([0, 3 * e23, 0, 4 * e23], normal_k),                   # |q| = 5.96e-7 < eps
        (normal_q, [3 * e22, 0, 4 * e22, 0]),                   # |k| = 1.19e-6 > eps
        ([0, 0, 0, 0], [0, 0, 0, 0]),                           # both zero
        ([e23, e23, e23, e23], [-e23, e23, -e23, e23]),         # |x| = 2.4e-7, both tiny
        (normal_q, normal_k),
    ]
    T = len(rows)
    q = np.array([r[0] for r in rows], np.float64).reshape(T, Hk, dk)
    k = np.array([r[1] for r in rows], np.float64).reshape(T, Hk, dk)
    rng = np.random.default_rng(17)
    v = rng.integers(-4, 5, (T, Hv, dv)) / 2.0
    g = rng.choice([0.5, 0.75, 1.0], (T, Hv))
    beta = rng.choice([0.25, 0.5, 1.0], (T, Hv))
    S0 = rng.integers(-3, 4, (1, Hv, dv, dk)) / 4.0
    cu = np.array([0, T], np.int32)
    out, final, caps = oracle.gdn_forward(q, k, v, g, beta, cu, gate_mode="precomputed", initial_state=S0,
                                          capacity=T)
    W = oracle.capsule_width(Hk, Hv, dk, dv)
    kn_caps = caps[0, :, Hv:Hv + Hk * dk]
    u_caps = caps[0, :, Hv + Hk * dk:W].reshape(T, Hv, dv)

    # by hand: the clamp's effect on the normalised key
    assert np.array_equal(kn_caps[1], np.zeros(dk)) and np.array_equal(kn_caps[6], np.zeros(dk))
    np.testing.assert_allclose(kn_caps[3], np.array([3, 4, 0, 0]) * e23 / 1e-6, rtol=1e-15)
    np.testing.assert_allclose(kn_caps[5], np.array([3, 0, 4, 0]) / 5.0, rtol=1e-15)
    np.testing.assert_allclose(kn_caps[7], np.array([-1, 1, -1, 1]) * e23 / 1e-6, rtol=1e-15)
    # zero key: the delta is beta v exactly, and the state is only decayed
    assert np.array_equal(u_caps[1], beta[1][:, None] * v[1])
    _, s0, _ = oracle.gdn_forward(q[:1], k[:1], v[:1], g[:1], beta[:1], np.array([0, 1]),
                                  gate_mode="precomputed", initial_state=S0)
    _, s1, _ = oracle.gdn_forward(q[:2], k[:2], v[:2], g[:2], beta[:2], np.array([0, 2]),
                                  gate_mode="precomputed", initial_state=S0)
    assert np.array_equal(s1[0], g[1][:, None, None] * s0[0])
    # zero query: a zero output
    assert np.array_equal(out[2], np.zeros((Hv, dv))) and np.array_equal(out[6], np.zeros((Hv, dv)))

    # everything against the exact rational evaluation with the clamped vectors
    qns = [_exact_unit(q[t, 0]) for t in range(T)]
    kns = [_exact_unit(k[t, 0]) for t in range(T)]
    for h in range(Hv):
        outs, Sx, us = _brute_units(qns, kns, [[Fr(x) for x in v[t, h]] for t in range(T)],
                                    [Fr(g[t, h]) for t in range(T)], [Fr(beta[t, h]) for t in range(T)],
                                    [[Fr(x) for x in row] for row in S0[0, h]], Fr(1, 2))
        assert max_rel(final[0, h], np.array([[float(x) for x in r] for r in Sx])) <= 1e-13
        for t in range(T):
            ex_o = np.array([float(x) for x in outs[t]])
            assert np.max(np.abs(out[t, h] - ex_o)) <= 1e-13 * max(1.0, np.max(np.abs(ex_o)))
            assert np.max(np.abs(u_caps[t, h] - np.array([float(x) for x in us[t]]))) <= 1e-13


def test_chunked_evaluator_clamps_like_the_sequential_oracle():
    """The chunked (WY) evaluator with runs of zero and sub-eps keys and queries
    inside and across chunks equals the sequential oracle."""
    lengths = [40, 23]
    q, k, v, a, b, A_log, dt_bias, S0, cu = _rand_batch(33, lengths, 1, 2, 16, 8)
    k[3] = 0.0
    k[10:14] = 0.0
    q[5:9] = 0.0
    k[20] *= 1e-8 / np.linalg.norm(k[20])
    q[21] *= 3e-7 / np.linalg.norm(q[21])
    k[41] *= 5e-7 / np.linalg.norm(k[41])
    out, final, caps = oracle.gdn_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias,
                                          initial_state=S0, capacity=max(lengths))
    for chunk in (1, 8, 64):
        o2, f2, u2 = chunked.chunked_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias,
                                             initial_state=S0, chunk=chunk)
        assert max_rel(o2, out) <= 1e-10
        assert max_rel(f2, final) <= 1e-10
    assert np.array_equal(out[5:9], np.zeros_like(out[5:9]))


# ---------------------------------------------------------------- invariants

def _rand_batch(seed, lengths, Hk, Hv, dk, dv, state=True):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    q = rng.standard_normal((T, Hk, dk))
    k = rng.standard_normal((T, Hk, dk))
    v = rng.standard_normal((T, Hv, dv))
    a = rng.standard_normal((T, Hv))
    b = rng.standard_normal((T, Hv))
    A_log = np.log(rng.uniform(1, 16, Hv))
    dt_bias = np.log(np.expm1(rng.uniform(1e-3, 0.1, Hv)))
    S0 = rng.standard_normal((len(lengths), Hv, dv, dk)) * 0.02 if state else None
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q, k, v, a, b, A_log, dt_bias, S0, cu


def test_identity_gates_leave_state_unchanged():
    q, k, v, a, b, A_log, dt_bias, S0, cu = _rand_batch(11, [7, 3], 2, 4, 8, 8)
    ones = np.ones_like(a)
    zeros = np.zeros_like(b)
    out, final, _ = oracle.gdn_forward(q, k, v, ones, zeros, cu, gate_mode="precomputed", initial_state=S0)
    assert np.array_equal(final, S0)
    # the read-out is then a plain matrix-vector product with the fixed state
    qn = q / np.linalg.norm(q, axis=-1, keepdims=True)
    for s in range(2):
        for t in range(cu[s], cu[s + 1]):
            for h in range(4):
                ref = (S0[s, h] @ qn[t, h // 2]) / math.sqrt(8)
                assert np.allclose(out[t, h], ref, rtol=1e-13, atol=1e-16)


def test_orthonormal_keys_recall_values():
    """g = 1, beta = 1, orthonormal keys: after writing (k_i, v_i), S k_i = v_i."""
    rng = np.random.default_rng(5)
    dk, dv, n = 16, 8, 10
    for keys in (np.eye(dk)[:n], np.linalg.qr(rng.standard_normal((dk, dk)))[0][:, :n].T):
        q = rng.standard_normal((n, 1, dk))
        k = keys.reshape(n, 1, dk)
        v = rng.standard_normal((n, 1, dv))
        S0 = rng.standard_normal((1, 1, dv, dk))
        _, final, _ = oracle.gdn_forward(q, k, v, np.ones((n, 1)), np.ones((n, 1)), np.array([0, n]),
                                         gate_mode="precomputed", initial_state=S0)
        recalled = final[0, 0] @ keys.T  # [dv, n]
        # standard-basis keys: one rounding of s + (v - s) per entry; otherwise FP64 noise
        tol = 1e-15 if np.array_equal(keys, np.eye(dk)[:n]) else 1e-12
        assert np.max(np.abs(recalled.T - v[:, 0])) <= tol * np.max(np.abs(v))


def test_pack_equals_one_by_one_bitwise():
    lengths = [17, 1, 0, 33, 5]
    q, k, v, a, b, A_log, dt_bias, S0, cu = _rand_batch(21, lengths, 2, 6, 16, 8)
    out, final, caps = oracle.gdn_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias,
                                          initial_state=S0, capacity=8)
    for s, L in enumerate(lengths):
        t0, t1 = cu[s], cu[s + 1]
        o1, f1, c1 = oracle.gdn_forward(q[t0:t1], k[t0:t1], v[t0:t1], a[t0:t1], b[t0:t1],
                                        np.array([0, L]), A_log=A_log, dt_bias=dt_bias,
                                        initial_state=S0[s:s + 1], capacity=8)
        assert np.array_equal(out[t0:t1], o1)
        assert np.array_equal(final[s], f1[0])
        assert np.array_equal(caps[s], c1[0], equal_nan=True)


@pytest.mark.parametrize("chunk", [1, 3, 16, 64])
def test_chunked_equals_sequential(chunk):
    lengths = [70, 9, 130]
    q, k, v, a, b, A_log, dt_bias, S0, cu = _rand_batch(31, lengths, 2, 4, 16, 12)
    out, final, caps = oracle.gdn_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias,
                                          initial_state=S0, capacity=max(lengths))
    o2, f2, u2 = chunked.chunked_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias,
                                         initial_state=S0, chunk=chunk)
    assert max_rel(o2, out) <= 1e-10
    assert max_rel(f2, final) <= 1e-10
    Hv, Hk, dk, dv = 4, 2, 16, 12
    for s, L in enumerate(lengths):
        u_oracle = caps[s, :L, Hv + Hk * dk:].reshape(L, Hv, dv)
        assert max_rel(u2[cu[s]:cu[s + 1]], u_oracle) <= 1e-10


def test_replay_reproduces_sequential_state_for_every_prefix():
    L = 9
    q, k, v, a, b, A_log, dt_bias, S0, cu = _rand_batch(41, [L], 2, 6, 8, 8)
    _, _, caps = oracle.gdn_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias,
                                    initial_state=S0, capacity=L)
    banks = np.concatenate([S0, np.zeros_like(S0)])
    for j in range(L + 1):
        _, fj, _ = oracle.gdn_forward(q[:j], k[:j], v[:j], a[:j], b[:j], np.array([0, j]), A_log=A_log,
                                      dt_bias=dt_bias, initial_state=S0)
        replayed = oracle.gdn_replay(banks, [0], [1], caps, [j], num_k_heads=2)
        assert max_rel(replayed[1], fj[0]) <= 1e-12
        assert np.array_equal(replayed[0], S0[0])  # the source bank is untouched


def test_pure_decay():
    """beta = 0: S_T = (prod g) S_0 and o_t = scale (prod_{s<=t} g_s) S_0 qn_t."""
    rng = np.random.default_rng(3)
    T, dk, dv = 12, 8, 4
    q = rng.standard_normal((T, 1, dk))
    k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = rng.uniform(0.5, 1.0, (T, 1))
    S0 = rng.standard_normal((1, 1, dv, dk))
    out, final, _ = oracle.gdn_forward(q, k, v, g, np.zeros((T, 1)), np.array([0, T]),
                                       gate_mode="precomputed", initial_state=S0)
    cum = np.cumprod(g[:, 0])
    assert max_rel(final[0, 0], cum[-1] * S0[0, 0]) <= 1e-14
    qn = q[:, 0] / np.linalg.norm(q[:, 0], axis=-1, keepdims=True)
    ref = cum[:, None] * (qn @ S0[0, 0].T) / math.sqrt(dk)
    assert max_rel(out[:, 0], ref) <= 1e-13


def test_gqa_equals_repeated_key_heads():
    """Value head h reads key head h // (Hv/Hk): GQA equals plain multi-head with
    each key head repeated for its value heads."""
    q, k, v, a, b, A_log, dt_bias, S0, cu = _rand_batch(51, [6, 4], 2, 6, 8, 8)
    o1, f1, _ = oracle.gdn_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias, initial_state=S0)
    qr, kr = np.repeat(q, 3, axis=1), np.repeat(k, 3, axis=1)
    o2, f2, _ = oracle.gdn_forward(qr, kr, v, a, b, cu, A_log=A_log, dt_bias=dt_bias, initial_state=S0)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)


def test_slots_place_state():
    q, k, v, a, b, A_log, dt_bias, S0, cu = _rand_batch(61, [3, 2], 1, 2, 8, 4)
    pool = np.random.default_rng(0).standard_normal((5, 2, 4, 8))
    slots = np.array([4, 1], np.int32)
    pool[4], pool[1] = S0[0], S0[1]
    o1, f1, _ = oracle.gdn_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias, initial_state=S0)
    o2, f2, _ = oracle.gdn_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias, initial_state=pool,
                                   state_slots=slots)
    assert np.array_equal(o1, o2)
    assert np.array_equal(f2[4], f1[0]) and np.array_equal(f2[1], f1[1])
    for untouched in (0, 2, 3):
        assert np.array_equal(f2[untouched], pool[untouched])


def test_bad_packing_and_slots_are_rejected():
    q, k, v, a, b, A_log, dt_bias, S0, cu = _rand_batch(71, [3, 2], 1, 1, 4, 4)
    with pytest.raises(oracle.OracleError):
        oracle.gdn_forward(q, k, v, a, b, np.array([0, 4, 3]), A_log=A_log, dt_bias=dt_bias)
    with pytest.raises(oracle.OracleError):
        oracle.gdn_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias, initial_state=S0,
                           state_slots=[0, 2])


# ---------------------------------------------------------------- closed forms

def test_dense_checkpoint_footprint_matches_pages():
    """The pages: a four-slot window over 48 GDN layers at the Qwen3.8 geometry
    costs 576 MiB of dense FP32 checkpoints; one state is Hv x dv x dk FP32."""
    fx = json.load(open(os.path.join(GOLDEN, "footprint.json")))
    _, final, _ = oracle.gdn_forward(np.zeros((0, 16, 128)), np.zeros((0, 16, 128)), np.zeros((0, 48, 128)),
                                     np.zeros((0, 48)), np.zeros((0, 48)), np.array([0]),
                                     A_log=np.zeros(48), dt_bias=np.zeros(48), num_state_slots=1)
    one_state = final.astype(np.float32).nbytes  # one request-layer state in FP32
    assert fx["slots"] * fx["layers"] * one_state == fx["bytes"]
    # the compact capsule per token-layer at the same geometry
    assert oracle.capsule_width(16, 48, 128, 128) * 4 == 32960


# ---------------------------------------------------------------- causal conv

def test_conv_matches_library_convolution():
    """Zero history, one sequence: the conv is numpy's full convolution with the
    reversed taps, truncated causally, then SiLU."""
    rng = np.random.default_rng(9)
    T, C, K = 23, 5, 4
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, K))
    bias = rng.standard_normal(C)
    out, st, _ = oracle.conv_forward(x, w, np.array([0, T]), np.zeros((1, C, K - 1)), bias=bias)
    for c in range(C):
        pre = np.convolve(x[:, c], w[c, ::-1])[:T] + bias[c]
        assert np.allclose(out[:, c], pre / (1 + np.exp(-pre)), rtol=1e-13, atol=1e-14)
        assert np.array_equal(st[0, c], x[T - K + 1:, c])


def test_conv_all_ones_decode():
    """All-ones taps, inputs and history: every output is silu(K + bias)."""
    C, K = 3, 4
    out, st, _ = oracle.conv_forward(np.ones((1, C)), np.ones((C, K)), np.array([0, 1]), np.ones((1, C, K - 1)),
                                     bias=np.full(C, 0.5))
    pre = K + 0.5
    assert np.allclose(out, pre / (1 + math.exp(-pre)), rtol=1e-15)


def test_conv_sequential_prefix_equivalence_and_replay():
    """Running a sequence in two pieces with the carried state equals running it
    whole; replaying the captured values of the first n tokens reproduces the
    state after n tokens."""
    rng = np.random.default_rng(10)
    T, C, K = 12, 6, 4
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, K))
    st0 = rng.standard_normal((1, C, K - 1))
    o_all, st_all, vals = oracle.conv_forward(x, w, np.array([0, T]), st0, capacity=T)
    o_a, st_a, _ = oracle.conv_forward(x[:5], w, np.array([0, 5]), st0)
    o_b, st_b, _ = oracle.conv_forward(x[5:], w, np.array([0, T - 5]), st_a)
    assert np.array_equal(np.concatenate([o_a, o_b]), o_all)
    assert np.array_equal(st_b, st_all)
    pool = np.concatenate([st0, np.zeros_like(st0)])
    for n in range(T + 1):
        _, st_n, _ = oracle.conv_forward(x[:n], w, np.array([0, n]), st0)
        rep = oracle.conv_replay(pool, [0], [1], vals, [n])
        assert np.array_equal(rep[1], st_n[0])


def test_conv_capture_count_bounds_the_capture():
    """The optional per-request capture count limits the compact capture to
    the first capture_count[b] appended inputs; counts above the capacity are
    rejected."""
    rng = np.random.default_rng(12)
    lengths, C, K, cap = [5, 2, 6], 3, 4, 4
    T = sum(lengths)
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, K))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    st = rng.standard_normal((3, C, K - 1))
    _, _, full = oracle.conv_forward(x, w, cu, st, capacity=cap)
    _, _, part = oracle.conv_forward(x, w, cu, st, capacity=cap, capture_count=[2, 4, 0])
    for s, n in enumerate([2, 4, 0]):
        m = min(n, lengths[s])
        assert np.array_equal(part[s, :m], full[s, :m])
        assert np.all(np.isnan(part[s, m:]))
    with pytest.raises(oracle.OracleError):
        oracle.conv_forward(x, w, cu, st, capacity=cap, capture_count=[5, 0, 0])
