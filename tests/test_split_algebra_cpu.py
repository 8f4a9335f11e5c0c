"""The algebra of the sequence-parallel (split) plan, checked in FP64 with
the oracle alone (CPU only).

Per value head each token maps the state affinely,
S -> S g (I - beta kn kn^T) + beta v kn^T, so over a segment that starts with
state S1:  S_t = S1 A_t + B_t,  where B_t is the segment run from a zero
state and A_t the segment run from the identity (dk = dv) with v = 0.  The
outputs split the same way: o_t = o_t(zero) + S1 o_t(identity), and the
final state is S1 A_last + B_last.  These are the three runs and two
combinations the split plan evaluates; here each run is the oracle's own
token-by-token recurrence, compared with the oracle over the whole sequence.
"""
import numpy as np
import pytest

import oracle
from gated_delta_rule_gateddeltanet_gb300 import workloads as wl


def _run(inp, lo, hi, state, v=None):
    """The oracle over tokens [lo, hi) of the single sequence in ``inp``."""
    sl = slice(lo, hi)
    vv = inp.v[sl] if v is None else v
    return oracle.gdn_forward(inp.q[sl], inp.k[sl], vv, inp.a[sl], inp.b[sl], np.array([0, hi - lo], np.int32),
                              A_log=inp.A_log, dt_bias=inp.dt_bias, initial_state=state)


@pytest.mark.parametrize("T,cut", [(150, 64), (97, 96), (40, 1)])
def test_segments_combine_into_the_sequential_result(T, cut):
    d = 16
    inp = wl.make_inputs(810 + T, [T], Hk=2, Hv=4, dk=d, dv=d, io_dtype=np.float64, state_std=0.3)
    Hv = 4
    o_full, f_full, _ = _run(inp, 0, T, inp.initial_state)
    o1, S1, _ = _run(inp, 0, cut, inp.initial_state)
    oz, Bf, _ = _run(inp, cut, T, np.zeros_like(inp.initial_state))
    eye = np.broadcast_to(np.eye(d), (1, Hv, d, d)).copy()
    oi, Af, _ = _run(inp, cut, T, eye, v=np.zeros_like(inp.v[cut:T]))
    # outputs: o_t = o_t(zero) + S1 o_t(identity), per head
    corr = np.einsum("hij,thj->thi", S1[0], oi)
    scale = max(1.0, np.abs(o_full).max())
    assert np.abs(o1 - o_full[:cut]).max() <= 1e-12 * scale
    assert np.abs(oz + corr - o_full[cut:]).max() <= 1e-12 * scale
    # final state: S1 A + B
    fin = np.einsum("hij,hjm->him", S1[0], Af[0]) + Bf[0]
    assert np.abs(fin - f_full[0]).max() <= 1e-12 * max(1.0, np.abs(f_full).max())


def test_identity_run_needs_the_v_term_removed():
    """With v left in, the identity run adds B_t a second time (the check
    above would fail): the decomposition is not an artefact of the inputs."""
    d, T, cut = 16, 80, 40
    inp = wl.make_inputs(830, [T], Hk=1, Hv=1, dk=d, dv=d, io_dtype=np.float64, state_std=0.3)
    o_full, _, _ = _run(inp, 0, T, inp.initial_state)
    _, S1, _ = _run(inp, 0, cut, inp.initial_state)
    oz, _, _ = _run(inp, cut, T, np.zeros_like(inp.initial_state))
    oi_wrong, _, _ = _run(inp, cut, T, np.eye(d)[None, None].copy())
    wrong = oz + np.einsum("hij,thj->thi", S1[0], oi_wrong)
    assert np.abs(wrong - o_full[cut:]).max() > 1e-3 * np.abs(o_full).max()
