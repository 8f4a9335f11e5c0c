"""Seeded random sweep of gdn_forward against the FP64 oracle: every case
draws head sizes (dk, dv independently in {32, 64, 128}), a GQA ratio, a
ragged batch (empty, one-token, short and multi-chunk spans), the I/O dtype,
raw or precomputed gates, the plan, in-place or out-of-place states with
scattered slots, an optional initial state and a capsule capacity, so that
the kernels meet combinations no hand-written case lists.

Tolerances (max |gpu - oracle| / max |oracle| per tensor): where a tensor-core
chunked kernel may run (automatic plan with a span past the recurrent limit,
forced chunked plan) 2e-3 on outputs, final states and capsule deltas; on the
recurrent plan FP32-level, 1e-5 on states and deltas and on FP32 outputs, and
2e-3 on FP16 outputs (one FP16 rounding).  Capsule decays and keys: 1e-5.
Slots no sequence names stay bit for bit as they were.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import max_rel
from gpu_common import run_gpu, capsule_parts, dev

from gated_delta_rule_gateddeltanet_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

N_CASES = 32
RECURRENT_LIMIT = {128: 32}  # the automatic plan's recurrent limit at dk = dv = 128 (256 below)


def _case(i):
    rng = np.random.default_rng(5000 + i)
    dk = int(rng.choice([32, 64, 128], p=[0.25, 0.25, 0.5]))
    dv = dk if rng.random() < 0.6 else int(rng.choice([32, 64, 128]))
    Hk = int(rng.choice([1, 2, 4]))
    Hv = Hk * int(rng.choice([1, 2, 3]))
    B = int(rng.integers(1, 7))
    kinds = rng.choice(["empty", "one", "short", "mid", "long"], size=B, p=[0.1, 0.25, 0.3, 0.2, 0.15])
    span = {"empty": (0, 1), "one": (1, 2), "short": (2, 9), "mid": (9, 41), "long": (41, 300)}
    lengths = [int(rng.integers(*span[k])) for k in kinds]
    io = np.float16 if rng.random() < 0.6 else np.float32
    plan = str(rng.choice(["auto", "recurrent", "chunked"], p=[0.5, 0.25, 0.25]))
    gates = "raw" if rng.random() < 0.75 else "precomputed"
    in_place = bool(rng.random() < 0.5)
    extra = int(rng.integers(0, 4))
    num_slots = B + extra
    slots = rng.permutation(num_slots)[:B].astype(np.int32)
    state_std = 0.02 if rng.random() < 0.8 else None
    cap = int(rng.choice([0, 1, 4, 70]))
    return dict(seed=6000 + i, dk=dk, dv=dv, Hk=Hk, Hv=Hv, lengths=lengths, io=io, plan=plan, gates=gates,
                in_place=in_place, num_slots=num_slots, slots=slots, state_std=state_std, cap=cap)


def _ids():
    out = []
    for i in range(N_CASES):
        c = _case(i)
        out.append(f"{i}-d{c['dk']}x{c['dv']}-H{c['Hk']}x{c['Hv']}-{c['plan']}-{c['gates']}-"
                   f"{'f16' if c['io'] == np.float16 else 'f32'}-{'inplace' if c['in_place'] else 'oop'}")
    return out


@pytest.mark.parametrize("i", range(N_CASES), ids=_ids())
def test_random_configuration_matches_oracle(i):
    c = _case(i)
    inp = wl.make_inputs(c["seed"], c["lengths"], Hk=c["Hk"], Hv=c["Hv"], dk=c["dk"], dv=c["dv"], io_dtype=c["io"],
                         state_std=c["state_std"], num_slots=c["num_slots"], capacity=c["cap"],
                         state_slots=c["slots"])
    a = b = None
    if c["gates"] == "precomputed":  # multiplicative decays and betas, zero and one included
        rng = np.random.default_rng(c["seed"] + 1)
        a = rng.uniform(0.3, 1.0, size=inp.a.shape).astype(np.float32)
        b = rng.uniform(0.0, 1.0, size=inp.b.shape).astype(np.float32)
        if a.size:
            a.flat[0], b.flat[-1] = 1.0, 0.0
    slots_total = c["num_slots"]
    final_state = None
    if inp.initial_state is None:  # a pool to hold the final states (the oracle starts from zeros)
        final_state = torch.full((slots_total, c["Hv"], c["dv"], c["dk"]), float("nan"), dtype=torch.float32,
                                 device=dev())
    gpu = run_gpu(inp, plan=c["plan"], gate_mode=c["gates"], a=a, b=b, in_place=c["in_place"],
                  final_state=final_state)
    ref = oracle.gdn_forward(inp.q, inp.k, inp.v, inp.a if a is None else a, inp.b if b is None else b,
                             inp.cu_seqlens, A_log=inp.A_log, dt_bias=inp.dt_bias, gate_mode=c["gates"],
                             initial_state=inp.initial_state, state_slots=inp.state_slots,
                             num_state_slots=slots_total, capacity=c["cap"])
    out, final, caps = gpu
    o_ref, f_ref, c_ref = ref

    longest = max(c["lengths"])
    limit = RECURRENT_LIMIT.get(c["dk"], 256) if c["dk"] == c["dv"] else 256
    tensor_cores = c["plan"] == "chunked" or (c["plan"] == "auto" and longest > limit)
    tol_state = 2e-3 if tensor_cores else 1e-5
    tol_out = 2e-3 if (tensor_cores or c["io"] == np.float16) else 1e-5
    assert max_rel(out, o_ref) <= tol_out, max_rel(out, o_ref)
    named = c["slots"]
    assert max_rel(final[named], f_ref[named]) <= tol_state, max_rel(final[named], f_ref[named])
    others = np.setdiff1d(np.arange(slots_total), named)
    if inp.initial_state is not None and others.size:
        assert np.array_equal(final[others], inp.initial_state[others].astype(np.float64))
    if c["cap"] > 0:
        g, kn, u = capsule_parts(caps, c["Hk"], c["Hv"], c["dk"], c["dv"])
        gr, knr, ur = capsule_parts(c_ref, c["Hk"], c["Hv"], c["dk"], c["dv"])
        for s, L in enumerate(c["lengths"]):
            n = min(L, c["cap"])
            if n:
                assert max_rel(g[s, :n], gr[s, :n]) <= 1e-5
                assert max_rel(kn[s, :n], knr[s, :n]) <= 1e-5
                assert max_rel(u[s, :n], ur[s, :n]) <= tol_state, max_rel(u[s, :n], ur[s, :n])


@pytest.mark.parametrize("plan", ["auto", "recurrent", "chunked"])
@pytest.mark.parametrize("d", [128, 32])
@pytest.mark.parametrize("in_place", [True, False])
def test_all_empty_batch(plan, d, in_place):
    """Every sequence empty (T = 0): no outputs; each named slot's final state
    is its initial state, in place or copied; capsule rows stay untouched."""
    inp = wl.make_inputs(6100 + d, [0, 0, 0], Hk=2, Hv=4, dk=d, dv=d, io_dtype=np.float16, state_std=0.02,
                         num_slots=5, capacity=3, state_slots=[4, 0, 2])
    out, final, caps = run_gpu(inp, plan=plan, in_place=in_place)
    assert out.shape[0] == 0
    assert np.array_equal(final, inp.initial_state.astype(np.float64))
