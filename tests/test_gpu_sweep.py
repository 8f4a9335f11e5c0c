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


# ---------------------------------------------------------------- prefix replay

def _replay_case(i):
    rng = np.random.default_rng(7000 + i)
    dk = int(rng.choice([32, 64, 128]))
    dv = dk if rng.random() < 0.6 else int(rng.choice([32, 64, 128]))
    Hk = int(rng.choice([1, 2, 4]))
    Hv = Hk * int(rng.choice([1, 2, 3]))
    R = int(rng.integers(1, 9))
    cap = int(rng.integers(1, 7))
    S = 2 * R + 1 + int(rng.integers(0, 4))  # room for R + 1 candidate sources and R destinations
    perm = rng.permutation(S)
    src = rng.choice(perm[:R + 1], size=R).astype(np.int32)  # sources may repeat (read only)
    dst = perm[R + 1:2 * R + 1].astype(np.int32)  # distinct, never another request's source
    for j in range(R):
        if rng.random() < 0.2:
            dst[j] = src[j]  # in-place replay of a request onto its own source
    if len(set(dst.tolist())) < R or any(dst[j] in np.delete(src, j) for j in range(R)):
        dst = perm[R + 1:2 * R + 1].astype(np.int32)
    n = rng.integers(0, cap + 1, size=R).astype(np.int32)
    return dict(seed=7100 + i, dk=dk, dv=dv, Hk=Hk, Hv=Hv, R=R, cap=cap, S=S, src=src, dst=dst, n=n)


@pytest.mark.parametrize("i", range(16))
def test_random_replay_matches_oracle(i):
    """Random head sizes, GQA ratios, request counts, capacities, accepted
    lengths (0 = copy) and slot layouts (sources shared, in-place replays);
    FP32-level (1e-5) on the written slots, every other slot bit for bit."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    import oracle as orc
    c = _replay_case(i)
    rng = np.random.default_rng(c["seed"])
    banks = (rng.standard_normal((c["S"], c["Hv"], c["dv"], c["dk"])) * 0.02).astype(np.float32)
    W = gdn.capsule_width(c["Hk"], c["Hv"], c["dk"], c["dv"])
    caps = np.empty((c["R"], c["cap"], W), np.float32)
    caps[:, :, :c["Hv"]] = rng.uniform(0.5, 1.0, size=(c["R"], c["cap"], c["Hv"]))
    caps[:, :, c["Hv"]:c["Hv"] + c["Hk"] * c["dk"]] = rng.standard_normal((c["R"], c["cap"], c["Hk"] * c["dk"])) / np.sqrt(c["dk"])
    caps[:, :, c["Hv"] + c["Hk"] * c["dk"]:] = rng.standard_normal((c["R"], c["cap"], c["Hv"] * c["dv"])) * 0.1
    want = orc.gdn_replay(banks, c["src"], c["dst"], caps, c["n"], num_k_heads=c["Hk"])
    got_t = torch.from_numpy(banks.copy()).to(dev())
    gdn.gdn_replay_prefix(got_t, torch.from_numpy(c["src"]).to(dev()), torch.from_numpy(c["dst"]).to(dev()),
                          torch.from_numpy(caps).to(dev()), torch.from_numpy(c["n"]).to(dev()), num_k_heads=c["Hk"])
    torch.cuda.synchronize()
    got = got_t.double().cpu().numpy()
    for j, d in enumerate(c["dst"]):
        assert max_rel(got[d], want[d]) <= 1e-5, (j, max_rel(got[d], want[d]))
    others = np.setdiff1d(np.arange(c["S"]), c["dst"])
    assert np.array_equal(got[others], banks[others].astype(np.float64))


# ---------------------------------------------------------------- causal conv and its replay

def _conv_case(i):
    rng = np.random.default_rng(8000 + i)
    io = np.float16 if rng.random() < 0.6 else np.float32
    C = int(rng.choice([8, 64, 520, 1032]))
    K = int(rng.choice([2, 3, 4]))
    B = int(rng.integers(1, 10))
    kinds = rng.choice(["empty", "one", "short", "long"], size=B, p=[0.1, 0.35, 0.35, 0.2])
    span = {"empty": (0, 1), "one": (1, 2), "short": (2, 9), "long": (9, 150)}
    lengths = [int(rng.integers(*span[k])) for k in kinds]
    longest = max(lengths)
    hint = int(rng.choice([0, max(longest, 1), 8, max(longest, 1) + int(rng.integers(0, 5))]))
    if hint and hint < longest:
        hint = longest
    S = B + int(rng.integers(0, 4))
    slots = rng.permutation(S)[:B].astype(np.int32)
    cap = int(rng.choice([0, 1, 3, 6]))
    cc = rng.integers(0, cap + 1, size=B).astype(np.int32) if (cap and rng.random() < 0.5) else None
    return dict(seed=8100 + i, io=io, C=C, K=K, lengths=lengths, hint=hint, S=S, slots=slots, cap=cap, cc=cc,
                in_place=bool(rng.random() < 0.5), state=bool(rng.random() < 0.8), bias=bool(rng.random() < 0.7))


@pytest.mark.parametrize("i", range(24))
def test_random_conv_matches_oracle(i):
    """Random channel counts, kernel sizes, ragged batches, max_seqlen hints
    (0, exact, 8, above), scattered slots, capture capacities and counts, in
    place or not, with or without an initial state and bias: outputs at 2e-3
    (fp16) / 1e-5 (FP32), states and captured inputs bit for bit, untouched
    slots and capture rows unchanged."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    import oracle as orc
    c = _conv_case(i)
    rng = np.random.default_rng(c["seed"])
    T = sum(c["lengths"])
    x = rng.standard_normal((T, c["C"])).astype(c["io"])
    w = (rng.standard_normal((c["C"], c["K"])) / 2).astype(np.float32)
    bias = (rng.standard_normal(c["C"]) / 4).astype(np.float32) if c["bias"] else None
    st = rng.standard_normal((c["S"], c["C"], c["K"] - 1)).astype(c["io"]) if c["state"] else None
    cu = np.concatenate([[0], np.cumsum(c["lengths"])]).astype(np.int32)
    st0 = st if st is not None else np.zeros((c["S"], c["C"], c["K"] - 1))
    want = orc.conv_forward(x, w, cu, st0, bias=bias, state_slots=c["slots"], capacity=c["cap"],
                            capture_count=c["cc"])
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    tdt = torch.float16 if c["io"] == np.float16 else torch.float32
    init = t(st)
    if c["in_place"] and init is not None:
        final = init
    else:
        final = t(st0.astype(c["io"])) if st is None else init.clone()
        if st is None:
            final.fill_(float("nan"))  # only the named slots must be written
    vals = torch.zeros((len(c["lengths"]), max(c["cap"], 1), c["C"]), dtype=tdt, device=dev()) if c["cap"] else None
    out, fin, cap_out = gdn.varlen_causal_conv_with_state(
        t(x), t(w), t(cu), bias=t(bias), initial_state=init, final_state=final, state_slots=t(c["slots"]),
        capture_count=t(c["cc"]), capacity=c["cap"], state_update=vals, num_state_slots=c["S"], max_seqlen=c["hint"])
    torch.cuda.synchronize()
    tol = 2e-3 if c["io"] == np.float16 else 1e-5
    assert max_rel(out.double().cpu().numpy(), want[0]) <= tol
    fin = fin.double().cpu().numpy()
    assert np.array_equal(fin[c["slots"]], want[1][c["slots"]])
    others = np.setdiff1d(np.arange(c["S"]), c["slots"])
    if st is not None and others.size:
        assert np.array_equal(fin[others], st[others].astype(np.float64))
    if c["cap"]:
        got_v = cap_out.double().cpu().numpy()
        for s_, L in enumerate(c["lengths"]):
            m = min(L, c["cap"], c["cc"][s_] if c["cc"] is not None else c["cap"])
            assert np.array_equal(got_v[s_, :m], want[2][s_, :m])
            assert np.all(got_v[s_, m:] == 0)


@pytest.mark.parametrize("i", range(8))
def test_random_conv_replay_matches_oracle(i):
    """Random channel counts, kernel sizes, request counts and accepted lengths:
    the replayed states equal the oracle's bit for bit, sources untouched."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    import oracle as orc
    rng = np.random.default_rng(8500 + i)
    io = np.float16 if i % 2 == 0 else np.float32
    C = int(rng.choice([8, 64, 520])) if io == np.float16 else int(rng.choice([4, 64, 516]))
    K = int(rng.choice([2, 3, 4]))
    R = int(rng.integers(1, 9))
    cap = int(rng.integers(1, 7))
    S = 2 * R + 1
    perm = rng.permutation(S)
    src, dst = perm[:R].astype(np.int32), perm[R:2 * R].astype(np.int32)
    n = rng.integers(0, cap + 1, size=R).astype(np.int32)
    states = rng.standard_normal((S, C, K - 1)).astype(io)
    vals = rng.standard_normal((R, cap, C)).astype(io)
    want = orc.conv_replay(states, src, dst, vals, n)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    st_t = t(states)
    gdn.causal_conv_replay_prefix(st_t, t(src), t(dst), t(vals), t(n))
    torch.cuda.synchronize()
    assert np.array_equal(st_t.double().cpu().numpy(), want)


# ---------------------------------------------------------------- device status on every path

STATUS_PATHS = {
    "decode": dict(lengths=[1, 1, 1], d=128, plan="auto"),
    "verify": dict(lengths=[4, 3, 6], d=128, plan="recurrent"),
    "mixed": dict(lengths=[4, 3, 6], d=64, plan="recurrent"),
    "two_phase": dict(lengths=[80, 70, 40], d=128, plan="chunked"),
    "single_kernel": dict(lengths=[80, 70, 40], d=128, plan="chunked", single=True),
    "split": dict(lengths=[2100, 70, 40], d=128, plan="chunked_split"),
}


@pytest.mark.parametrize("path", list(STATUS_PATHS))
def test_status_flags_skip_only_the_bad_sequence(path):
    """A sequence whose slot is out of range, or whose cu_seqlens entries run
    backwards, sets its status bit and is skipped: its slot keeps the initial
    state and the other sequences' states are those of the valid call, bit
    for bit (each chain is evaluated alone)."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    from gpu_common import single_kernel_workspace
    spec = STATUS_PATHS[path]
    d = spec["d"]
    inp = wl.make_inputs(6500, spec["lengths"], Hk=1, Hv=2, dk=d, dv=d, io_dtype=np.float16, state_std=0.02,
                         num_slots=4, state_slots=[0, 1, 2])
    ws = (lambda x: single_kernel_workspace(x)) if spec.get("single") else (lambda x: None)
    _, good, _ = run_gpu(inp, plan=spec["plan"], in_place=False, workspace=ws(inp))
    init = inp.initial_state.astype(np.float64)

    status = torch.zeros(1, dtype=torch.int32, device=dev())
    bad_slot = wl.GdnInputs(inp.q, inp.k, inp.v, inp.a, inp.b, inp.A_log, inp.dt_bias, inp.cu_seqlens,
                            inp.initial_state, np.array([0, 9, 2], np.int32))
    _, fin, _ = run_gpu(bad_slot, plan=spec["plan"], in_place=False, status=status, workspace=ws(bad_slot))
    assert status.item() == gdn.DEVERR["state_slot"]
    assert np.array_equal(fin[0], good[0]) and np.array_equal(fin[2], good[2])
    assert np.array_equal(fin[1], init[1]) and np.array_equal(fin[3], init[3])

    status.zero_()
    cu = inp.cu_seqlens.copy()
    cu[2] = cu[1] - 1  # sequence 1 ends before it starts; sequence 2 starts one token early
    bad_cu = wl.GdnInputs(inp.q, inp.k, inp.v, inp.a, inp.b, inp.A_log, inp.dt_bias, cu, inp.initial_state,
                          inp.state_slots)
    _, fin, _ = run_gpu(bad_cu, plan=spec["plan"], in_place=False, status=status, workspace=ws(bad_cu))
    assert status.item() & gdn.DEVERR["cu_seqlens"]
    assert np.array_equal(fin[0], good[0])
    assert np.array_equal(fin[1], init[1])


@pytest.mark.parametrize("path", list(STATUS_PATHS))
def test_empty_sequence_with_bad_slot_flagged(path):
    """An empty sequence whose slot is out of range sets the bit on every path
    (no kernel may rely on visiting a sequence through its tokens)."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    from gpu_common import single_kernel_workspace
    spec = STATUS_PATHS[path]
    d = spec["d"]
    inp = wl.make_inputs(6600, spec["lengths"] + [0], Hk=1, Hv=2, dk=d, dv=d, io_dtype=np.float16, state_std=0.02,
                         num_slots=4, state_slots=[0, 1, 2, 7])
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    ws = single_kernel_workspace(inp) if spec.get("single") else None
    _, fin, _ = run_gpu(inp, plan=spec["plan"], in_place=False, status=status, workspace=ws)
    assert status.item() == gdn.DEVERR["state_slot"]
    assert np.array_equal(fin[3], inp.initial_state[3].astype(np.float64))


@pytest.mark.parametrize("path", list(STATUS_PATHS))
def test_extreme_raw_gates_match_oracle(path):
    """Raw gate inputs far out in both tails (a, b in {-60, -5, 0, 5, 60} with
    A_log up to log 16): decays that underflow to exactly 0 (the state
    restarts), decays of 1 - 1e-27, betas of 0 and 1, on every path, against
    the oracle at the path's tolerance; nothing becomes NaN."""
    from gpu_common import single_kernel_workspace
    import oracle as orc
    spec = STATUS_PATHS[path]
    d = spec["d"]
    inp = wl.make_inputs(6700, spec["lengths"], Hk=1, Hv=2, dk=d, dv=d, io_dtype=np.float16, state_std=0.02,
                         capacity=8)
    rng = np.random.default_rng(6701)
    vals = np.array([-60.0, -5.0, 0.0, 5.0, 60.0], np.float32)
    a = rng.choice(vals, size=inp.a.shape).astype(np.float32)
    b = rng.choice(vals, size=inp.b.shape).astype(np.float32)
    A_log = np.log(np.array([1.0, 16.0], np.float32)).astype(np.float32)
    extreme = wl.GdnInputs(inp.q, inp.k, inp.v, a, b, A_log, inp.dt_bias, inp.cu_seqlens, inp.initial_state,
                           inp.state_slots, inp.capacity)
    ws = single_kernel_workspace(extreme) if spec.get("single") else None
    out, fin, caps = run_gpu(extreme, plan=spec["plan"], in_place=False, workspace=ws)
    ref = orc.gdn_forward(extreme.q, extreme.k, extreme.v, a, b, extreme.cu_seqlens, A_log=A_log,
                          dt_bias=extreme.dt_bias, initial_state=extreme.initial_state, capacity=8)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(fin))
    tensor_cores = spec["plan"] not in ("recurrent", "auto")  # the auto plan here runs the decode kernel
    assert max_rel(out, ref[0]) <= 2e-3, max_rel(out, ref[0])  # fp16 outputs: one fp16 rounding
    tol_state = 2e-3 if tensor_cores else 1e-5
    assert max_rel(fin, ref[1]) <= tol_state, max_rel(fin, ref[1])
    g, kn, u = capsule_parts(caps, 1, 2, d, d)
    gr, knr, ur = capsule_parts(ref[2], 1, 2, d, d)
    for s_, L in enumerate(spec["lengths"]):
        n = min(L, 8)
        assert max_rel(g[s_, :n], gr[s_, :n]) <= 1e-5
        assert max_rel(u[s_, :n], ur[s_, :n]) <= tol_state


# ---------------------------------------------------------------- dense rank-4 inputs and the split plan

@pytest.mark.parametrize("i", range(8))
def test_random_dense_equals_packed_and_oracle(i):
    """gdn_forward_dense on random batch and sequence sizes, head sizes and
    plans: bit for bit the packed call on the same tokens, and the oracle at
    the plan's tolerance."""
    from test_gpu_dense import _run_both
    rng = np.random.default_rng(9000 + i)
    dk = int(rng.choice([32, 64, 128]))
    dv = dk if rng.random() < 0.7 else int(rng.choice([32, 64, 128]))
    B = int(rng.integers(1, 5))
    S = int(rng.choice([1, 3, 17, 70, 130]))
    plan = str(rng.choice(["auto", "recurrent", "chunked"]))
    io = np.float16 if rng.random() < 0.6 else np.float32
    Hk = int(rng.choice([1, 2]))
    inp = wl.make_inputs(9100 + i, [S] * B, Hk=Hk, Hv=Hk * int(rng.choice([1, 3])), dk=dk, dv=dv, io_dtype=io,
                         state_std=0.02 if rng.random() < 0.8 else None)
    od, fd, op, fp = _run_both(inp, B, S, plan)
    assert np.array_equal(od, op) and np.array_equal(fd, fp)
    o_ref, f_ref, _ = oracle.gdn_forward(inp.q, inp.k, inp.v, inp.a, inp.b, inp.cu_seqlens, A_log=inp.A_log,
                                         dt_bias=inp.dt_bias, initial_state=inp.initial_state,
                                         num_state_slots=B)
    limit = 32 if dk == dv == 128 else 256
    tc = plan == "chunked" or (plan == "auto" and S > limit)
    assert max_rel(od, o_ref) <= (2e-3 if (tc or io == np.float16) else 1e-5)
    assert max_rel(fd, f_ref) <= (2e-3 if tc else 1e-5)


@pytest.mark.parametrize("i", range(4))
def test_random_split_plan_matches_oracle(i):
    """The sequence-parallel split plan on random batches: one or two
    sequences around and past the split threshold (1984 tokens) among short
    ones, fp16 or FP32, a capture capacity that allows the split or forbids it
    (captured tokens past the first half), at 2e-3 against the oracle."""
    rng = np.random.default_rng(9500 + i)
    longs = [int(rng.integers(1900, 2700)) for _ in range(int(rng.integers(1, 3)))]
    shorts = [int(rng.integers(0, 200)) for _ in range(int(rng.integers(0, 3)))]
    lengths = list(rng.permutation(longs + shorts))
    io = np.float16 if rng.random() < 0.5 else np.float32
    cap = int(rng.choice([0, 4, 1500]))
    inp = wl.make_inputs(9600 + i, lengths, Hk=1, Hv=2, dk=128, dv=128, io_dtype=io, state_std=0.02, capacity=cap)
    out, fin, caps = run_gpu(inp, plan="chunked_split", in_place=bool(i % 2))
    o_ref, f_ref, c_ref = oracle.gdn_forward(inp.q, inp.k, inp.v, inp.a, inp.b, inp.cu_seqlens, A_log=inp.A_log,
                                             dt_bias=inp.dt_bias, initial_state=inp.initial_state, capacity=cap)
    assert max_rel(out, o_ref) <= 2e-3, max_rel(out, o_ref)
    assert max_rel(fin, f_ref) <= 2e-3, max_rel(fin, f_ref)
    if cap:
        _, _, u = capsule_parts(caps, 1, 2, 128, 128)
        _, _, ur = capsule_parts(c_ref, 1, 2, 128, 128)
        for s_, L in enumerate(lengths):
            n = min(L, cap)
            if n:
                assert max_rel(u[s_, :n], ur[s_, :n]) <= 2e-3


@pytest.mark.parametrize("d", [128, 64])
def test_as_many_tokens_as_sequences_with_multi_token_spans(d):
    """T == B does not mean one token per span: with empty sequences beside
    multi-token ones, every span must still get the bits it gets alone (the
    decode kernel takes the spans of at most one token, the short-span kernel
    the others), and the results match the oracle."""
    lengths = [2, 0, 3, 0, 1, 0]  # T = 6 = B
    inp = wl.make_inputs(6800 + d, lengths, Hk=1, Hv=2, dk=d, dv=d, io_dtype=np.float16, state_std=0.02,
                         capacity=4)
    out, fin, caps = run_gpu(inp, in_place=False)
    o_ref, f_ref, _ = oracle.gdn_forward(inp.q, inp.k, inp.v, inp.a, inp.b, inp.cu_seqlens, A_log=inp.A_log,
                                         dt_bias=inp.dt_bias, initial_state=inp.initial_state, capacity=4)
    assert max_rel(out, o_ref) <= 2e-3 and max_rel(fin, f_ref) <= 1e-5
    cu = inp.cu_seqlens
    for s_, L in enumerate(lengths):
        one = wl.GdnInputs(inp.q[cu[s_]:cu[s_ + 1]], inp.k[cu[s_]:cu[s_ + 1]], inp.v[cu[s_]:cu[s_ + 1]],
                           inp.a[cu[s_]:cu[s_ + 1]], inp.b[cu[s_]:cu[s_ + 1]], inp.A_log, inp.dt_bias,
                           np.array([0, L], np.int32), inp.initial_state[s_:s_ + 1], None, 4)
        o1, f1, c1 = run_gpu(one, in_place=False)
        assert np.array_equal(out[cu[s_]:cu[s_ + 1]], o1), s_
        assert np.array_equal(fin[s_], f1[0]), s_
        assert np.array_equal(caps[s_, :min(L, 4)], c1[0, :min(L, 4)]), s_
