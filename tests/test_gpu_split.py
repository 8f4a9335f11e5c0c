"""GPU parity of the sequence-parallel chunked plan (GDN_PLAN_CHUNKED_SPLIT)
against the FP64 oracle, through the C ABI.

Under this plan a sequence of more than 1984 tokens (32 or more 64-token
chunks) runs as its first half from the initial state and its second half
twice, from a zero state and from the identity; two combining kernels add
S1 times the identity run's outputs to the second half's outputs and form
S1 A + B as the final state.  The cases cover split and unsplit sequences in
one batch (including 1984 and 1985 tokens, the two sides of the rule), ragged
last chunks, slow decays under which the final state depends strongly on S1
(so a wrong combination cannot hide behind fast forgetting), no initial
state, no final-state buffer, state slots with a bad slot, bitwise equality
of a packed batch with its sequences run alone, and the full head geometry
(Hk = 16, Hv = 48) with the oracle on one key head's value heads.

Tolerance: 2e-3 max-relative as for the chunked path; the combination adds a
tensor-core product with fp16 operands and a second rounding of second-half
outputs to the I/O type.
"""
import numpy as np
import pytest
import torch

from helpers import max_rel
from gpu_common import run_gpu, run_oracle, dev

from gated_delta_rule_gateddeltanet_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _check(inp, gpu, ref):
    out, final, _ = gpu
    o_ref, f_ref, _ = ref
    assert max_rel(out, o_ref) <= TOL, max_rel(out, o_ref)
    slots = np.arange(inp.B) if inp.state_slots is None else inp.state_slots
    assert max_rel(final[slots], f_ref[slots]) <= TOL, max_rel(final[slots], f_ref[slots])


def _slow_gates(inp, seed):
    """g in [0.999, 1], beta in [0, 0.05]: the state entering the second half
    still weighs about half of the final state after 2000 tokens."""
    rng = np.random.default_rng(seed)
    T, Hv = inp.a.shape
    g = rng.uniform(0.999, 1.0, size=(T, Hv)).astype(np.float32)
    beta = rng.uniform(0.0, 0.05, size=(T, Hv)).astype(np.float32)
    return g, beta


@pytest.mark.parametrize("io", [np.float16, np.float32])
def test_split_plan_matches_oracle(io):
    lengths = [2100, 300, 0, 4217]  # 2100 and 4217 tokens are split
    inp = wl.make_inputs(900, lengths, Hk=2, Hv=4, dk=128, dv=128, io_dtype=io, state_std=0.05)
    _check(inp, run_gpu(inp, plan="chunked_split"), run_oracle(inp))


def test_split_rule_edges_and_many_split_sequences():
    """1984 tokens (31 chunks) stay whole, 1985 (32 chunks) are split; seven
    split sequences between unsplit and empty ones."""
    lengths = [2000, 50, 2100, 0, 2500, 10, 1985, 1984, 3000, 65, 2048, 129]
    inp = wl.make_inputs(901, lengths, Hk=1, Hv=2, dk=128, dv=128, io_dtype=np.float16, state_std=0.05)
    _check(inp, run_gpu(inp, plan="chunked_split", in_place=False), run_oracle(inp))


def test_split_plan_slow_decay():
    inp = wl.make_inputs(902, [2500, 1990], Hk=1, Hv=2, dk=128, dv=128, io_dtype=np.float16, state_std=0.05)
    g, beta = _slow_gates(inp, 903)
    gpu = run_gpu(inp, plan="chunked_split", gate_mode="precomputed", a=g, b=beta, in_place=False)
    ref = run_oracle(inp, gate_mode="precomputed", a=g, b=beta)
    _check(inp, gpu, ref)
    # the first sequence's final state is far from what its second half alone
    # gives from a zero state (B): the S1 A term is large here
    lo, hi = 64 * 20, 2500  # 40 chunks, split after chunk 20
    half = wl.GdnInputs(inp.q[lo:hi], inp.k[lo:hi], inp.v[lo:hi], inp.a[lo:hi], inp.b[lo:hi], inp.A_log,
                        inp.dt_bias, np.array([0, hi - lo], np.int32), None)
    _, f_half, _ = run_oracle(half, gate_mode="precomputed", a=g[lo:hi], b=beta[lo:hi])
    assert max_rel(f_half[0], ref[1][0]) > 0.1


def test_split_zero_state_and_no_final_state():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    from gpu_common import to_dev
    inp = wl.make_inputs(904, [2200, 700], Hk=2, Hv=4, dk=128, dv=128, io_dtype=np.float16)
    gpu = run_gpu(inp, plan="chunked_split", in_place=False)
    _check(inp, gpu, run_oracle(inp))
    out, final, _ = gdn.gdn_forward(to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.a), to_dev(inp.b),
                                    to_dev(inp.cu_seqlens), A_log=to_dev(inp.A_log), dt_bias=to_dev(inp.dt_bias),
                                    plan="chunked_split", write_final_state=False)
    torch.cuda.synchronize()
    assert final is None
    assert np.array_equal(out.double().cpu().numpy(), gpu[0])


def test_split_pack_equals_one_by_one_bitwise():
    lengths = [2050, 70, 3000]
    inp = wl.make_inputs(905, lengths, Hk=2, Hv=4, dk=128, dv=128, io_dtype=np.float16, state_std=0.05)
    out, final, _ = run_gpu(inp, plan="chunked_split", in_place=False)
    cu = inp.cu_seqlens
    for s, L in enumerate(lengths):
        t0, t1 = cu[s], cu[s + 1]
        one = wl.GdnInputs(inp.q[t0:t1], inp.k[t0:t1], inp.v[t0:t1], inp.a[t0:t1], inp.b[t0:t1], inp.A_log,
                           inp.dt_bias, np.array([0, L], np.int32), inp.initial_state[s:s + 1], None)
        o1, f1, _ = run_gpu(one, plan="chunked_split", in_place=False)
        assert np.array_equal(out[t0:t1], o1)
        assert np.array_equal(final[s], f1[0])


def test_split_slots_and_bad_slot():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    inp = wl.make_inputs(906, [2100, 90, 2300], Hk=1, Hv=2, dk=128, dv=128, io_dtype=np.float16, state_std=0.05,
                         num_slots=6, state_slots=[4, 1, 2])
    out, final, _ = run_gpu(inp, plan="chunked_split", in_place=False)
    _check(inp, (out, final, None), run_oracle(inp))
    for untouched in (0, 3, 5):
        assert np.array_equal(final[untouched], inp.initial_state[untouched].astype(np.float64))
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    bad = wl.GdnInputs(inp.q, inp.k, inp.v, inp.a, inp.b, inp.A_log, inp.dt_bias, inp.cu_seqlens,
                       inp.initial_state, np.array([4, 1, 9], np.int32))
    out2, final2, _ = run_gpu(bad, plan="chunked_split", in_place=False, status=status)
    assert status.item() & gdn.DEVERR["state_slot"]
    assert np.array_equal(final2[4], final[4]) and np.array_equal(final2[1], final[1])
    n0 = inp.cu_seqlens[2]
    assert np.array_equal(out2[:n0], out[:n0])


def test_split_full_heads_sampled():
    """One 16,417-token sequence at Hk = 16, Hv = 48, d = 128, fp16, with an
    initial state; the oracle runs key head 5 and its value heads 15-17."""
    T = 16417
    inp = wl.make_inputs(907, [T], Hk=16, Hv=48, dk=128, dv=128, io_dtype=np.float16, state_std=0.02)
    out, final, _ = run_gpu(inp, plan="chunked_split", in_place=False)
    kh, hs = 5, slice(15, 18)
    c = np.ascontiguousarray
    sub = wl.GdnInputs(c(inp.q[:, kh:kh + 1]), c(inp.k[:, kh:kh + 1]), c(inp.v[:, hs]), c(inp.a[:, hs]),
                       c(inp.b[:, hs]), c(inp.A_log[hs]), c(inp.dt_bias[hs]), inp.cu_seqlens,
                       c(inp.initial_state[:, hs]))
    o_ref, f_ref, _ = run_oracle(sub)
    assert max_rel(out[:, hs], o_ref) <= TOL
    assert max_rel(final[:, hs], f_ref) <= TOL


def test_long_prefill_full_size_sampled():
    """The long-prefill measurement itself: one 262,144-token sequence at
    Hk = 16, Hv = 48, d = 128, fp16, zero initial state, the bench's own
    inputs and launch (split plan).  The oracle runs key head 5 and its
    value heads 15-17 over all 262,144 tokens (each chain is independent of
    the other heads)."""
    import bench
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    q, k, v, aa, bb, A_log, dt_bias, cu = bench.long_prefill_inputs(dev())
    Hv = v.shape[1]
    final = torch.zeros((1, Hv, 128, 128), dtype=torch.float32, device=dev())
    out, final, _ = gdn.gdn_forward(q, k, v, aa, bb, cu, A_log=A_log, dt_bias=dt_bias, final_state=final,
                                    plan="chunked_split")
    torch.cuda.synchronize()
    kh, hs = 5, slice(15, 18)
    h = lambda x: np.ascontiguousarray(x.cpu().numpy())
    sub = wl.GdnInputs(h(q[:, kh:kh + 1]), h(k[:, kh:kh + 1]), h(v[:, hs]), h(aa[:, hs]), h(bb[:, hs]),
                       h(A_log[hs]), h(dt_bias[hs]), h(cu), None)
    o_ref, f_ref, _ = run_oracle(sub)
    assert max_rel(out[:, hs].double().cpu().numpy(), o_ref) <= TOL
    assert max_rel(final[:, hs].double().cpu().numpy(), f_ref) <= TOL


@pytest.mark.parametrize("cap", [1000, 1500])
def test_split_plan_with_capsules(cap):
    """Capsules under the split plan.  Only tokens whose state is exact have a
    delta, so a sequence is split only when its captured tokens (the first
    `cap`) lie in its first half: with cap = 1000 both long sequences (first
    halves of 1088 and 2112 tokens) are split; with cap = 1500 the
    2100-token one runs whole and gives bitwise the chunked plan's results."""
    from gpu_common import capsule_parts
    lengths = [2100, 300, 4217]
    inp = wl.make_inputs(908, lengths, Hk=2, Hv=4, dk=128, dv=128, io_dtype=np.float16, state_std=0.05,
                         capacity=cap)
    gpu = run_gpu(inp, plan="chunked_split", in_place=False)
    ref = run_oracle(inp)
    _check(inp, gpu, ref)
    Hk, Hv, dk, dv = inp.dims
    g, kn, u = capsule_parts(gpu[2], Hk, Hv, dk, dv)
    gr, knr, ur = capsule_parts(ref[2], Hk, Hv, dk, dv)
    for s, L in enumerate(lengths):
        n = min(L, cap)
        assert max_rel(g[s, :n], gr[s, :n]) <= 1e-5
        assert max_rel(kn[s, :n], knr[s, :n]) <= 1e-5
        assert max_rel(u[s, :n], ur[s, :n]) <= TOL, (s, max_rel(u[s, :n], ur[s, :n]))
    if cap == 1500:  # the first sequence was not split: the chunked plan's bits
        whole = run_gpu(inp, plan="chunked", in_place=False)
        n0 = inp.cu_seqlens[1]
        assert np.array_equal(gpu[0][:n0], whole[0][:n0])
        assert np.array_equal(gpu[1][0], whole[1][0])
        assert np.array_equal(gpu[2][0], whole[2][0])
