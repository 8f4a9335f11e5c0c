"""GPU parity of the recurrent (decode / short-span) path and of prefix replay
against the FP64 oracle, through the C ABI.

Tolerances (max |gpu - oracle| / max |oracle| per tensor):
  FP32 recurrent arithmetic: 1e-5 on outputs, states and capsules.
  FP16 I/O: 2e-3 on the FP16 outputs (one FP16 rounding is 2^-11 of the
  element), 1e-5 on the FP32 state and capsules (inputs are widened exactly).
Bit-exact: cu_seqlens indexing (pack vs. one-by-one), slot placement, the
replayed prefix (untouched banks stay byte-identical).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import max_rel
from gpu_common import run_gpu, run_oracle, to_dev, dev, capsule_parts

from gated_delta_rule_gateddeltanet_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL32 = 1e-5
TOL16_OUT = 2e-3


def _check(inp, gpu, ref, fp16, cap=None):
    out, final, caps = gpu
    o_ref, f_ref, c_ref = ref
    assert max_rel(out, o_ref) <= (TOL16_OUT if fp16 else TOL32)
    slots = np.arange(inp.B) if inp.state_slots is None else inp.state_slots
    assert max_rel(final[slots], f_ref[slots]) <= TOL32
    cap = inp.capacity if cap is None else cap
    if cap > 0:
        lens = np.diff(inp.cu_seqlens)
        for s in range(inp.B):
            n = min(int(lens[s]), cap)
            if n:
                assert max_rel(caps[s, :n], c_ref[s, :n]) <= TOL32


def test_pr_ref_fp32_with_capsules():
    inp = wl.pr_ref()
    _check(inp, run_gpu(inp), run_oracle(inp), fp16=False)


def test_decode_step_full_size():
    """64 requests x 1 token, Hk=16, Hv=48, d=128, fp16, random state, in place."""
    inp = wl.decode_step()
    _check(inp, run_gpu(inp, capacity=1), run_oracle(inp, capacity=1), fp16=True, cap=1)


@pytest.mark.parametrize("io", [np.float16, np.float32])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 32), (32, 64)])
def test_ragged_batch_all_head_dims(io, dk, dv):
    lengths = [1, 7, 0, 19, 33, 2]
    inp = wl.make_inputs(77 + dk + dv, lengths, Hk=2, Hv=6, dk=dk, dv=dv, io_dtype=io, state_std=0.02,
                         capacity=5)
    _check(inp, run_gpu(inp, plan="recurrent"), run_oracle(inp), fp16=(io == np.float16))


def test_precomputed_gates():
    inp = wl.make_inputs(5, [9, 4], Hk=2, Hv=4, dk=128, dv=128, io_dtype=np.float32, state_std=0.02, capacity=3)
    rng = np.random.default_rng(6)
    g = rng.uniform(0.0, 1.0, inp.a.shape).astype(np.float32)
    g[0, :] = 0.0
    g[1, :] = 1.0
    beta = rng.uniform(0.0, 1.0, inp.b.shape).astype(np.float32)
    _check(inp, run_gpu(inp, gate_mode="precomputed", a=g, b=beta),
           run_oracle(inp, gate_mode="precomputed", a=g, b=beta), fp16=False)


def test_identity_gates_leave_state_bitwise():
    inp = wl.make_inputs(8, [5, 3], Hk=1, Hv=3, dk=128, dv=64, io_dtype=np.float16, state_std=0.02)
    ones = np.ones_like(inp.a)
    zeros = np.zeros_like(inp.b)
    _, final, _ = run_gpu(inp, gate_mode="precomputed", a=ones, b=zeros, in_place=False)
    assert np.array_equal(final, inp.initial_state.astype(np.float64))


def test_pack_equals_one_by_one_bitwise():
    lengths = [3, 1, 12, 0, 8]
    inp = wl.make_inputs(9, lengths, Hk=2, Hv=6, dk=128, dv=128, io_dtype=np.float16, state_std=0.02, capacity=4)
    out, final, caps = run_gpu(inp, in_place=False)
    cu = inp.cu_seqlens
    for s, L in enumerate(lengths):
        t0, t1 = cu[s], cu[s + 1]
        one = wl.GdnInputs(inp.q[t0:t1], inp.k[t0:t1], inp.v[t0:t1], inp.a[t0:t1], inp.b[t0:t1], inp.A_log,
                           inp.dt_bias, np.array([0, L], np.int32), inp.initial_state[s:s + 1], None, 4)
        o1, f1, c1 = run_gpu(one, in_place=False)
        assert np.array_equal(out[t0:t1], o1)
        assert np.array_equal(final[s], f1[0])
        n = min(L, 4)
        assert np.array_equal(caps[s, :n], c1[0, :n])


def test_in_place_equals_out_of_place_bitwise():
    inp = wl.make_inputs(10, [4, 4, 4], Hk=2, Hv=4, dk=128, dv=128, io_dtype=np.float16, state_std=0.02)
    a = run_gpu(inp, in_place=True)
    b = run_gpu(inp, in_place=False)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_state_slots_and_untouched_slots():
    lengths = [2, 5, 1]
    inp = wl.make_inputs(11, lengths, Hk=2, Hv=4, dk=64, dv=64, io_dtype=np.float32, state_std=0.02,
                         num_slots=7, state_slots=[5, 0, 3], capacity=2)
    out, final, caps = run_gpu(inp, in_place=False)
    ref = run_oracle(inp)
    _check(inp, (out, final, caps), ref, fp16=False)
    for untouched in (1, 2, 4, 6):
        assert np.array_equal(final[untouched], inp.initial_state[untouched].astype(np.float64))


def test_zero_initial_state_and_empty_sequences():
    inp = wl.make_inputs(12, [0, 6, 0], Hk=2, Hv=2, dk=128, dv=128, io_dtype=np.float32)
    out, final, _ = run_gpu(inp, in_place=False)
    o_ref, f_ref, _ = run_oracle(inp)
    assert max_rel(out, o_ref) <= TOL32
    assert max_rel(final, f_ref) <= TOL32
    assert np.all(final[0] == 0) and np.all(final[2] == 0)


def test_capsule_layout_semantics():
    """Decay per value head, the unit key per key head (shared by its value
    heads), the delta per value head; and S_t = g S_{t-1} + u kn^T holds."""
    inp = wl.make_inputs(13, [3], Hk=2, Hv=6, dk=64, dv=32, io_dtype=np.float32, state_std=0.02, capacity=3)
    _, _, caps = run_gpu(inp, in_place=False)
    g, kn, u = capsule_parts(caps, 2, 6, 64, 32)
    assert np.allclose(np.linalg.norm(kn, axis=-1), 1.0, atol=1e-6)
    q64 = inp.k.astype(np.float64)
    assert np.allclose(kn[0], q64 / np.linalg.norm(q64, axis=-1, keepdims=True), atol=1e-6)
    S = inp.initial_state[0].astype(np.float64)
    for t in range(3):
        for h in range(6):
            S[h] = g[0, t, h] * S[h] + np.outer(u[0, t, h], kn[0, t, h // 3])
    _, f_ref, _ = run_oracle(inp, capacity=0)
    assert max_rel(S, f_ref[0]) <= TOL32


def test_spec_verify_and_replay():
    """16 requests x 4 draft tokens with capsules, then replay of the accepted
    prefixes from the committed bank (slots 0..15) into the inactive bank
    (slots 16..31)."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    inp = wl.spec_verify()
    Hk, Hv, dk, dv = inp.dims
    pool = to_dev(inp.initial_state)
    committed = pool.clone()
    out, final, caps = run_gpu(inp, in_place=False, final_state=pool.clone())
    ref = run_oracle(inp)
    _check(inp, (out, final, caps), ref, fp16=True)

    caps_dev = to_dev(caps.astype(np.float32))
    acc = inp.extra["accept_len"]
    gdn.gdn_replay_prefix(committed, to_dev(inp.extra["src_slots"]), to_dev(inp.extra["dst_slots"]), caps_dev,
                          to_dev(acc), num_k_heads=Hk)
    torch.cuda.synchronize()
    got = committed.double().cpu().numpy()
    want = oracle.gdn_replay(inp.initial_state, inp.extra["src_slots"], inp.extra["dst_slots"],
                             caps.astype(np.float32), acc, num_k_heads=Hk)
    assert max_rel(got[16:], want[16:]) <= TOL32
    # the committed bank is byte-identical after the replay
    assert np.array_equal(got[:16], inp.initial_state[:16].astype(np.float64))
    # replaying the full draft equals the forward's final state; zero accepted is a copy
    for j in range(16):
        if acc[j] == 0:
            assert np.array_equal(got[16 + j], inp.initial_state[j].astype(np.float64))
        if acc[j] == 4:
            assert max_rel(got[16 + j], ref[1][j]) <= TOL32


def test_replay_every_prefix_matches_sequential_state():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    L = 6
    inp = wl.make_inputs(14, [L], Hk=2, Hv=6, dk=128, dv=128, io_dtype=np.float16, state_std=0.02, capacity=L)
    _, _, caps = run_gpu(inp, in_place=False)
    caps_dev = to_dev(caps.astype(np.float32)).expand(L + 1, L, caps.shape[2]).contiguous()
    banks = torch.zeros((2 * (L + 1), 6, 128, 128), dtype=torch.float32, device=dev())
    banks[:L + 1] = to_dev(inp.initial_state)
    gdn.gdn_replay_prefix(banks, to_dev(np.arange(L + 1, dtype=np.int32)),
                          to_dev(np.arange(L + 1, 2 * L + 2, dtype=np.int32)), caps_dev,
                          to_dev(np.arange(L + 1, dtype=np.int32)), num_k_heads=2)
    torch.cuda.synchronize()
    got = banks.double().cpu().numpy()
    for j in range(L + 1):
        sub = wl.GdnInputs(inp.q[:j], inp.k[:j], inp.v[:j], inp.a[:j], inp.b[:j], inp.A_log, inp.dt_bias,
                           np.array([0, j], np.int32), inp.initial_state, None, 0)
        _, f_ref, _ = run_oracle(sub)
        assert max_rel(got[L + 1 + j], f_ref[0]) <= TOL32


def test_replay_in_place():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    inp = wl.make_inputs(15, [4, 4], Hk=1, Hv=2, dk=128, dv=128, io_dtype=np.float32, state_std=0.02, capacity=4)
    _, final_ref, caps = run_gpu(inp, in_place=False)
    banks = to_dev(inp.initial_state)
    gdn.gdn_replay_prefix(banks, to_dev(np.array([0, 1], np.int32)), to_dev(np.array([0, 1], np.int32)),
                          to_dev(caps.astype(np.float32)), to_dev(np.array([4, 0], np.int32)), num_k_heads=1)
    torch.cuda.synchronize()
    got = banks.double().cpu().numpy()
    assert max_rel(got[0], final_ref[0]) <= TOL32
    assert np.array_equal(got[1], inp.initial_state[1].astype(np.float64))


def test_device_status_word_flags_bad_data_and_skips():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    inp = wl.make_inputs(16, [3, 2, 3], Hk=1, Hv=2, dk=64, dv=64, io_dtype=np.float32, state_std=0.02)
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    bad_cu = wl.GdnInputs(inp.q, inp.k, inp.v, inp.a, inp.b, inp.A_log, inp.dt_bias,
                          np.array([0, 3, 1, 8], np.int32), inp.initial_state)
    _, final, _ = run_gpu(bad_cu, status=status, in_place=False)
    assert status.item() & gdn.DEVERR["cu_seqlens"]
    assert np.array_equal(final[1], inp.initial_state[1].astype(np.float64))  # skipped sequence untouched
    status.zero_()
    bad_slot = wl.GdnInputs(inp.q, inp.k, inp.v, inp.a, inp.b, inp.A_log, inp.dt_bias, inp.cu_seqlens,
                            inp.initial_state, np.array([0, 9, 2], np.int32))
    run_gpu(bad_slot, status=status, in_place=False)
    assert status.item() & gdn.DEVERR["state_slot"]
    status.zero_()
    banks = to_dev(inp.initial_state)
    caps = torch.zeros((2, 2, gdn.capsule_width(1, 2, 64, 64)), dtype=torch.float32, device=dev())
    gdn.gdn_replay_prefix(banks, to_dev(np.array([0, 1], np.int32)), to_dev(np.array([2, 2], np.int32)), caps,
                          to_dev(np.array([3, 0], np.int32)), num_k_heads=1, status=status)
    torch.cuda.synchronize()
    assert status.item() & gdn.DEVERR["accept_len"]
    status.zero_()
    gdn.gdn_replay_prefix(banks, to_dev(np.array([0, 5], np.int32)), to_dev(np.array([1, 2], np.int32)), caps,
                          to_dev(np.array([1, 1], np.int32)), num_k_heads=1, status=status)
    torch.cuda.synchronize()
    assert status.item() & gdn.DEVERR["replay_slot"]


def test_bf16_rejected_on_device():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    q = torch.zeros((1, 1, 32), dtype=torch.bfloat16, device=dev())
    z = torch.zeros((1, 1), dtype=torch.float32, device=dev())
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_forward(q, q, torch.zeros((1, 1, 32), dtype=torch.bfloat16, device=dev()), z, z,
                        torch.tensor([0, 1], dtype=torch.int32, device=dev()),
                        A_log=torch.zeros(1, device=dev()), dt_bias=torch.zeros(1, device=dev()))
    assert e.value.code == 2


def test_fused_qkv_views():
    """q, k, v may be strided views of one fused projection [T, (2 Hk dk + Hv dv)]."""
    inp = wl.make_inputs(17, [5, 6], Hk=2, Hv=4, dk=64, dv=64, io_dtype=np.float16, state_std=0.02)
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    T = inp.T
    fused = np.concatenate([inp.q.reshape(T, -1), inp.k.reshape(T, -1), inp.v.reshape(T, -1)], axis=1)
    f = to_dev(fused)
    q = f[:, :128].view(T, 2, 64)
    k = f[:, 128:256].view(T, 2, 64)
    v = f[:, 256:].view(T, 4, 64)
    final = to_dev(inp.initial_state)
    out, final, _ = gdn.gdn_forward(q, k, v, to_dev(inp.a), to_dev(inp.b), to_dev(inp.cu_seqlens),
                                    A_log=to_dev(inp.A_log), dt_bias=to_dev(inp.dt_bias), initial_state=final,
                                    final_state=final)
    torch.cuda.synchronize()
    o_ref, f_ref, _ = run_oracle(inp)
    assert max_rel(out.double().cpu().numpy(), o_ref) <= TOL16_OUT
    assert max_rel(final.double().cpu().numpy(), f_ref) <= TOL32


def test_varlen_prefill_recurrent_plan_full_size():
    """8 sequences of U[256, 4096] tokens (Hk=16, Hv=48, d=128, fp16, zero
    state) on the forced recurrent plan."""
    inp = wl.varlen_prefill()
    _check(inp, run_gpu(inp, plan="recurrent"), run_oracle(inp), fp16=True)


def test_prepared_forward_call_equals_gdn_forward():
    """ForwardCall resolves the arguments once; repeated launches on refilled
    input buffers give bitwise the results of gdn_forward on the same data."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    inps = [wl.decode_step(seed=900 + i, requests=8) for i in range(3)]
    x = inps[0]
    bufs = {n: to_dev(getattr(x, n)).clone() for n in ("q", "k", "v", "a", "b")}
    cu = to_dev(x.cu_seqlens)
    state = to_dev(x.initial_state)
    call = gdn.ForwardCall(bufs["q"], bufs["k"], bufs["v"], bufs["a"], bufs["b"], cu, A_log=to_dev(x.A_log),
                           dt_bias=to_dev(x.dt_bias), initial_state=state, final_state=state, max_seqlen=1)
    ref_state = state.clone()
    for inp in inps:
        for n in bufs:
            bufs[n].copy_(to_dev(getattr(inp, n)))
        out, fin, _ = call.launch()
        o2, f2, _ = gdn.gdn_forward(to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.a), to_dev(inp.b), cu,
                                    A_log=to_dev(x.A_log), dt_bias=to_dev(x.dt_bias), initial_state=ref_state,
                                    final_state=ref_state, max_seqlen=1)
        torch.cuda.synchronize()
        assert torch.equal(out, o2) and torch.equal(fin, f2)


@pytest.mark.parametrize("plan,lengths", [("recurrent", [4] * 16), ("chunked", [100, 70, 3])])
def test_no_final_state_changes_nothing_else(plan, lengths):
    """With no final-state buffer the kernels write no state; outputs and
    capsules are bitwise those of the same call with a final state."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    inp = wl.make_inputs(520, lengths, Hk=2, Hv=6, dk=128, dv=128, io_dtype=np.float16, state_std=0.02,
                         capacity=4)
    args = lambda: (to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.a), to_dev(inp.b), to_dev(inp.cu_seqlens))
    init = to_dev(inp.initial_state)
    o1, f1, c1 = gdn.gdn_forward(*args(), A_log=to_dev(inp.A_log), dt_bias=to_dev(inp.dt_bias), initial_state=init,
                                 final_state=torch.empty_like(init), capacity=4, plan=plan)
    o2, f2, c2 = gdn.gdn_forward(*args(), A_log=to_dev(inp.A_log), dt_bias=to_dev(inp.dt_bias), initial_state=init,
                                 capacity=4, plan=plan, write_final_state=False)
    torch.cuda.synchronize()
    assert f2 is None
    assert torch.equal(o1, o2) and torch.equal(c1, c2)
    assert torch.equal(init, to_dev(inp.initial_state))  # the input state is untouched
