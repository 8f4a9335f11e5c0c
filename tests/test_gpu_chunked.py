"""GPU parity of the tcgen05 chunked-prefill path against the FP64 oracle.

Both chunked evaluations are covered: the two-phase one (a parallel per-chunk
kernel, then the state-passing kernel), which gdn_forward runs with the
workspace gdn_forward_workspace_size asks for, and the single-kernel one,
which it runs when the workspace only holds the chain list.

Tolerance: 2e-3 max-relative (max |gpu - oracle| / max |oracle| per tensor) on
outputs, final states and capsule deltas -- the tensor cores take fp16
operands (normalised q and k, the fp16 copy of the state, the delta terms and
the triangular inverse), each rounding being 2^-11 relative, with FP32
accumulation and an FP32 state.  Bit-exact: a packed batch against each
sequence run alone (each chain is evaluated by one CTA in a fixed order).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import max_rel
from gpu_common import run_gpu, run_oracle, to_dev, dev, capsule_parts, single_kernel_workspace

from gated_delta_rule_gateddeltanet_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _check(inp, gpu, ref, cap=None):
    out, final, caps = gpu
    o_ref, f_ref, c_ref = ref
    assert max_rel(out, o_ref) <= TOL, max_rel(out, o_ref)
    slots = np.arange(inp.B) if inp.state_slots is None else inp.state_slots
    assert max_rel(final[slots], f_ref[slots]) <= TOL, max_rel(final[slots], f_ref[slots])
    cap = inp.capacity if cap is None else cap
    if cap > 0:
        Hk, Hv, dk, dv = inp.dims
        lens = np.diff(inp.cu_seqlens)
        g, kn, u = capsule_parts(caps, Hk, Hv, dk, dv)
        gr, knr, ur = capsule_parts(c_ref, Hk, Hv, dk, dv)
        for s in range(inp.B):
            n = min(int(lens[s]), cap)
            if n:
                assert max_rel(g[s, :n], gr[s, :n]) <= 1e-5
                assert max_rel(kn[s, :n], knr[s, :n]) <= 1e-5
                assert max_rel(u[s, :n], ur[s, :n]) <= TOL, max_rel(u[s, :n], ur[s, :n])


LENGTHS = [0, 1, 63, 64, 65, 130, 200, 7]
PATHS = ["two_phase", "single_kernel"]


def _ws(path, inp):
    return single_kernel_workspace(inp) if path == "single_kernel" else None


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("io", [np.float16, np.float32])
def test_forced_chunked_ragged_with_state_and_capsules(io, path):
    inp = wl.make_inputs(201, LENGTHS, Hk=2, Hv=6, dk=128, dv=128, io_dtype=io, state_std=0.02, capacity=70)
    _check(inp, run_gpu(inp, plan="chunked", in_place=False, workspace=_ws(path, inp)), run_oracle(inp))


@pytest.mark.parametrize("path", PATHS)
def test_forced_chunked_zero_initial_state(path):
    inp = wl.make_inputs(202, [129, 3, 64], Hk=1, Hv=3, dk=128, dv=128, io_dtype=np.float16)
    _check(inp, run_gpu(inp, plan="chunked", in_place=False, workspace=_ws(path, inp)), run_oracle(inp))


def test_two_phase_gqa_ratios_and_many_chunks():
    """Key heads shared by 1, 2 and 4 value heads; a 20-chunk sequence next to
    sequences that end one token into a chunk and one token short of it."""
    for Hk, Hv, seed in ((3, 3, 211), (2, 4, 212), (1, 4, 213)):
        inp = wl.make_inputs(seed, [1280, 129, 127, 40], Hk=Hk, Hv=Hv, dk=128, dv=128, io_dtype=np.float16,
                             state_std=0.02, capacity=130)
        _check(inp, run_gpu(inp, in_place=True), run_oracle(inp))


def test_auto_plan_mixes_both_kernels():
    lengths = [1, 5, 33, 100, 32, 0, 257]
    inp = wl.make_inputs(203, lengths, Hk=2, Hv=4, dk=128, dv=128, io_dtype=np.float16, state_std=0.02,
                         capacity=40)
    _check(inp, run_gpu(inp, in_place=True), run_oracle(inp))


@pytest.mark.parametrize("path", PATHS)
def test_chunked_precomputed_gate_extremes(path):
    """Decays of exactly 0 and 1 and beta of 0 and 1 inside chunks."""
    inp = wl.make_inputs(204, [150, 70], Hk=1, Hv=2, dk=128, dv=128, io_dtype=np.float32, state_std=0.02)
    rng = np.random.default_rng(5)
    g = rng.uniform(0.5, 1.0, inp.a.shape).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, inp.b.shape).astype(np.float32)
    g[10, :] = 0.0
    g[100:140, 0] = 1.0
    g[60, 1] = 0.0
    beta[20:30, :] = 0.0
    beta[31, :] = 1.0
    _check(inp, run_gpu(inp, plan="chunked", gate_mode="precomputed", a=g, b=beta, in_place=False,
                        workspace=_ws(path, inp)),
           run_oracle(inp, gate_mode="precomputed", a=g, b=beta))


@pytest.mark.parametrize("path", PATHS)
def test_chunked_pack_equals_one_by_one_bitwise(path):
    lengths = [40, 100, 70, 33]
    inp = wl.make_inputs(205, lengths, Hk=2, Hv=6, dk=128, dv=128, io_dtype=np.float16, state_std=0.02,
                         capacity=8)
    out, final, caps = run_gpu(inp, in_place=False, workspace=_ws(path, inp))
    cu = inp.cu_seqlens
    for s, L in enumerate(lengths):
        t0, t1 = cu[s], cu[s + 1]
        one = wl.GdnInputs(inp.q[t0:t1], inp.k[t0:t1], inp.v[t0:t1], inp.a[t0:t1], inp.b[t0:t1], inp.A_log,
                           inp.dt_bias, np.array([0, L], np.int32), inp.initial_state[s:s + 1], None, 8)
        o1, f1, c1 = run_gpu(one, in_place=False, workspace=_ws(path, one))
        assert np.array_equal(out[t0:t1], o1)
        assert np.array_equal(final[s], f1[0])
        assert np.array_equal(caps[s], c1[0])


@pytest.mark.parametrize("path", PATHS)
def test_chunked_slots_and_status(path):
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    inp = wl.make_inputs(206, [80, 90, 40], Hk=1, Hv=2, dk=128, dv=128, io_dtype=np.float16, state_std=0.02,
                         num_slots=6, state_slots=[4, 1, 2])
    out, final, _ = run_gpu(inp, plan="chunked", in_place=False, workspace=_ws(path, inp))
    _check(inp, (out, final, None), run_oracle(inp))
    for untouched in (0, 3, 5):
        assert np.array_equal(final[untouched], inp.initial_state[untouched].astype(np.float64))
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    bad = wl.GdnInputs(inp.q, inp.k, inp.v, inp.a, inp.b, inp.A_log, inp.dt_bias, inp.cu_seqlens,
                       inp.initial_state, np.array([4, 9, 2], np.int32))
    _, final2, _ = run_gpu(bad, plan="chunked", in_place=False, status=status, workspace=_ws(path, bad))
    assert status.item() & gdn.DEVERR["state_slot"]
    assert np.array_equal(final2[4], final[4]) and np.array_equal(final2[2], final[2])


def test_missing_workspace_is_rejected():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    inp = wl.make_inputs(207, [100], Hk=1, Hv=1, dk=128, dv=128, io_dtype=np.float16)
    t = lambda x: to_dev(x)
    final = torch.zeros((1, 1, 128, 128), device=dev())
    args, _, keep = gdn.build_forward_args(t(inp.q), t(inp.k), t(inp.v), t(inp.a), t(inp.b), t(inp.cu_seqlens),
                                           A_log=t(inp.A_log), dt_bias=t(inp.dt_bias), final_state=final)
    lib = gdn.load_library()
    assert lib.gdn_forward(ctypes.byref(args), None) == 5


def test_varlen_prefill_full_size():
    """8 packed sequences of U[256, 4096] tokens, Hk=16, Hv=48, d=128, fp16,
    zero initial state: every sequence takes the chunked kernel."""
    inp = wl.varlen_prefill()
    _check(inp, run_gpu(inp, in_place=False), run_oracle(inp))


def test_spec_verify_auto_equals_recurrent():
    """4-token drafts stay on the recurrent kernel under the automatic plan,
    with or without the max_seqlen hint."""
    inp = wl.spec_verify()
    a = run_gpu(inp, in_place=False)
    b = run_gpu(inp, in_place=False, plan="recurrent")
    c = run_gpu(inp, in_place=False, max_seqlen=4)
    for x, y, z in zip(a, b, c):
        assert np.array_equal(x, y) and np.array_equal(x, z)


def test_serving_mix_sampled():
    """32 x 2048-token prefill, then 256 single-token decode steps on the
    resulting states.  Every sequence runs on the GPU; the oracle checks 3 of
    the 32 sequences (chains are independent) through the prefill and all 256
    decode steps."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    pre = wl.serving_mix_prefill()
    Hk, Hv, dk, dv = pre.dims
    state = torch.zeros((pre.B, Hv, dv, dk), dtype=torch.float32, device=dev())
    out, _, _ = gdn.gdn_forward(to_dev(pre.q), to_dev(pre.k), to_dev(pre.v), to_dev(pre.a), to_dev(pre.b),
                                to_dev(pre.cu_seqlens), A_log=to_dev(pre.A_log), dt_bias=to_dev(pre.dt_bias),
                                initial_state=state, final_state=state, max_seqlen=2048)
    sample = [0, 13, 31]
    L = 2048
    o_pre = out.double().cpu().numpy()
    sub = wl.GdnInputs(*(np.concatenate([x[s * L:(s + 1) * L] for s in sample]) for x in (pre.q, pre.k, pre.v,
                                                                                          pre.a, pre.b)),
                       pre.A_log, pre.dt_bias, wl.cu_from_lengths([L] * len(sample)), None)
    o_ref, f_ref, _ = run_oracle(sub)
    got = np.concatenate([o_pre[s * L:(s + 1) * L] for s in sample])
    assert max_rel(got, o_ref) <= TOL
    assert max_rel(state.double().cpu().numpy()[sample], f_ref) <= TOL
    ref_state = f_ref
    outs_gpu, outs_ref = [], []
    for step in range(256):
        d = wl.serving_mix_decode(step, pre)
        o, _, _ = gdn.gdn_forward(to_dev(d.q), to_dev(d.k), to_dev(d.v), to_dev(d.a), to_dev(d.b),
                                  to_dev(d.cu_seqlens), A_log=to_dev(d.A_log), dt_bias=to_dev(d.dt_bias),
                                  initial_state=state, final_state=state, max_seqlen=1)
        if step % 32 == 0 or step == 255:
            outs_gpu.append(o.double().cpu().numpy()[sample])
        ds = wl.GdnInputs(d.q[sample], d.k[sample], d.v[sample], d.a[sample], d.b[sample], d.A_log, d.dt_bias,
                          wl.cu_from_lengths([1] * len(sample)), ref_state)
        o_r, ref_state, _ = run_oracle(ds)
        if step % 32 == 0 or step == 255:
            outs_ref.append(o_r)
    torch.cuda.synchronize()
    assert max_rel(np.array(outs_gpu), np.array(outs_ref)) <= TOL
    assert max_rel(state.double().cpu().numpy()[sample], ref_state) <= TOL


@pytest.mark.parametrize("path", PATHS)
def test_chunked_many_sequences(path):
    """3000 sequences (33 to 200 tokens, one empty) on the chunked path: the
    planning kernel's longest-first list and per-sequence chunk offsets span
    many threads and warps of its prefix sum."""
    rng = np.random.default_rng(214)
    lengths = rng.integers(33, 201, 3000)
    lengths[1234] = 0
    inp = wl.make_inputs(215, lengths, Hk=1, Hv=1, dk=128, dv=128, io_dtype=np.float16, state_std=0.02,
                         capacity=2)
    _check(inp, run_gpu(inp, plan="chunked", in_place=False, workspace=_ws(path, inp)), run_oracle(inp))


def test_pages_ragged_batch_is_bitwise_the_prompts_alone():
    """The validation case of "Add GatedDeltaNet evaluation export for Qwen
    hybrid models" (reviewer validation): a batch of 17-, 512- and 1993-token
    prompts gives bit-identical outputs to the same prompts run alone.  Under
    the automatic plan the 17-token prompt takes the tensor-core short-span
    kernel and the others the chunked kernels, in the batch and alone."""
    lengths = [17, 512, 1993]
    inp = wl.make_inputs(216, lengths, Hk=2, Hv=6, dk=128, dv=128, io_dtype=np.float16, state_std=0.02)
    out, final, _ = run_gpu(inp, in_place=False)
    cu = inp.cu_seqlens
    for s, L in enumerate(lengths):
        t0, t1 = cu[s], cu[s + 1]
        one = wl.GdnInputs(inp.q[t0:t1], inp.k[t0:t1], inp.v[t0:t1], inp.a[t0:t1], inp.b[t0:t1], inp.A_log,
                           inp.dt_bias, np.array([0, L], np.int32), inp.initial_state[s:s + 1], None)
        o1, f1, _ = run_gpu(one, in_place=False)
        assert np.array_equal(out[t0:t1], o1)
        assert np.array_equal(final[s], f1[0])
    _check(inp, (out, final, None), run_oracle(inp))


# Head sizes 32 and 64 (and mixed dk != dv) run the two-phase evaluation on the
# d = 128 operand tiles zero-padded: features past dk and state rows past dv
# are zero in every operand, so the same tensor-core products give the
# smaller heads' results; only the first dk / dv entries are read or written.
SMALL = [(64, 64), (32, 32), (64, 128), (128, 64), (32, 128), (128, 32)]


@pytest.mark.parametrize("dk,dv", SMALL)
@pytest.mark.parametrize("io", [np.float16, np.float32])
def test_forced_chunked_small_head_sizes(io, dk, dv):
    inp = wl.make_inputs(220 + dk + dv, LENGTHS, Hk=2, Hv=6, dk=dk, dv=dv, io_dtype=io, state_std=0.02,
                         capacity=70)
    _check(inp, run_gpu(inp, plan="chunked", in_place=False), run_oracle(inp))


@pytest.mark.parametrize("dk,dv", [(64, 64), (32, 32)])
def test_auto_plan_small_heads_takes_the_chunked_path(dk, dv):
    """Long sequences at d = 32 / 64 under the automatic plan (the binding
    passes the workspace gdn_forward_workspace_size asks for): short ones stay
    on the recurrent kernels, long ones go to the chunked kernels; one key
    head with a single value head (Hk = Hv = 1) puts the last head's boxes
    past the end of the q / k / v rows."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    for Hk, Hv, seed in ((2, 4, 230), (1, 1, 231)):
        lengths = [300, 17, 1000, 64, 2]
        inp = wl.make_inputs(seed + dk, lengths, Hk=Hk, Hv=Hv, dk=dk, dv=dv, io_dtype=np.float16, state_std=0.02,
                             capacity=20)
        a = gdn.build_forward_args(to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.a), to_dev(inp.b),
                                   to_dev(inp.cu_seqlens), A_log=to_dev(inp.A_log), dt_bias=to_dev(inp.dt_bias))[0]
        assert gdn.workspace_size(a) > 0  # the chunked kernels may run
        _check(inp, run_gpu(inp, in_place=True), run_oracle(inp))
        # pack = one by one, bitwise (each sequence's plan depends on its own length)
        out, final, caps = run_gpu(inp, in_place=False)
        cu = inp.cu_seqlens
        for s, L in enumerate(lengths):
            t0, t1 = cu[s], cu[s + 1]
            one = wl.GdnInputs(inp.q[t0:t1], inp.k[t0:t1], inp.v[t0:t1], inp.a[t0:t1], inp.b[t0:t1], inp.A_log,
                               inp.dt_bias, np.array([0, L], np.int32), inp.initial_state[s:s + 1], None, 20)
            o1, f1, c1 = run_gpu(one, in_place=False)
            assert np.array_equal(out[t0:t1], o1)
            assert np.array_equal(final[s], f1[0])
            assert np.array_equal(caps[s], c1[0])


def test_split_plan_small_heads_runs_unsplit():
    """Below d = 128 the split plan splits nothing (its identity run is built
    for 128): the results are the chunked plan's, bitwise."""
    inp = wl.make_inputs(240, [2500, 90], Hk=2, Hv=4, dk=64, dv=64, io_dtype=np.float16, state_std=0.05,
                         capacity=8)
    a = run_gpu(inp, plan="chunked_split", in_place=False)
    b = run_gpu(inp, plan="chunked", in_place=False)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    _check(inp, a, run_oracle(inp))
