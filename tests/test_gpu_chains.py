"""GPU parity of chains of calls launched back to back, each reading what the
previous one wrote, with no host synchronisation in between, against the
FP64 oracle run step by step.

The library's kernels are launched as programmatic dependents of the kernel
before them on the stream: a kernel's CTAs may be resident while the
previous kernel finishes, and each waits for that kernel's completion before
its first read.  These chains check that ordering on every producer ->
consumer pair the path has: decode step -> decode step on the same state
(in place), the chunked prefill's plan -> prep -> scan (and the split plan's
combining kernels) -> decode on its final states, and verify -> replay ->
decode from the replayed bank.  Tolerances as elsewhere: 1e-5 for FP32
recurrent results, 2e-3 for fp16 outputs and the tensor-core chunked path.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import max_rel
from gpu_common import to_dev, dev

from gated_delta_rule_gateddeltanet_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _gdn():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    return gdn


def _decode_inputs(seed, B, Hk, Hv, d, A_log, dt_bias):
    inp = wl.make_inputs(seed, [1] * B, Hk=Hk, Hv=Hv, dk=d, dv=d, io_dtype=np.float16)
    inp.A_log, inp.dt_bias = A_log, dt_bias
    return inp


def test_decode_steps_in_place_back_to_back():
    gdn = _gdn()
    B, Hk, Hv, d, steps = 24, 2, 6, 128, 8
    first = wl.make_inputs(1401, [1] * B, Hk=Hk, Hv=Hv, dk=d, dv=d, io_dtype=np.float16, state_std=0.02)
    state = to_dev(first.initial_state)
    ins = [first] + [_decode_inputs(1402 + i, B, Hk, Hv, d, first.A_log, first.dt_bias) for i in range(steps - 1)]
    outs = []
    for x in ins:  # no synchronisation between the steps
        o, _, _ = gdn.gdn_forward(to_dev(x.q), to_dev(x.k), to_dev(x.v), to_dev(x.a), to_dev(x.b),
                                  to_dev(x.cu_seqlens), A_log=to_dev(x.A_log), dt_bias=to_dev(x.dt_bias),
                                  initial_state=state, final_state=state, max_seqlen=1)
        outs.append(o)
    torch.cuda.synchronize()
    ref_state = first.initial_state.astype(np.float64)
    for x, o in zip(ins, outs):
        o_ref, ref_state, _ = oracle.gdn_forward(x.q, x.k, x.v, x.a, x.b, x.cu_seqlens, A_log=x.A_log,
                                                 dt_bias=x.dt_bias, initial_state=ref_state)
        assert max_rel(o.double().cpu().numpy(), o_ref) <= 2e-3
    assert max_rel(state.double().cpu().numpy(), ref_state) <= 1e-5


@pytest.mark.parametrize("plan", ["auto", "chunked_split"])
def test_prefill_then_decode_back_to_back(plan):
    """The chunked prefill's kernels (plan, prep, scan; with the split plan
    also the two combining kernels) write the final states that the next
    call's decode kernel reads."""
    gdn = _gdn()
    Hk, Hv, d = 2, 4, 128
    lengths = [2100, 300, 65]  # the first sequence is split under the split plan
    pre = wl.make_inputs(1410, lengths, Hk=Hk, Hv=Hv, dk=d, dv=d, io_dtype=np.float16, state_std=0.02)
    B = len(lengths)
    state = to_dev(pre.initial_state)
    o_pre, _, _ = gdn.gdn_forward(to_dev(pre.q), to_dev(pre.k), to_dev(pre.v), to_dev(pre.a), to_dev(pre.b),
                                  to_dev(pre.cu_seqlens), A_log=to_dev(pre.A_log), dt_bias=to_dev(pre.dt_bias),
                                  initial_state=state, final_state=state, plan=plan)
    decs = [_decode_inputs(1411 + i, B, Hk, Hv, d, pre.A_log, pre.dt_bias) for i in range(3)]
    outs = []
    for x in decs:
        o, _, _ = gdn.gdn_forward(to_dev(x.q), to_dev(x.k), to_dev(x.v), to_dev(x.a), to_dev(x.b),
                                  to_dev(x.cu_seqlens), A_log=to_dev(x.A_log), dt_bias=to_dev(x.dt_bias),
                                  initial_state=state, final_state=state, max_seqlen=1)
        outs.append(o)
    torch.cuda.synchronize()
    o_ref, ref_state, _ = oracle.gdn_forward(pre.q, pre.k, pre.v, pre.a, pre.b, pre.cu_seqlens, A_log=pre.A_log,
                                             dt_bias=pre.dt_bias, initial_state=pre.initial_state)
    assert max_rel(o_pre.double().cpu().numpy(), o_ref) <= 2e-3
    for x, o in zip(decs, outs):
        o_ref, ref_state, _ = oracle.gdn_forward(x.q, x.k, x.v, x.a, x.b, x.cu_seqlens, A_log=x.A_log,
                                                 dt_bias=x.dt_bias, initial_state=ref_state)
        assert max_rel(o.double().cpu().numpy(), o_ref) <= 2e-3
    assert max_rel(state.double().cpu().numpy(), ref_state) <= 2e-3


def test_verify_replay_decode_back_to_back():
    """Verify (capsules) -> replay of the accepted prefixes into the inactive
    bank -> a decode step reading the replayed bank, twice over with the banks
    swapped, with no synchronisation in between."""
    gdn = _gdn()
    R, D, Hk, Hv, d = 8, 4, 2, 6, 128
    rng = np.random.default_rng(1420)
    banks_h = (rng.standard_normal((2 * R, Hv, d, d)) * 0.02).astype(np.float32)
    banks = to_dev(banks_h)
    src, dst = np.arange(R, dtype=np.int32), np.arange(R, 2 * R, dtype=np.int32)
    ver0 = wl.make_inputs(1421, [D] * R, Hk=Hk, Hv=Hv, dk=d, dv=d, io_dtype=np.float16)
    A_log, dt_bias = ver0.A_log, ver0.dt_bias
    ref = banks_h.astype(np.float64)
    results = []
    for rnd in range(2):
        ver = ver0 if rnd == 0 else wl.make_inputs(1422, [D] * R, Hk=Hk, Hv=Hv, dk=d, dv=d, io_dtype=np.float16)
        n = rng.integers(0, D + 1, R).astype(np.int32)
        dec = _decode_inputs(1430 + rnd, R, Hk, Hv, d, A_log, dt_bias)
        o_ver, _, caps = gdn.gdn_forward(to_dev(ver.q), to_dev(ver.k), to_dev(ver.v), to_dev(ver.a), to_dev(ver.b),
                                         to_dev(ver.cu_seqlens), A_log=to_dev(A_log), dt_bias=to_dev(dt_bias),
                                         initial_state=banks, state_slots=to_dev(src), num_state_slots=2 * R,
                                         capacity=D, max_seqlen=D, write_final_state=False)
        gdn.gdn_replay_prefix(banks, to_dev(src), to_dev(dst), caps, to_dev(n), num_k_heads=Hk)
        o_dec, _, _ = gdn.gdn_forward(to_dev(dec.q), to_dev(dec.k), to_dev(dec.v), to_dev(dec.a), to_dev(dec.b),
                                      to_dev(dec.cu_seqlens), A_log=to_dev(A_log), dt_bias=to_dev(dt_bias),
                                      initial_state=banks, final_state=banks, state_slots=to_dev(dst),
                                      num_state_slots=2 * R, max_seqlen=1)
        results.append((ver, n, dec, src.copy(), dst.copy(), o_ver, caps, o_dec))
        src, dst = dst, src  # publish: the updated bank becomes the committed one
    torch.cuda.synchronize()
    for ver, n, dec, s_, d_, o_ver, caps, o_dec in results:
        o_ref, _, c_ref = oracle.gdn_forward(ver.q, ver.k, ver.v, ver.a, ver.b, ver.cu_seqlens, A_log=A_log,
                                             dt_bias=dt_bias, initial_state=ref, state_slots=s_,
                                             num_state_slots=2 * R, capacity=D)
        assert max_rel(o_ver.double().cpu().numpy(), o_ref) <= 2e-3
        assert max_rel(caps.double().cpu().numpy(), c_ref) <= 1e-5
        ref = oracle.gdn_replay(ref, s_, d_, c_ref, n, num_k_heads=Hk)
        o_ref, ref, _ = oracle.gdn_forward(dec.q, dec.k, dec.v, dec.a, dec.b, dec.cu_seqlens, A_log=A_log,
                                           dt_bias=dt_bias, initial_state=ref, state_slots=d_, num_state_slots=2 * R)
        assert max_rel(o_dec.double().cpu().numpy(), o_ref) <= 2e-3
    assert max_rel(banks.double().cpu().numpy(), ref) <= 1e-5
