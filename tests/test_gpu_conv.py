"""GPU parity of the packed causal convolution, its compact capture and its
replay against the FP64 oracle, through the C ABI.

Tolerance (max-relative per tensor): FP32 I/O 1e-5; FP16 outputs 2e-3 (one
FP16 rounding).  The state and the captured values are copies of inputs, so
they must match bit for bit; so must a replay of captured values.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import max_rel
from gpu_common import to_dev, dev

pytestmark = pytest.mark.gpu


def _inputs(seed, lengths, C, K, io, slots=None, num_slots=None, state=True):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    x = rng.standard_normal((T, C)).astype(io)
    w = (rng.standard_normal((C, K)) / 2).astype(np.float32)
    bias = (rng.standard_normal(C) / 4).astype(np.float32)
    S = num_slots or len(lengths)
    st = rng.standard_normal((S, C, K - 1)).astype(io) if state else None
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return x, w, bias, st, cu


def _gpu(x, w, bias, st, cu, *, cap=0, capture_count=None, slots=None, in_place=True, activation="silu",
         num_slots=None, status=None, max_seqlen=0):
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    init = to_dev(st)
    S = st.shape[0] if st is not None else (num_slots or len(cu) - 1)
    C, K = w.shape
    if in_place and init is not None:
        final = init
    else:
        final = torch.full((S, C, K - 1), float("nan"), dtype=torch.float16 if x.dtype == np.float16 else
                           torch.float32, device=dev())
        if init is not None:
            final.copy_(init)
    out, final, vals = gdn.varlen_causal_conv_with_state(
        to_dev(x), to_dev(w), to_dev(cu), bias=to_dev(bias), initial_state=init, final_state=final,
        state_slots=to_dev(slots), capture_count=to_dev(capture_count), capacity=cap, activation=activation,
        status=status, num_state_slots=S, max_seqlen=max_seqlen)
    torch.cuda.synchronize()
    return (out.double().cpu().numpy(), final.double().cpu().numpy(),
            None if vals is None else vals.double().cpu().numpy())


def _oracle(x, w, bias, st, cu, *, cap=0, capture_count=None, slots=None, num_slots=None):
    S = st.shape[0] if st is not None else (num_slots or len(cu) - 1)
    C, K = w.shape
    st0 = st if st is not None else np.zeros((S, C, K - 1))
    return oracle.conv_forward(x, w, cu, st0, bias=bias, state_slots=slots, capacity=cap,
                               capture_count=capture_count)


@pytest.mark.parametrize("io", [np.float16, np.float32])
@pytest.mark.parametrize("K", [4, 3, 2])
def test_conv_ragged_many_token_blocks(io, K):
    lengths = [300, 5, 1, 0, 70, 2, 1700]  # long sequences span many token blocks
    x, w, bias, st, cu = _inputs(40 + K, lengths, 512, K, io)
    cap = 6
    cc = np.array([6, 3, 0, 2, 6, 1, 4], np.int32)
    got = _gpu(x, w, bias, st, cu, cap=cap, capture_count=cc)
    want = _oracle(x, w, bias, st, cu, cap=cap, capture_count=cc)
    tol = 2e-3 if io == np.float16 else 1e-5
    assert max_rel(got[0], want[0]) <= tol
    assert np.array_equal(got[1], want[1])  # the state is a copy of inputs
    for s, L in enumerate(lengths):
        n = min(L, cap, cc[s])
        assert np.array_equal(got[2][s, :n], want[2][s, :n])
        assert np.all(got[2][s, n:] == 0)  # rows past the capture stay untouched (zero-initialised)


def test_conv_out_of_place_zero_state_and_slots():
    lengths = [64, 3, 129]
    x, w, bias, _, cu = _inputs(50, lengths, 256, 4, np.float32, state=False)
    got = _gpu(x, w, bias, None, cu, in_place=False, num_slots=3)
    want = _oracle(x, w, bias, None, cu, num_slots=3)
    assert max_rel(got[0], want[0]) <= 1e-5
    assert np.array_equal(got[1], want[1])
    x, w, bias, st, cu = _inputs(51, lengths, 256, 4, np.float16, num_slots=6)
    slots = np.array([5, 0, 3], np.int32)
    got = _gpu(x, w, bias, st, cu, slots=slots, in_place=False)
    want = _oracle(x, w, bias, st, cu, slots=slots)
    assert max_rel(got[0], want[0]) <= 2e-3
    assert np.array_equal(got[1], want[1])  # written slots and untouched ones


def test_conv_qwen_geometry_decode_and_prefill():
    """The conv in front of the GatedDeltaNet of the Qwen3.5/3.8 linear-attention
    layers: channels = 2*16*128 + 48*128 = 10240, kernel 4, fp16: a 64 x 1-token
    decode step and an 8-sequence varlen prefill."""
    from gated_delta_rule_gateddeltanet_gb300 import workloads as wl
    C = 10240
    x, w, bias, st, cu = _inputs(52, [1] * 64, C, 4, np.float16)
    want = _oracle(x, w, bias, st, cu, cap=1)
    runs = []
    for hint in (0, 1):  # a max_seqlen hint of 1 runs the short-sequence kernel (no state-rolling launch)
        got = _gpu(x, w, bias, st, cu, cap=1, max_seqlen=hint)
        assert max_rel(got[0], want[0]) <= 2e-3 and np.array_equal(got[1], want[1])
        assert np.array_equal(got[2], want[2])
        runs.append(got)
    for a, b in zip(*runs):  # the hint changes the launch shape, never a bit of the results
        assert np.array_equal(a, b)
    lengths = wl.varlen_prefill_lengths()
    x, w, bias, st, cu = _inputs(53, lengths, C, 4, np.float16)
    got = _gpu(x, w, bias, st, cu)
    want = _oracle(x, w, bias, st, cu)
    assert max_rel(got[0], want[0]) <= 2e-3 and np.array_equal(got[1], want[1])


def test_conv_pack_equals_one_by_one_bitwise():
    lengths = [17, 512, 1, 93]
    x, w, bias, st, cu = _inputs(54, lengths, 1024, 4, np.float16)
    got = _gpu(x, w, bias, st, cu, cap=4, in_place=False)
    for s, L in enumerate(lengths):
        t0, t1 = cu[s], cu[s + 1]
        one = _gpu(x[t0:t1], w, bias, st[s:s + 1], np.array([0, L], np.int32), cap=4, in_place=False)
        assert np.array_equal(got[0][t0:t1], one[0])
        assert np.array_equal(got[1][s], one[1][0])
        assert np.array_equal(got[2][s], one[2][0])


def test_conv_replay_every_prefix():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    L, C, K = 6, 256, 4
    x, w, bias, st, cu = _inputs(55, [L], C, K, np.float16)
    _, _, vals = _gpu(x, w, bias, st, cu, cap=L, in_place=False)
    R = L + 1
    states = torch.zeros((2 * R, C, K - 1), dtype=torch.float16, device=dev())
    states[:R] = to_dev(st)
    vals_dev = to_dev(vals.astype(np.float16)).expand(R, L, C).contiguous()
    gdn.causal_conv_replay_prefix(states, to_dev(np.arange(R, dtype=np.int32)),
                                  to_dev(np.arange(R, 2 * R, dtype=np.int32)), vals_dev,
                                  to_dev(np.arange(R, dtype=np.int32)))
    torch.cuda.synchronize()
    got = states.double().cpu().numpy()
    for n in range(R):
        _, st_n, _ = oracle.conv_forward(x[:n], w, np.array([0, n]), st, bias=bias)
        assert np.array_equal(got[R + n], st_n[0])
        assert np.array_equal(got[n], st[0].astype(np.float64))  # sources untouched


def test_conv_status_flags():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    x, w, bias, st, cu = _inputs(56, [4, 3], 64, 4, np.float32)
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    _gpu(x, w, bias, st, cu, cap=2, capture_count=np.array([3, 1], np.int32), status=status)
    assert status.item() & gdn.DEVERR["capture_count"]
    status.zero_()
    _gpu(x, w, bias, st, cu, slots=np.array([0, 7], np.int32), status=status)
    assert status.item() & gdn.DEVERR["state_slot"]


@pytest.mark.parametrize("io", [np.float16, np.float32])
@pytest.mark.parametrize("K", [4, 3, 2])
@pytest.mark.parametrize("in_place", [True, False])
def test_conv_short_sequences_kernel(io, K, in_place):
    """max_seqlen hints of 1 .. 8 run one thread per (sequence pair, 4 channels):
    ragged 0-8 token sequences (odd count, so the last pair is half empty),
    scattered slots, per-request capture counts; results equal the oracle's and,
    bit for bit, the token-block kernel's (hint 0)."""
    lengths = [1, 0, 8, 3, 1, 5, 0, 2, 7, 4, 1]
    S = 16
    x, w, bias, st, cu = _inputs(70 + K, lengths, 520, K, io, num_slots=S)
    slots = np.array([9, 2, 15, 0, 4, 11, 7, 3, 13, 6, 1], np.int32)
    cap = 5
    cc = np.array([1, 0, 5, 2, 1, 3, 0, 2, 4, 5, 0], np.int32)
    want = _oracle(x, w, bias, st, cu, cap=cap, capture_count=cc, slots=slots)
    tol = 2e-3 if io == np.float16 else 1e-5
    runs = []
    for hint in (8, 0):
        got = _gpu(x, w, bias, st, cu, cap=cap, capture_count=cc, slots=slots, in_place=in_place, max_seqlen=hint)
        assert max_rel(got[0], want[0]) <= tol
        assert np.array_equal(got[1], want[1])  # written slots, and untouched ones
        for s_, L in enumerate(lengths):
            n = min(L, cap, cc[s_])
            assert np.array_equal(got[2][s_, :n], want[2][s_, :n])
            assert np.all(got[2][s_, n:] == 0)
        runs.append(got)
    for a, b in zip(*runs):
        assert np.array_equal(a, b)


def test_conv_short_kernel_zero_state_and_hint_exceeded():
    """No initial state (zeros; empty sequences still get their zero state out of
    place), and a hint that a sequence exceeds (a caller error): the short kernel
    loads the rows past its prefetch and stays exact."""
    lengths = [0, 2, 1, 13, 0, 6]
    x, w, bias, _, cu = _inputs(80, lengths, 256, 4, np.float16, state=False)
    want = _oracle(x, w, bias, None, cu, num_slots=6)
    for hint in (2, 8):
        got = _gpu(x, w, bias, None, cu, in_place=False, num_slots=6, max_seqlen=hint)
        assert max_rel(got[0], want[0]) <= 2e-3
        assert np.array_equal(got[1], want[1])
        ref = _gpu(x, w, bias, None, cu, in_place=False, num_slots=6, max_seqlen=0)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_conv_short_kernel_status_flags():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    x, w, bias, st, cu = _inputs(81, [1, 1, 1], 64, 4, np.float32)
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    _gpu(x, w, bias, st, cu, cap=1, capture_count=np.array([1, 2, 0], np.int32), status=status, max_seqlen=1)
    assert status.item() == gdn.DEVERR["capture_count"]
    status.zero_()
    _gpu(x, w, bias, st, cu, slots=np.array([0, 7, 1], np.int32), status=status, max_seqlen=1)
    assert status.item() == gdn.DEVERR["state_slot"]


@pytest.mark.parametrize("hint", [0, 1])
def test_conv_all_empty_batch(hint):
    """Every sequence empty (T = 0): no outputs, states kept (copied out of place)."""
    x, w, bias, st, cu = _inputs(82, [0, 0, 0], 64, 4, np.float16)
    for in_place in (True, False):
        got = _gpu(x, w, bias, st, cu, in_place=in_place, max_seqlen=hint)
        assert got[0].shape[0] == 0
        assert np.array_equal(got[1], st.astype(np.float64))


@pytest.mark.parametrize("hint", [0, 4])
def test_conv_bad_sequence_flagged_and_skipped(hint):
    """A backwards cu_seqlens entry: the bit is set, that sequence's slot keeps
    its state, and the valid sequences match the valid call bit for bit (token-
    block kernel and short-sequence kernel)."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    x, w, bias, st, cu = _inputs(83, [3, 2, 4], 64, 4, np.float16)
    good = _gpu(x, w, bias, st, cu, in_place=False, max_seqlen=hint)
    bad_cu = cu.copy()
    bad_cu[2] = bad_cu[1] - 1  # sequence 1 ends before it starts
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    got = _gpu(x, w, bias, st, bad_cu, in_place=False, status=status, max_seqlen=hint)
    assert status.item() & gdn.DEVERR["cu_seqlens"]
    assert np.array_equal(got[1][0], good[1][0])
    assert np.array_equal(got[1][1], st[1].astype(np.float64))


def test_conv_replay_status_flags():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    rng = np.random.default_rng(84)
    C, K = 64, 4
    states = to_dev(rng.standard_normal((4, C, K - 1)).astype(np.float16))
    before = states.clone()
    vals = to_dev(rng.standard_normal((2, 3, C)).astype(np.float16))
    i32 = lambda *v: to_dev(np.array(v, np.int32))
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    gdn.causal_conv_replay_prefix(states, i32(0, 1), i32(2, 3), vals, i32(4, 1), status=status)  # n > capacity
    torch.cuda.synchronize()
    assert status.item() == gdn.DEVERR["accept_len"]
    assert torch.equal(states[2], before[2])  # the bad request is skipped
    status.zero_()
    before = states.clone()
    gdn.causal_conv_replay_prefix(states, i32(0, 7), i32(2, 3), vals, i32(1, 1), status=status)  # source out of range
    torch.cuda.synchronize()
    assert status.item() == gdn.DEVERR["replay_slot"]
    assert torch.equal(states[3], before[3])


@pytest.mark.parametrize("hint", [0, 2])
def test_conv_empty_sequence_with_bad_slot_flagged(hint):
    """An empty sequence (no tokens for the token-block kernel to visit) whose
    slot is out of range still sets the bit."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    x, w, bias, st, cu = _inputs(85, [2, 0, 2], 64, 4, np.float16)
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    _gpu(x, w, bias, st, cu, slots=np.array([0, 7, 2], np.int32), in_place=False, status=status, max_seqlen=hint)
    assert status.item() == gdn.DEVERR["state_slot"]
