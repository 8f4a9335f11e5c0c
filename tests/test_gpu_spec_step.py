"""The speculative step captured in one CUDA graph (conv with capture ->
gdn_forward with capsules on the fused q|k|v view of the conv output ->
conv replay and GDN replay of the accepted prefix).

The graph replays the same kernels with the same arguments as the eager
calls, so over several steps (different accepted lengths, banks published in
between) every output, capture and state bank must be bitwise equal to the
eager sequence.  The eager calls are each checked against the FP64 oracle in
their own test files.  With every draft accepted, the replayed states equal
the verify pass's own final states.

The composed step is also checked against the FP64 oracle's own chain on the
same host inputs, over several published steps ("Replay compact fixed state
for hybrid decoding", Summary / Key changes: verify the drafts from the
committed state with compact capture, then replay the accepted prefix into
the inactive bank): the oracle convolution with capture, its output rounded
to fp16 (the convolution's output type) and sliced into q | k | v for the
oracle GDN forward with capsules, then the oracle's conv and GDN replays of
the accepted lengths, carried from step to step in the oracle's own banks.
Tolerances: the conv captures and conv states are copies of fp16 inputs, so
they must match bit for bit; fp16 outputs (conv and GDN) 2e-3; capsule
decays 1e-5 (they depend on the gate inputs alone); capsule keys and deltas
and the replayed FP32 GDN states 2e-3 in the composed chain (the GPU's FP32
convolution and the oracle's FP64 one can round an fp16 output to
neighbouring values, which moves a key or a delta by up to 2^-11 relative),
and 1e-5 when the oracle GDN is fed the conv output the GPU computed.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import max_rel
from gpu_common import dev

pytestmark = pytest.mark.gpu

R, D, Hk, Hv, d = 4, 4, 2, 6, 128
C = 2 * Hk * d + Hv * d


def _make(seed, keep=False):
    from gated_delta_rule_gateddeltanet_gb300.spec_step import SpeculativeStep
    g = torch.Generator().manual_seed(seed)
    w = torch.randn((C, 4), generator=g).mul_(0.5).to(dev())
    bias = torch.randn(C, generator=g).mul_(0.1).to(dev())
    conv_bank = torch.randn((2 * R, C, 3), generator=g).to(torch.float16).to(dev())
    gdn_bank = torch.randn((2 * R, Hv, d, d), generator=g).mul_(0.02).to(dev())
    A_log = torch.log(torch.empty(Hv).uniform_(1, 16, generator=g)).to(dev())
    dt_bias = torch.log(torch.expm1(torch.empty(Hv).uniform_(1e-3, 0.1, generator=g))).to(dev())
    return SpeculativeStep(w, bias, conv_bank, A_log, dt_bias, gdn_bank, num_k_heads=Hk, drafts=D,
                           keep_verify_state=keep)


def _inputs(step):
    g = torch.Generator().manual_seed(100 + step)
    x = torch.randn((R * D, C), generator=g).to(torch.float16)
    a = torch.randn((R * D, Hv), generator=g)
    b = torch.randn((R * D, Hv), generator=g)
    n = torch.randint(0, D + 1, (R,), generator=g, dtype=torch.int32)
    return x, a, b, n


@pytest.mark.parametrize("keep", [False, True])
def test_graph_step_equals_eager_over_published_steps(keep):
    eager, graphed = _make(7, keep), _make(7, keep)
    graphed.capture()
    for step in range(3):
        x, a, b, n = _inputs(step)
        for s in (eager, graphed):
            s.x.copy_(x); s.a.copy_(a); s.b.copy_(b); s.accept_len.copy_(n)
        eager.run_eager()
        graphed.replay()
        torch.cuda.synchronize()
        for name in ("out", "y", "capsules", "conv_values", "conv_bank", "gdn_bank"):
            assert torch.equal(getattr(eager, name), getattr(graphed, name)), (step, name)
        assert eager.status.item() == 0 and graphed.status.item() == 0
        eager.publish()
        graphed.publish()


def test_all_accepted_replay_reproduces_the_verify_states():
    s = _make(8, keep=True).capture()
    x, a, b, _ = _inputs(9)
    s.x.copy_(x); s.a.copy_(a); s.b.copy_(b); s.accept_len.fill_(D)
    s.replay()
    torch.cuda.synchronize()
    src, dst = s.src.long(), s.dst.long()
    assert torch.equal(s.conv_bank[dst], s.conv_scratch[src])
    rel = (s.gdn_bank[dst] - s.gdn_scratch[src]).abs().max() / s.gdn_scratch[src].abs().max()
    assert rel.item() <= 1e-6
    # nothing accepted: the inactive slots become copies of the committed ones
    s.publish()
    s.accept_len.zero_()
    s.replay()
    torch.cuda.synchronize()
    assert torch.equal(s.conv_bank[s.dst.long()], s.conv_bank[s.src.long()])
    assert torch.equal(s.gdn_bank[s.dst.long()], s.gdn_bank[s.src.long()])


def test_graph_step_matches_the_oracle_chain_over_published_steps():
    from gated_delta_rule_gateddeltanet_gb300.spec_step import SpeculativeStep
    rng = np.random.default_rng(31)
    w = (rng.standard_normal((C, 4)) * 0.5).astype(np.float32)
    bias = (rng.standard_normal(C) * 0.1).astype(np.float32)
    conv_ref = rng.standard_normal((2 * R, C, 3)).astype(np.float16).astype(np.float64)
    gdn_ref = (rng.standard_normal((2 * R, Hv, d, d)) * 0.02).astype(np.float32).astype(np.float64)
    A_log = np.log(rng.uniform(1, 16, Hv)).astype(np.float32)
    dt_bias = np.log(np.expm1(rng.uniform(1e-3, 0.1, Hv))).astype(np.float32)
    t = lambda x, dt=None: torch.from_numpy(np.ascontiguousarray(x if dt is None else x.astype(dt))).to(dev())
    s = SpeculativeStep(t(w), t(bias), t(conv_ref, np.float16), t(A_log), t(dt_bias), t(gdn_ref, np.float32),
                        num_k_heads=Hk, drafts=D).capture()
    src, dst = np.arange(R), np.arange(R, 2 * R)
    cu = np.arange(0, R * D + 1, D, dtype=np.int32)
    accepted = [[0, 4, 2, 1], [3, 0, 4, 4], [1, 2, 0, 3], [4, 4, 4, 4]]
    hd = Hk * d
    for step, n in enumerate(accepted):
        x = rng.standard_normal((R * D, C)).astype(np.float16)
        a = rng.standard_normal((R * D, Hv)).astype(np.float32)
        b = rng.standard_normal((R * D, Hv)).astype(np.float32)
        n = np.array(n, np.int32)
        s.x.copy_(t(x)); s.a.copy_(t(a)); s.b.copy_(t(b)); s.accept_len.copy_(t(n))
        committed_before = s.gdn_bank[t(src).long()].clone()
        s.replay()
        torch.cuda.synchronize()
        assert s.status.item() == 0

        # the oracle's chain on the same host inputs, from its own banks
        y_ref, _, vals_ref = oracle.conv_forward(x, w, cu, conv_ref, bias=bias, state_slots=src, capacity=D)
        y16 = y_ref.astype(np.float16)  # the convolution's output type
        q16, k16 = y16[:, :hd].reshape(-1, Hk, d), y16[:, hd:2 * hd].reshape(-1, Hk, d)
        v16 = y16[:, 2 * hd:].reshape(-1, Hv, d)
        o_ref, _, caps_ref = oracle.gdn_forward(q16, k16, v16, a, b, cu, A_log=A_log, dt_bias=dt_bias,
                                                initial_state=gdn_ref, state_slots=src, capacity=D)
        conv_next = oracle.conv_replay(conv_ref, src, dst, vals_ref, n)
        gdn_next = oracle.gdn_replay(gdn_ref, src, dst, caps_ref, n, num_k_heads=Hk)

        g = lambda name: getattr(s, name).double().cpu().numpy()
        y, out, caps, vals = g("y"), g("out"), g("capsules"), g("conv_values")
        conv_bank, gdn_bank = g("conv_bank"), g("gdn_bank")
        assert max_rel(y, y_ref) <= 2e-3, (step, max_rel(y, y_ref))
        assert np.array_equal(vals, vals_ref), step
        assert np.array_equal(conv_bank[dst], conv_next[dst]), step
        assert np.array_equal(conv_bank[src], conv_ref[src]), step
        assert max_rel(out, o_ref) <= 2e-3, (step, max_rel(out, o_ref))
        W0 = Hv + Hk * d
        assert max_rel(caps[:, :, :Hv], caps_ref[:, :, :Hv]) <= 1e-5, step
        assert max_rel(caps[:, :, Hv:W0], caps_ref[:, :, Hv:W0]) <= 2e-3, step
        assert max_rel(caps[:, :, W0:], caps_ref[:, :, W0:]) <= 2e-3, step
        assert max_rel(gdn_bank[dst], gdn_next[dst]) <= 2e-3, (step, max_rel(gdn_bank[dst], gdn_next[dst]))
        # the committed bank is never written
        assert torch.equal(s.gdn_bank[t(src).long()], committed_before)

        # stage-wise: the oracle GDN fed the GPU's own conv output, at the FP32 bound (the
        # committed slots read here are unchanged by the step)
        yq, yk = y[:, :hd].reshape(-1, Hk, d), y[:, hd:2 * hd].reshape(-1, Hk, d)
        o_s, _, caps_s = oracle.gdn_forward(yq, yk, y[:, 2 * hd:].reshape(-1, Hv, d), a, b, cu, A_log=A_log,
                                            dt_bias=dt_bias, initial_state=gdn_bank,
                                            state_slots=src, capacity=D)
        assert max_rel(out, o_s) <= 2e-3
        assert max_rel(caps, caps_s) <= 1e-5, (step, max_rel(caps, caps_s))
        bank_s = oracle.gdn_replay(gdn_bank, src, dst, caps_s, n, num_k_heads=Hk)
        assert max_rel(gdn_bank[dst], bank_s[dst]) <= 1e-5, (step, max_rel(gdn_bank[dst], bank_s[dst]))

        conv_ref, gdn_ref = conv_next, gdn_next
        s.publish()
        src, dst = dst, src
