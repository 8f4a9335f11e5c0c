"""The speculative step captured in one CUDA graph (conv with capture ->
gdn_forward with capsules on the fused q|k|v view of the conv output ->
conv replay and GDN replay of the accepted prefix).

The graph replays the same kernels with the same arguments as the eager
calls, so over several steps (different accepted lengths, banks published in
between) every output, capture and state bank must be bitwise equal to the
eager sequence.  The eager calls are each checked against the FP64 oracle in
their own test files.  With every draft accepted, the replayed states equal
the verify pass's own final states.
"""
import numpy as np
import pytest
import torch

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
