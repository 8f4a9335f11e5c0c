"""The Python binding checks every buffer's shape against the call's geometry
before it reaches the C ABI (which takes raw pointers and cannot): a slot
list, gate array, state pool, output or capsule buffer of the wrong extent
raises ValueError.  CPU tensors: each case raises before any library call."""
import numpy as np
import pytest
import torch

import gated_delta_rule_gateddeltanet_gb300 as gdn

T, B, Hk, Hv, d, S = 6, 2, 2, 4, 32, 3


def _fwd(**over):
    z = lambda *s, dt=torch.float32: torch.zeros(s, dtype=dt)
    kw = dict(q=z(T, Hk, d, dt=torch.float16), k=z(T, Hk, d, dt=torch.float16), v=z(T, Hv, d, dt=torch.float16),
              a=z(T, Hv), b=z(T, Hv), cu_seqlens=torch.tensor([0, 4, 6], dtype=torch.int32),
              A_log=z(Hv), dt_bias=z(Hv), initial_state=z(S, Hv, d, d), final_state=z(S, Hv, d, d),
              state_slots=torch.tensor([2, 0], dtype=torch.int32), output=z(T, Hv, d, dt=torch.float16),
              capacity=2, state_update=z(B, 2, gdn.capsule_width(Hk, Hv, d, d)))
    kw.update(over)
    q, k, v, a, b, cu = (kw.pop(n) for n in ("q", "k", "v", "a", "b", "cu_seqlens"))
    return gdn.build_forward_args(q, k, v, a, b, cu, **kw)


@pytest.mark.parametrize("name,bad", [
    ("k", torch.zeros(T - 1, Hk, d, dtype=torch.float16)),
    ("v", torch.zeros(T + 1, Hv, d, dtype=torch.float16)),
    ("a", torch.zeros(T, Hv - 1)),
    ("b", torch.zeros(T - 1, Hv)),
    ("A_log", torch.zeros(Hv + 1)),
    ("dt_bias", torch.zeros(Hv - 1)),
    ("state_slots", torch.tensor([0], dtype=torch.int32)),
    ("initial_state", torch.zeros(S, Hv, d, d + 32)),
    ("final_state", torch.zeros(S - 1, Hv, d, d)),
    ("output", torch.zeros(T - 1, Hv, d, dtype=torch.float16)),
    ("state_update", torch.zeros(B, 3, gdn.capsule_width(Hk, Hv, d, d))),
])
def test_forward_rejects_wrong_shapes(name, bad):
    _fwd()  # the consistent call resolves
    with pytest.raises(ValueError, match=name):
        _fwd(**{name: bad})


def test_forward_accepts_larger_pools_and_buffers():
    """A state pool with more slots than the call addresses (e.g. both banks of
    a speculative step) and an output or capsule buffer with spare rows are
    valid: only their leading extent may exceed the call's."""
    W = gdn.capsule_width(Hk, Hv, d, d)
    _fwd(initial_state=torch.zeros(2 * S, Hv, d, d), final_state=torch.zeros(S + 1, Hv, d, d),
         output=torch.zeros(T + 2, Hv, d, dtype=torch.float16), state_update=torch.zeros(B + 1, 2, W),
         num_state_slots=S)


def test_forward_rejects_two_dimensional_cu_seqlens():
    with pytest.raises(ValueError, match="cu_seqlens"):
        _fwd(cu_seqlens=torch.tensor([[0, 4, 6]], dtype=torch.int32))


C, K = 16, 4


def _conv(**over):
    kw = dict(x=torch.zeros(T, C, dtype=torch.float16), weight=torch.zeros(C, K),
              cu_seqlens=torch.tensor([0, 4, 6], dtype=torch.int32), bias=torch.zeros(C),
              initial_state=torch.zeros(S, C, K - 1, dtype=torch.float16),
              final_state=torch.zeros(S, C, K - 1, dtype=torch.float16),
              state_slots=torch.tensor([1, 2], dtype=torch.int32),
              capture_count=torch.tensor([1, 2], dtype=torch.int32), capacity=2,
              state_update=torch.zeros(B, 2, C, dtype=torch.float16), output=torch.zeros(T, C, dtype=torch.float16))
    kw.update(over)
    x, w, cu = (kw.pop(n) for n in ("x", "weight", "cu_seqlens"))
    return gdn.build_conv_args(x, w, cu, **kw)


@pytest.mark.parametrize("name,bad", [
    ("weight", torch.zeros(C + 8, K)),
    ("bias", torch.zeros(C - 8)),
    ("state_slots", torch.tensor([1, 2, 0], dtype=torch.int32)),
    ("capture_count", torch.tensor([1], dtype=torch.int32)),
    ("initial_state", torch.zeros(S, C, K, dtype=torch.float16)),
    ("final_state", torch.zeros(S, C + 8, K - 1, dtype=torch.float16)),
    ("output", torch.zeros(T - 1, C, dtype=torch.float16)),
    ("state_update", torch.zeros(B - 1, 2, C, dtype=torch.float16)),
])
def test_conv_rejects_wrong_shapes(name, bad):
    _conv()
    key = {"weight": "weight"}.get(name, name)
    with pytest.raises(ValueError, match=key):
        _conv(**{name: bad})


@pytest.mark.parametrize("which", ["dst_slots", "accept_len", "state_update"])
def test_replays_reject_wrong_lengths(which):
    R, cap = 3, 2
    W = gdn.capsule_width(Hk, Hv, d, d)
    i32 = lambda *v: torch.tensor(v, dtype=torch.int32)
    args = dict(src_slots=i32(0, 1, 2), dst_slots=i32(3, 4, 5), accept_len=i32(1, 0, 2),
                state_update=torch.zeros(R, cap, W))
    args[which] = {"dst_slots": i32(3, 4), "accept_len": i32(1, 0, 2, 1),
                   "state_update": torch.zeros(R - 1, cap, W)}[which]
    with pytest.raises(ValueError, match=which):
        gdn.gdn_replay_prefix(torch.zeros(6, Hv, d, d), args["src_slots"], args["dst_slots"], args["state_update"],
                              args["accept_len"], num_k_heads=Hk)
    cargs = dict(src_slots=i32(0, 1, 2), dst_slots=i32(3, 4, 5), accept_len=i32(1, 0, 2),
                 state_update=torch.zeros(R, cap, C, dtype=torch.float16))
    cargs[which] = {"dst_slots": i32(3), "accept_len": i32(1, 0),
                    "state_update": torch.zeros(R, cap, C + 8, dtype=torch.float16)}[which]
    with pytest.raises(ValueError, match=which):
        gdn.causal_conv_replay_prefix(torch.zeros(6, C, K - 1, dtype=torch.float16), cargs["src_slots"],
                                      cargs["dst_slots"], cargs["state_update"], cargs["accept_len"])
