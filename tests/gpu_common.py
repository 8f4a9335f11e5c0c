"""Helpers for the GPU parity tests: move seeded host inputs to the GPU, run
the library through its binding, run the oracle on the same host arrays."""
import numpy as np
import torch

import oracle


def dev():
    return torch.device("cuda:0")


def to_dev(x, dtype=None):
    if x is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(dev())


def single_kernel_workspace(inp):
    """A workspace that holds only the chain list ((B + 2) int32): gdn_forward
    then runs the single-kernel chunked evaluation instead of the two-phase one."""
    n = ((inp.B + 2) * 4 + 255) // 256 * 256
    return torch.zeros(n, dtype=torch.uint8, device=dev())


def run_gpu(inp, *, plan="auto", capacity=None, gate_mode="raw", a=None, b=None, in_place=True,
            status=None, final_state=None, max_seqlen=0, workspace=None):
    """Runs gdn_forward on ``inp`` (a workloads.GdnInputs); returns numpy arrays.
    ``workspace=None`` lets the binding allocate what gdn_forward_workspace_size
    asks for (the two-phase chunked evaluation)."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    cap = inp.capacity if capacity is None else capacity
    Hk, Hv, dk, dv = inp.dims
    init = to_dev(inp.initial_state)
    if final_state is None:
        if in_place and init is not None:
            final_state = init
        else:
            slots = inp.initial_state.shape[0] if inp.initial_state is not None else inp.B
            final_state = torch.full((slots, Hv, dv, dk), float("nan"), dtype=torch.float32, device=dev())
            if init is not None:
                final_state.copy_(init)
    out, final, caps = gdn.gdn_forward(
        to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.a if a is None else a),
        to_dev(inp.b if b is None else b), to_dev(inp.cu_seqlens), A_log=to_dev(inp.A_log),
        dt_bias=to_dev(inp.dt_bias), gate_mode=gate_mode, initial_state=init, final_state=final_state,
        state_slots=to_dev(inp.state_slots), capacity=cap, plan=plan, status=status,
        num_state_slots=final_state.shape[0], max_seqlen=max_seqlen, workspace=workspace)
    torch.cuda.synchronize()
    return (out.double().cpu().numpy(), final.double().cpu().numpy(),
            None if caps is None else caps.double().cpu().numpy())


def run_oracle(inp, *, capacity=None, gate_mode="raw", a=None, b=None):
    cap = inp.capacity if capacity is None else capacity
    return oracle.gdn_forward(inp.q, inp.k, inp.v, inp.a if a is None else a, inp.b if b is None else b,
                              inp.cu_seqlens, A_log=inp.A_log, dt_bias=inp.dt_bias, gate_mode=gate_mode,
                              initial_state=inp.initial_state, state_slots=inp.state_slots,
                              num_state_slots=(inp.initial_state.shape[0] if inp.initial_state is not None
                                               else None), capacity=cap)


def capsule_parts(caps, Hk, Hv, dk, dv):
    """Split [B, cap, W] capsule rows into (g [B,cap,Hv], kn [B,cap,Hk,dk], u [B,cap,Hv,dv])."""
    B, cap, _ = caps.shape
    g = caps[:, :, :Hv]
    kn = caps[:, :, Hv:Hv + Hk * dk].reshape(B, cap, Hk, dk)
    u = caps[:, :, Hv + Hk * dk:].reshape(B, cap, Hv, dv)
    return g, kn, u
