"""gdn_forward_no_alloc: the forward pass for hosts that cannot give the
operator any device memory beyond its declared inputs and outputs (an
inference runtime's custom-operator interface, a serving loop with a fixed
memory plan) or cannot afford a cudaMalloc on the call path.  It must give
the same results as gdn_forward with a caller workspace, call after call,
although every call reuses the same fixed scratch array inside the library.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import max_rel
from gpu_common import to_dev, dev

from gated_delta_rule_gateddeltanet_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 2e-3  # the chunked path's tolerance


def _run(entry, inp, use_workspace):
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    lib = gdn.load_library()
    Hk, Hv, dk, dv = inp.dims
    state = to_dev(inp.initial_state)
    out = torch.full((inp.T, Hv, dv), float("nan"), dtype=torch.float16, device=dev())
    caps = torch.zeros((inp.B, inp.capacity, gdn.capsule_width(Hk, Hv, dk, dv)), device=dev())
    args, _, keep = gdn.build_forward_args(
        to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.a), to_dev(inp.b), to_dev(inp.cu_seqlens),
        A_log=to_dev(inp.A_log), dt_bias=to_dev(inp.dt_bias), initial_state=state, final_state=state, output=out,
        state_update=caps, capacity=inp.capacity)
    ws = None
    if use_workspace:
        n = gdn.workspace_size(args)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev())
        args.workspace, args.workspace_bytes = ctypes.c_void_p(ws.data_ptr()), n
    rc = getattr(lib, entry)(ctypes.byref(args), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, rc
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), state.double().cpu().numpy(), caps.double().cpu().numpy()


def test_no_alloc_matches_gdn_forward_on_consecutive_calls():
    # two different batches, both long enough to run the chunked kernel, so
    # the second call finds the first call's leftovers in the shared scratch
    batches = [
        wl.make_inputs(301, [300, 45, 1, 129, 0, 64], Hk=2, Hv=6, dk=128, dv=128, io_dtype=np.float16,
                       state_std=0.02, capacity=8),
        wl.make_inputs(302, [70, 200, 33], Hk=1, Hv=3, dk=128, dv=128, io_dtype=np.float16, state_std=0.02,
                       capacity=4),
    ]
    for inp in batches:
        want = _run("gdn_forward", inp, use_workspace=True)
        got = _run("gdn_forward_no_alloc", inp, use_workspace=False)
        for g, w in zip(got, want):
            assert max_rel(g, w) <= TOL
        assert np.all(np.isfinite(got[0]))


def test_no_alloc_all_short_batch_needs_no_scratch():
    # every sequence takes the recurrent kernels, which use no workspace: the
    # call must not look the scratch array up and must match gdn_forward
    inp = wl.make_inputs(303, [1, 4, 32, 0, 17, 2], Hk=2, Hv=6, dk=128, dv=128, io_dtype=np.float16,
                         state_std=0.02, capacity=4)
    for _ in range(2):
        want = _run("gdn_forward", inp, use_workspace=True)
        got = _run("gdn_forward_no_alloc", inp, use_workspace=False)
        for g, w in zip(got, want):
            assert max_rel(g, w) <= TOL


def test_no_alloc_python_wrapper_matches_gdn_forward():
    # the binding's wrapper: it drops any workspace argument and lets the
    # argument builder allocate the outputs, then calls the no-alloc entry
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    inp = wl.make_inputs(304, [150, 3, 90], Hk=2, Hv=6, dk=128, dv=128, io_dtype=np.float16, state_std=0.02,
                         capacity=5)
    kw = dict(A_log=to_dev(inp.A_log), dt_bias=to_dev(inp.dt_bias), capacity=inp.capacity)
    ins = [to_dev(x) for x in (inp.q, inp.k, inp.v, inp.a, inp.b, inp.cu_seqlens)]
    for _ in range(2):
        s0, s1 = to_dev(inp.initial_state), to_dev(inp.initial_state)
        want = gdn.gdn_forward(*ins, initial_state=s0, final_state=s0, **kw)
        got = gdn.gdn_forward_no_alloc(*ins, initial_state=s1, final_state=s1,
                                       workspace=torch.empty(16, dtype=torch.uint8, device=dev()), **kw)
        torch.cuda.synchronize()
        for g, w in zip(got, want):
            assert max_rel(g.double().cpu().numpy(), w.double().cpu().numpy()) <= TOL


def test_no_alloc_rejects_batches_beyond_its_scratch():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    lib = gdn.load_library()
    a = gdn.ForwardArgs()
    a.num_seqs, a.total_tokens, a.num_k_heads, a.num_v_heads = 4095, 4095 * 40, 16, 48
    a.head_dim_k = a.head_dim_v = 128
    a.num_state_slots, a.io_dtype = 4095, 1
    # rejected on the host before anything is read or launched
    assert lib.gdn_forward_no_alloc(ctypes.byref(a), None) == 5
