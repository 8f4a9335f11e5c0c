"""GPU checks of the rank-4 (dense) entry point and of the state-layout
conversion.

Dense inputs [B, S, H, D] are the packed layout with B sequences of S tokens
each, so gdn_forward_dense must give bitwise the results of gdn_forward with
cu_seqlens = {0, S, ..., B S} on every plan; against the FP64 oracle it is held
to the packed tolerances (1e-5 for FP32 arithmetic on the recurrent kernel,
2e-3 where tensor cores take fp16 operands).  gdn_state_transpose is a pure
copy: bit-exact against numpy's transpose, and K-major -> V-major -> K-major
returns the input bitwise.
"""
import numpy as np
import pytest
import torch

from helpers import max_rel
from gpu_common import run_oracle, to_dev, dev, single_kernel_workspace

from gated_delta_rule_gateddeltanet_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _dense_inputs(seed, B, S, Hk, Hv, d, io, state=True):
    return wl.make_inputs(seed, [S] * B, Hk=Hk, Hv=Hv, dk=d, dv=d, io_dtype=io, state_std=0.02 if state else None)


def _run_both(inp, B, S, plan, workspace=None):
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    Hk, Hv, dk, dv = inp.dims
    r4 = lambda x: to_dev(x).reshape(B, S, *x.shape[1:])
    init = to_dev(inp.initial_state) if inp.initial_state is not None else None
    fd = torch.full((B, Hv, dv, dk), float("nan"), device=dev()) if init is None else init.clone()
    od, fd, _ = gdn.gdn_forward_dense(r4(inp.q), r4(inp.k), r4(inp.v), r4(inp.a), r4(inp.b),
                                      A_log=to_dev(inp.A_log), dt_bias=to_dev(inp.dt_bias), initial_state=init,
                                      final_state=fd, plan=plan, workspace=workspace)
    fp = torch.full((B, Hv, dv, dk), float("nan"), device=dev()) if init is None else init.clone()
    op, fp, _ = gdn.gdn_forward(to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.a), to_dev(inp.b),
                                to_dev(inp.cu_seqlens), A_log=to_dev(inp.A_log), dt_bias=to_dev(inp.dt_bias),
                                initial_state=init, final_state=fp, plan=plan, workspace=workspace)
    torch.cuda.synchronize()
    return (od.reshape(B * S, Hv, dv).double().cpu().numpy(), fd.double().cpu().numpy(),
            op.double().cpu().numpy(), fp.double().cpu().numpy())


@pytest.mark.parametrize("B,S,plan,tol", [(6, 4, "auto", 1e-5), (3, 200, "auto", 2e-3), (2, 130, "chunked", 2e-3),
                                          (5, 1, "recurrent", 1e-5), (2, 2100, "chunked_split", 2e-3)])
def test_dense_equals_packed_and_oracle(B, S, plan, tol):
    io = np.float32 if tol == 1e-5 else np.float16
    inp = _dense_inputs(301 + S, B, S, 2, 6, 128, io)
    od, fd, op, fp = _run_both(inp, B, S, plan)
    assert np.array_equal(od, op) and np.array_equal(fd, fp)
    o_ref, f_ref, _ = run_oracle(inp)
    assert max_rel(od, o_ref) <= tol
    assert max_rel(fd, f_ref) <= tol


def test_dense_single_kernel_workspace_and_zero_state():
    B, S = 2, 100
    inp = _dense_inputs(310, B, S, 1, 3, 128, np.float16, state=False)
    od, fd, op, fp = _run_both(inp, B, S, "chunked", workspace=single_kernel_workspace(inp))
    assert np.array_equal(od, op) and np.array_equal(fd, fp)
    o_ref, f_ref, _ = run_oracle(inp)
    assert max_rel(od, o_ref) <= 2e-3 and max_rel(fd, f_ref) <= 2e-3


def test_dense_rejects_cu_seqlens_and_bad_length():
    import ctypes
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    inp = _dense_inputs(311, 2, 8, 1, 1, 32, np.float32)
    t = lambda x: to_dev(x)
    args, _, keep = gdn.build_forward_args(t(inp.q), t(inp.k), t(inp.v), t(inp.a), t(inp.b), t(inp.cu_seqlens),
                                           A_log=t(inp.A_log), dt_bias=t(inp.dt_bias))
    lib = gdn.load_library()
    assert lib.gdn_forward_dense(ctypes.byref(args), 8, None) == 8   # cu_seqlens given
    args.cu_seqlens = None
    assert lib.gdn_forward_dense(ctypes.byref(args), 7, None) == 3   # 2 x 7 != 16 tokens
    assert lib.gdn_forward_dense(ctypes.byref(args), 8, None) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("rows,cols,num", [(128, 128, 96), (64, 128, 7), (32, 64, 3), (33, 70, 2)])
def test_state_transpose_is_an_exact_transpose(rows, cols, num):
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    x = np.random.default_rng(rows + cols).standard_normal((num, rows, cols)).astype(np.float32)
    y = gdn.state_transpose(to_dev(x))
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), np.swapaxes(x, 1, 2))
    back = gdn.state_transpose(y)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), x)


def test_dense_with_k_major_states():
    """The dense export's flow: K-major states [B, Hv, dk, dv] converted to
    V-major, the rank-4 forward, and the result converted back."""
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    B, S = 4, 70
    inp = _dense_inputs(312, B, S, 2, 4, 128, np.float16)
    k_major = np.ascontiguousarray(np.swapaxes(inp.initial_state, 2, 3))  # [B, Hv, dk, dv]
    v_major = gdn.state_transpose(to_dev(k_major))
    r4 = lambda x: to_dev(x).reshape(B, S, *x.shape[1:])
    out, final, _ = gdn.gdn_forward_dense(r4(inp.q), r4(inp.k), r4(inp.v), r4(inp.a), r4(inp.b),
                                          A_log=to_dev(inp.A_log), dt_bias=to_dev(inp.dt_bias),
                                          initial_state=v_major, final_state=v_major)
    final_k = gdn.state_transpose(final).cpu().double().numpy()
    torch.cuda.synchronize()
    o_ref, f_ref, _ = run_oracle(inp)
    assert max_rel(out.reshape(B * S, 4, 128).double().cpu().numpy(), o_ref) <= 2e-3
    assert max_rel(final_k, np.swapaxes(f_ref, 2, 3)) <= 2e-3
