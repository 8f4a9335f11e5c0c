"""GPU parity of the tensor-core evaluation of multi-token short spans (the
mixed recurrent kernel) against the FP64 oracle, through the C ABI.

The cases follow that kernel's structure: many work items per persistent CTA
(the next item's rows arrive while one computes; consecutive value heads of
one key head reuse the key-side staging), one-token and empty spans between
longer ones inside a CTA's range of items, 64-row blocks cut short by dv = 32
(the row boxes then reach into the next head's rows or past the array), spans
up to the 32-token recurrent limit (eight 4-token groups, the last one
ragged), and gates at their extremes.  Tolerances as for the CUDA-core
recurrent path: 1e-5 (max-relative) for FP32 results, 2e-3 for FP16 outputs.
"""
import numpy as np
import pytest

from helpers import max_rel
from gpu_common import run_gpu, run_oracle

from gated_delta_rule_gateddeltanet_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL32 = 1e-5
TOL16_OUT = 2e-3


def _check(inp, gpu, ref, fp16):
    out, final, caps = gpu
    o_ref, f_ref, c_ref = ref
    assert max_rel(out, o_ref) <= (TOL16_OUT if fp16 else TOL32)
    slots = np.arange(inp.B) if inp.state_slots is None else inp.state_slots
    assert max_rel(final[slots], f_ref[slots]) <= TOL32
    if inp.capacity > 0:
        lens = np.diff(inp.cu_seqlens)
        for s in range(inp.B):
            n = min(int(lens[s]), inp.capacity)
            if n:
                assert max_rel(caps[s, :n], c_ref[s, :n]) <= TOL32


def test_many_items_per_cta_with_one_token_and_empty_spans():
    """300 sequences of 0..5 tokens at Hk=4, Hv=12: 7200 (sequence, head, row
    block) items, about a dozen per CTA, with CUDA-core items (0 or 1 token)
    between tensor-core ones."""
    lengths = np.random.default_rng(600).integers(0, 6, 300)
    inp = wl.make_inputs(601, lengths, Hk=4, Hv=12, dk=128, dv=128, io_dtype=np.float16, state_std=0.02,
                         capacity=4)
    _check(inp, run_gpu(inp), run_oracle(inp), fp16=True)


@pytest.mark.parametrize("dk", [32, 64, 128])
def test_row_blocks_cut_short_by_dv(dk):
    """dv = 32: each 64-row block holds 32 rows; the row boxes' other 32 rows
    are the next head's (or past the end of the state array) and unused."""
    dv = 32
    inp = wl.make_inputs(610 + dk + dv, [3, 4, 2, 5, 4], Hk=2, Hv=6, dk=dk, dv=dv, io_dtype=np.float32,
                         state_std=0.02, capacity=3)
    _check(inp, run_gpu(inp, in_place=False), run_oracle(inp), fp16=False)


def test_spans_up_to_the_recurrent_limit():
    """32 tokens is the longest span the automatic plan keeps on the recurrent
    kernel: eight groups of four; 31 and 29 end in a ragged group."""
    inp = wl.make_inputs(620, [32, 31, 29, 2, 1], Hk=2, Hv=4, dk=128, dv=128, io_dtype=np.float16,
                         state_std=0.02, capacity=32)
    _check(inp, run_gpu(inp), run_oracle(inp), fp16=True)


def test_extreme_gates_multi_token():
    """Precomputed gates at the ends of their range inside 4-token groups:
    g = 0 (the state is forgotten mid-group), g = 1e-30 (products of decays
    underflow), g = 1; beta = 0 (no write) and beta = 1."""
    inp = wl.make_inputs(630, [4, 4, 3, 4, 2], Hk=2, Hv=4, dk=128, dv=128, io_dtype=np.float32, state_std=0.02,
                         capacity=4)
    rng = np.random.default_rng(631)
    T, Hv = inp.a.shape
    g = rng.choice(np.array([0.0, 1e-30, 1e-5, 0.5, 1.0], np.float32), size=(T, Hv)).astype(np.float32)
    beta = rng.choice(np.array([0.0, 0.25, 1.0], np.float32), size=(T, Hv)).astype(np.float32)
    _check(inp, run_gpu(inp, gate_mode="precomputed", a=g, b=beta),
           run_oracle(inp, gate_mode="precomputed", a=g, b=beta), fp16=False)


def test_zero_initial_state_multi_token_fp16():
    """No initial state: the rows start at zero (no row copies are issued)."""
    inp = wl.make_inputs(640, [4, 3, 4, 2], Hk=2, Hv=6, dk=128, dv=128, io_dtype=np.float16, capacity=4)
    _check(inp, run_gpu(inp), run_oracle(inp), fp16=True)


@pytest.mark.parametrize("pad", [0, 3])
def test_d128_spans_from_fused_views(pad):
    """d = 128 (the tcgen05 short-span kernel): q, k, v as strided views of one
    fused projection [T, 2 Hk dk + Hv dv + pad] fp16.  pad = 0: the first
    group's q, k, v rows arrive by tensor copies from the strided views; pad = 3:
    the row stride (in bytes) is not a multiple of 16, so they are read with
    plain loads.  Spans: a two-group span (6 tokens, capsules for the first 4),
    full and ragged groups, one token and empty, in place."""
    import torch
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    from gpu_common import to_dev
    lengths = [6, 4, 3, 1, 0, 4, 2]
    Hk, Hv, d = 2, 4, 128
    inp = wl.make_inputs(650 + pad, lengths, Hk=Hk, Hv=Hv, dk=d, dv=d, io_dtype=np.float16, state_std=0.02,
                         capacity=4)
    T = inp.T
    width = 2 * Hk * d + Hv * d
    fused = np.zeros((T, width + pad), np.float16)
    fused[:, :Hk * d] = inp.q.reshape(T, -1)
    fused[:, Hk * d:2 * Hk * d] = inp.k.reshape(T, -1)
    fused[:, 2 * Hk * d:width] = inp.v.reshape(T, -1)
    f = to_dev(fused)
    q = f[:, :Hk * d].view(T, Hk, d) if pad == 0 else f[:, :Hk * d].unflatten(1, (Hk, d))
    k = f[:, Hk * d:2 * Hk * d].unflatten(1, (Hk, d))
    v = f[:, 2 * Hk * d:width].unflatten(1, (Hv, d))
    state = to_dev(inp.initial_state)
    out, final, caps = gdn.gdn_forward(q, k, v, to_dev(inp.a), to_dev(inp.b), to_dev(inp.cu_seqlens),
                                       A_log=to_dev(inp.A_log), dt_bias=to_dev(inp.dt_bias), initial_state=state,
                                       final_state=state, capacity=4)
    torch.cuda.synchronize()
    gpu = (out.double().cpu().numpy(), final.double().cpu().numpy(), caps.double().cpu().numpy())
    _check(inp, gpu, run_oracle(inp), fp16=True)
