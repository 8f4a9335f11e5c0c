"""GPU parity, against the FP64 oracle, of the fused q/k L2 normalisation at
its degenerate inputs: zero keys and queries and vectors shorter than the
clamp eps = 1e-6 (x / max(|x|, eps)), on every kernel that normalises.

The normalisation is fused into the operator ("[CUDA] Add compact
GatedDeltaNet operator", Description: fused Qwen normalisation).  A zero key
leaves kn = 0, so the delta is beta v and the state is only decayed; a zero
query gives a zero output; a sub-eps vector becomes a short, non-unit
direction.  In the chunked paths such a key travels through the fp16 key
tiles, the triangular system and the tensor-memory state, so each kernel is
driven with them:

* the CUDA-core decode kernel (every span one token),
* the tensor-core short-span kernel (spans of 2-32 tokens),
* the two-phase and the single-kernel chunked evaluations,
* the sequence-parallel split plan.

Planted rows: whole zero rows of q, of k and of both, runs of zero keys across
a chunk boundary, and sub-eps rows (fp16: entries of +-2^-24, the smallest
fp16 subnormal, norm 6.7e-7 at dk = 128, or 2^-23 on a few lanes; fp32: random
directions of norm 1e-8 and 5e-7), plus rows just above eps.  Tolerances are
the paths' own: 1e-5 max-relative for FP32 recurrent results, 2e-3 for fp16
outputs and for the tensor-core chunked paths.  A zero query's output is
checked to be exactly zero.
"""
import numpy as np
import pytest

from helpers import max_rel
from gpu_common import run_gpu, run_oracle, single_kernel_workspace

from gated_delta_rule_gateddeltanet_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL32 = 1e-5
TOL16 = 2e-3


def _plant(inp, seed, run=None):
    """Overwrites rows of q and k with zero, sub-eps and just-above-eps
    vectors; returns the token indices whose query rows are zero (per key
    head: a list of (t, kh))."""
    rng = np.random.default_rng(seed)
    T, Hk, dk = inp.q.shape
    fp16 = inp.q.dtype == np.float16
    e24 = np.float16(2.0 ** -24) if fp16 else None

    def tiny(n):
        if fp16:
            x = rng.choice([-1.0, 1.0], n) * float(e24)          # norm 2^-24 sqrt(n) < eps for n <= 128
            return x.astype(np.float16)
        d = rng.standard_normal(n)
        return (d / np.linalg.norm(d) * rng.choice([1e-8, 5e-7])).astype(np.float32)

    def sparse_tiny(n):
        x = np.zeros(n)
        idx = rng.choice(n, 3, replace=False)
        x[idx] = rng.choice([-1.0, 1.0], 3) * 2.0 ** -23      # norm 2.1e-7
        return x.astype(inp.q.dtype)

    def above(n):
        d = rng.standard_normal(n)
        x = d / np.linalg.norm(d) * 4e-6                       # four times eps: normalised as usual
        return x.astype(inp.q.dtype)

    zero_q = []
    kinds = ["zero_q", "zero_k", "zero_both", "tiny_q", "tiny_k", "sparse_tiny_k", "tiny_both", "above_k"]
    picks = rng.choice(T * Hk, size=min(T * Hk, max(8, T * Hk // 6)), replace=False)
    for i, p in enumerate(picks):
        t, kh = divmod(int(p), Hk)
        kind = kinds[i % len(kinds)]
        if kind in ("zero_q", "zero_both"):
            inp.q[t, kh] = 0
            zero_q.append((t, kh))
        if kind in ("zero_k", "zero_both"):
            inp.k[t, kh] = 0
        if kind in ("tiny_q", "tiny_both"):
            inp.q[t, kh] = tiny(dk)
        if kind in ("tiny_k", "tiny_both"):
            inp.k[t, kh] = tiny(dk)
        if kind == "sparse_tiny_k":
            inp.k[t, kh] = sparse_tiny(dk)
        if kind == "above_k":
            inp.k[t, kh] = above(dk)
    if run is not None:  # a run of zero keys (and zero queries in the middle of it)
        t0, t1 = run
        inp.k[t0:t1] = 0
        inp.q[t0 + 2:t0 + 5] = 0
        zero_q += [(t, kh) for t in range(t0 + 2, t0 + 5) for kh in range(Hk)]
    return zero_q


def _check(inp, gpu, ref, tol_out, tol_state, tol_u, zero_q):
    out, final, caps = gpu
    o_ref, f_ref, c_ref = ref
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(final))
    assert max_rel(out, o_ref) <= tol_out, max_rel(out, o_ref)
    slots = np.arange(inp.B) if inp.state_slots is None else inp.state_slots
    assert max_rel(final[slots], f_ref[slots]) <= tol_state, max_rel(final[slots], f_ref[slots])
    Hk, Hv, dk, dv = inp.dims
    r = Hv // Hk
    for t, kh in zero_q:
        assert np.all(out[t, kh * r:(kh + 1) * r] == 0.0), (t, kh)
    if caps is not None and inp.capacity > 0:
        lens = np.diff(inp.cu_seqlens)
        for s in range(inp.B):
            n = min(int(lens[s]), inp.capacity)
            if not n:
                continue
            W0 = Hv + Hk * dk
            assert max_rel(caps[s, :n, :Hv], c_ref[s, :n, :Hv]) <= 1e-5
            assert max_rel(caps[s, :n, Hv:W0], c_ref[s, :n, Hv:W0]) <= 1e-5
            assert max_rel(caps[s, :n, W0:], c_ref[s, :n, W0:]) <= tol_u, max_rel(caps[s, :n, W0:],
                                                                                   c_ref[s, :n, W0:])


@pytest.mark.parametrize("io", [np.float16, np.float32])
def test_decode_kernel_zero_and_tiny_rows(io):
    inp = wl.make_inputs(1201, [1] * 24, Hk=2, Hv=6, dk=128, dv=128, io_dtype=io, state_std=0.02, capacity=1)
    zq = _plant(inp, 1)
    fp16 = io == np.float16
    _check(inp, run_gpu(inp, in_place=False), run_oracle(inp), TOL16 if fp16 else TOL32, TOL32, TOL32, zq)


@pytest.mark.parametrize("io", [np.float16, np.float32])
def test_short_span_kernel_zero_and_tiny_rows(io):
    lengths = [4, 4, 1, 17, 32, 2, 0, 9]
    inp = wl.make_inputs(1202, lengths, Hk=2, Hv=6, dk=128, dv=128, io_dtype=io, state_std=0.02, capacity=8)
    zq = _plant(inp, 2, run=(9, 17))  # zero keys across the 17-token span's groups
    fp16 = io == np.float16
    _check(inp, run_gpu(inp, in_place=False), run_oracle(inp), TOL16 if fp16 else TOL32, TOL32, TOL32, zq)


@pytest.mark.parametrize("path", ["two_phase", "single_kernel"])
@pytest.mark.parametrize("io", [np.float16, np.float32])
def test_chunked_paths_zero_and_tiny_rows(io, path):
    lengths = [130, 65, 7, 64]
    inp = wl.make_inputs(1203, lengths, Hk=2, Hv=6, dk=128, dv=128, io_dtype=io, state_std=0.02, capacity=70)
    zq = _plant(inp, 3, run=(56, 72))  # a run of zero keys across the first chunk boundary
    ws = single_kernel_workspace(inp) if path == "single_kernel" else None
    _check(inp, run_gpu(inp, plan="chunked", in_place=False, workspace=ws), run_oracle(inp),
           TOL16, TOL16, TOL16, zq)


def test_split_plan_zero_and_tiny_rows():
    lengths = [2100, 300]  # the first sequence is split into halves
    inp = wl.make_inputs(1204, lengths, Hk=2, Hv=4, dk=128, dv=128, io_dtype=np.float16, state_std=0.05)
    zq = _plant(inp, 4, run=(1080, 1100))  # zero keys where the second half starts
    _check(inp, run_gpu(inp, plan="chunked_split", in_place=False), run_oracle(inp), TOL16, TOL16, TOL16, zq)
