"""GPU parity at the boundary's largest batch: 65,535 sequences per call (the
most `gdn_forward` and `gdn_replay_prefix` accept; it is also the decode
kernel's grid height), against the FP64 oracle.

One token per sequence at Hk = Hv = 1, dk = dv = 32 keeps the state pool at
268 MB while every sequence index, state slot and capsule row up to the
limit is exercised; a shuffled slot list checks placement far from the
identity.  Tolerances as for the FP32 recurrent path (1e-5 max-relative);
untouched slots and the replay's source bank are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import max_rel
from gpu_common import run_gpu, run_oracle, to_dev, dev

from gated_delta_rule_gateddeltanet_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

B_MAX = 65535


def test_decode_at_the_largest_batch():
    rng = np.random.default_rng(1301)
    slots = rng.permutation(B_MAX + 7)[:B_MAX].astype(np.int32)  # 7 slots stay untouched
    inp = wl.make_inputs(1301, [1] * B_MAX, Hk=1, Hv=1, dk=32, dv=32, io_dtype=np.float32, state_std=0.02,
                         num_slots=B_MAX + 7, capacity=1, state_slots=slots)
    out, final, caps = run_gpu(inp, in_place=False)
    o_ref, f_ref, c_ref = run_oracle(inp)
    assert max_rel(out, o_ref) <= 1e-5
    assert max_rel(final[slots], f_ref[slots]) <= 1e-5
    assert max_rel(caps, c_ref) <= 1e-5
    untouched = np.setdiff1d(np.arange(B_MAX + 7), slots)
    assert untouched.size == 7
    assert np.array_equal(final[untouched], inp.initial_state[untouched].astype(np.float64))


def test_replay_at_the_largest_batch():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    rng = np.random.default_rng(1302)
    Hk = Hv = 1
    d = 32
    W = gdn.capsule_width(Hk, Hv, d, d)
    caps = rng.standard_normal((B_MAX, 2, W)).astype(np.float32)
    caps[:, :, :Hv] = rng.uniform(0.5, 1.0, (B_MAX, 2, Hv))  # decays
    kn = caps[:, :, Hv:Hv + d]
    caps[:, :, Hv:Hv + d] = kn / np.linalg.norm(kn, axis=-1, keepdims=True)
    banks = (rng.standard_normal((2 * B_MAX, Hv, d, d)) * 0.02).astype(np.float32)
    src = np.arange(B_MAX, dtype=np.int32)
    dst = np.arange(B_MAX, 2 * B_MAX, dtype=np.int32)
    n = rng.integers(0, 3, B_MAX).astype(np.int32)
    bank_d = to_dev(banks)
    gdn.gdn_replay_prefix(bank_d, to_dev(src), to_dev(dst), to_dev(caps), to_dev(n), num_k_heads=Hk)
    torch.cuda.synchronize()
    got = bank_d.double().cpu().numpy()
    ref = oracle.gdn_replay(banks, src, dst, caps, n, num_k_heads=Hk)
    assert max_rel(got[dst], ref[dst]) <= 1e-5
    assert np.array_equal(got[src], banks[src].astype(np.float64))  # the committed bank is untouched
    zero = dst[n == 0]
    assert np.array_equal(got[zero], banks[src[n == 0]].astype(np.float64))  # nothing accepted: a copy
