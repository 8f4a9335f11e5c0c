"""Debug builds (GDN_DEBUG_CHECKS): the precondition that one call's requests
use distinct state slots is checked on the device and reported as
GDN_DEVERR_DUP_SLOT; distinct slots raise nothing, and the results are those
of the release library bit for bit (the check launches ahead of the work and
changes none of it)."""
import numpy as np
import pytest
import torch

from gpu_common import dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    from gated_delta_rule_gateddeltanet_gb300 import build
    return gdn.load_library(build.build(debug=True))


@pytest.fixture
def use_debug(debug_lib, monkeypatch):
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    gdn.load_library()  # the release library stays loaded for comparisons
    release = gdn._lib
    monkeypatch.setattr(gdn, "_lib", debug_lib)
    return release


def _forward_inputs(seed, lengths, Hk=2, Hv=4, d=32):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    q = rng.standard_normal((T, Hk, d)).astype(np.float32)
    k = rng.standard_normal((T, Hk, d)).astype(np.float32)
    v = rng.standard_normal((T, Hv, d)).astype(np.float32)
    a = rng.standard_normal((T, Hv)).astype(np.float32)
    b = rng.standard_normal((T, Hv)).astype(np.float32)
    A_log = np.log(rng.uniform(1, 16, Hv)).astype(np.float32)
    dt_bias = np.log(np.expm1(rng.uniform(1e-3, 0.1, Hv))).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return [to_dev(x) for x in (q, k, v, a, b, cu, A_log, dt_bias)]


def _forward(gdn, slots, S=6, lengths=(3, 1, 5)):
    q, k, v, a, b, cu, A_log, dt_bias = _forward_inputs(90, list(lengths))
    Hv, d = v.shape[1], v.shape[2]
    init = to_dev(np.random.default_rng(91).standard_normal((S, Hv, d, d)).astype(np.float32) * 0.02)
    final = init.clone()
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    out, fin, _ = gdn.gdn_forward(q, k, v, a, b, cu, A_log=A_log, dt_bias=dt_bias, initial_state=init,
                                  final_state=final, state_slots=to_dev(np.array(slots, np.int32)),
                                  num_state_slots=S, status=status)
    torch.cuda.synchronize()
    return out, fin, status.item()


def test_forward_duplicate_slots_flagged(use_debug, monkeypatch):
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    _, _, st = _forward(gdn, [4, 1, 4])
    assert st == gdn.DEVERR["dup_slot"]
    out, fin, st = _forward(gdn, [4, 1, 0])
    assert st == 0
    monkeypatch.setattr(gdn, "_lib", use_debug)  # the release library
    ref_out, ref_fin, st = _forward(gdn, [4, 1, 0])
    assert st == 0
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)


def test_replay_duplicate_destinations_flagged(use_debug):
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    Hk, Hv, d, cap, R = 1, 2, 32, 3, 3
    W = gdn.capsule_width(Hk, Hv, d, d)
    rng = np.random.default_rng(92)
    banks = to_dev(rng.standard_normal((8, Hv, d, d)).astype(np.float32))
    caps = to_dev(rng.standard_normal((R, cap, W)).astype(np.float32) * 0.1)
    n = to_dev(np.array([1, 2, 0], np.int32))
    for src, dst, want in (([0, 1, 2], [5, 6, 5], True),   # two requests write slot 5
                           ([0, 1, 2], [5, 0, 7], True),   # request 1 writes slot 0, which request 0 reads
                           ([0, 1, 2], [0, 6, 7], False),  # a request may replay onto its own source
                           ([0, 1, 2], [5, 6, 7], False)):
        status = torch.zeros(1, dtype=torch.int32, device=dev())
        gdn.gdn_replay_prefix(banks.clone(), to_dev(np.array(src, np.int32)), to_dev(np.array(dst, np.int32)), caps,
                              n, num_k_heads=Hk, status=status)
        torch.cuda.synchronize()
        assert status.item() == (gdn.DEVERR["dup_slot"] if want else 0), (src, dst)


def test_conv_and_conv_replay_duplicate_slots_flagged(use_debug):
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    rng = np.random.default_rng(93)
    C, K = 64, 4
    x = to_dev(rng.standard_normal((5, C)).astype(np.float16))
    w = to_dev(rng.standard_normal((C, K)).astype(np.float32))
    cu = to_dev(np.array([0, 2, 3, 5], np.int32))
    for slots, want in (([1, 3, 1], True), ([1, 3, 0], False)):
        for hint in (0, 2):  # token-block and short-sequence kernels
            st = to_dev(rng.standard_normal((4, C, K - 1)).astype(np.float16))
            status = torch.zeros(1, dtype=torch.int32, device=dev())
            gdn.varlen_causal_conv_with_state(x, w, cu, initial_state=st, final_state=st, capacity=2,
                                              state_slots=to_dev(np.array(slots, np.int32)), status=status,
                                              num_state_slots=4, max_seqlen=hint)
            torch.cuda.synchronize()
            assert status.item() == (gdn.DEVERR["dup_slot"] if want else 0), (slots, hint)
    states = to_dev(rng.standard_normal((6, C, K - 1)).astype(np.float16))
    vals = to_dev(rng.standard_normal((2, 2, C)).astype(np.float16))
    n = to_dev(np.array([1, 2], np.int32))
    for dst, want in (([4, 4], True), ([4, 5], False)):
        status = torch.zeros(1, dtype=torch.int32, device=dev())
        gdn.causal_conv_replay_prefix(states, to_dev(np.array([0, 1], np.int32)), to_dev(np.array(dst, np.int32)),
                                      vals, n, status=status)
        torch.cuda.synchronize()
        assert status.item() == (gdn.DEVERR["dup_slot"] if want else 0), dst
