"""CPU-side checks of the C ABI: the library builds and loads, exports every
entry point include/gdn.h declares, the ctypes mirror of gdn_forward_args has
the C layout, and host-visible argument errors return before any launch.
No call here reaches a kernel."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_gateddeltanet_gb300 import build
    build.build()
    import gated_delta_rule_gateddeltanet_gb300 as g
    return g.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gdn_forward", "gdn_forward_workspace_size", "gdn_replay_prefix", "gdn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)


def test_debug_library_builds_and_exports_every_declared_symbol(lib):
    """libgdn_debug.so (the precondition checks of GDN_DEBUG_CHECKS) builds
    from the same sources and exports the same entry points."""
    from gated_delta_rule_gateddeltanet_gb300 import build
    path = build.build(debug=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in declared_functions():
        assert n in exported, n


def test_forward_args_layout_matches_c(tmp_path):
    import gated_delta_rule_gateddeltanet_gb300 as g
    fields = [f for f, _ in g.ForwardArgs._fields_]
    src = tmp_path / "layout.c"
    body = "\n".join(f'printf("{f} %zu\\n", offsetof(gdn_forward_args, {f}));' for f in fields)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gdn.h"\nint main(void){\n'
                   + body + '\nprintf("sizeof %zu\\n", sizeof(gdn_forward_args));\nreturn 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    for f in fields:
        assert int(got[f]) == getattr(g.ForwardArgs, f).offset, f
    assert int(got["sizeof"]) == ctypes.sizeof(g.ForwardArgs)


def _args(**kw):
    import gated_delta_rule_gateddeltanet_gb300 as g
    a = g.ForwardArgs()
    a.num_seqs, a.total_tokens, a.num_k_heads, a.num_v_heads = 2, 4, 16, 48
    a.head_dim_k = a.head_dim_v = 128
    a.num_state_slots, a.io_dtype = 2, 1
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: every case below fails its host check first
    for f in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "cu_seqlens", "final_state", "output"):
        setattr(a, f, fake)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(io_dtype=2), 2),                   # BF16 rejected
    (dict(io_dtype=7), 2),
    (dict(num_v_heads=40), 3),               # Hv not a multiple of Hk
    (dict(head_dim_k=96), 3),
    (dict(head_dim_v=256), 3),
    (dict(state_update_capacity=-1), 3),
    (dict(num_state_slots=1), 3),            # identity slots need >= B slots
    (dict(q_stride=100), 3),                 # shorter than Hk*dk
    (dict(scale=float("nan")), 3),
    (dict(gate_mode=5), 8),
    (dict(plan=9), 8),
    (dict(A_log=None), 1),                   # raw gates need A_log and dt_bias
    (dict(cu_seqlens=None), 1),             # (final_state may be NULL: no state is written)
    (dict(state_update_capacity=4), 1),      # capsules requested without a buffer
    (dict(final_state=ctypes.c_void_p(0x1004)), 4),
])
def test_forward_rejects_bad_arguments_before_launch(lib, kw, code):
    a = _args(**kw)
    assert lib.gdn_forward(ctypes.byref(a), None) == code


def test_forward_null_args_and_workspace_query(lib):
    assert lib.gdn_forward(None, None) == 1
    a = _args()
    n = ctypes.c_size_t(123)
    assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
    assert n.value >= 0
    assert lib.gdn_forward_workspace_size(ctypes.byref(a), None) == 1


def test_empty_batch_is_a_no_op(lib):
    a = _args(num_seqs=0, total_tokens=0)
    assert lib.gdn_forward(ctypes.byref(a), None) == 0


def test_replay_rejects_bad_arguments(lib):
    f = lib.gdn_replay_prefix
    fake = ctypes.c_void_p(0x1000)
    assert f(fake, 4, 2, 16, 40, 128, 128, fake, fake, fake, 4, fake, None, None) == 3
    assert f(fake, 4, 2, 16, 48, 128, 100, fake, fake, fake, 4, fake, None, None) == 3
    assert f(None, 4, 2, 16, 48, 128, 128, fake, fake, fake, 4, fake, None, None) == 1
    assert f(fake, 4, 2, 16, 48, 128, 128, fake, fake, None, 4, fake, None, None) == 1
    assert f(ctypes.c_void_p(0x1008), 4, 2, 16, 48, 128, 128, fake, fake, fake, 4, fake, None, None) == 4
    assert f(fake, 4, 0, 16, 48, 128, 128, None, None, None, 0, None, None, None) == 0


def test_status_strings(lib):
    for code in range(9):
        assert lib.gdn_status_string(code)
    assert lib.gdn_status_string(99) == b"unknown status"


def test_capsule_width_matches_pages_geometry():
    import gated_delta_rule_gateddeltanet_gb300 as g
    # 48 value heads, 16 key heads, d = 128: 8240 floats = 32,960 bytes per token-layer
    assert g.capsule_width(16, 48, 128, 128) * 4 == 32960


def test_workspace_size_follows_the_plan(lib):
    n = ctypes.c_size_t(0)
    # decode-sized batch (T <= 32): recurrent only, no workspace
    a = _args(num_seqs=16, total_tokens=16, num_state_slots=16)
    assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0 and n.value == 0
    # long batch at d = 128: the two-phase chunked evaluation may run -> a header
    # ((7 + 8B) int32 rounded up to 1 KiB) plus, for each of at most T/64 + B
    # chunks, a 32 KiB record per key head and a 17,408-byte record per value head
    def two_phase(B, T, Hk, Hv):
        return ((7 + 8 * B) * 4 + 1023) // 1024 * 1024 + (T // 64 + B) * (Hk * 32768 + Hv * 17408)
    a = _args(num_seqs=8, total_tokens=17000, num_state_slots=8)
    assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
    assert n.value == two_phase(8, 17000, a.num_k_heads, a.num_v_heads)
    a = _args(num_seqs=100, total_tokens=17000, num_state_slots=100)
    assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
    assert n.value == two_phase(100, 17000, a.num_k_heads, a.num_v_heads)
    # the varlen prefill geometry (8 sequences, 15,991 tokens, Hk=16, Hv=48): ~414 MB
    a = _args(num_seqs=8, total_tokens=15991, num_state_slots=8, num_k_heads=16, num_v_heads=48)
    assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
    assert n.value == 1024 + 257 * (16 * 32768 + 48 * 17408)
    # a max_seqlen hint of at most 32 keeps the batch recurrent
    a = _args(num_seqs=64, total_tokens=64, num_state_slots=64, max_seqlen=1)
    assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0 and n.value == 0
    # forced recurrent plan: none
    a = _args(num_seqs=8, total_tokens=17000, num_state_slots=8, plan=1)
    assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0 and n.value == 0
    # head sizes 32 / 64 run the same two-phase evaluation on zero-padded tiles: the same records
    for dk, dv in ((64, 128), (32, 32), (128, 64)):
        a = _args(num_seqs=8, total_tokens=17000, num_state_slots=8, head_dim_k=dk, head_dim_v=dv)
        assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
        assert n.value == two_phase(8, 17000, a.num_k_heads, a.num_v_heads)


def test_split_plan_workspace_and_restrictions(lib):
    n = ctypes.c_size_t(0)
    base = ((7 + 8 * 8) * 4 + 1023) // 1024 * 1024 + (17000 // 64 + 8) * (16 * 32768 + 48 * 17408)
    # + three FP32 states per value head for each sequence that can be split
    # (at most min(B, T / 1985)) + T/2 + 64 rows of identity-run outputs
    for io, esz in ((1, 2), (0, 4)):
        a = _args(num_seqs=8, total_tokens=17000, num_state_slots=8, plan=3, io_dtype=io)
        assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
        assert n.value == base + 8 * 3 * 48 * 128 * 128 * 4 + (17000 // 2 + 64) * 48 * 128 * esz
    # too short to split anything: the plain two-phase size
    a = _args(num_seqs=2, total_tokens=1984, num_state_slots=2, plan=3)
    assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
    assert n.value == 1024 + (1984 // 64 + 2) * (16 * 32768 + 48 * 17408)
    assert lib.gdn_forward(ctypes.byref(_args(plan=3, head_dim_k=64)), None) == 5  # runs unsplit: needs workspace
    # below 128 nothing is split: the plain two-phase size
    a = _args(num_seqs=8, total_tokens=17000, num_state_slots=8, plan=3, head_dim_k=64, head_dim_v=64)
    assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0 and n.value == base
    # capsules are allowed (captured tokens come from first halves); this call has no workspace
    assert lib.gdn_forward(ctypes.byref(_args(plan=3, state_update_capacity=4, state_update=ctypes.c_void_p(0x1000))),
                           None) == 5
    assert lib.gdn_forward(ctypes.byref(_args(plan=3)), None) == 5                            # no workspace
    assert lib.gdn_forward(ctypes.byref(_args(plan=4)), None) == 8
    # the no-alloc entry has no form of the split plan: refused before any lookup or launch
    assert lib.gdn_forward_no_alloc(ctypes.byref(_args(plan=3)), None) == 7
    assert lib.gdn_forward_no_alloc(ctypes.byref(_args(plan=3, num_seqs=1, total_tokens=3000,
                                                       num_state_slots=1)), None) == 7


def test_forced_chunked_plan_needs_workspace(lib):
    # every head size has the two-phase form; without its workspace a forced plan is refused
    assert lib.gdn_forward(ctypes.byref(_args(plan=2, head_dim_k=64)), None) == 5
    assert lib.gdn_forward(ctypes.byref(_args(plan=2, head_dim_v=32)), None) == 5
    assert lib.gdn_forward(ctypes.byref(_args(max_seqlen=-1)), None) == 3
    # forced chunked plan without workspace
    assert lib.gdn_forward(ctypes.byref(_args(plan=2)), None) == 5


def _conv_args(**kw):
    import gated_delta_rule_gateddeltanet_gb300 as g
    a = g.ConvArgs()
    a.num_seqs, a.total_tokens, a.channels, a.kernel_size = 2, 8, 10240, 4
    a.num_state_slots, a.io_dtype, a.activation = 2, 1, 1
    fake = ctypes.c_void_p(0x1000)
    for f in ("x", "weight", "cu_seqlens", "final_state", "output"):
        setattr(a, f, fake)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(io_dtype=2), 2),                 # BF16 rejected
    (dict(channels=10), 3),                # not a multiple of 8 fp16 channels
    (dict(kernel_size=5), 3),
    (dict(kernel_size=1), 3),
    (dict(state_update_capacity=-1), 3),
    (dict(x_stride=100), 3),
    (dict(num_state_slots=1), 3),
    (dict(activation=3), 8),
    (dict(weight=None), 1),
    (dict(cu_seqlens=None), 1),
    (dict(state_update_capacity=2), 1),    # capture requested without a buffer
    (dict(x=ctypes.c_void_p(0x1008)), 4),
    (dict(x_stride=10244), 4),             # 10244 fp16 = 20488 bytes, not a multiple of 16
])
def test_conv_rejects_bad_arguments_before_launch(lib, kw, code):
    a = _conv_args(**kw)
    assert lib.varlen_causal_conv_with_state(ctypes.byref(a), None) == code


def test_conv_args_layout_matches_c(tmp_path):
    import gated_delta_rule_gateddeltanet_gb300 as g
    fields = [f for f, _ in g.ConvArgs._fields_]
    src = tmp_path / "layout.c"
    body = "\n".join(f'printf("{f} %zu\\n", offsetof(gdn_conv_args, {f}));' for f in fields)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gdn.h"\nint main(void){\n'
                   + body + '\nprintf("sizeof %zu\\n", sizeof(gdn_conv_args));\nreturn 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    for f in fields:
        assert int(got[f]) == getattr(g.ConvArgs, f).offset, f
    assert int(got["sizeof"]) == ctypes.sizeof(g.ConvArgs)


def test_conv_replay_rejects_bad_arguments(lib):
    f = lib.causal_conv_replay_prefix
    fake = ctypes.c_void_p(0x1000)
    assert f(fake, 4, 2, 10240, 4, 2, fake, fake, fake, 4, fake, None, None) == 2
    assert f(fake, 4, 2, 10, 4, 1, fake, fake, fake, 4, fake, None, None) == 3
    assert f(fake, 4, 2, 10240, 7, 1, fake, fake, fake, 4, fake, None, None) == 3
    assert f(None, 4, 2, 10240, 4, 1, fake, fake, fake, 4, fake, None, None) == 1
    assert f(fake, 4, 2, 10240, 4, 1, fake, fake, None, 4, fake, None, None) == 1
    assert f(fake, 4, 0, 10240, 4, 1, None, None, None, 0, None, None, None) == 0


def test_dense_and_transpose_reject_bad_arguments_before_launch(lib):
    # rank-4 entry point: cu_seqlens must be absent, and B * S must equal T
    a = _args(num_seqs=2, total_tokens=8)
    assert lib.gdn_forward_dense(ctypes.byref(a), 4, None) == 8          # cu_seqlens given
    a.cu_seqlens = None
    assert lib.gdn_forward_dense(ctypes.byref(a), 3, None) == 3          # 2 x 3 != 8
    assert lib.gdn_forward_dense(ctypes.byref(a), -1, None) == 3
    assert lib.gdn_forward_dense(None, 4, None) == 1
    a = _args(num_seqs=2, total_tokens=8, io_dtype=2)
    a.cu_seqlens = None
    assert lib.gdn_forward_dense(ctypes.byref(a), 4, None) == 2          # BF16 still rejected
    a = _args(num_seqs=0, total_tokens=0)
    a.cu_seqlens = None
    assert lib.gdn_forward_dense(ctypes.byref(a), 5, None) == 0          # empty batch: nothing to do
    # state transpose
    P = ctypes.c_void_p
    assert lib.gdn_state_transpose(P(0x1000), P(0x100000), -1, 128, 128, None) == 3
    assert lib.gdn_state_transpose(P(0x1000), P(0x100000), 0, 128, 128, None) == 0   # nothing to move
    assert lib.gdn_state_transpose(None, P(0x100000), 4, 128, 128, None) == 1
    # 4 matrices of 128 x 128 floats = 256 KiB: destinations inside that range overlap the source
    assert lib.gdn_state_transpose(P(0x100000), P(0x100000 + 4096), 4, 128, 128, None) == 8


def test_split_workspace_bounds_hold_for_any_lengths(lib):
    """The split plan's workspace holds three states per head for at most
    min(B, T / 1985) split sequences and T/2 + 64 identity-run rows: for any
    mix of lengths, the sequences the rule splits (32 or more chunks, cut
    after ceil(chunks / 2)) stay within both, and gdn_forward_workspace_size
    reports exactly that room."""
    rng = __import__("numpy").random.default_rng(17)
    n = ctypes.c_size_t(0)
    cases = [[1985] * 7, [1984] * 9, [64 * 33 + 1, 1985, 3], [262144], [4096, 4095, 4097, 1]]
    cases += [list(rng.integers(0, 9000, rng.integers(1, 40))) for _ in range(200)]
    for lengths in cases:
        B, T = len(lengths), int(sum(lengths))
        if T == 0:
            continue
        chunks = [(L + 63) // 64 for L in lengths]
        split = [c >= 32 for c in chunks]
        seg2 = sum(L - 64 * ((c + 1) // 2) for L, c, s in zip(lengths, chunks, split) if s)
        nsplit = sum(split)
        max_split = min(B, T // (64 * 31 + 1))
        assert nsplit <= max_split, lengths
        assert seg2 <= T // 2 + 64, lengths
        a = _args(num_seqs=B, total_tokens=T, num_state_slots=B, plan=3)
        assert lib.gdn_forward_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
        base = ((7 + 8 * B) * 4 + 1023) // 1024 * 1024 + (T // 64 + B) * (16 * 32768 + 48 * 17408)
        extra = max_split * 3 * 48 * 128 * 128 * 4 + (T // 2 + 64) * 48 * 128 * 2 if max_split > 0 else 0
        assert n.value == base + extra, lengths
