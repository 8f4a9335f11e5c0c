"""GatedDeltaNet oracle: plain FP64 CPU evaluation of the gated delta rule.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package entry point's smoke
check and the benchmark's CPU-baseline leg import this package.  The product
path (the CUDA library and its Python binding) never imports, loads or calls
it, and the two share no code: the arithmetic lives in ``gdn_oracle.c``
(compiled here with gcc, nothing from the CUDA build) and in ``chunked.py``.

What each function follows (page title, then section):

* ``gdn_forward`` -- the per-token gated delta rule with native Qwen gate
  arithmetic, the V-major FP32 state and the three outputs
  ``[output, final_state, state_update]`` ("[CUDA] Add compact GatedDeltaNet
  operator", Description; "Add GatedDeltaNet evaluation export for Qwen hybrid
  models", What changed).
* ``gdn_replay`` -- replay of an accepted capsule prefix into an inactive bank
  ("Replay compact fixed state for hybrid decoding", Summary, Key changes).
* ``conv_forward`` / ``conv_replay`` -- the packed depthwise causal
  convolution with carried state and compact value capture ("[CUDA] Add
  compact GatedDeltaNet operator", embedded commit "Add compact
  VarlenCausalConv state updates", Description).

Pins (tests/test_oracle_*.py): an exact rational brute force of the unrolled
transition on tiny inputs, exact-gate special cases, the invariants (identity
gates, orthonormal keys, pack vs. one-by-one, chunked vs. sequential, replay
vs. sequential state), pure decay, and the pages' 576 MiB footprint.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (FP64, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
               "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32 = ctypes.c_int
            lib.gdn_oracle_forward.restype = i32
            lib.gdn_oracle_forward.argtypes = [i32] * 7 + [P] * 7 + [i32, ctypes.c_double] + [P] * 6 + [i32]
            lib.gdn_oracle_replay.restype = i32
            lib.gdn_oracle_replay.argtypes = [P, i32, i32, i32, i32, i32, i32, P, P, P, i32, P]
            lib.conv_oracle_forward.restype = i32
            lib.conv_oracle_forward.argtypes = [i32] * 5 + [P] * 8 + [i32, P]
            lib.gdn_oracle_threads.restype = i32
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all host cores)."""
    return int(_load().gdn_oracle_threads())


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def gdn_forward(q, k, v, a, b, cu_seqlens, *, A_log=None, dt_bias=None, gate_mode="raw",
                scale=None, initial_state=None, state_slots=None, num_state_slots=None,
                capacity=0):
    """FP64 gated delta rule over packed varlen tokens.

    q, k: [T, Hk, dk]; v: [T, Hv, dv]; a, b: [T, Hv] (raw gate inputs, or the
    effective decay and beta when ``gate_mode="precomputed"``); A_log, dt_bias:
    [Hv]; cu_seqlens: [B+1]; initial_state: [slots, Hv, dv, dk] or None (zeros);
    state_slots: [B] or None (identity).  Inputs are widened exactly to FP64.

    Returns ``(output [T,Hv,dv], final_state [slots,Hv,dv,dk],
    state_update [B,capacity,W] or None)``, all FP64.  Capsule rows that no
    token fills are NaN.
    """
    q, k, v, a, b = (_f64(x) for x in (q, k, v, a, b))
    cu = _i32(cu_seqlens)
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    B = cu.shape[0] - 1
    slots = _i32(state_slots)
    if num_state_slots is None:
        num_state_slots = initial_state.shape[0] if initial_state is not None else B
    init = _f64(initial_state)
    final = np.zeros((num_state_slots, Hv, dv, dk)) if init is None else init.copy()
    out = np.zeros((T, Hv, dv))
    W = Hv + Hk * dk + Hv * dv
    caps = np.full((B, capacity, W), np.nan) if capacity > 0 else None
    mode = {"raw": 0, "precomputed": 1}[gate_mode]
    if mode == 0 and (A_log is None or dt_bias is None):
        raise OracleError("raw gates need A_log and dt_bias")
    A_log = _f64(A_log)
    dt_bias = _f64(dt_bias)
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(dk)
    rc = _load().gdn_oracle_forward(B, T, Hk, Hv, dk, dv, num_state_slots, _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), mode, float(scale),
                                    _ptr(cu), _ptr(slots), _ptr(init), _ptr(final), _ptr(out),
                                    _ptr(caps), int(capacity))
    if rc != 0:
        raise OracleError(f"gdn_oracle_forward failed with code {rc}")
    return out, final, caps


def gdn_replay(banks, src_slots, dst_slots, capsules, accept_len, *, num_k_heads):
    """FP64 prefix replay; returns the updated banks (a new array).

    banks: [slots, Hv, dv, dk]; capsules: [R, cap, W]; accept_len: [R] in [0, cap].
    """
    banks = _f64(banks).copy()
    caps = _f64(capsules)
    src, dst, n = _i32(src_slots), _i32(dst_slots), _i32(accept_len)
    S, Hv, dv, dk = banks.shape
    R, cap, _ = caps.shape
    rc = _load().gdn_oracle_replay(_ptr(banks), S, R, int(num_k_heads), Hv, dk, dv, _ptr(src), _ptr(dst),
                                   _ptr(caps), cap, _ptr(n))
    if rc != 0:
        raise OracleError(f"gdn_oracle_replay failed with code {rc}")
    return banks


def conv_forward(x, w, cu_seqlens, conv_state, *, bias=None, state_slots=None, capacity=0, capture_count=None):
    """FP64 packed depthwise causal conv + SiLU with carried state.

    x: [T, C]; w: [C, K]; conv_state: [slots, C, K-1] (oldest first);
    capture_count: optional [B], each in [0, capacity].
    Returns ``(out [T,C], new_conv_state, values [B,cap,C] or None)``; capture
    rows that no token fills are NaN.
    """
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    cu, slots = _i32(cu_seqlens), _i32(state_slots)
    cc = _i32(capture_count)
    T, C = x.shape
    K = w.shape[1]
    state = _f64(conv_state).copy()
    B = cu.shape[0] - 1
    out = np.zeros((T, C))
    values = np.full((B, capacity, C), np.nan) if capacity > 0 else None
    rc = _load().conv_oracle_forward(B, T, C, K, state.shape[0], _ptr(x), _ptr(w), _ptr(bias), _ptr(cu),
                                     _ptr(slots), _ptr(state), _ptr(out), _ptr(values), int(capacity), _ptr(cc))
    if rc != 0:
        raise OracleError(f"conv_oracle_forward failed with code {rc}")
    return out, state, values


def conv_replay(conv_states, src_slots, dst_slots, values, accept_len):
    """Replay of the compact conv capture: the new state is the last K-1 entries
    of (state of src, followed by the first n captured inputs).  Plain Python."""
    st = _f64(conv_states).copy()
    vals = _f64(values)
    out = st.copy()
    Km1 = st.shape[2]
    for j, (s, d, n) in enumerate(zip(src_slots, dst_slots, accept_len)):
        hist = np.concatenate([st[s], vals[j, :n, :].T], axis=1)  # [C, Km1 + n]
        out[d] = hist[:, hist.shape[1] - Km1:]
    return out


def capsule_width(Hk: int, Hv: int, dk: int, dv: int) -> int:
    """Floats per captured token: decay per value head, shared key per key head,
    delta per value head."""
    return Hv + Hk * dk + Hv * dv
