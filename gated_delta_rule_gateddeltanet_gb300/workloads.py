"""Seeded synthetic inputs for the GatedDeltaNet path.

This module only draws random numbers (numpy ``default_rng``); it holds none of
the method's arithmetic.  The same host arrays feed the CUDA path and the FP64
oracle.  Distributions follow the workloads of the pages' operator: packed THD
q/k/v ~ N(0, 1); raw gate inputs a, b ~ N(0, 1) in FP32; per-head
A_log = log(U(1, 16)) and dt_bias = log(expm1(U(1e-3, 0.1))) (the inverse
softplus of a small positive step); FP32 V-major states ~ N(0, 0.02^2).

Named workloads (sizes as in the docstrings of each function):
``pr_ref`` (T=64, 2 heads, d=32, fp32), ``decode_step`` (64 x 1 token,
Hk=16, Hv=48, d=128, fp16), ``varlen_prefill`` (8 sequences of U[256, 4096]
tokens), ``spec_verify`` (16 x 4 draft tokens + accepted prefixes U{0..4}),
``serving_mix`` (32 x 2048-token prefill, then 256 decode steps).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEEDS = {"pr_ref": 1001, "decode_step": 1002, "varlen_prefill": 1003, "spec_verify": 1004,
         "serving_mix": 1005}


@dataclass
class GdnInputs:
    q: np.ndarray            # [T, Hk, dk] io dtype
    k: np.ndarray            # [T, Hk, dk]
    v: np.ndarray            # [T, Hv, dv]
    a: np.ndarray            # [T, Hv] float32 raw
    b: np.ndarray            # [T, Hv] float32 raw
    A_log: np.ndarray        # [Hv] float32
    dt_bias: np.ndarray      # [Hv] float32
    cu_seqlens: np.ndarray   # [B+1] int32
    initial_state: np.ndarray | None  # [slots, Hv, dv, dk] float32 or None
    state_slots: np.ndarray | None = None
    capacity: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def T(self):
        return self.q.shape[0]

    @property
    def B(self):
        return self.cu_seqlens.shape[0] - 1

    @property
    def dims(self):
        return self.q.shape[1], self.v.shape[1], self.q.shape[2], self.v.shape[2]


def _normal(rng, shape, dtype):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return x.astype(dtype, copy=False)


def cu_from_lengths(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu


def gate_params(rng, Hv):
    A_log = np.log(rng.uniform(1.0, 16.0, size=Hv)).astype(np.float32)
    dt_bias = np.log(np.expm1(rng.uniform(1e-3, 0.1, size=Hv))).astype(np.float32)
    return A_log, dt_bias


def make_inputs(seed, lengths, *, Hk, Hv, dk, dv, io_dtype=np.float16, state_std=None,
                num_slots=None, capacity=0, state_slots=None) -> GdnInputs:
    """Draw one packed batch.  ``state_std=None`` means a zero (absent) initial state."""
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in lengths]
    T = int(sum(lengths))
    B = len(lengths)
    q = _normal(rng, (T, Hk, dk), io_dtype)
    k = _normal(rng, (T, Hk, dk), io_dtype)
    v = _normal(rng, (T, Hv, dv), io_dtype)
    a = _normal(rng, (T, Hv), np.float32)
    b = _normal(rng, (T, Hv), np.float32)
    A_log, dt_bias = gate_params(rng, Hv)
    slots = num_slots if num_slots is not None else B
    init = None
    if state_std is not None:
        init = (rng.standard_normal(size=(slots, Hv, dv, dk), dtype=np.float32) * np.float32(state_std))
    ss = None if state_slots is None else np.asarray(state_slots, dtype=np.int32)
    return GdnInputs(q, k, v, a, b, A_log, dt_bias, cu_from_lengths(lengths), init, ss, capacity)


def pr_ref(seed=SEEDS["pr_ref"]) -> GdnInputs:
    """1 sequence, T=64, Hk=Hv=2, dk=dv=32, fp32 I/O, zero initial state,
    capsules for all 64 tokens."""
    return make_inputs(seed, [64], Hk=2, Hv=2, dk=32, dv=32, io_dtype=np.float32, capacity=64)


def decode_step(seed=SEEDS["decode_step"], requests=64) -> GdnInputs:
    """64 requests x 1 token, Hk=16, Hv=48, dk=dv=128, fp16 q/k/v, random
    FP32 state N(0, 0.02^2) of shape [64, 48, 128, 128]."""
    return make_inputs(seed, [1] * requests, Hk=16, Hv=48, dk=128, dv=128, io_dtype=np.float16,
                       state_std=0.02)


def varlen_prefill_lengths(seed=SEEDS["varlen_prefill"], n=8):
    return np.random.default_rng(seed).integers(256, 4097, n)


def varlen_prefill(seed=SEEDS["varlen_prefill"]) -> GdnInputs:
    """8 packed sequences with lengths U[256, 4096], Hk=16, Hv=48, d=128, fp16,
    zero initial state (chunk size 64 on the tensor-core path)."""
    lengths = varlen_prefill_lengths(seed)
    return make_inputs(seed + 1, lengths, Hk=16, Hv=48, dk=128, dv=128, io_dtype=np.float16)


def spec_verify(seed=SEEDS["spec_verify"], requests=16, draft=4) -> GdnInputs:
    """16 requests x 4 draft tokens (T=64), Hk=16, Hv=48, d=128, fp16, random
    committed FP32 state, capsules for every draft token.  ``extra`` holds the
    accepted prefix lengths U{0..4} and the source/destination banks of the
    replay: committed bank = slots [0, 16), inactive bank = slots [16, 32)."""
    inp = make_inputs(seed, [draft] * requests, Hk=16, Hv=48, dk=128, dv=128, io_dtype=np.float16,
                      state_std=0.02, num_slots=2 * requests, capacity=draft,
                      state_slots=np.arange(requests))
    rng = np.random.default_rng(seed + 7)
    inp.extra["accept_len"] = rng.integers(0, draft + 1, requests).astype(np.int32)
    inp.extra["src_slots"] = np.arange(requests, dtype=np.int32)
    inp.extra["dst_slots"] = np.arange(requests, 2 * requests, dtype=np.int32)
    return inp


def serving_mix_prefill(seed=SEEDS["serving_mix"], sequences=32, length=2048) -> GdnInputs:
    """32 x 2048-token packed fp16 prefill, Hk=16, Hv=48, d=128, zero initial state."""
    return make_inputs(seed, [length] * sequences, Hk=16, Hv=48, dk=128, dv=128, io_dtype=np.float16)


def serving_mix_decode(step, prefill: GdnInputs, seed=SEEDS["serving_mix"]) -> GdnInputs:
    """Fresh single-token inputs for decode step ``step`` (0..255) of the serving
    mix, one token per sequence of ``prefill``.  The per-head gate parameters
    belong to the layer, so they are the prefill's; the state is the prefill's
    final state (not drawn here)."""
    inp = make_inputs(seed * 1000 + 17 + step, [1] * prefill.B, Hk=16, Hv=48, dk=128, dv=128,
                      io_dtype=np.float16)
    inp.A_log = prefill.A_log
    inp.dt_bias = prefill.dt_bias
    return inp
