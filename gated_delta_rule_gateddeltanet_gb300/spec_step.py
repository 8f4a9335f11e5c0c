"""One speculative-decoding step of a GatedDeltaNet layer, captured once in a
CUDA graph and replayed.

Source: "Replay compact fixed state for hybrid decoding" (Summary, Key
changes): per step the engine runs the drafted tokens through the layer from
the committed fixed state, captures compact per-token updates (the conv
inputs and the GDN capsules), and replays only the accepted prefix into the
inactive state bank before publishing it.  "[CUDA] Add compact GatedDeltaNet
operator" (embedded commit "Add compact VarlenCausalConv state updates") gives
the conv side: capture of the appended inputs, [batch, capacity, channels].

At the Qwen decode geometry the four kernels of a step run for tens of
microseconds in total, so host launch overhead is a large part of a step.
Here the step is four C-ABI calls with arguments built once, recorded into a
CUDA graph:

  1. varlen_causal_conv_with_state: x -> y = silu(conv(x)), from the committed
     conv states (slots ``src``), capturing every draft token's input;
  2. gdn_forward on y viewed as the fused [q | k | v] projection (token stride
     C = 2 Hk d + Hv d), raw gates a, b, from the committed GDN states, with a
     capsule per draft token;
  3. causal_conv_replay_prefix and 4. gdn_replay_prefix: the accepted prefix
     (``accept_len``, device data the caller writes before each replay) into
     the inactive slots ``dst`` of both banks.

The conv replay needs only the conv call's capture, so it runs on a side
stream beside the GDN replay; the main stream waits for it at the end of the
step.  It forks after the GDN forward rather than before it: the verify
kernel runs two register-heavy CTAs per SM, and conv-replay CTAs resident
beside it delayed their placement (the step took 41.0 µs with the fork
before the forward, 39.1 µs with it after).

Every per-step quantity is device memory read at replay time (inputs, gate
inputs, slot lists, accepted lengths), so one graph serves every step: the
caller writes the step's inputs and accepted lengths, replays, and publishes
by swapping ``src`` and ``dst`` (``publish()``).  The speculative final conv
states go to a scratch pool and the GDN verify writes no final state at all
(gdn_forward with no final-state buffer); the committed bank is never written.
"""
from __future__ import annotations

import ctypes

import torch

from . import DTYPE, GdnError, build_conv_args, build_forward_args, capsule_width, load_library, workspace_size


class SpeculativeStep:
    """R requests x D draft tokens through conv + GatedDeltaNet with compact
    capture, then replay of the accepted prefix, as one CUDA graph.

    conv_bank: [2R, C, K-1] (io dtype) and gdn_bank: [2R, Hv, d, d] fp32 hold
    the committed and inactive states; ``src``/``dst`` (device int32 [R])
    name each request's committed and inactive slot (initially 0..R-1 and
    R..2R-1).  ``keep_verify_state=True`` also writes the verify pass's own
    final GDN states to ``gdn_scratch``.  Inputs per step: ``x`` [R*D, C], ``a``, ``b`` [R*D, Hv] (raw
    gate inputs) and ``accept_len`` [R] int32 in [0, D], all device tensors
    owned by this object (write into them, then call ``replay()``).
    Outputs: ``out`` [R*D, Hv, d] and the captures ``conv_values``,
    ``capsules``.
    """

    def __init__(self, conv_weight, conv_bias, conv_bank, A_log, dt_bias, gdn_bank, *, num_k_heads, drafts,
                 activation="silu", keep_verify_state=False):
        dev = conv_bank.device
        self.dev = dev
        two_r, C, km1 = conv_bank.shape
        R = two_r // 2
        Hk = num_k_heads
        _, Hv, d, d2 = gdn_bank.shape
        if d != d2 or C != 2 * Hk * d + Hv * d or gdn_bank.shape[0] != two_r:
            raise ValueError("conv channels must be 2 Hk d + Hv d and both banks must hold 2R slots")
        dt = conv_bank.dtype
        T = R * drafts
        self.R, self.D, self.Hk, self.Hv, self.d, self.C = R, drafts, Hk, Hv, d, C
        self.conv_bank, self.gdn_bank = conv_bank, gdn_bank
        self.src = torch.arange(R, dtype=torch.int32, device=dev)
        self.dst = torch.arange(R, 2 * R, dtype=torch.int32, device=dev)
        self.accept_len = torch.zeros(R, dtype=torch.int32, device=dev)
        self.x = torch.zeros((T, C), dtype=dt, device=dev)
        self.a = torch.zeros((T, Hv), dtype=torch.float32, device=dev)
        self.b = torch.zeros((T, Hv), dtype=torch.float32, device=dev)
        self.cu = torch.arange(0, T + 1, drafts, dtype=torch.int32, device=dev)
        self.y = torch.empty((T, C), dtype=dt, device=dev)
        self.out = torch.empty((T, Hv, d), dtype=dt, device=dev)
        self.conv_values = torch.zeros((R, drafts, C), dtype=dt, device=dev)
        self.capsules = torch.zeros((R, drafts, capsule_width(Hk, Hv, d, d)), dtype=torch.float32, device=dev)
        self.conv_scratch = torch.empty_like(conv_bank)
        # the verify pass's own final GDN states are not needed (the accepted
        # prefix is replayed from the committed state), so none are written
        # unless asked for
        self.gdn_scratch = torch.empty_like(gdn_bank) if keep_verify_state else None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

        self.conv_args, _, k1 = build_conv_args(
            self.x, conv_weight, self.cu, bias=conv_bias, initial_state=conv_bank, final_state=self.conv_scratch,
            state_slots=self.src, capacity=drafts, activation=activation, output=self.y,
            state_update=self.conv_values, status=self.status, num_state_slots=two_r, max_seqlen=drafts)
        q = self.y[:, :Hk * d].view(T, Hk, d)
        k = self.y[:, Hk * d:2 * Hk * d].view(T, Hk, d)
        v = self.y[:, 2 * Hk * d:].view(T, Hv, d)
        self.fwd_args, _, k2 = build_forward_args(
            q, k, v, self.a, self.b, self.cu, A_log=A_log, dt_bias=dt_bias, initial_state=gdn_bank,
            final_state=self.gdn_scratch, state_slots=self.src, output=self.out, state_update=self.capsules,
            capacity=drafts, status=self.status, num_state_slots=two_r, max_seqlen=drafts,
            write_final_state=keep_verify_state)
        need = workspace_size(self.fwd_args)
        self.workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        if need:
            self.fwd_args.workspace, self.fwd_args.workspace_bytes = ctypes.c_void_p(self.workspace.data_ptr()), need
        self._keep = (k1, k2, q, k, v, conv_weight, conv_bias, A_log, dt_bias)
        self.lib = load_library()
        self.graph = None
        self._side = torch.cuda.Stream(dev)
        self._conv_done, self._side_done = torch.cuda.Event(), torch.cuda.Event()

    def run_eager(self, stream=None):
        """The four calls on ``stream`` (default: current), the conv replay
        forked onto a side stream after the GDN forward and joined at the end."""
        main = stream if stream is not None else torch.cuda.current_stream(self.dev)
        s = ctypes.c_void_p(main.cuda_stream)
        lib = self.lib
        p = lambda t: ctypes.c_void_p(t.data_ptr())
        rc = lib.varlen_causal_conv_with_state(ctypes.byref(self.conv_args), s)
        if rc:
            raise GdnError(rc, "varlen_causal_conv_with_state")
        rc = lib.gdn_forward(ctypes.byref(self.fwd_args), s)
        if rc:
            raise GdnError(rc, "gdn_forward")
        # the conv replay forks here, beside the GDN replay: beside the verify its CTAs
        # would take SM room the verify's two register-heavy CTAs per SM need
        self._conv_done.record(main)
        self._side.wait_event(self._conv_done)
        two_r, C, km1 = self.conv_bank.shape
        rc = lib.causal_conv_replay_prefix(p(self.conv_bank), two_r, self.R, C, km1 + 1, DTYPE[self.conv_bank.dtype],
                                           p(self.src), p(self.dst), p(self.conv_values), self.D, p(self.accept_len),
                                           p(self.status), ctypes.c_void_p(self._side.cuda_stream))
        if rc:
            raise GdnError(rc, "causal_conv_replay_prefix")
        self._side_done.record(self._side)
        rc = lib.gdn_replay_prefix(p(self.gdn_bank), two_r, self.R, self.Hk, self.Hv, self.d, self.d, p(self.src),
                                   p(self.dst), p(self.capsules), self.D, p(self.accept_len), p(self.status), s)
        if rc:
            raise GdnError(rc, "gdn_replay_prefix")
        main.wait_event(self._side_done)

    def capture(self):
        """Records the step into a CUDA graph, after one eager warm-up step on
        a side stream (the state banks are restored after it, so capturing
        changes no state)."""
        saved = (self.conv_bank.clone(), self.gdn_bank.clone(), self.accept_len.clone())
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(side):
            self.run_eager(side)
        torch.cuda.current_stream(self.dev).wait_stream(side)
        self.conv_bank.copy_(saved[0])
        self.gdn_bank.copy_(saved[1])
        self.accept_len.copy_(saved[2])
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.run_eager(torch.cuda.current_stream(self.dev))
        return self

    def replay(self):
        if self.graph is None:
            self.capture()
        self.graph.replay()

    def publish(self):
        """After a step: the inactive slots become the committed ones."""
        tmp = self.src.clone()
        self.src.copy_(self.dst)
        self.dst.copy_(tmp)
