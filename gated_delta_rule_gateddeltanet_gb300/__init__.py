"""GB300 GatedDeltaNet: Python binding of the libgdn.so C ABI.

This module only marshals arguments: it checks tensor dtypes and devices,
allocates outputs that the caller did not pass (with torch, on the tensors'
device), fills the ``gdn_forward_args`` struct of ``include/gdn.h`` and calls
the library on the current torch stream.  Every step of the computation runs
in the library's CUDA kernels.  There is no CPU fallback: if ``libgdn.so`` is
missing or cannot be loaded, importing the entry points raises.

Entry points (same names as the C ABI):
    gdn_forward(...)        -> (output, final_state, state_update)
    gdn_replay_prefix(...)  -> state_banks (updated in place)
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB as LIB_PATH

__all__ = ["gdn_forward", "ForwardCall", "gdn_forward_dense", "state_transpose", "gdn_forward_no_alloc", "gdn_replay_prefix", "varlen_causal_conv_with_state",
           "causal_conv_replay_prefix", "GdnError", "load_library", "capsule_width",
           "STATUS", "DEVERR", "PLAN"]

STATUS = {0: "GDN_OK", 1: "GDN_ERR_NULL", 2: "GDN_ERR_DTYPE", 3: "GDN_ERR_SHAPE", 4: "GDN_ERR_ALIGN",
          5: "GDN_ERR_WORKSPACE", 6: "GDN_ERR_CUDA", 7: "GDN_ERR_UNSUPPORTED", 8: "GDN_ERR_ARG"}
DEVERR = {"cu_seqlens": 0x1, "state_slot": 0x2, "accept_len": 0x4, "replay_slot": 0x8, "timeout": 0x10,
          "capture_count": 0x20, "dup_slot": 0x40}
ACTIVATION = {"none": 0, "silu": 1}
PLAN = {"auto": 0, "recurrent": 1, "chunked": 2, "chunked_split": 3}
DTYPE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
GATE_MODE = {"raw": 0, "precomputed": 1}


class GdnError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


class ForwardArgs(ctypes.Structure):
    """Mirror of ``gdn_forward_args`` (include/gdn.h)."""
    _fields_ = [
        ("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32), ("num_k_heads", ctypes.c_int32),
        ("num_v_heads", ctypes.c_int32), ("head_dim_k", ctypes.c_int32), ("head_dim_v", ctypes.c_int32),
        ("num_state_slots", ctypes.c_int32), ("io_dtype", ctypes.c_int32), ("gate_mode", ctypes.c_int32),
        ("plan", ctypes.c_int32), ("scale", ctypes.c_float), ("state_update_capacity", ctypes.c_int32),
        ("max_seqlen", ctypes.c_int32),
        ("q_stride", ctypes.c_int64), ("k_stride", ctypes.c_int64), ("v_stride", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("cu_seqlens", ctypes.c_void_p), ("state_slots", ctypes.c_void_p),
        ("initial_state", ctypes.c_void_p), ("final_state", ctypes.c_void_p), ("output", ctypes.c_void_p),
        ("state_update", ctypes.c_void_p), ("status", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


class ConvArgs(ctypes.Structure):
    """Mirror of ``gdn_conv_args`` (include/gdn.h)."""
    _fields_ = [
        ("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32), ("channels", ctypes.c_int32),
        ("kernel_size", ctypes.c_int32), ("num_state_slots", ctypes.c_int32), ("io_dtype", ctypes.c_int32),
        ("activation", ctypes.c_int32), ("state_update_capacity", ctypes.c_int32), ("max_seqlen", ctypes.c_int32),
        ("x_stride", ctypes.c_int64),
        ("x", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("bias", ctypes.c_void_p),
        ("cu_seqlens", ctypes.c_void_p), ("state_slots", ctypes.c_void_p), ("capture_count", ctypes.c_void_p),
        ("initial_state", ctypes.c_void_p), ("final_state", ctypes.c_void_p), ("output", ctypes.c_void_p),
        ("state_update", ctypes.c_void_p), ("status", ctypes.c_void_p),
    ]


_lib = None


def load_library(path: str | None = None):
    """Load libgdn.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libgdn.so is not built ({p}); run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.gdn_forward.restype = i32
    lib.gdn_forward.argtypes = [ctypes.POINTER(ForwardArgs), P]
    lib.gdn_forward_workspace_size.restype = i32
    lib.gdn_forward_workspace_size.argtypes = [ctypes.POINTER(ForwardArgs), ctypes.POINTER(ctypes.c_size_t)]
    lib.gdn_replay_prefix.restype = i32
    lib.gdn_replay_prefix.argtypes = [P, i32, i32, i32, i32, i32, i32, P, P, P, i32, P, P, P]
    lib.gdn_forward_no_alloc.restype = i32
    lib.gdn_forward_no_alloc.argtypes = [ctypes.POINTER(ForwardArgs), P]
    lib.varlen_causal_conv_with_state.restype = i32
    lib.varlen_causal_conv_with_state.argtypes = [ctypes.POINTER(ConvArgs), P]
    lib.causal_conv_replay_prefix.restype = i32
    lib.causal_conv_replay_prefix.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, i32, P, P, P]
    lib.gdn_forward_dense.restype = i32
    lib.gdn_forward_dense.argtypes = [ctypes.POINTER(ForwardArgs), i32, P]
    lib.gdn_state_transpose.restype = i32
    lib.gdn_state_transpose.argtypes = [P, P, ctypes.c_int64, i32, i32, P]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_status_string.argtypes = [i32]
    if path is None:
        _lib = lib
    return lib


def capsule_width(num_k_heads: int, num_v_heads: int, head_dim_k: int, head_dim_v: int) -> int:
    """Floats per capsule row: decay per value head, unit key per key head, delta per value head."""
    return num_v_heads + num_k_heads * head_dim_k + num_v_heads * head_dim_v


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(t, name, dtype=None, device=None, contiguous=True):
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _shape(t, name, shape, leading_at_least=False):
    """Raise unless ``t`` (if given) has ``shape``: the C ABI takes raw
    pointers, so the binding is where a buffer's extent is checked against the
    call's geometry, before any launch.  With ``leading_at_least`` the first
    extent may be larger (a state pool or output buffer with more rows than the
    call addresses); the inner extents must match."""
    if t is None:
        return
    want = tuple(int(x) for x in shape)
    got = tuple(t.shape)
    ok = (len(got) == len(want) and got[1:] == want[1:] and
          (got[0] >= want[0] if leading_at_least else got[0] == want[0]))
    if not ok:
        lead = "at least " if leading_at_least else ""
        raise ValueError(f"{name} must have shape {want} ({lead}{want[0]} rows), got {got}")


def _token_stride(t, name, inner):
    """Elements between consecutive tokens of a [T, H, d] view whose inner two
    dims are contiguous (allows slices of a fused qkv projection)."""
    if t.dim() != 3:
        raise ValueError(f"{name} must be [T, H, d]")
    if t.numel() == 0:  # no tokens (every sequence empty): nothing is read, any strides do
        return inner
    if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError(f"{name}: heads and channels must be contiguous inside a token")
    return t.stride(0) if t.shape[0] > 1 else inner


def build_forward_args(q, k, v, a, b, cu_seqlens, *, A_log=None, dt_bias=None, gate_mode="raw",
                       initial_state=None, final_state=None, state_slots=None, output=None,
                       state_update=None, capacity=0, scale=0.0, plan="auto", status=None,
                       num_state_slots=None, workspace=None, max_seqlen=0, num_seqs=None,
                       write_final_state=True):
    """Fill a ForwardArgs struct from tensors; returns (args, outputs, keepalive).
    ``cu_seqlens=None`` (rank-4 calls) takes the batch size from ``num_seqs``.
    ``write_final_state=False`` passes no final-state buffer: the kernels then
    write no state (the returned final_state is None)."""
    dev = q.device
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    B = cu_seqlens.shape[0] - 1 if cu_seqlens is not None else int(num_seqs)
    if q.dtype not in DTYPE:
        raise TypeError(f"unsupported dtype {q.dtype}")
    for name, t in (("k", k), ("v", v)):
        _check(t, name, dtype=q.dtype, device=dev, contiguous=False)
    for name, t in (("a", a), ("b", b), ("A_log", A_log), ("dt_bias", dt_bias)):
        _check(t, name, dtype=torch.float32, device=dev)
    _check(cu_seqlens, "cu_seqlens", dtype=torch.int32, device=dev)
    _check(state_slots, "state_slots", dtype=torch.int32, device=dev)
    _check(status, "status", dtype=torch.int32, device=dev)
    if cu_seqlens is not None and cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be one-dimensional [B + 1]")
    _shape(k, "k", (T, Hk, dk))
    if v.dim() != 3 or v.shape[0] != T:
        raise ValueError(f"v must be [T = {T}, Hv, dv], got {tuple(v.shape)}")
    _shape(a, "a", (T, Hv))
    _shape(b, "b", (T, Hv))
    _shape(A_log, "A_log", (Hv,))
    _shape(dt_bias, "dt_bias", (Hv,))
    _shape(state_slots, "state_slots", (B,))
    if status is not None and status.numel() < 1:
        raise ValueError("status must hold one int32")
    if num_state_slots is None:
        if initial_state is not None:
            num_state_slots = initial_state.shape[0]
        elif final_state is not None:
            num_state_slots = final_state.shape[0]
        else:
            num_state_slots = B
    if not write_final_state:
        final_state = None
    elif final_state is None:
        final_state = (torch.empty if initial_state is not None else torch.zeros)(
            (num_state_slots, Hv, dv, dk), dtype=torch.float32, device=dev)
        if initial_state is not None:
            final_state.copy_(initial_state)
    _check(initial_state, "initial_state", dtype=torch.float32, device=dev)
    _check(final_state, "final_state", dtype=torch.float32, device=dev)
    _shape(initial_state, "initial_state", (num_state_slots, Hv, dv, dk), leading_at_least=True)
    _shape(final_state, "final_state", (num_state_slots, Hv, dv, dk), leading_at_least=True)
    if output is None:
        output = torch.empty((T, Hv, dv), dtype=q.dtype, device=dev)
    _check(output, "output", dtype=q.dtype, device=dev)
    _shape(output, "output", (T, Hv, dv), leading_at_least=True)
    W = capsule_width(Hk, Hv, dk, dv)
    if capacity > 0 and state_update is None:
        state_update = torch.zeros((B, capacity, W), dtype=torch.float32, device=dev)
    _check(state_update, "state_update", dtype=torch.float32, device=dev)
    if capacity > 0:
        _shape(state_update, "state_update", (B, capacity, W), leading_at_least=True)

    args = ForwardArgs()
    args.num_seqs, args.total_tokens, args.num_k_heads, args.num_v_heads = B, T, Hk, Hv
    args.head_dim_k, args.head_dim_v, args.num_state_slots = dk, dv, int(num_state_slots)
    args.io_dtype = DTYPE[q.dtype]
    args.gate_mode = GATE_MODE[gate_mode]
    args.plan = PLAN[plan]
    args.scale = float(scale or 0.0)
    args.state_update_capacity = int(capacity)
    args.max_seqlen = int(max_seqlen or 0)
    args.q_stride = _token_stride(q, "q", Hk * dk)
    args.k_stride = _token_stride(k, "k", Hk * dk)
    args.v_stride = _token_stride(v, "v", Hv * dv)
    args.q, args.k, args.v = _ptr(q), _ptr(k), _ptr(v)
    args.a, args.b = _ptr(a), _ptr(b)
    args.A_log, args.dt_bias = _ptr(A_log), _ptr(dt_bias)
    args.cu_seqlens, args.state_slots = _ptr(cu_seqlens), _ptr(state_slots)
    # final_state was seeded from initial_state above when the caller passed no output buffer
    args.initial_state = _ptr(initial_state)
    args.final_state = _ptr(final_state)
    args.output = _ptr(output)
    args.state_update = _ptr(state_update) if capacity > 0 else None
    args.status = _ptr(status)
    if workspace is not None:
        args.workspace, args.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    keep = (q, k, v, a, b, A_log, dt_bias, cu_seqlens, state_slots, initial_state, status, workspace)
    return args, (output, final_state, state_update), keep


def workspace_size(args: ForwardArgs) -> int:
    n = ctypes.c_size_t(0)
    rc = load_library().gdn_forward_workspace_size(ctypes.byref(args), ctypes.byref(n))
    if rc != 0:
        raise GdnError(rc, "gdn_forward_workspace_size")
    return int(n.value)


def gdn_forward(q, k, v, a, b, cu_seqlens, *, A_log=None, dt_bias=None, gate_mode="raw",
                initial_state=None, final_state=None, state_slots=None, output=None,
                state_update=None, capacity=0, scale=0.0, plan="auto", status=None,
                num_state_slots=None, workspace=None, max_seqlen=0, write_final_state=True):
    """Gated delta rule over a packed varlen batch (C ABI ``gdn_forward``).

    q, k: [T, Hk, dk] fp16/fp32 CUDA; v: [T, Hv, dv]; a, b: [T, Hv] fp32 (raw
    gate inputs, or g and beta with ``gate_mode="precomputed"``); A_log, dt_bias:
    [Hv] fp32; cu_seqlens: [B+1] int32.  ``initial_state`` [slots, Hv, dv, dk]
    fp32 or None (zeros); ``final_state`` may be the same tensor (in place).
    ``max_seqlen``: an upper bound on the longest sequence (0 = unknown), a
    hint that lets decode-sized batches skip the chunked kernel.  Workspace is
    allocated here when the call needs some and none is passed.
    Returns ``(output, final_state, state_update)``; state_update is
    [B, capacity, W] fp32 or None.
    """
    lib = load_library()
    args, outs, keep = build_forward_args(q, k, v, a, b, cu_seqlens, A_log=A_log, dt_bias=dt_bias,
                                          gate_mode=gate_mode, initial_state=initial_state,
                                          final_state=final_state, state_slots=state_slots, output=output,
                                          state_update=state_update, capacity=capacity, scale=scale, plan=plan,
                                          status=status, num_state_slots=num_state_slots, workspace=workspace,
                                          max_seqlen=max_seqlen, write_final_state=write_final_state)
    need = workspace_size(args)
    if need > 0 and workspace is None:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
        args.workspace, args.workspace_bytes = ctypes.c_void_p(ws.data_ptr()), need
        keep = keep + (ws,)
    rc = lib.gdn_forward(ctypes.byref(args), _stream_handle(q.device))
    if rc != 0:
        raise GdnError(rc, "gdn_forward")
    return outs


class ForwardCall:
    """A gdn_forward call whose arguments are resolved once: the same device
    buffers (inputs, states, outputs, workspace) serve every launch, and
    ``launch()`` is a single C-ABI call with no argument marshalling.  Suits a
    serving loop that refills fixed input buffers every step (e.g. by copies
    from pinned host memory) and calls the operator on them.  Arguments as for
    ``gdn_forward``; the tensors must stay alive and in place while the object
    is used.  ``outputs`` is ``(output, final_state, state_update)``."""

    def __init__(self, q, k, v, a, b, cu_seqlens, **kw):
        workspace = kw.pop("workspace", None)
        self.args, self.outputs, keep = build_forward_args(q, k, v, a, b, cu_seqlens, workspace=workspace, **kw)
        need = workspace_size(self.args)
        if need > 0 and workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            self.args.workspace, self.args.workspace_bytes = ctypes.c_void_p(workspace.data_ptr()), need
        self._keep = keep + (workspace,)
        self._lib = load_library()
        self._ref = ctypes.byref(self.args)
        self._device = q.device

    def launch(self, stream=None):
        """Runs the call on ``stream`` (a torch.cuda.Stream; default: the current stream)."""
        h = ctypes.c_void_p((stream or torch.cuda.current_stream(self._device)).cuda_stream)
        rc = self._lib.gdn_forward(self._ref, h)
        if rc != 0:
            raise GdnError(rc, "gdn_forward")
        return self.outputs


def gdn_forward_dense(q, k, v, a, b, *, workspace=None, **kw):
    """Rank-4 inputs (C ABI ``gdn_forward_dense``): q, k [B, S, Hk, dk], v
    [B, S, Hv, dv], a, b [B, S, Hv], contiguous.  Other keyword arguments as
    for ``gdn_forward`` (states stay V-major [slots, Hv, dv, dk]; see
    ``state_transpose`` for the dense export's K-major layout).  Returns
    ``(output [B, S, Hv, dv], final_state, state_update)``."""
    lib = load_library()
    B, S = q.shape[0], q.shape[1]
    flat = lambda t: None if t is None else t.reshape(B * S, *t.shape[2:])
    output = kw.pop("output", None)
    if output is not None:
        output = output.view(B * S, *output.shape[2:])
    args, (out, final, caps), keep = build_forward_args(flat(q), flat(k), flat(v), flat(a), flat(b), None,
                                                        output=output, workspace=workspace, num_seqs=B, **kw)
    need = workspace_size(args)
    if need > 0 and workspace is None:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
        args.workspace, args.workspace_bytes = ctypes.c_void_p(ws.data_ptr()), need
        keep = keep + (ws,)
    rc = lib.gdn_forward_dense(ctypes.byref(args), S, _stream_handle(q.device))
    if rc != 0:
        raise GdnError(rc, "gdn_forward_dense")
    return out.view(B, S, *out.shape[1:]), final, caps


def state_transpose(src, dst=None):
    """Transposes the last two dims of an FP32 CUDA tensor (C ABI
    ``gdn_state_transpose``): K-major [.., dk, dv] <-> V-major [.., dv, dk]."""
    _check(src, "src", dtype=torch.float32)
    rows, cols = src.shape[-2], src.shape[-1]
    if dst is None:
        dst = torch.empty(*src.shape[:-2], cols, rows, dtype=torch.float32, device=src.device)
    _check(dst, "dst", dtype=torch.float32, device=src.device)
    num = src.numel() // max(rows * cols, 1) if rows * cols else 0
    rc = load_library().gdn_state_transpose(_ptr(src), _ptr(dst), num, rows, cols, _stream_handle(src.device))
    if rc != 0:
        raise GdnError(rc, "gdn_state_transpose")
    return dst


def gdn_forward_no_alloc(q, k, v, a, b, cu_seqlens, **kw):
    """``gdn_forward`` through the C ABI ``gdn_forward_no_alloc``: the chunked
    kernel's workspace comes from a fixed array inside the library, for hosts
    that cannot hand the operator extra device memory.  Same arguments and
    results as ``gdn_forward`` (``workspace`` is ignored); at most
    ``GDN_NO_ALLOC_MAX_SEQS`` (4094) sequences when the chunked kernel may run.
    Calls that overlap on the GPU share that array and must not be made."""
    lib = load_library()
    kw.pop("workspace", None)
    args, outs, keep = build_forward_args(q, k, v, a, b, cu_seqlens, **kw)
    rc = lib.gdn_forward_no_alloc(ctypes.byref(args), _stream_handle(q.device))
    if rc != 0:
        raise GdnError(rc, "gdn_forward_no_alloc")
    return outs


def gdn_replay_prefix(state_banks, src_slots, dst_slots, state_update, accept_len, *, num_k_heads,
                      status=None):
    """Replay an accepted capsule prefix into the destination banks, in place
    (C ABI ``gdn_replay_prefix``).  state_banks: [slots, Hv, dv, dk] fp32;
    state_update: [R, capacity, W] fp32; src/dst/accept_len: [R] int32."""
    lib = load_library()
    S, Hv, dv, dk = state_banks.shape
    R = src_slots.shape[0]
    cap = state_update.shape[1] if state_update is not None else 0
    dev = state_banks.device
    _check(state_banks, "state_banks", dtype=torch.float32, device=dev)
    for name, t in (("src_slots", src_slots), ("dst_slots", dst_slots), ("accept_len", accept_len),
                    ("status", status)):
        _check(t, name, dtype=torch.int32, device=dev)
    _check(state_update, "state_update", dtype=torch.float32, device=dev)
    if src_slots.dim() != 1:
        raise ValueError("src_slots must be one-dimensional [R]")
    _shape(dst_slots, "dst_slots", (R,))
    _shape(accept_len, "accept_len", (R,))
    if state_update is not None:
        _shape(state_update, "state_update", (R, cap, capsule_width(num_k_heads, Hv, dk, dv)), leading_at_least=True)
    rc = lib.gdn_replay_prefix(_ptr(state_banks), S, R, int(num_k_heads), Hv, dk, dv, _ptr(src_slots),
                               _ptr(dst_slots), _ptr(state_update), cap, _ptr(accept_len), _ptr(status),
                               _stream_handle(dev))
    if rc != 0:
        raise GdnError(rc, "gdn_replay_prefix")
    return state_banks


def build_conv_args(x, weight, cu_seqlens, *, bias=None, initial_state=None, final_state=None, state_slots=None,
                    capture_count=None, capacity=0, activation="silu", output=None, state_update=None,
                    status=None, num_state_slots=None, max_seqlen=0):
    """Fill a ConvArgs struct from tensors; returns (args, outputs, keepalive)."""
    dev = x.device
    T, C = x.shape
    K = weight.shape[1]
    B = cu_seqlens.shape[0] - 1
    if x.dtype not in DTYPE:
        raise TypeError(f"unsupported dtype {x.dtype}")
    if x.numel() > 0 and x.stride(1) != 1:  # (no tokens: nothing is read)
        raise ValueError("x: channels must be contiguous")
    _check(weight, "weight", dtype=torch.float32, device=dev)
    _check(bias, "bias", dtype=torch.float32, device=dev)
    for name, t in (("cu_seqlens", cu_seqlens), ("state_slots", state_slots), ("capture_count", capture_count),
                    ("status", status)):
        _check(t, name, dtype=torch.int32, device=dev)
    if cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be one-dimensional [B + 1]")
    _shape(weight, "weight", (C, K))
    _shape(bias, "bias", (C,))
    _shape(state_slots, "state_slots", (B,))
    _shape(capture_count, "capture_count", (B,))
    if num_state_slots is None:
        src = initial_state if initial_state is not None else final_state
        num_state_slots = src.shape[0] if src is not None else B
    if final_state is None:
        final_state = (initial_state.clone() if initial_state is not None else
                       torch.zeros((num_state_slots, C, K - 1), dtype=x.dtype, device=dev))
    for name, t in (("initial_state", initial_state), ("final_state", final_state)):
        _check(t, name, dtype=x.dtype, device=dev)
    if output is None:
        output = torch.empty((T, C), dtype=x.dtype, device=dev)
    if capacity > 0 and state_update is None:
        state_update = torch.zeros((B, capacity, C), dtype=x.dtype, device=dev)
    _check(output, "output", dtype=x.dtype, device=dev)
    _check(state_update, "state_update", dtype=x.dtype, device=dev)
    _shape(initial_state, "initial_state", (num_state_slots, C, K - 1), leading_at_least=True)
    _shape(final_state, "final_state", (num_state_slots, C, K - 1), leading_at_least=True)
    _shape(output, "output", (T, C), leading_at_least=True)
    if capacity > 0:
        _shape(state_update, "state_update", (B, capacity, C), leading_at_least=True)
    a = ConvArgs()
    a.num_seqs, a.total_tokens, a.channels, a.kernel_size = B, T, C, K
    a.num_state_slots, a.io_dtype = int(num_state_slots), DTYPE[x.dtype]
    a.activation, a.state_update_capacity = ACTIVATION[activation], int(capacity)
    a.max_seqlen = int(max_seqlen or 0)
    a.x_stride = x.stride(0) if T > 1 else C
    a.x, a.weight, a.bias = _ptr(x), _ptr(weight), _ptr(bias)
    a.cu_seqlens, a.state_slots, a.capture_count = _ptr(cu_seqlens), _ptr(state_slots), _ptr(capture_count)
    a.initial_state, a.final_state, a.output = _ptr(initial_state), _ptr(final_state), _ptr(output)
    a.state_update = _ptr(state_update) if capacity > 0 else None
    a.status = _ptr(status)
    keep = (x, weight, bias, cu_seqlens, state_slots, capture_count, initial_state, status)
    return a, (output, final_state, state_update), keep


def varlen_causal_conv_with_state(x, weight, cu_seqlens, **kw):
    """Packed depthwise causal conv (+ SiLU) with carried state (C ABI
    ``varlen_causal_conv_with_state``).  x: [T, C] fp16/fp32; weight: [C, K]
    fp32; optional bias [C]; initial_state / final_state [slots, C, K-1] in
    x's dtype (may be the same tensor); capture_count [B] int32.  Returns
    ``(output, final_state, state_update)``."""
    lib = load_library()
    args, outs, keep = build_conv_args(x, weight, cu_seqlens, **kw)
    rc = lib.varlen_causal_conv_with_state(ctypes.byref(args), _stream_handle(x.device))
    if rc != 0:
        raise GdnError(rc, "varlen_causal_conv_with_state")
    return outs


def causal_conv_replay_prefix(conv_states, src_slots, dst_slots, state_update, accept_len, *, status=None):
    """Replay accepted captured conv inputs into the destination states, in
    place (C ABI ``causal_conv_replay_prefix``).  conv_states: [slots, C, K-1];
    state_update: [R, capacity, C]; src/dst/accept_len: [R] int32."""
    lib = load_library()
    S, C, Km1 = conv_states.shape
    dev = conv_states.device
    _check(conv_states, "conv_states", device=dev)
    _check(state_update, "state_update", dtype=conv_states.dtype, device=dev)
    for name, t in (("src_slots", src_slots), ("dst_slots", dst_slots), ("accept_len", accept_len),
                    ("status", status)):
        _check(t, name, dtype=torch.int32, device=dev)
    cap = state_update.shape[1] if state_update is not None else 0
    R = src_slots.shape[0]
    if src_slots.dim() != 1:
        raise ValueError("src_slots must be one-dimensional [R]")
    _shape(dst_slots, "dst_slots", (R,))
    _shape(accept_len, "accept_len", (R,))
    if state_update is not None:
        _shape(state_update, "state_update", (R, cap, C), leading_at_least=True)
    rc = lib.causal_conv_replay_prefix(_ptr(conv_states), S, src_slots.shape[0], C, Km1 + 1, DTYPE[conv_states.dtype],
                                       _ptr(src_slots), _ptr(dst_slots), _ptr(state_update), cap, _ptr(accept_len),
                                       _ptr(status), _stream_handle(dev))
    if rc != 0:
        raise GdnError(rc, "causal_conv_replay_prefix")
    return conv_states
