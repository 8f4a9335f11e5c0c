"""Benchmark of the GatedDeltaNet hot path on GB300.

A step is one gdn_forward over the decode workload: 64 requests x 1 token,
Hk=16 key heads, Hv=48 value heads, dk=dv=128, fp16 q/k/v/output, raw FP32
gates, FP32 V-major state [64, 48, 128, 128] updated in place.  The state is
rotated over 4 pools of 192 MiB so every step streams it from HBM (the
working set, 768 MiB, is far larger than the 129 MB L2).

One JSON line is printed by rank 0 (see the keys at the end of main()).
``--impl reference`` times the FP64 CPU oracle on the same workload instead.
Under torchrun every rank runs its own 64 requests (weak scaling, no
collective on the data path); the barrier and the max over ranks are the only
communication.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN tokens/s and state HBM GB/s (% of roofline) at decode/prefill, 1×GB300"
WORKLOAD = "decode step: 64 requests x 1 token, Hk=16, Hv=48, dk=dv=128, fp16 I/O, fp32 state [64,48,128,128]"
NBUF = 4


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--no-extra", action="store_true", help="skip the prefill / verify+replay sub-measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) measurement")
    ap.add_argument("--only", choices=sorted(SUB_MEASUREMENTS),
                    help="run one sub-measurement alone on GPU 0 and print its JSON (for profiling)")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed plumbing

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            import torch
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = torch.device("cuda", self.local) if torch.cuda.is_available() else torch.device("cpu")
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = torch.device("cuda", self.local) if torch.cuda.is_available() else torch.device("cpu")
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def shard_seed(base: int, rank: int) -> int:
    """Each rank draws its own requests (weak scaling)."""
    return base + 7919 * rank


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid=None):
        self.proc = None
        self.path = None
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = [exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if device_uuid:
            cmd += ["-i", device_uuid]
        self.fh = open(self.path, "w")
        self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as fh:
            lines = fh.readlines()
        os.unlink(self.path)
        return self.summarise(lines)

    @staticmethod
    def summarise(lines):
        """Median and maximum SM clock and the throttle reasons seen in
        ``nvidia-smi --format=csv,noheader,nounits`` lines of FIELDS."""
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, fl in rows for n, f in zip(names, fl) if f.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- profiles

def recorded_traffic(kernel_src: str, name: str):
    """Per-launch DRAM bytes from the committed ncu summary of this kernel, or
    None when the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m_b or not m_h:
        return None
    if hashlib.sha256(open(kernel_src, "rb").read()).hexdigest() != m_h.group(1):
        return None
    return float(m_b.group(1))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------- GPU arm

def workload_config(R, Hk, Hv, dk, dv, world):
    """The ``config`` object of the JSON line; both arms report the same one."""
    return {"workload": WORKLOAD, "requests_per_gpu": R, "Hk": Hk, "Hv": Hv, "dk": dk, "dv": dv,
            "io_dtype": "fp16", "state_dtype": "fp32", "plan": "auto (recurrent for 1-token spans)",
            "l2": f"inputs larger than L2: {NBUF} rotating in-place state pools of 192 MiB",
            "parallelism": f"dp{world} (independent requests per GPU)"}


def decode_bytes_per_launch(R, Hk, Hv, dk, dv, io_bytes=2):
    """Algorithmic HBM bytes of one decode launch: the state read and written
    once, q, k, v, output in the I/O dtype, raw a and b in FP32."""
    state = 2 * Hv * dv * dk * 4
    io = 2 * Hk * dk * io_bytes + 2 * Hv * dv * io_bytes + 2 * Hv * 4
    return R * (state + io)


def run_gdn(a, dist: Dist):
    import torch
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    from gated_delta_rule_gateddeltanet_gb300 import workloads as wl

    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    lib = gdn.load_library()
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)

    # ---- inputs: NBUF rotating input sets and in-place state pools
    sets = []
    for i in range(NBUF):
        inp = wl.decode_step(seed=shard_seed(wl.SEEDS["decode_step"] + 100 * i, dist.rank))
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        d = dict(q=t(inp.q), k=t(inp.k), v=t(inp.v), a=t(inp.a), b=t(inp.b), A_log=t(inp.A_log),
                 dt_bias=t(inp.dt_bias), cu=t(inp.cu_seqlens), state=t(inp.initial_state),
                 out=torch.empty((inp.T, 48, 128), dtype=torch.float16, device=dev), inp=inp)
        args, _, keep = gdn.build_forward_args(d["q"], d["k"], d["v"], d["a"], d["b"], d["cu"], A_log=d["A_log"],
                                               dt_bias=d["dt_bias"], initial_state=d["state"],
                                               final_state=d["state"], output=d["out"], max_seqlen=1)
        d["args"], d["keep"] = args, keep
        sets.append(d)
    R = sets[0]["inp"].B
    Hk, Hv, dk, dv = sets[0]["inp"].dims

    def step(i):
        rc = lib.gdn_forward(ctypes.byref(sets[i % NBUF]["args"]), sh)
        if rc:
            raise gdn.GdnError(rc, "gdn_forward")

    for i in range(a.warmup):
        step(i)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(a.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    ck = clocks.stop()
    ms_local = e0.elapsed_time(e1)
    ms = dist.max(ms_local)
    ms_per_step = ms / a.steps
    tokens = dist.sum(R * a.steps)
    value = tokens / (ms / 1e3)

    hbm_peak, tc_peak, peak_kind = measured_peaks()
    bytes_launch = decode_bytes_per_launch(R, Hk, Hv, dk, dv)
    achieved_gbs = bytes_launch / (ms_local / a.steps / 1e3) / 1e9
    traffic = recorded_traffic(os.path.join(ROOT, "gated_delta_rule_gateddeltanet_gb300", "csrc", "gdn_recurrent.cu"),
                               "decode_step.recurrent_kernel.ncu.md")
    roofline = {"bound": "hbm", "kernel": "recurrent_kernel<__half,128>", "achieved": round(achieved_gbs, 1),
                "peak": hbm_peak, "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                "unit": "GB/s", "frac": round(achieved_gbs / hbm_peak, 4), "traffic": traffic,
                "algorithmic_bytes_per_launch": bytes_launch,
                "launch_us": round(ms_local / a.steps * 1e3, 2)}

    # ---- e2e: host buffers through the public binding
    e2e = None if a.no_e2e else run_e2e(a, dist, sets, dev, stream)

    extra = {}
    if not a.no_extra and dist.rank == 0:
        extra["prefill"] = run_prefill(dev, stream)
        extra["spec_verify_replay"] = run_spec(dev, stream, lib, sh)
        extra["causal_conv"] = run_conv(dev, stream)
        extra["serving_mix"] = run_serving_mix(dev, stream, lib, sh)
        extra["state_transpose"] = run_transpose(dev, stream, lib, sh)
        extra["spec_step_graph"] = run_spec_step(dev, stream)
        extra["long_prefill"] = run_long_prefill(dev, stream)

    cpu = None
    if not a.no_cpu and dist.rank == 0 and dist.world == 1:
        cpu = run_cpu_baseline(sets[0]["inp"])

    if dist.rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": dist.world,
                "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms_per_step, 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded numpy: q,k,v ~ N(0,1) fp16; a,b ~ N(0,1); A_log=log U(1,16); "
                        "dt_bias=log expm1 U(1e-3,0.1); state ~ N(0,0.02^2))",
                "config": workload_config(R, Hk, Hv, dk, dv, dist.world),
                "state_gbs": round(2 * R * Hv * dv * dk * 4 / (ms_local / a.steps / 1e3) / 1e9, 1),
                "roofline": roofline, "e2e": e2e, "gpu_launches": a.steps, "clocks": ck,
                "cpu_baseline": cpu}
        line.update(extra)
        print(json.dumps(line), flush=True)


def run_e2e(a, dist, sets, dev, stream):
    """Same metric through the public Python binding with host buffers: every
    step copies that step's q, k, v, a, b and cu_seqlens from pinned host memory
    into fixed device buffers, launches a prepared ``gdn.ForwardCall`` on them
    and reads the output back to pinned host memory.  The state stays resident
    in HBM (a fixed-state pool).  ``per_call_binding`` is the same loop through
    ``gdn.gdn_forward``, which marshals every argument on every call."""
    import torch
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    host, devb, calls = [], [], []
    for d in sets:
        hs = {n: d[n].cpu().pin_memory() for n in ("q", "k", "v", "a", "b", "cu")}
        ho = torch.empty(d["out"].shape, dtype=d["out"].dtype).pin_memory()
        host.append((hs, ho))
        db = {n: torch.empty_like(d[n]) for n in ("q", "k", "v", "a", "b", "cu")}
        devb.append(db)
        calls.append(gdn.ForwardCall(db["q"], db["k"], db["v"], db["a"], db["b"], db["cu"], A_log=d["A_log"],
                                     dt_bias=d["dt_bias"], initial_state=d["state"], final_state=d["state"],
                                     output=d["out"], max_seqlen=1))
    h2d = sum(x.numel() * x.element_size() for x in host[0][0].values())
    d2h = host[0][1].numel() * host[0][1].element_size()
    steps = max(10, a.steps)

    def step_prepared(i):
        j = i % NBUF
        hs, ho = host[j]
        db = devb[j]
        for n in hs:
            db[n].copy_(hs[n], non_blocking=True)
        out = calls[j].launch(stream)[0]
        ho.copy_(out, non_blocking=True)

    def step_binding(i):
        j = i % NBUF
        hs, ho = host[j]
        db = devb[j]
        for n in hs:
            db[n].copy_(hs[n], non_blocking=True)
        d = sets[j]
        out, _, _ = gdn.gdn_forward(db["q"], db["k"], db["v"], db["a"], db["b"], db["cu"], A_log=d["A_log"],
                                    dt_bias=d["dt_bias"], initial_state=d["state"], final_state=d["state"],
                                    output=d["out"], max_seqlen=1)
        ho.copy_(out, non_blocking=True)

    def timed(step):
        for i in range(min(a.warmup, 50)):
            step(i)
        torch.cuda.synchronize()
        dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        return dist.max(e0.elapsed_time(e1))

    # pipelined: step i's input copies (copy stream) and step i-1's output read
    # (a second copy stream) overlap the kernel of the step before; each
    # buffer set is reused only after the work that last read it has finished
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_h2d = [torch.cuda.Event() for _ in range(NBUF)]
    ev_kernel = [torch.cuda.Event() for _ in range(NBUF)]
    ev_d2h = [torch.cuda.Event() for _ in range(NBUF)]
    used = [False] * NBUF

    def step_pipelined(i):
        j = i % NBUF
        hs, ho = host[j]
        db = devb[j]
        with torch.cuda.stream(h2d_stream):
            if used[j]:
                h2d_stream.wait_event(ev_kernel[j])  # the kernel that last read these device inputs
            for n in hs:
                db[n].copy_(hs[n], non_blocking=True)
            ev_h2d[j].record(h2d_stream)
        stream.wait_event(ev_h2d[j])
        if used[j]:
            stream.wait_event(ev_d2h[j])  # the output buffer's previous read is done
        out = calls[j].launch(stream)[0]
        ev_kernel[j].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(ev_kernel[j])
            ho.copy_(out, non_blocking=True)
            ev_d2h[j].record(d2h_stream)
        used[j] = True

    def timed_pipelined():
        for i in range(min(a.warmup, 50)):
            step_pipelined(i)
        torch.cuda.synchronize()
        dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_stream.wait_event(e0)
        for i in range(steps):
            step_pipelined(i)
        for j in range(NBUF):  # the timed region ends when every output has reached the host
            stream.wait_event(ev_d2h[j])
        e1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        return dist.max(e0.elapsed_time(e1))

    ms = timed_pipelined()
    ms_serial = timed(step_prepared)
    ms_binding = timed(step_binding)
    tokens = dist.sum(sets[0]["inp"].B * steps)
    return {"value": round(tokens / (ms / 1e3), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(ms / steps, 4),
            "path": "python binding ForwardCall.launch -> C ABI gdn_forward; per step 6 copies from pinned host "
                    "inputs (copy stream) and one to a pinned host output (second copy stream), overlapping the "
                    "neighbouring steps' kernels; state resident in HBM",
            "serial_one_stream": {"value": round(tokens / (ms_serial / 1e3), 1),
                                  "ms_per_step": round(ms_serial / steps, 4)},
            "per_call_binding": {"value": round(tokens / (ms_binding / 1e3), 1),
                                 "ms_per_step": round(ms_binding / steps, 4)}}


def _flush_l2(buf):
    buf.add_(1.0)


PREFILL_WARMUP, PREFILL_CALLS = 10, 50


def run_prefill(dev, stream):
    """Varlen prefill: 8 packed sequences of U[256, 4096] tokens, Hk=16, Hv=48,
    d=128, fp16, zero initial state; L2 flushed before each call."""
    import torch
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    from gated_delta_rule_gateddeltanet_gb300 import workloads as wl
    inp = wl.varlen_prefill()
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    q, k, v, aa, bb = t(inp.q), t(inp.k), t(inp.v), t(inp.a), t(inp.b)
    A_log, dt_bias, cu = t(inp.A_log), t(inp.dt_bias), t(inp.cu_seqlens)
    final = torch.zeros((inp.B, 48, 128, 128), dtype=torch.float32, device=dev)
    out = torch.empty((inp.T, 48, 128), dtype=torch.float16, device=dev)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)  # 256 MiB
    plan = "auto"
    maxlen = int(np.diff(inp.cu_seqlens).max())
    args, _, _ = gdn.build_forward_args(q, k, v, aa, bb, cu, A_log=A_log, dt_bias=dt_bias, final_state=final,
                                        output=out, plan=plan, max_seqlen=maxlen)
    ws_two_phase = torch.empty(gdn.workspace_size(args), dtype=torch.uint8, device=dev)
    ws_single = torch.empty(4096, dtype=torch.uint8, device=dev)  # the chain list only: single-kernel evaluation

    def timed(ws):
        # arguments resolved once: each timed call is one C-ABI call
        call = gdn.ForwardCall(q, k, v, aa, bb, cu, A_log=A_log, dt_bias=dt_bias, final_state=final, output=out,
                               plan=plan, max_seqlen=maxlen, workspace=ws)
        for _ in range(PREFILL_WARMUP):
            call.launch(stream)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(PREFILL_CALLS)]
        for e0, e1 in ev:
            _flush_l2(flush)
            e0.record(stream)
            call.launch(stream)
            e1.record(stream)
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)

    ms = timed(ws_two_phase)
    ms_single = timed(ws_single)
    T = inp.T
    lengths = [int(x) for x in np.diff(inp.cu_seqlens)]
    _, tc_peak, kind = measured_peaks()
    flops = prefill_algorithmic_flops(T)
    chunk_heads = sum((L + 63) // 64 for L in lengths) * 48
    executed = chunk_heads * PREFILL_MMA_FLOPS_PER_CHUNK_HEAD
    tflops = flops / (ms / 1e3) / 1e12
    return {"workload": "varlen prefill: 8 sequences, lengths U[256,4096] (seeded), Hk=16, Hv=48, d=128, fp16, "
                        "zero initial state", "tokens": int(T), "lengths": lengths,
            "plan": plan, "ms": round(ms, 4), "tokens_per_s": round(T / (ms / 1e3), 1), "l2": "flushed (256 MiB write)",
            "timing": f"median of {PREFILL_CALLS} calls after {PREFILL_WARMUP} warm-up calls, each bracketed by CUDA "
                      "events on the launch stream, arguments prepared once (ForwardCall)",
            "workspace_bytes": int(ws_two_phase.numel()),
            "single_kernel_ms": round(ms_single, 4),
            "roofline": {"bound": "tensor", "kernel": "wy_prep_kernel + wy_scan_kernel (two-phase chunked)",
                         "achieved": round(tflops, 2),
                         "peak": tc_peak, "peak_kind": f"{kind} dense bf16 burst (fp16 runs at the bf16 rate)",
                         "unit": "TFLOP/s", "frac": round(tflops / tc_peak, 4), "algorithmic_flops": flops,
                         "executed_mma_flops": executed,
                         "executed_tflops": round(executed / (ms / 1e3) / 1e12, 2),
                         "traffic": recorded_traffic(os.path.join(ROOT, "gated_delta_rule_gateddeltanet_gb300", "csrc",
                                                                  "gdn_chunked_wy.cu"),
                                                     "varlen_prefill.wy_kernels.ncu.md")}}


def long_prefill_inputs(dev, T=262144, Hk=16, Hv=48, d=128, seed=1006):
    """The long-prefill batch (one sequence of T tokens), drawn on the device
    from a seeded generator: q, k, v ~ N(0,1) fp16, raw a, b ~ N(0,1), and the
    gate parameters of the other workloads."""
    import torch
    from gated_delta_rule_gateddeltanet_gb300 import workloads as wl
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    rnd = lambda shape, dt: torch.randn(shape, generator=gen, device=dev, dtype=dt)
    q, k, v = rnd((T, Hk, d), torch.float16), rnd((T, Hk, d), torch.float16), rnd((T, Hv, d), torch.float16)
    aa, bb = rnd((T, Hv), torch.float32), rnd((T, Hv), torch.float32)
    A_log, dt_bias = (torch.from_numpy(x).to(dev) for x in wl.gate_params(np.random.default_rng(seed), Hv))
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    return q, k, v, aa, bb, A_log, dt_bias, cu


def run_long_prefill(dev, stream):
    """One 262,144-token sequence (the pages' 256k context), Hk=16, Hv=48,
    d=128, fp16, zero initial state, under the chunked plan (48 chains) and
    the sequence-parallel split plan (144 chains + the combining kernels).
    Inputs are drawn on the device from a seeded generator (5.4 GB, far
    larger than L2)."""
    import torch
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    q, k, v, aa, bb, A_log, dt_bias, cu = long_prefill_inputs(dev)
    T, Hk, d = q.shape
    Hv = v.shape[1]
    final = torch.zeros((1, Hv, d, d), dtype=torch.float32, device=dev)
    out = torch.empty((T, Hv, d), dtype=torch.float16, device=dev)
    res = {}
    for plan in ("chunked", "chunked_split"):
        args, _, _ = gdn.build_forward_args(q, k, v, aa, bb, cu, A_log=A_log, dt_bias=dt_bias, final_state=final,
                                            output=out, plan=plan)
        ws = torch.empty(gdn.workspace_size(args), dtype=torch.uint8, device=dev)
        run = lambda: gdn.gdn_forward(q, k, v, aa, bb, cu, A_log=A_log, dt_bias=dt_bias, final_state=final,
                                      output=out, plan=plan, workspace=ws)
        run()
        times = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        res[plan] = (statistics.median(times), int(ws.numel()))
        del ws
        torch.cuda.empty_cache()
    _, tc_peak, kind = measured_peaks()
    flops = prefill_algorithmic_flops(T)
    ms_seq, ws_seq = res["chunked"]
    ms_split, ws_split = res["chunked_split"]
    tflops = flops / (ms_split / 1e3) / 1e12
    return {"workload": "long prefill: 1 sequence of 262,144 tokens, Hk=16, Hv=48, d=128, fp16, zero initial state "
                        "(inputs drawn on the device, seed 1006)", "tokens": T,
            "chunked_ms": round(ms_seq, 3), "chunked_split_ms": round(ms_split, 3),
            "speedup": round(ms_seq / ms_split, 3), "tokens_per_s": round(T / (ms_split / 1e3), 1),
            "workspace_bytes": {"chunked": ws_seq, "chunked_split": ws_split},
            "roofline": {"bound": "tensor", "kernel": "split plan: prep + scan (144 chains) + correction + final",
                         "achieved": round(tflops, 2), "peak": tc_peak,
                         "peak_kind": f"{kind} dense bf16 burst (fp16 runs at the bf16 rate)", "unit": "TFLOP/s",
                         "frac": round(tflops / tc_peak, 4), "algorithmic_flops": flops}}


# Algorithmic FLOPs of the chunked evaluation per token and value head (chunk
# C = 64, d = 128, r = 3 value heads per key head): the state-passing products
# 6 d^2, the intra-chunk products C (2d/r + d + 2d) (K K^T and Q K^T shared by
# the r value heads of a key head), and the triangular inverse C^2 / 3.
PREFILL_FLOPS_PER_TOKEN_HEAD = 6 * 128 * 128 + 64 * (2 * 128 / 3 + 128 + 2 * 128) + 64 * 64 / 3
# tcgen05 FLOPs the two-phase path issues per (64-token chunk, value head): in
# the scan kernel MMA2 128x128x128, MMA3 and MMA4 128x64x64, MMA5 128x128x64;
# in the prep kernel [Q;K]K^T 128x64x128 once per key head (r = 3 value heads).
PREFILL_MMA_FLOPS_PER_CHUNK_HEAD = (2 * (128 * 128 * 128 + 2 * 128 * 64 * 64 + 128 * 128 * 64)
                                    + 2 * 128 * 64 * 128 // 3)


def prefill_algorithmic_flops(tokens, heads=48):
    return int(tokens * heads * PREFILL_FLOPS_PER_TOKEN_HEAD)


def run_spec(dev, stream, lib, sh):
    """Speculative verify (16 x 4 tokens with capsules) then replay of the
    accepted prefixes into the inactive bank; 4 rotating state pools."""
    import torch
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    from gated_delta_rule_gateddeltanet_gb300 import workloads as wl
    pools, fargs, rargs = [], [], []
    for i in range(NBUF):
        inp = wl.spec_verify(seed=wl.SEEDS["spec_verify"] + 100 * i)
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        pool = t(inp.initial_state)
        caps = torch.zeros((16, 4, gdn.capsule_width(16, 48, 128, 128)), dtype=torch.float32, device=dev)
        scratch = torch.empty_like(pool[:16])
        d = dict(q=t(inp.q), k=t(inp.k), v=t(inp.v), a=t(inp.a), b=t(inp.b), A_log=t(inp.A_log),
                 dt_bias=t(inp.dt_bias), cu=t(inp.cu_seqlens), slots=t(inp.state_slots),
                 out=torch.empty((inp.T, 48, 128), dtype=torch.float16, device=dev), pool=pool, caps=caps,
                 src=t(inp.extra["src_slots"]), dst=t(inp.extra["dst_slots"]), n=t(inp.extra["accept_len"]),
                 scratch=scratch)
        # verify writes the speculative final state to a scratch pool (slots 0..15 of `scratch`)
        args, _, keep = gdn.build_forward_args(d["q"], d["k"], d["v"], d["a"], d["b"], d["cu"], A_log=d["A_log"],
                                               dt_bias=d["dt_bias"], initial_state=pool, final_state=scratch,
                                               state_slots=None, output=d["out"], state_update=caps, capacity=4,
                                               num_state_slots=16, max_seqlen=4)
        # the same verify writing no final state (its capsules are what the replay needs)
        args_ns, _, keep_ns = gdn.build_forward_args(d["q"], d["k"], d["v"], d["a"], d["b"], d["cu"],
                                                     A_log=d["A_log"], dt_bias=d["dt_bias"], initial_state=pool,
                                                     state_slots=None, output=d["out"], state_update=caps,
                                                     capacity=4, num_state_slots=16, max_seqlen=4,
                                                     write_final_state=False)
        d["args"], d["keep"], d["acc"] = args, keep, int(inp.extra["accept_len"].sum())
        d["args_ns"], d["keep_ns"] = args_ns, keep_ns
        pools.append(d)

    cur = [sh]  # the stream the calls go to (the graph capture uses a side stream)

    def verify(i):
        rc = lib.gdn_forward(ctypes.byref(pools[i % NBUF]["args"]), cur[0])
        if rc:
            raise gdn.GdnError(rc, "gdn_forward")

    def verify_no_state(i):
        rc = lib.gdn_forward(ctypes.byref(pools[i % NBUF]["args_ns"]), cur[0])
        if rc:
            raise gdn.GdnError(rc, "gdn_forward")

    def replay(i):
        d = pools[i % NBUF]
        rc = lib.gdn_replay_prefix(ctypes.c_void_p(d["pool"].data_ptr()), 32, 16, 16, 48, 128, 128,
                                   ctypes.c_void_p(d["src"].data_ptr()), ctypes.c_void_p(d["dst"].data_ptr()),
                                   ctypes.c_void_p(d["caps"].data_ptr()), 4, ctypes.c_void_p(d["n"].data_ptr()),
                                   None, cur[0])
        if rc:
            raise gdn.GdnError(rc, "gdn_replay_prefix")

    res, host = {}, {}
    for name, fn in (("verify", verify), ("verify_no_state", verify_no_state), ("replay", replay)):
        for i in range(20):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # device time: 40 launches captured in one CUDA graph, replayed 10 times (median)
        n = 40
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        cur[0] = ctypes.c_void_p(side.cuda_stream)
        with torch.cuda.graph(graph, stream=side):
            for i in range(n):
                fn(i)
        cur[0] = sh
        graph.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(10):
            with torch.cuda.stream(side):
                e0.record()
                graph.replay()
                e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / n)
        res[name] = statistics.median(ts)
        del graph
        # the same calls launched one by one from the host (adds the per-call host time)
        m = 400
        e0.record(stream)
        for i in range(m):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        host[name] = e0.elapsed_time(e1) / m
    hbm_peak, _, kind = measured_peaks()
    state_bytes = 2 * 16 * 48 * 128 * 128 * 4
    cap_bytes = gdn.capsule_width(16, 48, 128, 128) * 4
    rep_bytes = state_bytes + statistics.mean(d["acc"] for d in pools) * cap_bytes
    ver_bytes = state_bytes + 64 * (33152 + cap_bytes)
    ver_ns_bytes = state_bytes // 2 + 64 * (33152 + cap_bytes)
    return {"workload": "spec verify + replay: 16 requests x 4 draft tokens, Hk=16, Hv=48, d=128, fp16, "
                        "capsules for all tokens, replay of U{0..4} accepted into the inactive bank",
            "timing": "device time: 40 launches in one CUDA graph, median of 10 replays; *_host_loop_us: the "
                      "same calls launched one by one through the C ABI",
            "verify_us": round(res["verify"] * 1e3, 2), "replay_us": round(res["replay"] * 1e3, 2),
            "verify_no_final_state_us": round(res["verify_no_state"] * 1e3, 2),
            "verify_host_loop_us": round(host["verify"] * 1e3, 2),
            "verify_no_final_state_host_loop_us": round(host["verify_no_state"] * 1e3, 2),
            "replay_host_loop_us": round(host["replay"] * 1e3, 2),
            "verify_tokens_per_s": round(64 / (res["verify"] / 1e3), 1),
            "replay_gbs": round(rep_bytes / (res["replay"] / 1e3) / 1e9, 1),
            "replay_frac_hbm": round(rep_bytes / (res["replay"] / 1e3) / 1e9 / hbm_peak, 4),
            "verify_gbs": round(ver_bytes / (res["verify"] / 1e3) / 1e9, 1),
            "verify_frac_hbm": round(ver_bytes / (res["verify"] / 1e3) / 1e9 / hbm_peak, 4),
            "verify_no_final_state_frac_hbm": round(ver_ns_bytes / (res["verify_no_state"] / 1e3) / 1e9 / hbm_peak, 4),
            "l2": f"{NBUF} rotating state pools of 96 MiB"}


def run_conv(dev, stream):
    """The packed causal conv in front of the GatedDeltaNet (channels 2*16*128
    + 48*128 = 10240, kernel 4, fp16, SiLU, state updated in place) on the
    decode step (64 x 1 token, capture of 1 token) and on the varlen prefill."""
    import torch
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    from gated_delta_rule_gateddeltanet_gb300 import workloads as wl
    C, K = 10240, 4
    hbm, _, kind = measured_peaks()
    res = {}
    for name, lengths, cap in (("decode", [1] * 64, 1), ("prefill", list(wl.varlen_prefill_lengths()), 0)):
        rng = np.random.default_rng(77)
        T, B = int(sum(lengths)), len(lengths)
        x = torch.from_numpy(rng.standard_normal((T, C), dtype=np.float32).astype(np.float16)).to(dev)
        w = torch.from_numpy(rng.standard_normal((C, K), dtype=np.float32)).to(dev)
        bias = torch.zeros(C, dtype=torch.float32, device=dev)
        cu = torch.from_numpy(wl.cu_from_lengths(lengths)).to(dev)
        states = [torch.zeros((B, C, K - 1), dtype=torch.float16, device=dev) for _ in range(NBUF)]
        out = torch.empty((T, C), dtype=torch.float16, device=dev)
        caps = torch.zeros((B, max(cap, 1), C), dtype=torch.float16, device=dev)
        lib = gdn.load_library()
        args = [gdn.build_conv_args(x, w, cu, bias=bias, initial_state=states[i], final_state=states[i], output=out,
                                    state_update=caps if cap else None, capacity=cap,
                                    max_seqlen=max(lengths))[0] for i in range(NBUF)]

        def run(i, s):
            rc = lib.varlen_causal_conv_with_state(ctypes.byref(args[i % NBUF]), ctypes.c_void_p(s.cuda_stream))
            if rc:
                raise gdn.GdnError(rc, "varlen_causal_conv_with_state")
        for i in range(5):
            run(i, stream)
        torch.cuda.synchronize()
        n = 200 if name == "decode" else 20
        # the launches are captured in a CUDA graph and replayed, so the host's
        # launch rate does not bound the few-microsecond decode case
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cs = torch.cuda.current_stream()
            for i in range(n):
                run(i, cs)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / n * 1e3
        nbytes = T * C * 2 * 2 + B * C * (K - 1) * 2 * 2 + T * min(cap, 1) * C * 2 + C * (K + 1) * 4
        res[name] = {"tokens": T, "us": round(us, 2), "tokens_per_s": round(T / (us / 1e6), 1),
                     "gbs": round(nbytes / (us / 1e6) / 1e9, 1), "frac_hbm": round(nbytes / (us / 1e6) / 1e9 / hbm, 4),
                     "algorithmic_bytes": nbytes}
    res["workload"] = ("causal conv: channels 10240, kernel 4, fp16, SiLU, in-place state; decode 64 x 1 token "
                       "(max_seqlen hint 1: one launch), prefill 8 x U[256,4096] tokens (conv + state roll: 2 launches); C ABI with "
                       "prebuilt arguments, launches captured in a CUDA graph and replayed")
    return res


def run_serving_mix(dev, stream, lib, sh):
    """32 x 2048-token packed prefill (zero initial state) followed by 256
    single-token decode steps on the resulting FP32 states, updated in place.
    Every decode step has fresh seeded inputs, copied to the device before the
    timed region; the launches go through the C ABI with prebuilt arguments."""
    import torch
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    from gated_delta_rule_gateddeltanet_gb300 import workloads as wl
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    pre = wl.serving_mix_prefill()
    B, L = pre.B, 2048
    state = torch.zeros((B, 48, 128, 128), dtype=torch.float32, device=dev)
    pout = torch.empty((pre.T, 48, 128), dtype=torch.float16, device=dev)
    keep = []
    pargs, _, k0 = gdn.build_forward_args(t(pre.q), t(pre.k), t(pre.v), t(pre.a), t(pre.b), t(pre.cu_seqlens),
                                          A_log=t(pre.A_log), dt_bias=t(pre.dt_bias), final_state=state,
                                          output=pout, max_seqlen=L)
    ws = torch.empty(gdn.workspace_size(pargs), dtype=torch.uint8, device=dev)
    pargs.workspace, pargs.workspace_bytes = ctypes.c_void_p(ws.data_ptr()), ws.numel()
    keep += [k0, ws]
    steps = 256
    dargs = []
    dout = torch.empty((B, 48, 128), dtype=torch.float16, device=dev)
    for s in range(steps):
        d = wl.serving_mix_decode(s, pre)
        args, _, kk = gdn.build_forward_args(t(d.q), t(d.k), t(d.v), t(d.a), t(d.b), t(d.cu_seqlens),
                                             A_log=t(d.A_log), dt_bias=t(d.dt_bias), initial_state=state,
                                             final_state=state, output=dout, max_seqlen=1)
        dargs.append(args)
        keep.append(kk)

    def call(args):
        rc = lib.gdn_forward(ctypes.byref(args), sh)
        if rc:
            raise gdn.GdnError(rc, "gdn_forward")

    def once():
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        state.zero_()
        ev[0].record(stream)
        call(pargs)
        ev[1].record(stream)
        for a in dargs:
            call(a)
        ev[2].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])

    once()  # warm-up
    runs = [once() for _ in range(3)]
    p_ms = statistics.median(r[0] for r in runs)
    d_ms = statistics.median(r[1] for r in runs)
    hbm, tc, kind = measured_peaks()
    dec_bytes = decode_bytes_per_launch(B, 16, 48, 128, 128)
    return {"workload": "serving mix: 32 x 2048-token packed prefill (fp16, Hk=16, Hv=48, d=128, zero initial "
                        "state) then 256 single-token decode steps on the resulting fp32 states, fresh seeded "
                        "inputs per step, state updated in place",
            "prefill_ms": round(p_ms, 3), "prefill_tokens_per_s": round(pre.T / (p_ms / 1e3), 1),
            "prefill_tflops": round(prefill_algorithmic_flops(pre.T) / (p_ms / 1e3) / 1e12, 2),
            "decode_ms_total": round(d_ms, 3), "decode_us_per_step": round(d_ms / steps * 1e3, 2),
            "decode_tokens_per_s": round(B * steps / (d_ms / 1e3), 1),
            "decode_frac_hbm": round(dec_bytes / (d_ms / steps / 1e3) / 1e9 / hbm, 4),
            "tokens_per_s": round((pre.T + B * steps) / ((p_ms + d_ms) / 1e3), 1),
            "launches": 2 + steps}


def run_transpose(dev, stream, lib, sh):
    """K-major <-> V-major conversion of the decode step's state pool
    (64 x 48 matrices of 128 x 128 FP32 = 192 MiB each way), 4 rotating pairs."""
    import torch
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    n = 64 * 48
    pairs = [(torch.randn((n, 128, 128), device=dev), torch.empty((n, 128, 128), device=dev)) for _ in range(NBUF)]

    def call(i):
        src, dst = pairs[i % NBUF]
        rc = lib.gdn_state_transpose(ctypes.c_void_p(src.data_ptr()), ctypes.c_void_p(dst.data_ptr()), n, 128, 128,
                                     sh)
        if rc:
            raise gdn.GdnError(rc, "gdn_state_transpose")
    for i in range(5):
        call(i)
    torch.cuda.synchronize()
    reps = 40
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(reps):
        call(i)
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    hbm, _, _ = measured_peaks()
    nbytes = 2 * n * 128 * 128 * 4
    return {"workload": "state layout conversion: 3072 matrices of 128 x 128 fp32 (the decode pool), 4 rotating pairs",
            "us": round(us, 2), "gbs": round(nbytes / (us / 1e6) / 1e9, 1),
            "frac_hbm": round(nbytes / (us / 1e6) / 1e9 / hbm, 4)}


def run_spec_step(dev, stream):
    """A whole speculative step of one layer (conv with capture -> gdn_forward
    with capsules on the fused q|k|v view -> conv replay -> GDN replay),
    16 requests x 4 drafts at the Qwen geometry, launched eagerly through the
    C ABI with prebuilt arguments vs replayed from one CUDA graph."""
    import torch
    from gated_delta_rule_gateddeltanet_gb300.spec_step import SpeculativeStep
    from gated_delta_rule_gateddeltanet_gb300 import workloads as wl
    R, D, Hk, Hv, d = 16, 4, 16, 48, 128
    C = 2 * Hk * d + Hv * d
    inp = wl.spec_verify()
    g = torch.Generator().manual_seed(11)
    s = SpeculativeStep(torch.randn((C, 4), generator=g).to(dev), torch.zeros(C, device=dev),
                        torch.randn((2 * R, C, 3), generator=g).to(torch.float16).to(dev),
                        torch.from_numpy(inp.A_log).to(dev), torch.from_numpy(inp.dt_bias).to(dev),
                        torch.randn((2 * R, Hv, d, d), generator=g).mul_(0.02).to(dev), num_k_heads=Hk, drafts=D)
    s.x.copy_(torch.randn((R * D, C), generator=g).to(torch.float16))
    s.a.copy_(torch.from_numpy(inp.a))
    s.b.copy_(torch.from_numpy(inp.b))
    s.accept_len.copy_(torch.from_numpy(inp.extra["accept_len"]))
    s.capture()
    res = {}
    for name, fn in (("eager_us", lambda: s.run_eager(stream)), ("graph_us", s.replay)):
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        n = 200
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = round(e0.elapsed_time(e1) / n * 1e3, 2)
    res["workload"] = ("speculative step of one layer: 16 requests x 4 drafts, conv (10240 channels, capture) + "
                       "gdn_forward (capsules) + conv replay (on a side stream, overlapping the GDN replay) + GDN replay of "
                       "U{0..4} accepted tokens; 4 launches eager (prebuilt C-ABI arguments) vs one CUDA-graph replay")
    res["tokens_per_s_graph"] = round(R * D / (res["graph_us"] / 1e6), 1)
    return res


# ---------------------------------------------------------------- CPU oracle (baseline and reference arm)

def oracle_decode_sample(inp, requests):
    """The first ``requests`` requests of a decode step, as oracle inputs."""
    cu = inp.cu_seqlens[:requests + 1]
    T = int(cu[-1])
    return dict(q=inp.q[:T], k=inp.k[:T], v=inp.v[:T], a=inp.a[:T], b=inp.b[:T], cu=cu,
                state=inp.initial_state[:requests], A_log=inp.A_log, dt_bias=inp.dt_bias)


def time_oracle_step(s):
    import oracle
    t0 = time.perf_counter()
    oracle.gdn_forward(s["q"], s["k"], s["v"], s["a"], s["b"], s["cu"], A_log=s["A_log"], dt_bias=s["dt_bias"],
                       initial_state=s["state"])
    return time.perf_counter() - t0


def run_cpu_baseline(inp, budget_s=12.0):
    import oracle
    oracle.build()
    full = oracle_decode_sample(inp, inp.B)
    t1 = time_oracle_step(full)
    reps = max(1, int(budget_s / max(t1, 1e-3)))
    total, n = 0.0, 0
    for _ in range(reps):
        total += time_oracle_step(full)
        n += 1
    return {"value": round(n * inp.B / total, 2), "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{n} full decode steps (64 requests x 1 token, all 48 heads) in {total:.1f} s, FP64 C oracle "
                      f"with OpenMP over (request, head) chains"}


# seconds of oracle work the reference arm spreads over its warm-up and timed steps
REFERENCE_BUDGET_S = 150.0


def run_reference(a, dist: Dist):
    if dist.rank != 0:
        return
    import oracle
    from gated_delta_rule_gateddeltanet_gb300 import workloads as wl
    oracle.build()
    inp = wl.decode_step()
    full = oracle_decode_sample(inp, inp.B)
    t_full = time_oracle_step(full)
    per_step = REFERENCE_BUDGET_S / max(1, a.steps + a.warmup)
    req = int(max(1, min(inp.B, math.floor(inp.B * per_step / max(t_full, 1e-6)))))
    s = oracle_decode_sample(inp, req)
    for _ in range(a.warmup):
        time_oracle_step(s)
    t = sum(time_oracle_step(s) for _ in range(a.steps))
    value = req * a.steps / t
    sample = (f"each step: the first {req} of the 64 requests of the decode step (1 token each, all 48 heads), "
              f"FP64 C oracle, OpenMP over (request, head) chains")
    line = {"metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": a.gpus, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": round(t / a.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(inp.B, *inp.dims, a.gpus),
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": oracle.threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# The sub-measurements reported beside the headline (see run_gdn), by name.
SUB_MEASUREMENTS = {"prefill": run_prefill, "spec_verify_replay": run_spec, "causal_conv": run_conv,
                    "serving_mix": run_serving_mix, "state_transpose": run_transpose,
                    "spec_step_graph": run_spec_step, "long_prefill": run_long_prefill}
NEEDS_LIB = {"spec_verify_replay", "serving_mix", "state_transpose"}


def run_only(name):
    """One sub-measurement alone (e.g. under a profiler), printed as JSON."""
    import torch
    import gated_delta_rule_gateddeltanet_gb300 as gdn
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib = gdn.load_library()
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    fn = SUB_MEASUREMENTS[name]
    res = fn(dev, stream, lib, sh) if name in NEEDS_LIB else fn(dev, stream)
    print(json.dumps({"only": name, name: res}), flush=True)


def main():
    a = parse()
    if a.only:
        run_only(a.only)
        return
    dist = Dist()
    try:
        if a.impl == "reference":
            run_reference(a, dist)
        else:
            run_gdn(a, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
