#!/usr/bin/env python3
"""Throughput of the linear-attention hot path on GB300, one JSON line on rank 0.

Headline step: one causal forward (keeping Out) plus one causal backward on the
training workload B=4, H=16, N=8192, D=M=64, bf16 storage, fp32 accumulation.
tokens/s counts (b, n) positions across all heads: B*N tokens per step.

Also measured in the same run (the "paths" object): the causal forward alone,
the long-sequence forward (B=1, H=16, N=65536, D=M=128), the non-causal fp32
forward and backward (B=8, H=8, N=4096, D=M=64), one decode step of 256 sequences x 16
heads (D=M=64, fp32 state), the softmax KV-cache decode step it replaces (the
same heads with a full 4096-position cache), gated retention (forward on the
training shape, one decode step), the degree-2 polynomial feature map (causal,
B=4 H=16 N=4096 D=32 M=64, against the FP32 FMA rate) and the 2048-token prefill that hands the
decode its state (the causal forward emitting the final S, Z of every head), each
with its fraction of the HBM roofline.

Timing: W untimed warm-up steps, then K steps between a barrier and a device
synchronize, timed with CUDA events on the launching stream; max over ranks.
The training inputs (4 x 64 MiB) exceed L2, so consecutive steps do not reuse
L2; the decode state (64 MiB) fits in L2, so the decode step is timed in steady
state over four independent states (256 MiB, back to back, no flush), with the
single step after an L2 flush reported beside it; the softmax KV-cache step
reads a 4.3 GB cache, far larger than L2; the polynomial path, whose inputs fit
in L2, flushes it before each call (a 256 MiB write, then a 256 MiB read, so
that the flush's own dirty lines are written back before the call).  Every
path's calls are enqueued back to back with no host wait between them.

--impl reference times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal linear-attn tokens/s (fwd, fwd+bwd, decode) and % of roofline"
HEADLINE = "causal_train_bf16"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- helpers

def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources the training step's kernels are built from (and the C ABI that launches them):
# the DRAM counters in profiles/traffic.json hold while these are unchanged.
TRAFFIC_SOURCES = ("causal_tc.cu", "causal_bwd_tc.cu", "tc_common.cuh", "tc_ptx.cuh", "la_common.cuh",
                   "la_launch.h", "la_api.cu")


def _csrc_hash() -> str:
    d = os.path.join(ROOT, "linear_attention_02_gb300", "csrc")
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _traffic(key: str):
    """DRAM bytes per launch from a committed ncu capture, or None if absent/stale."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(key)
    if not e or e.get("csrc_hash") != _csrc_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clocks and clock-event (throttle) reasons sampled during the timed region.

    Polls NVML (read-only queries through ctypes) every 0.5 ms on the GPU the
    process runs on, matched by PCI bus id; falls back to nvidia-smi at its
    100 ms minimum interval when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []  # (sm_mhz, max_mhz, reason_bits)
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None

    def _open_nvml(self):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return False
        handle = ctypes.c_void_p()
        bus = None
        try:
            pr = torch.cuda.get_device_properties(self.cuda_index)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
        except Exception:
            bus = None
        if bus is None or lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(handle)) != 0:
            if lib.nvmlDeviceGetHandleByIndex_v2(self.cuda_index, ctypes.byref(handle)) != 0:
                return False
        self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self._nvml, self._handle = lib, handle
        return True

    def _poll_nvml(self):
        import ctypes
        lib, h = self._nvml, self._handle
        cur, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(cur)) == 0 and
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0):
                r = self._reasons_fn(h, ctypes.byref(rs))
                self.samples.append((cur.value, mx.value, rs.value if r == 0 else 0))
            time.sleep(0.0005)

    def _poll_smi(self):
        cmd = ["nvidia-smi", "-i", str(self.cuda_index), "--query-gpu=clocks.sm,clocks.max.sm,"
               "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "100"]
        proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        while not self._stop.is_set():
            line = proc.stdout.readline()
            if not line:
                break
            parts = [x.strip() for x in line.split(",")]
            try:
                self.samples.append((float(parts[0]), float(parts[1]), int(parts[2], 16)))
            except (ValueError, IndexError):
                pass
        proc.terminate()

    def __enter__(self):
        try:
            use_nvml = self._open_nvml()
        except Exception:
            use_nvml = False
        self._thread = threading.Thread(target=self._poll_nvml if use_nvml else self._poll_smi,
                                        daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self._thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = set()
        for _, _, bits in self.samples:
            for b, name in self.REASONS.items():
                if bits & b:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x[0] for x in self.samples),
                "sm_max_mhz": max(x[1] for x in self.samples), "reasons": sorted(reasons),
                "samples": len(self.samples)}


# ------------------------------------------------------------- workloads

def _bytes_fwd(B, H, N, D, M, esz, den=False):
    # read Q, K, V; write Out (+ the fp32 normaliser per token)
    return B * H * N * ((2 * D + 2 * M) * esz + (4 if den else 0))


def _bytes_bwd(B, H, N, D, M, esz, with_out=True, den=False):
    # read Q, K, V, dOut (+ Out, + the fp32 normaliser per token); write dQ, dK, dV
    return B * H * N * ((2 * D + 2 * M + (M if with_out else 0) + 2 * D + M) * esz + (4 if den else 0))


def _bytes_decode(B, H, D, M, esz):
    return B * H * (2 * D * M * 4 + 2 * D * 4 + (2 * D + M) * esz + M * 4)


def _bf16_tensor_tflops():
    """Dense bf16 tensor-core peak: the measured burst cuBLAS figure (this path is timed alone),
    else the profiling recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def _time_events(torch, fn, reps, stream, flush=None):
    """Mean device ms of fn over reps, CUDA events on `stream`.

    The calls are enqueued one behind the other with no host wait in between: a wait
    lets the GPU go idle while the host makes the next call (Python, ctypes, the
    launches), and an event pair around that call would count the idle time.
    Without `flush` one event pair spans all reps; with it, each call has its own pair
    after its (untimed) flush, which keeps the GPU busy while the call is enqueued."""
    if flush is None:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / reps
    evs = []
    for _ in range(reps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / reps


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import linear_attention_02_gb300 as la
    from linear_attention_02_gb300 import synth

    hbm, peak_src = _peaks()
    stream = torch.cuda.current_stream()
    w = synth.WORKLOADS[HEADLINE]
    B, H, N, D, M = w.B, w.H, w.N, w.D, w.M
    seed = w.seed + 7919 * rank  # each rank its own batch (weak scaling)
    x = synth.qkv(B, H, N, D, M, w.dtype, seed, w.scale, with_grad=True, device="cuda")
    Q, K, V, G = x["Q"], x["K"], x["V"], x["G"]
    O = torch.empty_like(V)
    den = torch.empty((B, H, N), dtype=torch.float32, device="cuda")  # normaliser kept for the backward
    ckpt = torch.empty(la.la_causal_ckpt_floats(B, H, N, D, M), dtype=torch.float32, device="cuda")
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)

    ev = []

    def step(record=False):
        if record:
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
        la.la_forward_causal(Q, K, V, out=O, den=den, ckpt=ckpt)
        if record:
            e1.record(stream)
        la.la_backward_causal(Q, K, V, G, Out=O, dQ=dQ, dK=dK, dV=dV, Den=den, Ckpt=ckpt)
        if record:
            e2.record(stream)
            ev.append((e0, e1, e2))

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches0 = la.la_kernel_launch_count()
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step(record=True)
        t1.record(stream)
        torch.cuda.synchronize()
    launches = la.la_kernel_launch_count() - launches0
    ms_total = t0.elapsed_time(t1)
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in ev)
    bwd_ms = statistics.mean(b.elapsed_time(c) for _, b, c in ev)
    if world > 1:
        t = torch.tensor([ms_total], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
    ms_step = ms_total / args.steps
    tokens = B * N * world
    value = tokens / (ms_step / 1e3)

    # end to end: pinned host inputs -> device -> fwd + bwd -> host outputs, every step.
    # Pipelined over three streams with two device buffer sets: step k's input copy and
    # step k-1's output copy run while step k computes (separate copy engines), the way a
    # training loop feeds a device; every byte still crosses the link inside the timed region.
    hx = {k: v.cpu().pin_memory() for k, v in x.items()}
    slots = []
    for _ in range(2):
        dxs = {k: torch.empty_like(v) for k, v in x.items()}
        outs = [torch.empty_like(t) for t in (O, dQ, dK, dV)]
        slots.append((dxs, outs, [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]))
    hout = slots[0][2]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_cmp + ev_out:
        e.record(stream)

    def e2e_step(k):
        dxs, outs, houts = slots[k & 1]
        s_in.wait_event(ev_cmp[k & 1])          # step k - 2 is done with these inputs
        with torch.cuda.stream(s_in):
            for name in dxs:
                dxs[name].copy_(hx[name], non_blocking=True)
        ev_in[k & 1].record(s_in)
        stream.wait_event(ev_in[k & 1])
        stream.wait_event(ev_out[k & 1])        # step k - 2's outputs are read out
        Ok, dQk, dKk, dVk = outs
        la.la_forward_causal(dxs["Q"], dxs["K"], dxs["V"], out=Ok, den=den, ckpt=ckpt, stream=stream)
        la.la_backward_causal(dxs["Q"], dxs["K"], dxs["V"], dxs["G"], Out=Ok, dQ=dQk, dK=dKk, dV=dVk,
                              Den=den, Ckpt=ckpt, stream=stream)
        ev_cmp[k & 1].record(stream)
        s_out.wait_event(ev_cmp[k & 1])
        with torch.cuda.stream(s_out):
            for h, d in zip(houts, outs):
                h.copy_(d, non_blocking=True)
        ev_out[k & 1].record(s_out)

    for k in range(2):
        e2e_step(k)
    torch.cuda.synchronize()
    e2e_steps = max(4, min(args.steps, 20))
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for k in range(e2e_steps):
        e2e_step(k)
    s_out.wait_event(ev_cmp[(e2e_steps - 1) & 1])
    b.record(s_out)
    b.synchronize()
    e2e_ms = a.elapsed_time(b) / e2e_steps
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    h2d = sum(v.numel() * v.element_size() for v in hx.values())
    d2h = sum(h.numel() * h.element_size() for h in hout)

    esz = 2
    fwd_bytes = _bytes_fwd(B, H, N, D, M, esz, den=True)
    bwd_bytes = _bytes_bwd(B, H, N, D, M, esz, with_out=True, den=True)
    dom, dom_ms, dom_bytes = ("la_backward_causal", bwd_ms, bwd_bytes) if bwd_ms >= fwd_ms else \
        ("la_forward_causal", fwd_ms, fwd_bytes)
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm,
                "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "traffic": _traffic(f"{HEADLINE}/{dom}"),
                "algorithmic_bytes": dom_bytes, "avg_ms": round(dom_ms, 5)}

    paths = None
    clk_paths = None
    if not args.no_paths:
        with ClockSampler(local) as clk_paths:
            paths = measure_paths(torch, la, synth, stream, hbm, fwd_ms, bwd_ms, fwd_bytes, bwd_bytes,
                                  B * N)

    if world > 1:
        dist.barrier()
    out = None
    if rank == 0:
        clocks = clk.summary()
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"{HEADLINE}: causal linear attention fwd+bwd, B={B} H={H} "
                                   f"N={N} D=M={D}, bf16 storage, fp32 accumulation, "
                                   "phi=elu+1, Out, the normaliser and state checkpoints kept from the forward",
                       "global_batch": B * world, "seq_len": N, "heads": H, "head_dim": D,
                       "parallelism": f"replicas x{world} (independent batches, no collective)",
                       "l2": "inputs larger than L2 (4 x 64 MiB resident per rank)"},
            "roofline": roofline,
            "e2e": {"value": round(tokens / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms, 4),
                    "pipelining": "input copies, compute and output copies on three streams, "
                                  "two device buffer sets; every step's bytes cross inside the "
                                  "timed region"},
            "gpu_launches": launches,
            "clocks": clocks,
            "paths": paths,
            "clocks_paths": clk_paths.summary() if clk_paths is not None else None,
        }
        if not args.no_cpu:
            out["cpu_baseline"] = cpu_baseline(synth)
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return out


def measure_paths(torch, la, synth, stream, hbm, fwd_ms, bwd_ms, fwd_bytes, bwd_bytes, tok):
    res = {}

    def entry(ms, byts, tokens, extra=None):
        gbs = byts / (ms / 1e3) / 1e9
        d = {"ms": round(ms, 5), "tokens_per_s": round(tokens / (ms / 1e3), 1),
             "algorithmic_bytes": byts, "achieved_gbs": round(gbs, 1),
             "hbm_frac": round(gbs / hbm, 4)}
        if extra:
            d.update(extra)
        return d

    res["causal_train_bf16/fwd"] = entry(fwd_ms, fwd_bytes, tok)
    res["causal_train_bf16/bwd"] = entry(bwd_ms, bwd_bytes, tok)
    res["causal_train_bf16/fwd+bwd"] = entry(fwd_ms + bwd_ms, fwd_bytes + bwd_bytes, tok)

    w = synth.WORKLOADS["causal_long_bf16"]
    x = synth.qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.scale, device="cuda")
    O = torch.empty_like(x["V"])
    f = lambda: la.la_forward_causal(x["Q"], x["K"], x["V"], out=O)
    for _ in range(3):
        f()
    ms = _time_events(torch, f, 10, stream)
    res["causal_long_bf16/fwd"] = entry(ms, _bytes_fwd(w.B, w.H, w.N, w.D, w.M, 2), w.B * w.N)
    del x, O

    w = synth.WORKLOADS["noncausal_f32"]
    x = synth.qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.scale, device="cuda")
    O = torch.empty_like(x["V"])
    f = lambda: la.la_forward_noncausal(x["Q"], x["K"], x["V"], out=O)
    for _ in range(3):
        f()
    ms = _time_events(torch, f, 20, stream)
    res["noncausal_f32/fwd"] = entry(ms, _bytes_fwd(w.B, w.H, w.N, w.D, w.M, 4), w.B * w.N)
    # the non-causal backward on the same shape, taking the forward's output
    G = synth.randn((w.B, w.H, w.N, w.M), w.dtype, w.seed + 1, device="cuda")
    dQ, dK, dV = torch.empty_like(x["Q"]), torch.empty_like(x["K"]), torch.empty_like(x["V"])
    f = lambda: la.la_backward_noncausal(x["Q"], x["K"], x["V"], G, Out=O, dQ=dQ, dK=dK, dV=dV)
    for _ in range(3):
        f()
    ms = _time_events(torch, f, 20, stream)
    res["noncausal_f32/bwd"] = entry(ms, _bytes_bwd(w.B, w.H, w.N, w.D, w.M, 4, with_out=True),
                                     w.B * w.N)
    del x, O, G, dQ, dK, dV

    w = synth.WORKLOADS["decode_bf16"]
    B, H, D, M = w.B, w.H, w.D, w.M
    S = torch.randn(B, H, D, M, device="cuda").abs_()
    Z = torch.rand(B, H, D, device="cuda").add_(1.0)
    steps = [synth.decode_step_qkv(B, H, D, M, w.dtype, w.seed, t, device="cuda") for t in range(8)]
    out = torch.empty(B, H, M, device="cuda")
    flush_buf = torch.empty(256 * 1024 * 1024 // 4, device="cuda")
    it = [0]

    def dec():
        s = steps[it[0] % len(steps)]
        it[0] += 1
        la.la_decode_step(s["q"], s["k"], s["v"], S, Z, out=out)

    flush_rd = torch.empty(256 * 1024 * 1024 // 4, device="cuda")
    sink = torch.empty(1, device="cuda")

    def flush():
        # write a buffer larger than L2, then read another: the state is out of L2 and the
        # flush's own dirty lines are written back before the timed step starts
        flush_buf.fill_(1.0)
        torch.sum(flush_rd, dim=0, keepdim=True, out=sink)

    for _ in range(3):
        dec()
    # steady state with the state larger than L2: back-to-back steps cycling over four
    # independent 64 MiB states (four decode batches), no flush, so each step reads a state
    # last touched three steps before (not in L2) and the write-backs of earlier steps'
    # states land inside the timed loop, as in a serving loop over several batches
    sets = [(torch.randn(B, H, D, M, device="cuda").abs_(), torch.rand(B, H, D, device="cuda").add_(1.0))
            for _ in range(4)]
    cyc = [0]

    def dec_rr():
        Sx, Zx = sets[cyc[0] % 4]
        s = steps[cyc[0] % len(steps)]
        cyc[0] += 1
        la.la_decode_step(s["q"], s["k"], s["v"], Sx, Zx, out=out)

    for _ in range(8):
        dec_rr()
    n_rr = 64
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_ev.record(stream)
    for _ in range(n_rr):
        dec_rr()
    b_ev.record(stream)
    b_ev.synchronize()
    ms = a_ev.elapsed_time(b_ev) / n_rr
    ms_flush = _time_events(torch, dec, 50, stream, flush=flush)
    ms_wr = _time_events(torch, dec, 50, stream, flush=lambda: flush_buf.fill_(1.0))
    ms_warm = _time_events(torch, dec, 50, stream)
    res["decode_bf16/step"] = entry(ms, _bytes_decode(B, H, D, M, 2), B, {
        "l2": "steady state: 64 back-to-back steps over four 64 MiB states (256 MiB > L2), no flush",
        "ms_flush_write_then_read": round(ms_flush, 5),
        "ms_flush_write_only": round(ms_wr, 5),
        "ms_l2_warm": round(ms_warm, 5)})
    del sets
    lin_ms = ms
    del S, Z, out

    # the softmax KV-cache step on the same heads at the end of the decode run (a full
    # cache of prefill + steps positions): what the recurrent step replaces
    T_max = w.prefill + w.steps
    Kc = synth.randn((B, H, T_max, D), w.dtype, w.seed + 2, device="cuda")
    Vc = synth.randn((B, H, T_max, M), w.dtype, w.seed + 3, device="cuda")
    out = torch.empty(B, H, M, device="cuda")
    T = T_max - 1
    f = lambda: la.la_softmax_decode_step(steps[0]["q"], steps[0]["k"], steps[0]["v"], Kc, Vc, T, out=out)
    for _ in range(3):
        f()
    ms = _time_events(torch, f, 10, stream)
    sd_bytes = B * H * (T * (D + M) * 2 + (D + M) * 2 + (2 * D + M) * 2 + M * 4)
    res["softmax_kv_decode_bf16/step"] = entry(ms, sd_bytes, B, {
        "cache_positions": T + 1, "l2": "the 4.3 GB cache is far larger than L2",
        "time_vs_recurrent_step": round(ms / lin_ms, 2)})
    del Kc, Vc, out, steps, flush_buf, flush_rd, sink

    # retention (decayed, unnormalised linear attention): gated decays on the training
    # workload's shape, and one gated decode step of the decode workload's heads
    wt = synth.WORKLOADS[HEADLINE]
    x = synth.qkv(wt.B, wt.H, wt.N, wt.D, wt.M, wt.dtype, wt.seed, wt.scale, device="cuda")
    gates = synth.decays((wt.B, wt.H, wt.N), wt.seed + 5, 0.85, 1.0, device="cuda")
    O = torch.empty_like(x["V"])
    f = lambda: la.la_forward_retention(x["Q"], x["K"], x["V"], gates=gates, out=O)
    for _ in range(3):
        f()
    ms = _time_events(torch, f, 10, stream)
    res["retention_gated_bf16/fwd"] = entry(
        ms, _bytes_fwd(wt.B, wt.H, wt.N, wt.D, wt.M, 2) + wt.B * wt.H * wt.N * 4, wt.B * wt.N)
    del x, O, gates
    Srs = [torch.randn(B, H, D, M, device="cuda") for _ in range(4)]  # four states, 256 MiB > L2
    sq = synth.decode_step_qkv(B, H, D, M, w.dtype, w.seed, 0, device="cuda")
    gate = synth.decays((B, H), w.seed + 6, 0.85, 1.0, device="cuda")
    out = torch.empty(B, H, M, device="cuda")
    cyc = [0]

    def f():
        la.la_retention_decode_step(sq["q"], sq["k"], sq["v"], Srs[cyc[0] % 4], gate=gate, out=out)
        cyc[0] += 1

    for _ in range(8):
        f()
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_ev.record(stream)
    for _ in range(64):
        f()
    b_ev.record(stream)
    b_ev.synchronize()
    ms = a_ev.elapsed_time(b_ev) / 64
    res["retention_gated_bf16/decode_step"] = entry(
        ms, B * H * (2 * D * M * 4 + (2 * D + M) * 2 + 4 + M * 4), B,
        {"l2": "steady state: 64 back-to-back steps over four 64 MiB states (256 MiB > L2), no flush"})
    del Srs, sq, gate, out

    # the degree-2 polynomial feature map (C = D^2 = 1024 features), causal, bf16: both
    # contractions on the tensor core, measured against the dense bf16 peak
    # Its inputs (67 MB) fit in L2: each call follows an L2 flush that writes, then reads,
    # a 256 MiB buffer (so the flush's own dirty lines are written back before the call)
    Bp, Hp, Np, Dp, Mp = 4, 16, 4096, 32, 64
    x = synth.qkv(Bp, Hp, Np, Dp, Mp, "bf16", 1007, device="cuda")
    O = torch.empty_like(x["V"])
    f = lambda: la.la_forward_poly2(x["Q"], x["K"], x["V"], causal=True, out=O)
    fl_w = torch.empty(256 * 1024 * 1024 // 4, device="cuda")
    fl_r = torch.empty(256 * 1024 * 1024 // 4, device="cuda")
    fl_s = torch.empty(1, device="cuda")

    def poly_flush():
        fl_w.fill_(1.0)
        torch.sum(fl_r, dim=0, keepdim=True, out=fl_s)

    for _ in range(3):
        f()
    ms = _time_events(torch, f, 10, stream, flush=poly_flush)
    flops = Bp * Hp * Np * 4 * Dp * Dp * (Mp + 1)  # phi(Q) [S | Z] and phi(K)^T [V | 1] per token
    tc_peak, tc_src = _bf16_tensor_tflops()
    d = entry(ms, _bytes_fwd(Bp, Hp, Np, Dp, Mp, 2), Bp * Np)
    d.update({"bound": "tensor", "algorithmic_tflops": round(flops / (ms / 1e3) / 1e12, 2),
              "tensor_peak_tflops": round(tc_peak, 1), "peak_source": tc_src,
              "tensor_frac": round(flops / (ms / 1e3) / 1e12 / tc_peak, 4),
              "workload": f"B={Bp} H={Hp} N={Np} D={Dp} M={Mp} bf16, causal",
              "l2": "flushed before each call (256 MiB written, then read)"})
    res["poly2_causal_bf16/fwd"] = d
    del x, O, fl_w, fl_r, fl_s

    # the prefill that hands the decode its state: the causal forward over every sequence's
    # prompt, emitting the final S, Z of each head (inputs larger than L2)
    x = synth.qkv(B, H, w.prefill, D, M, w.dtype, w.seed, w.scale, device="cuda")
    O = torch.empty_like(x["V"])
    f = lambda: la.la_forward_causal(x["Q"], x["K"], x["V"], out=O, return_state=True)
    for _ in range(3):
        f()
    ms = _time_events(torch, f, 10, stream)
    res["decode_bf16/prefill"] = entry(ms, _bytes_fwd(B, H, w.prefill, D, M, 2) + B * H * (D * M + D) * 4,
                                       B * w.prefill)
    del x, O
    return res


def cpu_baseline(synth, steps: int = 1):
    """The fp64 oracle on host cores over a bounded sample of the headline workload."""
    import oracle
    w = synth.WORKLOADS[HEADLINE]
    cores = oracle.default_threads()
    heads = max(1, min(w.B * w.H, 2 * cores))
    x = synth.qkv(1, heads, w.N, w.D, w.M, w.dtype, w.seed, w.scale, with_grad=True)
    Q, K, V, G = (x[n] for n in ("Q", "K", "V", "G"))
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.causal_forward_recurrent(Q, K, V, nthreads=cores)
        oracle.causal_backward_cumsum(Q, K, V, G, nthreads=cores)
    dt = (time.perf_counter() - t0) / steps
    # heads / H of the B*N tokens of a step are covered per sample
    tokens = w.N * heads / w.H
    return {"value": round(tokens / dt, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{heads} heads x N={w.N} (D=M={w.D}) of the fwd+bwd step, fp64 recurrent "
                      f"forward + cumulative-sum backward, {dt:.2f} s per sample"}


def _synth_module():
    """The seeded input generator, loaded by path: importing it through the package
    would load the CUDA library, which the CPU-only reference arm must not touch."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_la_synth", os.path.join(ROOT, "linear_attention_02_gb300", "synth.py"))
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod  # its dataclasses look their module up by name
    spec.loader.exec_module(mod)
    return mod


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    synth = _synth_module()  # inputs only
    w = synth.WORKLOADS[HEADLINE]
    for _ in range(max(0, min(args.warmup, 1))):
        cpu_baseline(synth)
    t0 = time.perf_counter()
    samples = [cpu_baseline(synth) for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    v = statistics.mean(s["value"] for s in samples)
    out = {"impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(wall / max(args.steps, 1) * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": f"{HEADLINE}: causal linear attention fwd+bwd, B={w.B} H={w.H} "
                                  f"N={w.N} D=M={w.D}, bf16 inputs evaluated in fp64",
                      "global_batch": w.B, "seq_len": w.N},
           "cpu_baseline": {"value": round(v, 1), "unit": "tokens/s", "kind": "oracle",
                            "cores": samples[0]["cores"], "sample": samples[0]["sample"]},
           "e2e": {"value": round(v, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return out


# Small cases for kernel profiles (ncu): inputs larger than L2 (129 MB) but a few
# hundred MB on the device, each op run `reps` times after one warm-up call.
PROFILE_CASES = {
    "causal_train": "causal forward + backward, B=4 H=16 N=8192 D=M=64 bf16 (the headline step)",
    "causal_long_small": "causal forward, B=1 H=4 N=65536 D=M=128 bf16 (the long workload's kernel, 4 heads)",
    "noncausal_f32": "non-causal forward, B=8 H=8 N=4096 D=M=64 fp32",
    "noncausal_f32_bwd": "non-causal backward, B=8 H=8 N=4096 D=M=64 fp32, Out given",
    "decode": "decode step, 256 sequences x 16 heads, D=M=64, bf16 q/k/v, fp32 state",
    "softmax_decode": "softmax KV-cache step, 64 sequences x 16 heads, D=64, 4096-position cache",
    "retention_gated": "gated retention forward, B=4 H=16 N=8192 D=M=64 bf16",
    "poly2": "degree-2 polynomial map, causal, B=4 H=16 N=4096 D=32 M=64 bf16 (the bench workload)",
}


def run_profile(case: str, reps: int):
    """Runs one path `reps` times (after one warm-up call) for a profiler to capture."""
    import torch
    import linear_attention_02_gb300 as la
    from linear_attention_02_gb300 import synth
    torch.cuda.set_device(0)
    dev = "cuda"
    if case == "causal_train":
        w = synth.WORKLOADS["causal_train_bf16"]
        x = synth.qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.scale, with_grad=True, device=dev)
        den = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        ck = torch.empty(la.la_causal_ckpt_floats(w.B, w.H, w.N, w.D, w.M), dtype=torch.float32, device=dev)

        def f():
            O = la.la_forward_causal(x["Q"], x["K"], x["V"], den=den, ckpt=ck)
            la.la_backward_causal(x["Q"], x["K"], x["V"], x["G"], Out=O, Den=den, Ckpt=ck)
    elif case == "causal_long_small":
        x = synth.qkv(1, 4, 65536, 128, 128, "bf16", 1004, 0.5, device=dev)
        f = lambda: la.la_forward_causal(x["Q"], x["K"], x["V"])
    elif case in ("noncausal_f32", "noncausal_f32_bwd"):
        w = synth.WORKLOADS["noncausal_f32"]
        x = synth.qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.scale, with_grad=True, device=dev)
        O = la.la_forward_noncausal(x["Q"], x["K"], x["V"])
        if case == "noncausal_f32":
            f = lambda: la.la_forward_noncausal(x["Q"], x["K"], x["V"], out=O)
        else:
            f = lambda: la.la_backward_noncausal(x["Q"], x["K"], x["V"], x["G"], Out=O)
    elif case == "decode":
        S = torch.randn(256, 16, 64, 64, device=dev)
        Z = torch.rand(256, 16, 64, device=dev).add_(1.0)
        s_ = synth.decode_step_qkv(256, 16, 64, 64, "bf16", 1005, 0, device=dev)
        f = lambda: la.la_decode_step(s_["q"], s_["k"], s_["v"], S, Z)
    elif case == "softmax_decode":
        Kc = synth.randn((64, 16, 4096, 64), "bf16", 1007, device=dev)
        Vc = synth.randn((64, 16, 4096, 64), "bf16", 1008, device=dev)
        s_ = synth.decode_step_qkv(64, 16, 64, 64, "bf16", 1005, 0, device=dev)
        f = lambda: la.la_softmax_decode_step(s_["q"], s_["k"], s_["v"], Kc, Vc, 4095)
    elif case == "retention_gated":
        w = synth.WORKLOADS["causal_train_bf16"]
        x = synth.qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.scale, device=dev)
        gates = synth.decays((w.B, w.H, w.N), w.seed + 5, 0.85, 1.0, device=dev)
        f = lambda: la.la_forward_retention(x["Q"], x["K"], x["V"], gates=gates)
    elif case == "poly2":
        x = synth.qkv(4, 16, 4096, 32, 64, "bf16", 1007, device=dev)
        f = lambda: la.la_forward_poly2(x["Q"], x["K"], x["V"], causal=True)
    else:
        raise SystemExit(f"unknown profile case {case}; one of {sorted(PROFILE_CASES)}")
    f()
    torch.cuda.synchronize()
    for _ in range(reps):
        f()
    torch.cuda.synchronize()
    la.la_check_device_status()
    print(f"profile case {case}: {PROFILE_CASES[case]}, {reps} runs", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-paths", action="store_true", help="headline step only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--profile", choices=sorted(PROFILE_CASES),
                    help="run one path on a small case for a profiler, print no JSON line")
    ap.add_argument("--reps", type=int, default=2, help="runs of the --profile case")
    args = ap.parse_args()
    if args.profile:
        run_profile(args.profile, args.reps)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
