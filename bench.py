#!/usr/bin/env python
"""Benchmark of the chunked gated delta rule with state / W fake QDQ on GB300.

Default (``--mode fwdbwd``): one step = one pass of the hot path over one
global batch made of micro-batches of the forward+backward workload (B=8,
T=4096, H=16, Dk=Dv=128, E4M3 state and W QDQ, h0 ~ N(0, 0.1^2), dO and
dht as upstream gradients): per micro-batch the forward (saving the
backward's context) and the identity-STE backward.  The number of
micro-batches is chosen during warm-up so that a step lasts about 50 ms of
device time (stated in ``config``).  After the timed steps the forward alone
(no backward context) is timed on the single-layer workload (B=4, T=4096,
H=16, D=128): the configuration the forward's roofline target is set on,
reported as ``roofline``; the backward's roofline is ``roofline_bwd``.
``--mode fwd`` times the forward alone; ``--mode decode`` the decode QAT step
(256 sequences, one token each, carried fp32 states of 256 MiB);
``--mode kda`` the KDA recurrence and ``--mode two_precision`` the
two-precision profile (fp32 anchor, E4M3 read copy), both B=4, T=4096,
H=16; ``--mode two_precision_bwd`` that profile's training step (forward
saving the window anchors, then the window-wise adjoint).  Inputs are synthetic (seeded) and resident in HBM when the timed
region starts; every micro-batch's inputs exceed the 129 MB L2, so no flush
is needed between them.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(fp64 chunked reference) on a bounded sample of the same workload instead.
Under torchrun every rank runs its own batch (weak scaling, no collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN chunk fwd(+STE bwd) tokens/s at H=16,D=128,T=4096; % of roofline"


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def _max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    if torch.distributed.get_backend() == "gloo":
        device = torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled every millisecond
    through NVML (read-only queries) while the timed region runs; falls back to
    ``nvidia-smi -lms 200`` when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device):
        self.device = device
        self.samples = []      # (sm_mhz, max_mhz, reasons_mask)
        self.stop = threading.Event()
        self.nvml = None
        self.proc = None
        self.lines = []

    def _open_nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        prop = torch.cuda.get_device_properties(self.device)
        bus = ("%04x:%02x:%02x.0" % (getattr(prop, "pci_domain_id", 0), prop.pci_bus_id,
                                     prop.pci_device_id)).encode()
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
            cnt = ctypes.c_uint()
            if lib.nvmlDeviceGetCount_v2(ctypes.byref(cnt)) != 0 or cnt.value != 1 or \
                    lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                return None
        self._c = ctypes
        return lib, h

    def _poll(self):
        lib, h = self.nvml
        c = self._c
        sm, mx, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        fn_r = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, c.byref(sm)) == 0 and \
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, c.byref(mx)) == 0 and \
                    fn_r(h, c.byref(rs)) == 0:
                self.samples.append((sm.value, mx.value, rs.value))
            time.sleep(0.001)

    def __enter__(self):
        try:
            self.nvml = self._open_nvml()
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            self.th = threading.Thread(target=self._poll, daemon=True)
            self.th.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 2.0:
                time.sleep(0.001)
            self.samples.clear()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device.index), "--query-gpu=clocks.sm,clocks.max.sm,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
            time.sleep(0.5)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        names = [0x8, 0x40, 0x20, 0x4]
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            try:
                mask = sum(b for b, v in zip(names, f[2:6]) if v.lower() == "active")
                self.samples.append((float(f[0]), float(f[1]), mask))
            except (ValueError, IndexError):
                continue

    def __exit__(self, *a):
        self.stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if hasattr(self, "th"):
            self.th.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "nvml" if self.nvml else "nvidia-smi"}
        mask = 0
        for _, _, m in self.samples:
            mask |= m
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples),
                "reasons": sorted(v for b, v in self.REASONS.items() if mask & b),
                "samples": len(self.samples), "source": "nvml" if self.nvml else "nvidia-smi"}


def e2e_pipelined(dev, ws, steps, warmup, host_in, dev_in, run, res_h):
    """End-to-end timing through the public API from pinned host memory.

    Every step copies its inputs host -> device (``host_in[name]`` into
    ``dev_in[set][name]``), runs ``run(set)`` (the library calls; returns the
    device result tensors) and copies every result back into ``res_h[set]``.
    Three streams and two device buffer sets let step i's compute overlap the
    upload of step i+1 and the download of step i-1, as a pipelined user loop
    would; events order each buffer set's reuse.  Returns (pipelined ms per
    step, serial ms per step), both max over ranks; the serial figure runs the
    same steps on one stream, copies and compute back to back."""
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        st = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_cmp[st])          # step i-2 no longer reads this input set
            for n, t in dev_in[st].items():
                t.copy_(host_in[n], non_blocking=True)
            ev_in[st].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[st])
            s_cmp.wait_event(ev_out[st])         # step i-2's results have left this set
            outs = run(st)
            ev_cmp[st].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[st])
            for dst, src in zip(res_h[st], outs):
                dst.copy_(src, non_blocking=True)
            ev_out[st].record(s_out)

    def serial_step():
        for n, t in dev_in[0].items():
            t.copy_(host_in[n], non_blocking=True)
        for dst, src in zip(res_h[0], run(0)):
            dst.copy_(src, non_blocking=True)

    t = {}
    for kind in ("pipelined", "serial"):
        for i in range(max(2, warmup)):
            step(i) if kind == "pipelined" else serial_step()
        torch.cuda.synchronize()
        _barrier(ws)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if kind == "pipelined":
            a.record(s_in)
            for i in range(steps):
                step(i)
            s_in.wait_stream(s_out)
            b.record(s_in)
        else:
            a.record()
            for _ in range(steps):
                serial_step()
            b.record()
        torch.cuda.synchronize()
        t[kind] = _max_over_ranks(a.elapsed_time(b), ws, dev) / steps
    return t["pipelined"], t["serial"]


def _peaks(tensor_key="bf16_tflops"):
    """(HBM GB/s, dense bf16 TFLOP/s, source): the driver's measured peaks, else
    the fallback figures (6.8 TB/s, 1.9 PFLOP/s burst, 1.7 sustained)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk[tensor_key]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, (1900.0 if tensor_key == "bf16_tflops" else 1700.0), "fallback"


def _strip_comments(src):
    """C/C++/CUDA source without its comments and blank lines (string and
    character literals kept), so that a comment edit leaves the hash alone."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).splitlines()]
    return "\n".join(ln for ln in lines if ln)


def _source_hash(files):
    """Hash of the kernel sources' code (comments excluded) that a committed
    ncu summary was taken on."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def _traffic(profile_md, source_files, workload_key):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", profile_md)
    try:
        txt = open(path).read()
    except OSError:
        return None
    m_src = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", txt)
    m_tr = re.search(r"traffic_bytes_per_launch\[%s\]:\s*([0-9.eE+]+)" % re.escape(workload_key), txt)
    if not m_src or not m_tr or m_src.group(1) != _source_hash(source_files):
        return None
    return float(m_tr.group(1))


FWD_SOURCES = ["gated_delta_rule_54_gb300/csrc/fwd.cu", "gated_delta_rule_54_gb300/csrc/fwd_fused.cu",
               "gated_delta_rule_54_gb300/csrc/common.cuh", "gated_delta_rule_54_gb300/csrc/tc.cuh"]
BWD_SOURCES = ["gated_delta_rule_54_gb300/csrc/bwd.cu", "gated_delta_rule_54_gb300/csrc/bwd_tc.cu",
               "gated_delta_rule_54_gb300/csrc/bwd_scan_tc.cu", "gated_delta_rule_54_gb300/csrc/common.cuh",
               "gated_delta_rule_54_gb300/csrc/tc.cuh"]


def fwd_alg_bytes(w, save_ctx):
    """Algorithmic HBM bytes of one forward launch: inputs read once, outputs written once."""
    tok = w.B * w.T
    b = tok * w.Hk * w.Dk * 2 * 2            # q, k bf16
    b += tok * w.Hv * w.Dv * 2               # v bf16
    b += tok * w.Hv * 4 * 2                  # beta, g f32
    b += tok * w.Hv * w.Dv * 4               # o f32
    b += w.B * w.Hv * w.Dk * w.Dv * 4 * (2 if w.h0 else 1)   # h0 read, ht write
    if save_ctx:
        nch = w.B * (-(-w.T // 64))
        b += tok * w.Hv * w.Dk + nch * w.Hv * 4                          # W codes + scales
        b += nch * w.Hv * w.Dk * w.Dv + nch * w.Hv * (w.Dv // 64) * 4    # state codes + scales
    return b


def bwd_alg_bytes(w):
    """Algorithmic HBM bytes of one backward pass: q,k,v,beta,g,dO, saved context
    and dht read once; dq,dk,dv,dbeta,dg,dh0 written once."""
    tok = w.B * w.T
    nch = w.B * (-(-w.T // 64))
    b = tok * w.Hk * w.Dk * 2 * 2 + tok * w.Hv * w.Dv * 2 + tok * w.Hv * 4 * 2
    b += tok * w.Hv * w.Dv * 2                                           # dO bf16
    b += tok * w.Hv * w.Dk + nch * w.Hv * 4                              # W codes + scales
    b += nch * w.Hv * w.Dk * w.Dv + nch * w.Hv * (w.Dv // 64) * 4        # state codes + scales
    b += w.B * w.Hv * w.Dk * w.Dv * 4 * 2                                # dht in, dh0 out
    b += tok * w.Hk * w.Dk * 4 * 2 + tok * w.Hv * w.Dv * 4 + tok * w.Hv * 4 * 2  # grads out
    return b


def fwd_alg_flops(w):
    """Algorithmic forward FLOPs (triangular products at half): 9.0 MFLOP per
    64-token chunk-head at Dk = Dv = 128, i.e. 140.6 kFLOP per token-head."""
    C, Dk, Dv = 64, w.Dk, w.Dv
    per_chunk = (C * C * Dk + C ** 3 / 3 + C * C * Dk + C * C * Dv + 2 * C * Dk * Dv * 3
                 + C * C * Dk + C * C * Dv)
    return per_chunk / C * w.B * w.T * w.Hv


def bwd_alg_flops(w):
    """Algorithmic STE-backward FLOPs: six Dk x Dv products (dH and dDelta
    paths, 2 C Dk Dv each), ten C x C x D products (the gated attention and WY
    gradients) and the solve's gradient, per 64-token chunk-head: 18.6 MFLOP
    at Dk = Dv = 128 (291 kFLOP per token-head)."""
    C, Dk, Dv = 64, w.Dk, w.Dv
    per_chunk = 6 * 2 * C * Dk * Dv + 10 * C * C * (Dk + Dv) / 2 + 2 * C ** 3 / 3
    return per_chunk / C * w.B * w.T * w.Hv


def roofline_entry(alg_bytes, alg_flops, dur_ms, kernel, traffic, tensor_peak_key):
    """Roofline record of one call: the bound is the larger of bytes / HBM peak
    and FLOPs / bf16 tensor peak (measured peaks); achieved is in that bound's
    unit."""
    hbm, tensor, kind = _peaks(tensor_peak_key)
    t_mem = alg_bytes / (hbm * 1e9)
    t_tc = alg_flops / (tensor * 1e12)
    if t_mem >= t_tc:
        achieved = alg_bytes / (dur_ms / 1e3) / 1e9
        rec = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
               "frac": round(achieved / hbm, 4)}
    else:
        achieved = alg_flops / (dur_ms / 1e3) / 1e12
        rec = {"bound": "tensor", "achieved": round(achieved, 2), "peak": tensor, "unit": "TFLOP/s",
               "frac": round(achieved / tensor, 4)}
    rec.update({"traffic": traffic, "kernel": kernel, "peak_source": kind,
                "alg_bytes_per_launch": int(alg_bytes), "alg_flops_per_launch": int(alg_flops),
                "t_roof_us": round(max(t_mem, t_tc) * 1e6, 2), "launch_ms": round(dur_ms, 4)})
    return rec


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
STEP_TARGET_MS = 50.0   # micro-batches per step are chosen so that a step lasts about this long


def _gdn_buffers(w, dev, rank, bwd, save_ctx):
    from gated_delta_rule_54_gb300 import api, synth
    cpu = synth.make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
    p = api.make_problem(d["q"], d["k"], d["v"], None, 1.0, w.state_mode, w.w_mode,
                         save_ctx=save_ctx)
    d["o"] = torch.empty(w.B, w.T, w.Hv, w.Dv, device=dev)
    d["ht"] = torch.empty(w.B, w.Hv, w.Dk, w.Dv, device=dev)
    d["ctx"] = torch.empty(api.gdn_ctx_bytes(p), device=dev, dtype=torch.uint8)
    if bwd:
        gen = torch.Generator().manual_seed(1000 + rank)
        d["do"] = torch.randn(w.B, w.T, w.Hv, w.Dv, generator=gen).to(torch.bfloat16).to(dev)
        d["dht"] = (torch.randn(w.B, w.Hv, w.Dk, w.Dv, generator=gen) * 0.01).to(dev)
        d["ws"] = torch.empty(max(api.gdn_bwd_workspace_bytes(p), 1), device=dev, dtype=torch.uint8)
        f32 = dict(device=dev, dtype=torch.float32)
        d["grads"] = (torch.empty(d["q"].shape, **f32), torch.empty(d["k"].shape, **f32),
                      torch.empty(d["v"].shape, **f32), torch.empty(d["beta"].shape, **f32),
                      torch.empty(d["g"].shape, **f32), torch.empty(d["ht"].shape, **f32))
    return cpu, d


def run_ours(args, ws, rank, local):
    from gated_delta_rule_54_gb300 import api, synth
    from gated_delta_rule_54_gb300._lib import load

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    load()
    w = synth.WORKLOADS[args.workload]
    w = synth.Workload(**{**w.__dict__, "seed": w.seed + rank})
    bwd = args.mode == "fwdbwd"
    sm, wm = w.state_mode, w.w_mode
    bv, nd = args.block_v, args.neumann_degree
    # two buffer sets, used by alternate micro-batches
    sets = [_gdn_buffers(w, dev, rank, bwd, save_ctx=bwd) for _ in range(2)]
    cpu = sets[0][0]
    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    fwd_times, bwd_times = [], []

    def fwd(d):
        api.gdn_chunk_fwd_qdq(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], state_mode=sm,
                              w_mode=wm, out=(d["o"], d["ht"], d["ctx"]), save_ctx=bwd,
                              block_v=bv, neumann_degree=nd)

    def bwd_call(d):
        api.gdn_chunk_bwd_ste(d["q"], d["k"], d["v"], d["beta"], d["g"], d["ctx"], d["do"],
                              d["dht"], state_mode=sm, w_mode=wm, workspace=d["ws"],
                              out=d["grads"], block_v=bv, neumann_degree=nd)

    def step(micro, record=False):
        for m in range(micro):
            d = sets[m % 2][1]
            e0 = ev() if record else None
            if record:
                e0.record(stream)
            fwd(d)
            if record:
                e1 = ev()
                e1.record(stream)
                fwd_times.append((e0, e1))
            if bwd:
                bwd_call(d)
                if record:
                    e2 = ev()
                    e2.record(stream)
                    bwd_times.append((e1, e2))

    # warm-up, which also sizes the step: micro-batches of the workload until a
    # step lasts about STEP_TARGET_MS of device time (the clock sampler then
    # sees the GPU under load for the whole timed region)
    for _ in range(args.warmup):
        step(1)
    torch.cuda.synchronize()
    a, b = ev(), ev()
    a.record(stream)
    step(2)
    b.record(stream)
    torch.cuda.synchronize()
    one = a.elapsed_time(b) / 2
    micro = args.micro_batches or max(1, min(64, int(round(STEP_TARGET_MS / max(one, 1e-3)))))
    micro = int(_max_over_ranks(micro, ws, dev))
    step(micro)
    torch.cuda.synchronize()
    _barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        t_start, t_end = ev(), ev()
        t_start.record(stream)
        for _ in range(args.steps):
            step(micro, record=True)
        t_end.record(stream)
        torch.cuda.synchronize()
    _barrier(ws)
    ms_total = t_start.elapsed_time(t_end)
    ms_total = _max_over_ranks(ms_total, ws, dev)
    ms_step = ms_total / args.steps
    tokens = w.B * w.T * micro
    value = tokens * ws * args.steps / (ms_total / 1e3)
    fwd_ms = statistics.mean(x.elapsed_time(y) for x, y in fwd_times)
    bwd_ms = statistics.mean(x.elapsed_time(y) for x, y in bwd_times) if bwd else None
    launches_per_step = micro * (_fwd_launches(w, bv, nd) + (args.bwd_launches if bwd else 0))

    # the forward alone (no backward context) on the single-layer workload
    # (B=4, T=4096, H=16, D=128): the configuration the forward's roofline
    # target is set on; timed as its own loop after the step
    fl = synth.WORKLOADS["layer"] if w.Dk == 128 and not w.varlen_total else w
    fl = synth.Workload(**{**fl.__dict__, "seed": fl.seed + rank})
    _, dl = _gdn_buffers(fl, dev, rank, False, save_ctx=False)

    def fwd_only():
        api.gdn_chunk_fwd_qdq(dl["q"], dl["k"], dl["v"], dl["beta"], dl["g"], dl["h0"],
                              state_mode=fl.state_mode, w_mode=fl.w_mode,
                              out=(dl["o"], dl["ht"], dl["ctx"]), save_ctx=False,
                              block_v=bv, neumann_degree=nd)

    for _ in range(args.warmup):
        fwd_only()
    reps = max(args.steps, 50)
    a, b = ev(), ev()
    a.record(stream)
    for _ in range(reps):
        fwd_only()
    b.record(stream)
    torch.cuda.synchronize()
    fwd_only_ms = _max_over_ranks(a.elapsed_time(b) / reps, ws, dev)
    del dl

    fwd_kernel = ("gdn forward, forward only: chunk prep + fused scan/outputs"
                  if _fused(fl, bv, nd) else "gdn forward, forward only: prep, state scan, outputs")
    roof = roofline_entry(fwd_alg_bytes(fl, False), fwd_alg_flops(fl), fwd_only_ms, fwd_kernel,
                          _traffic("gdn_fwd_kernels_single_layer.md", FWD_SOURCES, "layer"),
                          "bf16_tflops")
    roof["workload"] = fl.name
    roof_bwd = None
    if bwd:
        roof_bwd = roofline_entry(bwd_alg_bytes(w), bwd_alg_flops(w), bwd_ms,
                                  "gdn backward (all launches of one call)",
                                  _traffic("gdn_bwd_kernels_single_layer.md", BWD_SOURCES, args.workload),
                                  "bf16_tflops_sustained")
        roof_bwd["workload"] = w.name
    roof_train_fwd = roofline_entry(fwd_alg_bytes(w, bwd), fwd_alg_flops(w), fwd_ms,
                                    "gdn forward inside the step" + (" (saving the backward's context)"
                                                                     if bwd else ""),
                                    None, "bf16_tflops_sustained")
    roof_train_fwd["workload"] = w.name

    # end to end through the public API from pinned host buffers (one
    # micro-batch per step: its inputs up, its results down)
    e2e = None
    if not args.no_e2e:
        d0 = sets[0][1]
        names = [n for n in ("q", "k", "v", "beta", "g", "h0") if cpu[n] is not None]
        host_in = {n: cpu[n].pin_memory() for n in names}
        if bwd:
            host_in["do"] = d0["do"].cpu().pin_memory()
            host_in["dht"] = d0["dht"].cpu().pin_memory()
        dev_in = [{n: torch.empty_like(t, device=dev) for n, t in host_in.items()} for _ in range(2)]
        ctxs = [sets[0][1]["ctx"], sets[1][1]["ctx"]]

        def result_set():
            r = [torch.empty_like(d0["o"]), torch.empty_like(d0["ht"])]
            if bwd:
                r += [torch.empty_like(t) for t in d0["grads"]]
            return r

        res_d = [result_set(), result_set()]
        res_h = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in r] for r in res_d]

        def run(st):
            x, r = dev_in[st], res_d[st]
            api.gdn_chunk_fwd_qdq(x["q"], x["k"], x["v"], x["beta"], x["g"], x.get("h0"),
                                  state_mode=sm, w_mode=wm, out=(r[0], r[1], ctxs[st]),
                                  save_ctx=bwd, block_v=bv, neumann_degree=nd)
            if bwd:
                api.gdn_chunk_bwd_ste(x["q"], x["k"], x["v"], x["beta"], x["g"], ctxs[st], x["do"],
                                      x["dht"], state_mode=sm, w_mode=wm, workspace=d0["ws"],
                                      out=tuple(r[2:]), block_v=bv, neumann_degree=nd)
            return r

        e_ms, s_ms = e2e_pipelined(dev, ws, args.steps, args.warmup, host_in, dev_in, run, res_h)
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in res_h[0])
        e2e = {"value": round(w.B * w.T * ws / (e_ms / 1e3), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e_ms, 4),
               "step": "one micro-batch of the workload",
               "schedule": "pipelined: step i+1's upload and step i-1's download overlap step i's "
                           "compute (three streams, two device buffer sets)",
               "serial_value": round(w.B * w.T * ws / (s_ms / 1e3), 1),
               "serial_ms_per_step": round(s_ms, 4)}

    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu_base = cpu_baseline(w, cpu, bwd, budget_s=args.cpu_budget)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), beta=sigmoid, g=-softplus)",
        "config": {"workload": w.name, "mode": args.mode, "B": w.B, "T": w.T, "Hk": w.Hk,
                   "Hv": w.Hv, "Dk": w.Dk, "Dv": w.Dv, "state_mode": sm, "w_mode": wm,
                   "chunk": 64, "block_v": bv,
                   "solve": "exact" if nd is None else "neumann degree %d" % nd,
                   "micro_batches_per_step": micro,
                   "global_batch_tokens": tokens * ws,
                   "l2": "inputs larger than L2 (no flush needed)",
                   "fwd_ms": round(fwd_ms, 4), "bwd_ms": round(bwd_ms, 4) if bwd else None,
                   "fwd_only_ms": round(fwd_only_ms, 4), "fwd_only_workload": fl.name,
                   "fwd_only_tflops_alg": round(fwd_alg_flops(fl) / (fwd_only_ms / 1e3) / 1e12, 2)},
        "clocks": clk.summary(), "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "roofline": roof, "roofline_bwd": roof_bwd, "roofline_step_fwd": roof_train_fwd,
        "cpu_baseline": cpu_base,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def cpu_baseline(w, cpu, bwd, budget_s=20.0):
    """The oracle, as it stands, on whole sequences of the workload (all heads),
    until the budget is used; tokens/s scaled from the sample.  Forward and
    backward: the fp64 chunked form with autograd.  Forward only: the fp64 token
    recurrence (C, OpenMP over (sequence, value head); it has no W site, so the
    state QDQ is its only quantizer)."""
    from oracle.chunked import chunked
    if not bwd:
        import oracle
        t0 = time.time()
        done = 0
        for n in range(w.B):
            sl = slice(n, n + 1)
            oracle.recurrent(*[cpu[x][sl] for x in ("q", "k", "v", "beta", "g")],
                             cpu["h0"][sl] if cpu["h0"] is not None else None,
                             state_mode=w.state_mode)
            done += 1
            if time.time() - t0 > budget_s * 0.5:
                break
        dt = time.time() - t0
        return {"value": round(done * w.T / dt, 2), "unit": "tokens/s",
                "cores": oracle.num_threads(), "kind": "oracle",
                "sample": "%d of %d sequences (T=%d, all %d heads), fp64 token recurrence "
                          "(C, OpenMP)" % (done, w.B, w.T, w.Hv)}
    t0 = time.time()
    done = 0
    for n in range(w.B):
        sl = slice(n, n + 1)
        args = [cpu[x][sl] for x in ("q", "k", "v", "beta", "g")]
        h0 = cpu["h0"][sl] if cpu["h0"] is not None else None
        if bwd:
            xs = [a.double().requires_grad_(True) for a in args] + (
                [h0.double().requires_grad_(True)] if h0 is not None else [None])
            o, ht = chunked(*xs, state_mode=w.state_mode, w_mode=w.w_mode)
            (o.sum() + ht.sum()).backward()
        else:
            chunked(*args, h0, state_mode=w.state_mode, w_mode=w.w_mode)
        done += 1
        if time.time() - t0 > budget_s * 0.5:
            break
    dt = time.time() - t0
    return {"value": round(done * w.T / dt, 2), "unit": "tokens/s", "cores": torch.get_num_threads(),
            "kind": "oracle",
            "sample": "%d of %d sequences (T=%d, all %d heads), fp64 chunked oracle %s" % (
                done, w.B, w.T, w.Hv, "fwd+autograd bwd" if bwd else "fwd")}


# ----------------------------------------------------------------------------
# decode QAT step (--mode decode)
# ----------------------------------------------------------------------------
DECODE_METRIC = "GDN decode QAT tokens/s at B=256,H=16,D=128 (one token per sequence); % of roofline"
DECODE_SOURCES = ["gated_delta_rule_54_gb300/csrc/decode.cu", "gated_delta_rule_54_gb300/csrc/common.cuh"]


def decode_alg_bytes(w):
    """Algorithmic HBM bytes of one decode launch: the carried state read and
    written once, the token's q, k, v, beta, g read and o written."""
    tok = w.B * w.T
    b = w.B * w.Hv * w.Dk * w.Dv * 4 * 2
    b += tok * (w.Hk * w.Dk * 2 * 2 + w.Hv * w.Dv * 2 + w.Hv * 4 * 2 + w.Hv * w.Dv * 4)
    return b


def run_decode(args, ws, rank, local):
    from gated_delta_rule_54_gb300 import api, synth
    from gated_delta_rule_54_gb300._lib import load

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    load()
    w = synth.WORKLOADS[args.workload]
    w = synth.Workload(**{**w.__dict__, "seed": w.seed + rank})
    cpu = synth.make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
    q, k, v, beta, g = d["q"], d["k"], d["v"], d["beta"], d["g"]
    # two state buffers used in turn: each step reads the state the last one wrote
    states = [d["h0"], torch.empty_like(d["h0"])]
    o = torch.empty(w.B, w.T, w.Hv, w.Dv, device=dev)
    sm = w.state_mode
    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    it = [0]

    def step():
        i = it[0]
        api.gdn_decode_qdq(q, k, v, beta, g, states[i % 2], state_mode=sm, state_out=states[1 - i % 2],
                           out=o)
        it[0] += 1

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    _barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
    _barrier(ws)
    ms_total = _max_over_ranks(a.elapsed_time(b), ws, dev)
    ms_step = ms_total / args.steps
    tokens = w.B * w.T
    value = tokens * ws * args.steps / (ms_total / 1e3)
    peak, _, peak_kind = _peaks()
    alg = decode_alg_bytes(w)
    achieved = alg / (ms_step / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": _traffic("gdn_decode_kernel_decode_step.md", DECODE_SOURCES, args.workload),
            "kernel": "gdn_decode_kernel", "peak_source": peak_kind,
            "alg_bytes_per_launch": alg, "launch_ms": round(ms_step, 4)}

    # end to end: the token's inputs from pinned host memory, o back; the
    # carried states stay resident on the device (a decode cache)
    e2e = None
    if not args.no_e2e:
        names = ("q", "k", "v", "beta", "g")
        host = {n: cpu[n].pin_memory() for n in names}
        o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        h2d = sum(host[n].numel() * host[n].element_size() for n in names)
        d2h = o_h.numel() * o_h.element_size()

        def e2e_step():
            for n in names:
                d[n].copy_(host[n], non_blocking=True)
            step()
            o_h.copy_(o, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        _barrier(ws)
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(args.steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e_ms = _max_over_ranks(a.elapsed_time(b), ws, dev)
        e2e = {"value": round(tokens * ws * args.steps / (e_ms / 1e3), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e_ms / args.steps, 4),
               "note": "carried states resident on the device"}

    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu_base = decode_cpu_baseline(w, cpu, budget_s=args.cpu_budget)
    line = {
        "metric": DECODE_METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), beta=sigmoid, "
                "g=-softplus, states N(0, 0.1^2))",
        "config": {"workload": w.name, "mode": "decode", "B": w.B, "T": w.T, "Hk": w.Hk,
                   "Hv": w.Hv, "Dk": w.Dk, "Dv": w.Dv, "state_mode": sm, "block_v": 64,
                   "readout": "pre",
                   "l2": "states (2 x 256 MiB, read and written in turn) larger than L2"},
        "clocks": clk.summary(), "e2e": e2e, "gpu_launches": args.steps, "roofline": roof,
        "cpu_baseline": cpu_base,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def decode_cpu_baseline(w, cpu, budget_s=20.0, rows=None):
    """The fp64 decode oracle, as it stands, on whole rows (all heads) until
    the budget is used; tokens/s scaled from the sample."""
    from oracle.decode import decode
    t0 = time.time()
    done = 0
    for n in range(w.B if rows is None else rows):
        sl = slice(n, n + 1)
        decode(*[cpu[x][sl] for x in ("q", "k", "v", "beta", "g", "h0")], state_mode=w.state_mode)
        done += 1
        if time.time() - t0 > budget_s * 0.5:
            break
    dt = time.time() - t0
    return {"value": round(done * w.T / dt, 2), "unit": "tokens/s", "cores": torch.get_num_threads(),
            "kind": "oracle",
            "sample": "%d of %d rows (one token, all %d heads), fp64 decode oracle" % (
                done, w.B, w.Hv)}


# ----------------------------------------------------------------------------
# token-serial recurrences: KDA (--mode kda) and the two-precision profile
# (--mode two_precision)
# ----------------------------------------------------------------------------
KDA_METRIC = "KDA recurrent fwd tokens/s at B=4,T=4096,H=16,D=128 (state QDQ every 64 tokens); % of roofline"
TP_METRIC = ("two-precision GDN fwd tokens/s at B=4,T=4096,H=16,D=128 (fp32 anchor, E4M3 read copy, "
             "16-token flush); % of roofline")
KDA_SOURCES = ["gated_delta_rule_54_gb300/csrc/kda.cu", "gated_delta_rule_54_gb300/csrc/common.cuh"]
TP_SOURCES = ["gated_delta_rule_54_gb300/csrc/two_precision.cu",
              "gated_delta_rule_54_gb300/csrc/two_precision.cuh",
              "gated_delta_rule_54_gb300/csrc/common.cuh"]
TP_FLUSH = 16


def token_serial_alg_bytes(w, g_per_channel):
    """Algorithmic HBM bytes of one launch: q, k, v, beta, g read once (g per key
    channel for KDA, per head otherwise), o written once, h0 read and ht written."""
    tok = w.B * w.T
    g = w.Hv * w.Dk * 4 if g_per_channel else w.Hv * 4
    b = tok * (w.Hk * w.Dk * 2 * 2 + w.Hv * w.Dv * 2 + w.Hv * 4 + g + w.Hv * w.Dv * 4)
    return b + w.B * w.Hv * w.Dk * w.Dv * 4 * 2


def kda_alg_bytes(w):
    return token_serial_alg_bytes(w, True)


class _TokenSerial:
    """What differs between the two token-serial benchmarks."""

    def __init__(self, mode):
        from gated_delta_rule_54_gb300 import api, synth
        self.mode = mode
        self.kda = mode == "kda"
        self.metric = KDA_METRIC if self.kda else TP_METRIC
        self.kernel = "kda_recurrent_kernel" if self.kda else "gdn_two_precision_kernel"
        self.profile = ("kda_recurrent_kernel_kda_layer.md" if self.kda
                        else "gdn_two_precision_kernel_two_precision_layer.md")
        self.sources = KDA_SOURCES if self.kda else TP_SOURCES
        self.make = synth.make_kda_inputs if self.kda else synth.make_inputs
        self.gname = "g_k" if self.kda else "g"
        self.api = api

    def call(self, w, x, out=None):
        if self.kda:
            return self.api.kda_recurrent_fwd_qdq(x["q"], x["k"], x["v"], x["beta"], x["g_k"],
                                                  x["h0"], state_mode=w.state_mode)
        return self.api.gdn_two_precision_fwd(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                                              read_mode=w.state_mode, flush=TP_FLUSH, out=out)

    def oracle(self, w, x):
        if self.kda:
            from oracle.kda import kda_recurrent
            return kda_recurrent(x["q"], x["k"], x["v"], x["beta"], x["g_k"], x["h0"],
                                 state_mode=w.state_mode)
        from oracle.two_precision import two_precision
        return two_precision(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                             read_mode=w.state_mode, flush=TP_FLUSH)

    def config(self, w):
        c = {"workload": w.name, "mode": self.mode, "B": w.B, "T": w.T, "Hk": w.Hk, "Hv": w.Hv,
             "Dk": w.Dk, "Dv": w.Dv}
        if self.kda:
            c.update(state_mode=w.state_mode, chunk=64, block_v=64)
        else:
            c.update(read_mode=w.state_mode, flush=TP_FLUSH, read_group="per value row, 128 key channels")
        c["l2"] = "inputs larger than L2 (no flush needed)"
        return c

    def data(self):
        g = "g per key channel" if self.kda else "g"
        return ("synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), beta=sigmoid, "
                "%s=-softplus(N(0,1)), h0 N(0, 0.1^2))" % g)

    def cpu_sample(self, w, cpu, Ts=256):
        sl = lambda t: t[:1, :Ts] if t is not None else None
        x = {n: sl(cpu[n]) for n in ("q", "k", "v", "beta", self.gname)}
        x["h0"] = cpu["h0"][:1] if cpu["h0"] is not None else None
        t0 = time.time()
        self.oracle(w, x)
        return Ts, time.time() - t0


def run_token_serial(args, ws, rank, local):
    from gated_delta_rule_54_gb300 import synth
    from gated_delta_rule_54_gb300._lib import load

    ts = _TokenSerial(args.mode)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    load()
    w = synth.WORKLOADS[args.workload]
    w = synth.Workload(**{**w.__dict__, "seed": w.seed + rank})
    cpu = ts.make(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    for _ in range(args.warmup):
        ts.call(w, d)
    torch.cuda.synchronize()
    _barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(args.steps):
            ts.call(w, d)
        b.record(stream)
        torch.cuda.synchronize()
    _barrier(ws)
    ms_total = _max_over_ranks(a.elapsed_time(b), ws, dev)
    ms_step = ms_total / args.steps
    tokens = w.B * w.T
    value = tokens * ws * args.steps / (ms_total / 1e3)
    peak, _, peak_kind = _peaks()
    alg = token_serial_alg_bytes(w, ts.kda)
    achieved = alg / (ms_step / 1e3) / 1e9

    # end to end through the public API from pinned host buffers (two-precision only)
    e2e = None
    if not args.no_e2e and not ts.kda:
        names = ("q", "k", "v", "beta", "g", "h0")
        host_in = {n: cpu[n].pin_memory() for n in names}
        dev_in = [{n: torch.empty_like(t, device=dev) for n, t in host_in.items()} for _ in range(2)]
        res_d = [[torch.empty(w.B, w.T, w.Hv, w.Dv, device=dev),
                  torch.empty(w.B, w.Hv, w.Dk, w.Dv, device=dev)] for _ in range(2)]
        res_h = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in r] for r in res_d]

        def run(st):
            ts.call(w, dev_in[st], out=tuple(res_d[st]))
            return res_d[st]

        e_ms, s_ms = e2e_pipelined(dev, ws, args.steps, args.warmup, host_in, dev_in, run, res_h)
        e2e = {"value": round(tokens * ws / (e_ms / 1e3), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host_in.values()),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in res_h[0]),
               "ms_per_step": round(e_ms, 4),
               "schedule": "pipelined: step i+1's upload and step i-1's download overlap step i's "
                           "compute (three streams, two device buffer sets)",
               "serial_value": round(tokens * ws / (s_ms / 1e3), 1),
               "serial_ms_per_step": round(s_ms, 4)}

    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline:
        Ts, dt = ts.cpu_sample(w, cpu)
        cpu_base = {"value": round(Ts / dt, 2), "unit": "tokens/s", "cores": torch.get_num_threads(),
                    "kind": "oracle",
                    "sample": "1 sequence x %d tokens, all %d heads, fp64 %s oracle" % (
                        Ts, w.Hv, "KDA" if ts.kda else "two-precision")}
    line = {
        "metric": ts.metric, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": ts.data(), "config": ts.config(w),
        "clocks": clk.summary(), "e2e": e2e, "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": _traffic(ts.profile, ts.sources, args.workload),
                     "kernel": ts.kernel, "peak_source": peak_kind,
                     "alg_bytes_per_launch": alg, "launch_ms": round(ms_step, 4)},
        "cpu_baseline": cpu_base,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# two-precision training step (--mode two_precision_bwd): the forward saving
# its window anchors, then the window-wise adjoint
# ----------------------------------------------------------------------------
TPB_METRIC = ("two-precision GDN fwd+bwd tokens/s at B=4,T=4096,H=16,D=128 (fp32 anchor, E4M3 "
              "read copy, 16-token flush, window-wise adjoint); % of roofline")
TPB_SOURCES = ["gated_delta_rule_54_gb300/csrc/two_precision_bwd.cu",
               "gated_delta_rule_54_gb300/csrc/two_precision.cuh",
               "gated_delta_rule_54_gb300/csrc/common.cuh"]


def tp_anchor_bytes(w, flush=TP_FLUSH):
    """The forward's saved anchors: one fp32 [Hv, Dk, Dv] per window slot."""
    return (w.B * w.T // flush + w.B) * w.Hv * w.Dk * w.Dv * 4


def tp_bwd_alg_bytes(w, flush=TP_FLUSH):
    """Algorithmic HBM bytes of one backward launch: q, k, v (bf16), beta, g,
    dO (f32) and the anchors read once; dq, dk, dv, dbeta, dg written once;
    dht read and dh0 written."""
    tok = w.B * w.T
    b = tok * (w.Hk * w.Dk * 2 * 2 + w.Hv * w.Dv * 2 + w.Hv * 4 * 2 + w.Hv * w.Dv * 4)
    b += tok * (w.Hk * w.Dk * 4 * 2 + w.Hv * w.Dv * 4 + w.Hv * 4 * 2)
    return b + tp_anchor_bytes(w, flush) + w.B * w.Hv * w.Dk * w.Dv * 4 * 2


def tp_upstream(w, seed):
    gen = torch.Generator().manual_seed(seed)
    do = torch.randn(w.B, w.T, w.Hv, w.Dv, generator=gen)
    dht = torch.randn(w.B, w.Hv, w.Dk, w.Dv, generator=gen) * 0.1
    return do, dht


def tp_bwd_cpu_sample(w, cpu, do, dht, Ts):
    """The oracle's autograd (fp64) on one sequence x Ts tokens, all heads."""
    from oracle.two_precision import two_precision_torch
    sl = lambda t: t[:1, :Ts]
    xs = [sl(cpu[n]).to(torch.float32).double().requires_grad_(True)
          for n in ("q", "k", "v", "beta", "g")]
    xs.append(cpu["h0"][:1].double().requires_grad_(True))
    t0 = time.time()
    o, ht = two_precision_torch(*xs, read_mode=w.state_mode, flush=TP_FLUSH)
    loss = (o * sl(do).double()).sum() + (ht * dht[:1].double()).sum()
    torch.autograd.grad(loss, xs)
    return Ts, time.time() - t0


def run_tp_bwd(args, ws, rank, local):
    from gated_delta_rule_54_gb300 import api, synth
    from gated_delta_rule_54_gb300._lib import load

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    load()
    w = synth.WORKLOADS[args.workload]
    w = synth.Workload(**{**w.__dict__, "seed": w.seed + rank})
    cpu = synth.make_inputs(w)
    do_h, dht_h = tp_upstream(w, 1000 + w.seed)
    names = ("q", "k", "v", "beta", "g", "h0")
    d = {n: cpu[n].to(dev) for n in names}
    d["do"], d["dht"] = do_h.to(dev), dht_h.to(dev)
    rm = w.state_mode
    f32 = dict(device=dev, dtype=torch.float32)

    def buffers():
        return {"o": torch.empty(w.B, w.T, w.Hv, w.Dv, **f32),
                "ht": torch.empty(w.B, w.Hv, w.Dk, w.Dv, **f32),
                "grads": (torch.empty(w.B, w.T, w.Hk, w.Dk, **f32),
                          torch.empty(w.B, w.T, w.Hk, w.Dk, **f32),
                          torch.empty(w.B, w.T, w.Hv, w.Dv, **f32),
                          torch.empty(w.B, w.T, w.Hv, **f32), torch.empty(w.B, w.T, w.Hv, **f32),
                          torch.empty(w.B, w.Hv, w.Dk, w.Dv, **f32))}

    def fwd(x, bufs):
        return api.gdn_two_precision_fwd(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                                         read_mode=rm, flush=TP_FLUSH, save_anchors=True,
                                         out=(bufs["o"], bufs["ht"]))

    def bwd(x, anchors, bufs):
        return api.gdn_two_precision_bwd(x["q"], x["k"], x["v"], x["beta"], x["g"], anchors,
                                         x["do"], x["dht"], read_mode=rm, flush=TP_FLUSH,
                                         out=bufs["grads"])

    bufs = buffers()

    def step(x, b):
        _, _, anchors = fwd(x, b)
        return bwd(x, anchors, b)

    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        step(d, bufs)
    torch.cuda.synchronize()
    _barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(args.steps):
            step(d, bufs)
        b.record(stream)
        torch.cuda.synchronize()
    _barrier(ws)
    ms_total = _max_over_ranks(a.elapsed_time(b), ws, dev)
    ms_step = ms_total / args.steps
    # the backward alone (its launches from one forward's anchors)
    _, _, anchors = fwd(d, bufs)
    for _ in range(2):
        bwd(d, anchors, bufs)
    torch.cuda.synchronize()
    a, b = ev(), ev()
    a.record(stream)
    for _ in range(args.steps):
        bwd(d, anchors, bufs)
    b.record(stream)
    torch.cuda.synchronize()
    bwd_ms = _max_over_ranks(a.elapsed_time(b), ws, dev) / args.steps
    tokens = w.B * w.T
    value = tokens * ws * args.steps / (ms_total / 1e3)
    peak, _, peak_kind = _peaks()
    alg = tp_bwd_alg_bytes(w)
    achieved = alg / (bwd_ms / 1e3) / 1e9
    G = w.Hv // w.Hk

    e2e = None
    if not args.no_e2e:
        host_in = {n: cpu[n].pin_memory() for n in names}
        host_in["do"], host_in["dht"] = do_h.pin_memory(), dht_h.pin_memory()
        dev_in = [{n: torch.empty_like(t, device=dev) for n, t in host_in.items()} for _ in range(2)]
        res_d = [buffers() for _ in range(2)]
        res_h = [[torch.empty(t.shape, dtype=t.dtype).pin_memory()
                  for t in (r["o"], r["ht"]) + r["grads"]] for r in res_d]

        def run(st):
            step(dev_in[st], res_d[st])
            return [res_d[st]["o"], res_d[st]["ht"]] + list(res_d[st]["grads"])

        e_ms, s_ms = e2e_pipelined(dev, ws, args.steps, args.warmup, host_in, dev_in, run, res_h)
        e2e = {"value": round(tokens * ws / (e_ms / 1e3), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host_in.values()),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in res_h[0]),
               "ms_per_step": round(e_ms, 4),
               "schedule": "pipelined: step i+1's upload and step i-1's download overlap step i's "
                           "compute (three streams, two device buffer sets)",
               "serial_value": round(tokens * ws / (s_ms / 1e3), 1),
               "serial_ms_per_step": round(s_ms, 4)}

    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline:
        Ts, dt = tp_bwd_cpu_sample(w, cpu, do_h, dht_h, 32)
        cpu_base = {"value": round(Ts / dt, 2), "unit": "tokens/s", "cores": torch.get_num_threads(),
                    "kind": "oracle",
                    "sample": "1 sequence x %d tokens, all %d heads, fp64 two-precision oracle "
                              "forward + autograd backward" % (Ts, w.Hv)}
    line = {
        "metric": TPB_METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), beta=sigmoid, "
                "g=-softplus(N(0,1)), h0 N(0, 0.1^2); dO N(0,1), dht N(0, 0.1^2))",
        "config": {"workload": w.name, "mode": "two_precision_bwd", "B": w.B, "T": w.T,
                   "Hk": w.Hk, "Hv": w.Hv, "Dk": w.Dk, "Dv": w.Dv, "read_mode": rm,
                   "flush": TP_FLUSH, "l2": "inputs larger than L2 (no flush needed)"},
        "clocks": clk.summary(), "e2e": e2e,
        "gpu_launches": args.steps * (2 + (2 if G > 1 else 0)),
        "fwd_ms": round(ms_step - bwd_ms, 4), "bwd_ms": round(bwd_ms, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": _traffic("gdn_two_precision_bwd_kernel_two_precision_layer.md",
                                         TPB_SOURCES, args.workload),
                     "kernel": "gdn_two_precision_bwd_kernel", "peak_source": peak_kind,
                     "alg_bytes_per_launch": alg, "launch_ms": round(bwd_ms, 4)},
        "cpu_baseline": cpu_base,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ----------------------------------------------------------------------------
def run_reference(args, ws, rank):
    if rank != 0:
        return
    from gated_delta_rule_54_gb300 import synth
    from oracle.chunked import chunked
    w = synth.WORKLOADS[args.workload]
    if args.mode == "decode":
        cpu = synth.make_inputs(synth.Workload(**{**w.__dict__, "B": 16}))
        for _ in range(args.warmup):
            decode_cpu_baseline(w, cpu, budget_s=1e9, rows=1)
        t0 = time.time()
        for _ in range(args.steps):
            decode_cpu_baseline(w, cpu, budget_s=1e9, rows=16)
        dt = time.time() - t0
        value = 16 * w.T * args.steps / dt
        sample = "16 rows x one token, all %d heads per step (fp64 decode oracle)" % w.Hv
        print(json.dumps({
            "impl": "reference", "metric": DECODE_METRIC, "value": round(value, 2),
            "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "mode": "decode", "B": w.B, "T": w.T, "Hk": w.Hk,
                       "Hv": w.Hv, "Dk": w.Dk, "Dv": w.Dv, "state_mode": w.state_mode},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s",
                             "cores": torch.get_num_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return
    if args.mode == "two_precision_bwd":
        cpu = synth.make_inputs(w)
        do_h, dht_h = tp_upstream(w, 1000 + w.seed)
        for _ in range(args.warmup):
            tp_bwd_cpu_sample(w, cpu, do_h, dht_h, 4)
        done = el = 0.0
        for _ in range(args.steps):
            n, dt = tp_bwd_cpu_sample(w, cpu, do_h, dht_h, 16)
            done += n
            el += dt
        value = done / el
        print(json.dumps({
            "impl": "reference", "metric": TPB_METRIC, "value": round(value, 2), "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "mode": "two_precision_bwd", "B": w.B, "T": w.T,
                       "Hk": w.Hk, "Hv": w.Hv, "Dk": w.Dk, "Dv": w.Dv, "read_mode": w.state_mode,
                       "flush": TP_FLUSH},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s",
                             "cores": torch.get_num_threads(), "kind": "oracle",
                             "sample": "1 sequence x 16 tokens, all %d heads per step (fp64 "
                                       "two-precision oracle forward + autograd backward)" % w.Hv},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return
    if args.mode in ("kda", "two_precision"):
        ts = _TokenSerial(args.mode)
        cpu = ts.make(w)
        for _ in range(args.warmup):
            ts.cpu_sample(w, cpu, Ts=64)
        done = el = 0.0
        for _ in range(args.steps):
            n, dt = ts.cpu_sample(w, cpu, Ts=256)
            done += n
            el += dt
        value = done / el
        sample = "1 sequence x 256 tokens, all %d heads per step (fp64 %s oracle)" % (
            w.Hv, "KDA" if ts.kda else "two-precision")
        print(json.dumps({
            "impl": "reference", "metric": ts.metric, "value": round(value, 2), "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": ts.config(w),
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s",
                             "cores": torch.get_num_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return
    bwd = args.mode == "fwdbwd"
    T_s = 1024   # bounded sample per step: one sequence, all heads, 1024 tokens
    ws_ = synth.Workload(**{**w.__dict__, "B": 1, "T": T_s})
    cpu = synth.make_inputs(ws_)
    xs = [cpu[x] for x in ("q", "k", "v", "beta", "g", "h0")]

    import oracle

    def step():
        if bwd:
            ys = [a.double().requires_grad_(True) if a is not None else None for a in xs]
            o, ht = chunked(*ys, state_mode=w.state_mode, w_mode=w.w_mode)
            (o.sum() + ht.sum()).backward()
        else:  # the forward baseline: the fp64 token recurrence in C
            oracle.recurrent(*xs, state_mode=w.state_mode)

    for _ in range(args.warmup):
        step()
    t0 = time.time()
    for _ in range(args.steps):
        step()
    dt = time.time() - t0
    value = T_s * args.steps / dt
    sample = "1 sequence x %d tokens, all %d heads per step (%s)" % (
        T_s, w.Hv, "fp64 chunked oracle, fwd+autograd bwd" if bwd
        else "fp64 token recurrence, C with OpenMP over (sequence, head)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "mode": args.mode, "B": w.B, "T": w.T, "Hk": w.Hk,
                       "Hv": w.Hv, "Dk": w.Dk, "Dv": w.Dv, "state_mode": w.state_mode,
                       "w_mode": w.w_mode},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s",
                             "cores": torch.get_num_threads() if bwd else oracle.num_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--mode", default=None,
                    choices=["fwd", "fwdbwd", "decode", "kda", "two_precision",
                             "two_precision_bwd"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--block-v", type=int, default=64, help="state-scale tile width")
    ap.add_argument("--neumann-degree", type=int, default=None,
                    help="Neumann approximate inverse of this degree instead of the exact solve")
    ap.add_argument("--micro-batches", type=int, default=0,
                    help="micro-batches of the workload per step (0: sized to ~50 ms per step)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.mode is None:
        args.mode = "fwdbwd" if _backward_available() else "fwd"
    if args.workload is None:
        args.workload = {"decode": "decode", "kda": "kda", "two_precision": "two_precision",
                         "two_precision_bwd": "two_precision",
                         "fwdbwd": "fwd_bwd"}.get(args.mode, "layer")
    args.bwd_launches = BWD_LAUNCHES
    ws, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    elif args.mode == "decode":
        run_decode(args, ws, rank, local)
    elif args.mode in ("kda", "two_precision"):
        run_token_serial(args, ws, rank, local)
    elif args.mode == "two_precision_bwd":
        run_tp_bwd(args, ws, rank, local)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        torch.distributed.destroy_process_group()


BWD_LAUNCHES = 2   # kernels one backward call launches (reverse scan + chunk gradients)


def _fused(w, block_v, neumann_degree):
    """The two-launch fused forward applies (as in the library's dispatch)."""
    return (w.Dk == 128 and w.Dv == 128 and w.state_mode != "none" and w.w_mode != "none"
            and block_v == 64 and neumann_degree is None)


def _fwd_launches(w, block_v, neumann_degree):
    """Kernels one forward call launches: chunk prep + fused scan/outputs, or
    chunk prep, state scan, outputs."""
    return 2 if _fused(w, block_v, neumann_degree) else 3


def _backward_available():
    return BWD_LAUNCHES > 0


if __name__ == "__main__":
    main()
