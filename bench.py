"""Benchmark of the fast-weight recurrence on GB300.

One timed "step" is one fw_prefill over the Falcon-1 bf16 workload
(B=8, H=16, T=4096, d=128, fp32 state; the chunked tensor-core kernel when it
takes the call), the path that runs every prefill row: feature map and
pairing, norms and gates, decay products, Gram and triangular solve,
residuals, outputs and state carry.  The JSON line also carries the other
workloads (linear attention, long context, fp32, decode) as sub-results.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica of the workload on its
own GPU (the chains are independent: no collective on the data path); the
value is all ranks' tokens over the slowest rank's time ("weak" scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_token_mixer_gb300 import inputs as I  # noqa: E402

HEADLINE = "falcon1_bf16"
METRIC = "fast-weight prefill tokens/s and decode steps/s on 1 GB300, % of roofline"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# FP32 FMA peak for a SIMT-bound kernel: 152 SMs x 128 FMA lanes x 2 flop x 2.07 GHz.
ALU_FP32_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


KERNEL_SOURCES = {
    "chunked prefill": ("fw_chunked.cu", "fw_sm100.cuh", "fw_internal.cuh"),
    "chunked prefill (two segments)": ("fw_chunked.cu", "fw_sm100.cuh", "fw_internal.cuh"),
    "chunked prefill (per channel)": ("fw_chunked_chan.cu", "fw_sm100.cuh", "fw_internal.cuh"),
    "recurrent (SIMT)": ("fw_recurrent.cu", "fw_internal.cuh"),
    "window prefill (SIMT)": ("fw_window_prefill.cu", "fw_window.cuh", "fw_sm100.cuh",
                              "fw_internal.cuh"),
    "decode step": ("fw_decode.cu",),
}


def sources_sha256(kernel):
    """Hash of the source files a kernel is built from (to tell whether a stored
    ncu traffic figure was taken on the kernel as it stands)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_token_mixer_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def stored_traffic(kernel, workload):
    """DRAM bytes read + written per launch from the committed ncu summary
    (profiles/traffic.json), or None when the kernel changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get("%s/%s" % (kernel, workload))
    except (OSError, ValueError):
        return None
    if not rec or rec.get("sources_sha256") != sources_sha256(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


def algorithmic_bytes_prefill(w):
    """Bytes a prefill must move: q, k, v read and o written once, beta and
    lambda read once (beta per value channel for Falcon-2), S0 read (when
    given) and S_T written once."""
    esz = 2 if w.dtype == torch.bfloat16 else 4
    ht = w.B * w.H * w.T
    gates = {"falcon1": 8, "falcon1a": 8, "falcon3": 8, "falcon3a": 8,
             "falcon2": 4 * w.d + 4, "falcon2a": 4 * w.d + 4}
    per_ht = 4 * w.d * esz + gates.get(w.mode, 0)
    state = w.B * w.H * w.d * w.d * 4
    return ht * per_ht + state * (2 if w.s0_std > 0 else 1)


def prefill_kernel(w, algo="auto", sms=152):
    """The kernel fw_prefill picks for a workload, as the library dispatches it:
    a step per value channel (Falcon-2 / 2A) on the per-channel chunked kernel
    where it takes the call (bf16, d = 128, phi = identity), else on the staged
    per-token kernel; the other modes on the chunked tensor-core kernel where it
    takes the call (bf16, d = 128; Falcon-1 / 1A only with phi = identity), else
    on the per-token kernel.  The chunked kernel runs each chain as two segments
    at once (plus a fix-up kernel) when at most a third of the sms SMs hold a
    chain and T >= 4096."""
    if algo == "recurrent":
        return "recurrent (SIMT)"
    tc = w.dtype == torch.bfloat16 and w.d == 128
    if w.mode in ("falcon2", "falcon2a"):
        if tc and w.phi == "identity":
            return "chunked prefill (per channel)"
        return "window prefill (SIMT)"
    chunked = tc and (w.mode == "linattn" or w.phi == "identity")
    if not chunked:
        return "recurrent (SIMT)"
    if 3 * w.B * w.H <= sms and w.T >= 4096:
        return "chunked prefill (two segments)"
    return "chunked prefill"


def matmul_flops_prefill(w, C=64):
    """Dense matmul FLOPs of the chunked forms per launch, on tcgen05: Falcon-1
    10 C d + 6 d^2 per head-token; linear attention and Falcon-1A (no
    residual, so no W, U or solve) 4 C d + 4 d^2 (Q X^T, P Y, Q S0, X^T Y);
    the per-channel kernel (Falcon-2) 4 C d + 6 d^2 (the Gram [X; Q] X^T,
    X S0, Q S0 and the state update; Falcon-2A 4 C d + 4 d^2, no X S0).  The
    per-channel kernel's cross-block sums on the warps' tf32 MMAs (112 d per
    head-token) are not counted.  None where the launch runs no tensor-core
    kernel."""
    k = prefill_kernel(w)
    ht = w.B * w.H * w.T
    if k == "chunked prefill (per channel)":
        return ht * (4 * C * w.d + (6 if w.mode == "falcon2" else 4) * w.d * w.d)
    if k not in ("chunked prefill", "chunked prefill (two segments)"):
        return None
    if w.mode == "falcon1":
        return ht * (10 * C * w.d + 6 * w.d * w.d)
    return ht * (4 * C * w.d + 4 * w.d * w.d)


MATMUL_NOTE = {"falcon1": "10Cd+6d^2", "falcon2": "4Cd+6d^2", "falcon2a": "4Cd+4d^2"}


# workloads the headline (fw_prefill) can run: the window family has its own call
PREFILL_WORKLOADS = sorted(n for n, w in I.WORKLOADS.items()
                           if w.mode not in ("falcon3", "falcon3a"))


def oracle_run(oracle, w, x, threads):
    """The fp64 oracle entry that computes workload w's mode, run on the input
    dict x.  Returns the name of the entry that ran."""
    if w.mode in ("falcon1", "falcon1a"):
        oracle.falcon1(x["q"], x["k"], x["v"], x["beta"], x["lam"], S0=x["S0"], phi=w.phi,
                       eps=w.eps, nthreads=threads, inner=(w.mode == "falcon1a"))
        return w.mode
    if w.mode in ("falcon2", "falcon2a"):
        oracle.falcon2(x["q"], x["k"], x["v"], x["beta"], x["lam"], S0=x["S0"], phi=w.phi,
                       eps=w.eps, nthreads=threads, inner=(w.mode == "falcon2a"))
        return w.mode
    if w.mode in ("falcon3", "falcon3a"):
        oracle.falcon3(x["q"], x["k"], x["v"], x["beta"], x["lam"], w.window, S0=x["S0"],
                       phi=w.phi, eps=w.eps, nthreads=threads, inner=(w.mode == "falcon3a"))
        return w.mode
    if w.mode == "linattn":
        oracle.linattn(x["q"], x["k"], x["v"], S0=x["S0"], phi=w.phi, nthreads=threads)
        return "linattn"
    raise ValueError("no oracle entry for mode %r" % w.mode)


def window_flops(w):
    """Flops of the Falcon-3 / 3A write by its definition, per head-token:
    W residual reads S^T x_j (Falcon-3 only), the rank-W write and the decay,
    and the read S^T q -- (2W + 2) d^2 multiply-adds (3A: W + 2), 2 flops each.
    The kernel forms the older pairs' reads by recursion, so it executes fewer.
    Falcon-2 / 2A (a step per value column) is the same count with W = 1."""
    reads = 0 if w.mode in ("falcon3a", "falcon2a") else w.window
    return w.B * w.H * w.T * 2 * (reads + w.window + 2) * w.d * w.d


def recurrence_flops(w):
    """Flops of the recurrence itself: about 6 d^2 per head-token."""
    return w.B * w.H * w.T * 6 * w.d * w.d


class Clocks:
    """Sample SM clocks and throttle reasons with nvidia-smi while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        mhz, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                mhz.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, p in zip(names, parts[3:7]):
                if p.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(mhz)}


def job_rate(ms_local, units_per_rank, world, dist=None, device=None):
    """Whole-job throughput over `world` ranks: the slowest rank's time (max over
    ranks) and all ranks' units divided by it.  Returns (ms_max, units per second)."""
    ms = float(ms_local)
    if dist is not None and world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, units_per_rank * world / (ms / 1e3)


def timed(fn, K, W, stream):
    """W untimed warm-up calls, then K calls each bracketed by CUDA events on
    the launching stream.  Returns (total ms of the region, per-call ms)."""
    for _ in range(W):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1), [a.elapsed_time(b) for a, b in ev]


def bench_prefill(w, K, W, dev, fw, algo="auto", rbw=False, same_pair=False):
    x = I.prefill_inputs(w, device=dev)
    o = torch.empty_like(x["q"])
    S_T = torch.empty(w.B, w.H, w.d, w.d, device=dev)
    stream = torch.cuda.current_stream()

    def fn():
        fw.prefill(x["q"], x["k"], x["v"], x["beta"], x["lam"], x["S0"], mode=w.mode,
                   phi=w.phi, eps=w.eps, algo=algo, o=o, S_T=S_T, stream=stream, rbw=rbw,
                   same_pair=same_pair)

    total, per = timed(fn, K, W, stream)
    fw.check(stream)
    kern_ms = statistics.mean(per)
    toks = w.B * w.T
    res = {
        "tokens_per_s": toks * K / (total / 1e3),
        "head_tokens_per_s": toks * w.H * K / (total / 1e3),
        "ms_per_step": total / K,
        "kernel_ms": kern_ms,
        "hbm_gbs": algorithmic_bytes_prefill(w) / (kern_ms / 1e3) / 1e9,
        "matmul_tflops": (matmul_flops_prefill(w) / (kern_ms / 1e3) / 1e12
                          if algo == "auto" and matmul_flops_prefill(w) else None),
        "recurrence_tflops": recurrence_flops(w) / (kern_ms / 1e3) / 1e12,
        "algo": algo,
        "kernel": prefill_kernel(w, algo),
    }
    if rbw or same_pair:
        res["flags"] = [f for f, on in (("rbw", rbw), ("same_pair", same_pair)) if on]
    elif algo == "auto" and res["kernel"] != "recurrent (SIMT)":
        # DRAM bytes of one launch from the committed ncu summary (None once the
        # kernel's sources changed since the capture)
        res["dram_bytes_per_launch"] = stored_traffic(res["kernel"], w.name)
    if res["kernel"] == "window prefill (SIMT)":
        # per-channel steps on the staged per-token kernel (window of one pair):
        # bound by FP32 ALU work, not by memory
        tf = window_flops(w) / (kern_ms / 1e3) / 1e12
        res["roofline"] = {"bound": "alu", "achieved": tf, "peak": ALU_FP32_TFLOPS,
                           "unit": "TFLOP/s", "frac": tf / ALU_FP32_TFLOPS,
                           "kernel": "window prefill (SIMT)",
                           "flops": "4 d^2 multiply-adds per head-token (2A: 3)"}
    return res, x


def bench_window(w, K, W, dev, fw):
    """Falcon-3 / 3A prefill through fw_window_prefill (window of w.window pairs)."""
    x = I.prefill_inputs(w, device=dev)
    o = torch.empty_like(x["q"])
    S_T = torch.empty(w.B, w.H, w.d, w.d, device=dev)
    win = fw.new_window(w.B, w.H, w.d, w.window, dev)
    stream = torch.cuda.current_stream()

    def fn():
        fw.window_prefill(x["q"], x["k"], x["v"], x["beta"], x["lam"], w.window, x["S0"],
                          mode=w.mode, phi=w.phi, eps=w.eps, o=o, S_T=S_T, win_out=win,
                          stream=stream)

    total, per = timed(fn, K, W, stream)
    fw.check(stream)
    kern_ms = statistics.mean(per)
    tf = window_flops(w) / (kern_ms / 1e3) / 1e12
    toks = w.B * w.T
    return {"tokens_per_s": toks * K / (total / 1e3), "ms_per_step": total / K,
            "kernel_ms": kern_ms, "window": w.window,
            "hbm_gbs": algorithmic_bytes_prefill(w) / (kern_ms / 1e3) / 1e9,
            "roofline": {"bound": "alu", "achieved": tf, "peak": ALU_FP32_TFLOPS,
                         "unit": "TFLOP/s", "frac": tf / ALU_FP32_TFLOPS,
                         "kernel": "window prefill (SIMT)",
                         "traffic": stored_traffic("window prefill (SIMT)", w.name),
                         "flops": "(2W+2) d^2 multiply-adds per head-token (3A: W+2)"}}


def bench_window_step(K_steps, W, dev, fw, window=4, mode="falcon3"):
    """Falcon-3 / 3A decode steps on the decode workload's states, alternating
    two carried windows."""
    cfg = I.DECODE
    Bn, H, d = cfg["batch"], cfg["H"], cfg["d"]
    x = I.decode_inputs(K_steps, Bn, H, d, device=dev)
    S = torch.zeros(Bn, H, d, d, device=dev)
    o = torch.empty(Bn, H, d, device=dev, dtype=torch.bfloat16)
    wins = [fw.new_window(Bn, H, d, window, dev), fw.new_window(Bn, H, d, window, dev)]
    stream = torch.cuda.current_stream()
    i = [0]

    def fn():
        s = i[0] % K_steps
        fw.window_step(x["q"][s], x["k_prev"][s], x["v"][s], x["beta"][s], x["lam"][s], S,
                       window, win_in=wins[i[0] & 1], win_out=wins[(i[0] + 1) & 1], mode=mode,
                       eps=cfg["eps"], o=o, stream=stream)
        i[0] += 1

    total, per = timed(fn, K_steps, W, stream)
    fw.check(stream)
    kern_ms = statistics.mean(per)
    # state read and written, carried window read and written, step vectors
    nbytes = Bn * H * (2 * d * d * 4 + 2 * (window - 1) * 2 * d * 4 + 4 * d * 2 + 8 + 8)
    return {"steps_per_s": K_steps / (total / 1e3), "tokens_per_s": Bn * K_steps / (total / 1e3),
            "kernel_ms": kern_ms, "hbm_gbs": nbytes / (kern_ms / 1e3) / 1e9,
            "bytes_per_step": nbytes, "steps": K_steps, "window": window, "mode": mode}


def e2e_prefill(w, K, W, dev, fw, x_dev):
    """Same metric through the public call with host buffers: every step copies
    its inputs from pinned host memory to the device, runs fw_prefill and
    reads o and S_T back into pinned host memory.  The steps are pipelined on
    three streams with two device buffer sets, so that step i+1's host-to-device
    copies and step i-1's device-to-host copies overlap step i's kernel; the
    timed region runs from the first copy in to the last copy out."""
    host = {k: (t.cpu().pin_memory() if t is not None else None) for k, t in x_dev.items()}
    dbuf = [{k: (torch.empty_like(t) if t is not None else None) for k, t in x_dev.items()}
            for _ in range(2)]
    outs = [(torch.empty_like(x_dev["q"]), torch.empty(w.B, w.H, w.d, w.d, device=dev))
            for _ in range(2)]
    o_h = torch.empty(x_dev["q"].shape, dtype=x_dev["q"].dtype).pin_memory()
    S_h = torch.empty((w.B, w.H, w.d, w.d), dtype=torch.float32).pin_memory()
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = o_h.numel() * o_h.element_size() + S_h.numel() * 4

    def run(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_run = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(n):
            d, (o, S_T) = dbuf[i & 1], outs[i & 1]
            if i >= 2:
                s_in.wait_event(ev_run[i - 2])      # step i-2's kernel has read this buffer set
            with torch.cuda.stream(s_in):
                for k, t in host.items():
                    if t is not None:
                        d[k].copy_(t, non_blocking=True)
            ev_in[i].record(s_in)
            s_run.wait_event(ev_in[i])
            if i >= 2:
                s_run.wait_event(ev_out[i - 2])     # step i-2's results are copied out
            fw.prefill(d["q"], d["k"], d["v"], d["beta"], d["lam"], d["S0"], mode=w.mode,
                       phi=w.phi, eps=w.eps, o=o, S_T=S_T, stream=s_run)
            ev_run[i].record(s_run)
            s_out.wait_event(ev_run[i])
            with torch.cuda.stream(s_out):
                o_h.copy_(o, non_blocking=True)
                S_h.copy_(S_T, non_blocking=True)
            ev_out[i].record(s_out)
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    run(W)
    total = run(K)
    fw.check(s_run)
    return {"value": w.B * w.T * K / (total / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": "copies in, kernel and copies out of consecutive steps overlap on three streams"}


def bench_decode(K_steps, W, dev, fw):
    cfg = I.DECODE
    Bn, H, d = cfg["batch"], cfg["H"], cfg["d"]
    x = I.decode_inputs(K_steps, Bn, H, d, device=dev)
    S = torch.zeros(Bn, H, d, d, device=dev)
    o = torch.empty(Bn, H, d, device=dev, dtype=torch.bfloat16)
    stream = torch.cuda.current_stream()
    i = [0]

    def fn():
        s = i[0] % K_steps
        fw.step(x["q"][s], x["k_prev"][s], x["v"][s], x["beta"][s], x["lam"][s], S,
                eps=cfg["eps"], o=o, stream=stream)
        i[0] += 1

    total, per = timed(fn, K_steps, W, stream)
    fw.check(stream)
    kern_ms = statistics.mean(per)
    nbytes = Bn * H * (2 * d * d * 4 + 4 * d * 2 + 8)
    res = {"steps_per_s": K_steps / (total / 1e3), "tokens_per_s": Bn * K_steps / (total / 1e3),
           "kernel_ms": kern_ms, "hbm_gbs": nbytes / (kern_ms / 1e3) / 1e9,
           "bytes_per_step": nbytes, "steps": K_steps}
    # the DRAM bytes ncu counted for one launch of this kernel (part of the state is
    # still in L2 from the previous step), and the rate on those bytes
    dram = stored_traffic("decode step", "decode")
    res["dram_bytes_per_launch"] = dram
    res["dram_gbs"] = dram / (kern_ms / 1e3) / 1e9 if dram else None
    return res


def cpu_baseline(w, x=None, budget_s=10.0):
    """The fp64 oracle as it stands, on this host's cores, on a bounded sample
    of the workload: the workload's own chains (x, the inputs the GPU leg
    timed, copied to the host; drawn here when None), full T, in groups of
    one chain per core, until every chain is done or about budget_s seconds
    of oracle time have passed."""
    import oracle
    oracle.build()
    n_all = w.B * w.H
    threads = oracle.default_threads()
    x = I.prefill_inputs(w) if x is None else {k: (t.cpu() if t is not None else None)
                                                for k, t in x.items()}
    flat = {k: (t.reshape((1, n_all) + tuple(t.shape[2:])) if t is not None else None)
            for k, t in x.items()}
    done, dt = 0, 0.0
    ran = None
    while done < n_all and dt < budget_s:
        n = min(threads, n_all - done)
        sub = {k: (t[:, done:done + n].contiguous() if t is not None else None)
               for k, t in flat.items()}
        t0 = time.perf_counter()
        ran = oracle_run(oracle, w, sub, threads)
        dt += time.perf_counter() - t0
        done += n
    # tokens/s of the whole workload: chains are independent, so the sample's
    # head-token rate carries over; one token = H head-tokens.
    ht_rate = done * w.T / dt
    return {"value": ht_rate / w.H, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "oracle": ran,
            "sample": "%d of %d chains (B*H) in groups of %d, full T=%d, d=%d, fp64, %.2f s"
                      % (done, n_all, threads, w.T, w.d, dt)}


def headline_config(w, world):
    """The `config` object of the bench line, shared by both arms."""
    return {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d_k": w.d, "d_v": w.d,
            "mode": w.mode, "state": "fp32", "global_batch": w.B * world,
            "seq_len": w.T, "parallelism": "replicas x%d (independent chains)" % world,
            "l2": "inputs larger than L2 (%.0f MB moved per step)"
                  % (algorithmic_bytes_prefill(w) / 1e6)}


def run_reference(args):
    """Reference arm: the fp64 oracle as it stands, timed on the host cores
    (rank 0 only; other ranks return without work)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = I.WORKLOADS[args.workload]
    threads = oracle.default_threads()
    n = max(1, min(w.B * w.H, threads))
    sub = I.prefill_inputs(w.with_shape(B=1, H=n))
    ran = []

    def fn():
        ran.append(oracle_run(oracle, w, sub, threads))

    for _ in range(args.warmup):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    dt = time.perf_counter() - t0
    val = n * w.T * args.steps / dt / w.H
    sample = "%d of %d chains per step (B*H), full T=%d, d=%d, fp64" % (n, w.B * w.H, w.T, w.d)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(w, args.gpus),
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "oracle": ran[-1], "sample": sample},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_sub(name, K, W, dev, fw, peaks):
    """One sub-benchmark alone (the same calls the full run makes)."""
    if name == "decode":
        r = bench_decode(K, W, dev, fw)
    elif name in ("decode_falcon3_w4", "decode_falcon3a_w4"):
        r = bench_window_step(K, W, dev, fw, window=4, mode=name.split("_")[1])
    elif name in I.WORKLOADS and I.WORKLOADS[name].mode in ("falcon3", "falcon3a"):
        return dict(bench_window(I.WORKLOADS[name], K, W, dev, fw), workload=name)
    elif name in I.WORKLOADS:
        r, _ = bench_prefill(I.WORKLOADS[name], K, W, dev, fw)
    else:
        raise SystemExit("unknown sub-benchmark %r" % name)
    r["hbm_frac"] = r["hbm_gbs"] / peaks["hbm"]
    if r.get("dram_gbs"):
        r["dram_frac"] = r["dram_gbs"] / peaks["hbm"]
    r["workload"] = name
    return r


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=PREFILL_WORKLOADS)
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline leg")
    ap.add_argument("--sub", default=None,
                    help="run one sub-benchmark of the 'workloads' object alone (a prefill "
                         "workload name, decode, decode_falcon3_w4 or decode_falcon3a_w4) and "
                         "print its result; for profiling")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        run_reference(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from linear_token_mixer_gb300 import build as B
    B.build()
    from linear_token_mixer_gb300 import fw
    fw.lib()
    peaks = _peaks()
    if args.sub:
        print(json.dumps(run_sub(args.sub, args.steps, args.warmup, dev, fw, peaks)), flush=True)
        return
    w = I.WORKLOADS[args.workload]

    # ---- headline: timed region bracketed by barrier + synchronize
    x = I.prefill_inputs(w, device=dev)
    o = torch.empty_like(x["q"])
    S_T = torch.empty(w.B, w.H, w.d, w.d, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        fw.prefill(x["q"], x["k"], x["v"], x["beta"], x["lam"], x["S0"], mode=w.mode,
                   phi=w.phi, eps=w.eps, o=o, S_T=S_T, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with Clocks(local) as clk:
        time.sleep(0.3)
        t_start = time.perf_counter()
        for a, b in ev:
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        t_host = time.perf_counter() - t_start
        # keep the GPU busy while the clock sampler catches at least a few samples
        if t_host < 0.5:
            t_end = time.perf_counter() + 0.5
            while time.perf_counter() < t_end:
                step()
            torch.cuda.synchronize()
    if dist:
        dist.barrier()
    fw.check(stream)
    per = [a.elapsed_time(b) for a, b in ev]
    ms_total, value = job_rate(ev[0][0].elapsed_time(ev[-1][1]), w.B * w.T * args.steps, world,
                               dist, dev)
    kern_ms = statistics.mean(per)

    algo_bytes = algorithmic_bytes_prefill(w)
    achieved_gbs = algo_bytes / (kern_ms / 1e3) / 1e9
    kname = prefill_kernel(w)
    if kname in ("chunked prefill", "chunked prefill (two segments)", "chunked prefill (per channel)"):
        roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": achieved_gbs / peaks["hbm"],
                "traffic": stored_traffic(kname, w.name),
                "kernel": kname, "peak_source": peaks["src"],
                "algorithmic_bytes_per_launch": algo_bytes}
    else:
        flops = window_flops(w) if kname == "window prefill (SIMT)" else recurrence_flops(w)
        tf = flops / (kern_ms / 1e3) / 1e12
        roof = {"bound": "alu", "achieved": tf, "peak": ALU_FP32_TFLOPS, "unit": "TFLOP/s",
                "frac": tf / ALU_FP32_TFLOPS,
                "traffic": stored_traffic(kname, w.name), "kernel": kname,
                "peak_source": "152 SMs x 128 FP32 lanes x 2 x 2.07 GHz"}
    mm = matmul_flops_prefill(w)
    mm_tf = mm / (kern_ms / 1e3) / 1e12 if mm else None

    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": headline_config(w, world),
        "roofline": roof,
        "tensor": ({"matmul_tflops": mm_tf, "peak": peaks["bf16"],
                    "frac": mm_tf / peaks["bf16"], "chunk": 64,
                    "note": "dense matmul FLOPs of the chunked form (%s per head-token)"
                            % MATMUL_NOTE.get(w.mode, "4Cd+4d^2")}
                   if mm_tf else None),
        "gpu_launches": args.steps,
        "kernel_ms": kern_ms,
    }

    if rank == 0:
        out["clocks"] = clk.summary()
        out["e2e"] = e2e_prefill(w, max(3, args.steps // 2), 3, dev, fw, x)
        if not args.no_cpu:
            out["cpu_baseline"] = cpu_baseline(w, x)
        if not args.no_extra:
            extra = {}
            for name in ("linattn_bf16", "falcon1_long", "falcon1_fp32", "falcon1a_bf16",
                         "falcon2_bf16"):
                wn = I.WORKLOADS[name]
                r, _ = bench_prefill(wn, 5 if name not in ("falcon1_long", "falcon2_bf16") else 3,
                                     3, dev, fw)
                r["hbm_frac"] = r["hbm_gbs"] / peaks["hbm"]
                extra[name] = r
            # the read-before-write / same-step-pair arms on the headline workload
            r, _ = bench_prefill(w, 5, 3, dev, fw, rbw=True, same_pair=True)
            r["hbm_frac"] = r["hbm_gbs"] / peaks["hbm"]
            extra[w.name + "+rbw+same_pair"] = r
            dec = bench_decode(I.DECODE["steps"], 3, dev, fw)
            dec["hbm_frac"] = dec["hbm_gbs"] / peaks["hbm"]
            dec["dram_frac"] = dec["dram_gbs"] / peaks["hbm"] if dec["dram_gbs"] else None
            extra["decode"] = dec
            # the window family (Falcon-3 / 3A, W = 4): prefill and decode step
            for name in ("falcon3_bf16", "falcon3a_bf16"):
                extra[name] = bench_window(I.WORKLOADS[name], 3, 3, dev, fw)
            for mode in ("falcon3", "falcon3a"):
                ds = bench_window_step(256, 3, dev, fw, window=4, mode=mode)
                ds["hbm_frac"] = ds["hbm_gbs"] / peaks["hbm"]
                extra["decode_%s_w4" % mode] = ds
            out["workloads"] = extra
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
