#!/usr/bin/env python3
"""Attention training-step benchmark on GB300.

Workload: causal attention forward + backward, batch 4 x N=8192, H=32, D=128,
bf16 Q/K/V/dO ~ N(0,1) (seed 5), scale D^-1/2; the batch is packed as four
sequences with cu_seqlens [0, 8192, 16384, 24576, 32768].  One step = one
forward (O stored in f32, lse) and one backward (Dr preprocess, dK/dV, dQ)
through the library's C ABI.

Metric: attention fwd+bwd TFLOP/s, with fwd = 4 N^2 D H / 2 per causal
sequence and bwd = 2.5 x fwd, summed over the batch; `value` is the whole-job
rate over all ranks (each rank runs the full batch: weak scaling, no
collective on the data path).

The default run also times the forward alone on the four smaller
configurations (causal N=256 fp16, full N=1024 fp16, varlen causal bf16, cross
f32 8192 x 2048) and adds them to the same line as a `workloads` record
(device time per call, TFLOP/s, algorithmic bytes and GB/s, roofline, clocks,
the oracle's rate); `--no-workloads` skips it.

Prints one JSON line.  `--impl reference` times the f64 CPU oracle instead,
on a bounded sample of the same workload.  `--workload <name>` measures the
forward alone on one of the smaller workloads (causal_fp16_n256,
full_fp16_n1024, varlen_causal_bf16, cross_f32_8192x2048, and
pruned_full_bf16_n8192 for `--prune-threshold`) with the same line;
`--workload csr_*` measures attention over a CSR relation (radius graphs).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "causal_train_bf16_b4_n8192"
METRIC = "attention fwd+bwd TFLOP/s (causal, B=4, N=8192, H=32, D=128, bf16)"
UNIT = "TFLOP/s"


def attention_flops(lengths_q, lengths_k, H, D, causal):
    """Algorithmic forward FLOPs: 4 Lq Lk D H per sequence, halved for causal."""
    f = 0.0
    for lq, lk in zip(lengths_q, lengths_k):
        f += 4.0 * lq * lk * D * H * (0.5 if causal else 1.0)
    return f


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a per-rank number over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: every rank processes `units_per_rank` (weak
    scaling); the job takes as long as its slowest rank."""
    return units_per_rank * world / (ms_max * 1e-3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p.get("hbm_gbs"), "bf16_tflops": p.get("bf16_tflops"),
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"),
                "sm_max_mhz": p.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


def spread(ms_list):
    """Median, minimum and maximum of per-step times (ms)."""
    return {"median": statistics.median(ms_list), "min": min(ms_list), "max": max(ms_list)}


def dtype_label(w) -> str:
    """The arithmetic type a workload computes in, for the JSON line ("e4m3+bf16"
    when fp8 queries and keys feed the score contraction)."""
    base = {"fp16": "f16", "bf16": "bf16", "f32": "f32"}[w.dtype]
    return ("e4m3+" if getattr(w, "qk_fp8", False) else "") + base


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key, src_hash):
    """DRAM bytes per launch from a committed ncu summary, if the kernel
    source has not changed since the counters were taken (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel_key)
    if not rec or rec.get("source_hash") != src_hash:
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms; the summary
    keeps the samples taken between start() and stop() (the timed region)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            # wait (up to 3 s) for the first sample so that the region is covered
            deadline = time.time() + 3.0
            while time.time() < deadline and os.path.getsize(self.file.name) == 0:
                time.sleep(0.02)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.06)  # one more sample after the region
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    @staticmethod
    def _when(stamp):
        import datetime
        try:
            return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        if not self.proc or not self.file:
            return None
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.file.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        parsed = []
        for r in rows:
            if len(r) < 10:
                continue
            try:
                parsed.append((self._when(r[0]), float(r[2]), float(r[3]), r[6:10]))
            except ValueError:
                continue
        inside = parsed
        if self.t0 is not None and self.t1 is not None:
            # the region plus one sampling period on each side
            inside = [x for x in parsed if x[0] is not None and self.t0 - 0.05 <= x[0] <= self.t1 + 0.05]
            if not inside:
                inside = parsed
        if not inside:
            return None
        reasons = {n for x in inside for n, val in zip(names, x[3]) if val.strip().lower() == "active"}
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": inside[-1][2],
                "reasons": sorted(reasons), "samples": len(inside)}


def time_oracle_sample(x, w, max_seconds=20.0):
    """Time the oracle's forward + backward on whole (sequence, head) pairs of
    the workload, adding pairs until about `max_seconds` of CPU work."""
    import numpy as np

    import oracle
    L = x["lengths_q"][0]
    pair_flops = attention_flops([L], [L], 1, w.D, w.causal) * 3.5
    done, spent, pairs = 0, 0.0, []
    rng = np.random.default_rng(0)
    while spent < max_seconds * 0.5 and done < 8:
        b, h = int(rng.integers(0, w.batch)), int(rng.integers(0, w.H))
        s0, s1 = b * L, (b + 1) * L
        q, k, v, dO = (x[n][s0:s1, h:h + 1] for n in ("q", "k", "v", "dO"))
        t0 = time.perf_counter()
        oracle.fwd(q, k, v, causal=True)
        oracle.bwd(q, k, v, dO, causal=True)
        spent += time.perf_counter() - t0
        done += 1
        pairs.append((b, h))
    return {"value": pair_flops * done / spent / 1e12, "unit": UNIT, "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{done} whole (sequence, head) pairs of the workload, fwd+bwd, "
                      f"N={L}, D={w.D}, causal: {spent:.1f} s"}


FWD_WORKLOADS = ("causal_fp16_n256", "full_fp16_n1024", "varlen_causal_bf16", "cross_f32_8192x2048",
                 "pruned_full_bf16_n8192", "causal_fp8qk_b4_n8192")
CSR_WORKLOADS = ("csr_gat_n512", "csr_radius_field_bf16", "csr_radius_dot_bf16")
L2_BYTES = 129 * 1024 * 1024


# the four smaller configurations, timed forward-only inside the default run
SUB_WORKLOADS = ("causal_fp16_n256", "full_fp16_n1024", "varlen_causal_bf16", "cross_f32_8192x2048")


def fwd_algorithmic_bytes(lengths_q, lengths_k, H, D, qk_es, v_es, o_es):
    """Bytes a forward must move at least: q, k and v read once, o and lse
    (f32) written once."""
    tq, tk = sum(lengths_q), sum(lengths_k)
    return (tq * qk_es + tk * qk_es + tk * v_es) * H * D + tq * H * D * o_es + 4 * tq * H


def copy_bandwidth(dev, nbytes=256 << 20, reps=4):
    """Pinned host <-> device copy bandwidth on this machine, GB/s: host to
    device alone, device to host alone, and both directions at once (two
    streams; the total of both)."""
    import torch
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    main = torch.cuda.current_stream(dev)
    sa, sb = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def run(h2d, d2h):
        ev = torch.cuda.Event()
        ev.record(main)
        for st, on, fn in ((sa, h2d, lambda: d_in.copy_(h_in, non_blocking=True)),
                           (sb, d2h, lambda: h_out.copy_(d_out, non_blocking=True))):
            if on:
                st.wait_event(ev)
                with torch.cuda.stream(st):
                    fn()
                done = torch.cuda.Event()
                done.record(st)
                main.wait_event(done)

    out = {}
    for name, h2d, d2h in (("h2d_gbs", True, False), ("d2h_gbs", False, True), ("both_gbs", True, True)):
        run(h2d, d2h)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(main)
        for _ in range(reps):
            run(h2d, d2h)
        t1.record(main)
        torch.cuda.synchronize()
        moved = nbytes * reps * (int(h2d) + int(d2h))
        out[name] = moved / (t0.elapsed_time(t1) * 1e-3) / 1e9
    return out


def time_oracle_fwd_rows(x, w, max_seconds=15.0):
    """Time the oracle's forward on randomly drawn query rows of the workload,
    adding rows until about `max_seconds` of CPU work; report the workload's
    FLOP rate over those rows."""
    import numpy as np

    import oracle
    lq, lk = x["lengths_q"], x["lengths_k"]
    cu = np.concatenate([[0], np.cumsum(lq)])
    rng = np.random.default_rng(0)
    done_rows, spent, flops = 0, 0.0, 0.0
    n = 64
    while spent < max_seconds * 0.5:
        toks = rng.integers(0, int(cu[-1]), n)
        heads = rng.integers(0, w.H, n)
        t0 = time.perf_counter()
        oracle.fwd_rows(x["q"], x["k"], x["v"], toks, heads, causal=w.causal,
                        cu_seqlens_q=x["cu_seqlens_q"], cu_seqlens_k=x["cu_seqlens_k"])
        spent += time.perf_counter() - t0
        seq = np.searchsorted(cu, toks, side="right") - 1
        for t, b in zip(toks, seq):
            keys = min(int(t - cu[b]) + 1, lk[b]) if w.causal else lk[b]
            flops += 4.0 * keys * w.D
        done_rows += n
        n = min(4 * n, 1 << 16)
    return {"value": flops / spent / 1e12, "unit": UNIT, "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{done_rows} random (query row, head) pairs of the workload, forward: "
                      f"{spent:.1f} s"}


def time_forward_launches(call, stream, flush, steps, warmup, local, sync_ranks=None):
    """Device time (ms, CUDA events on `stream`) of each of `steps` forward
    launches after `warmup` untimed ones, the L2 flushed before each launch when
    `flush` (a device buffer larger than L2) is given; nvidia-smi clocks are
    sampled during the timed launches.  Returns (per-launch ms, kernels
    launched, clock summary)."""
    import torch

    import online_softmax_attention_gb300 as attn
    for _ in range(warmup):
        call.run(stream)
    torch.cuda.synchronize()
    status = attn.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} ({attn.strerror(status)}) set during warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    n0 = attn.launch_count()
    if sync_ranks:
        sync_ranks()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.start()
        for e0, e1 in evs:
            if flush is not None:
                flush.zero_()
            e0.record(stream)
            call.run(stream)
            e1.record(stream)
        torch.cuda.synchronize()
        clk.stop()
    if sync_ranks:
        sync_ranks()
    launches = attn.launch_count() - n0
    status = attn.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} ({attn.strerror(status)}) set in the timed region")
    return [a.elapsed_time(b) for a, b in evs], launches, clk.summary()


def fwd_peak(family, w, peaks, dev):
    """(peak, bound, note) of a forward's roofline: the bf16 / f16 dense
    tensor peak (burst: a forward launch is timed alone), 4/3 of it with fp8
    scores, or the FP32 FFMA peak for the CUDA-core kernel."""
    import torch
    if family == "tc" and w.qk_fp8:
        # half the FLOPs (S = Q K^T) at the fp8 rate, 2x the 16-bit rate (nominal
        # ratio), half (P V) at the 16-bit rate: peak = 2 / (1/(2 P) + 1/P) = 4 P / 3
        return (peaks["bf16_tflops"] * 4.0 / 3.0, "tensor",
                f"mixed: fp8 score contraction at 2x and bf16 value contraction at 1x the "
                f"bf16 dense burst peak ({peaks['source']}), i.e. 4/3 of it")
    if family == "tc" and w.dtype == "f32":
        # f32 inputs on the tensor cores: each contraction is six bf16 products
        # of the operands' bf16 parts, so the tensor pipe does 6x the algorithmic work
        return (peaks["bf16_tflops"] / 6.0, "tensor",
                f"f32 by bf16 operand splitting: six bf16 products per contraction, 1/6 of the "
                f"bf16 dense burst peak ({peaks['source']})")
    if family == "tc":
        return peaks["bf16_tflops"], "tensor", f"bf16/f16 dense, burst ({peaks['source']})"
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return (sms * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12, "alu",
            f"FP32 FFMA: {sms} SMs x 128 lanes x 2 FLOP x {peaks['sm_max_mhz']:.0f} MHz")


def fwd_kernel_sources(family, dtype="bf16"):
    csrc = "online_softmax_attention_gb300/csrc/"
    shared = [csrc + "common.cuh", csrc + "internal.h"]
    if family == "tc":
        return [csrc + ("fwd_x3.cu" if dtype == "f32" else "fwd_tc.cu")] + shared + [csrc + "sm100.cuh"]
    return [csrc + "fwd_simt.cu"] + shared


def forward_record(name, dev, local, steps, warmup, oracle_seconds):
    """Forward-only measurement of one of the smaller configurations, for the
    `workloads` record of the default run: device time per forward call (L2
    flushed before each call when the inputs fit in L2), FLOP rate, algorithmic
    bytes and their rate, the roofline of the attention kernel, clocks, and the
    oracle's rate on a bounded sample of the same rows."""
    import torch

    import attn_inputs
    import online_softmax_attention_gb300 as attn
    w = attn_inputs.WORKLOADS[name]
    x = attn_inputs.make_workload(w)
    flops = attention_flops(x["lengths_q"], x["lengths_k"], w.H, w.D, w.causal)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    cq = x["cu_seqlens_q"].to(dev) if x["cu_seqlens_q"] is not None else None
    ck = x["cu_seqlens_k"].to(dev) if x["cu_seqlens_k"] is not None else None
    call = attn.FwdCall(q, k, v, causal=w.causal, cu_seqlens_q=cq, cu_seqlens_k=ck,
                        out_dtype=torch.float32 if w.dtype == "bf16" else None)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if in_bytes < L2_BYTES else None
    stream = torch.cuda.current_stream()
    per_launch, launches, clocks = time_forward_launches(call, stream, flush, steps, warmup, local)
    ms = statistics.median(per_launch)
    nbytes = fwd_algorithmic_bytes(x["lengths_q"], x["lengths_k"], w.H, w.D, q.element_size(),
                                   v.element_size(), call.o.element_size())
    family = call.selected_kernel()
    peaks = load_peaks()
    peak, bound, note = fwd_peak(family, w, peaks, dev)
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    traffic = recorded_traffic("fwd:" + name, source_hash(fwd_kernel_sources(family, w.dtype)))
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ffma_peak = sms * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
    rec = {
        "config": w.note, "kernel": family, "num_splits": call.num_splits(),
        "dtype": dtype_label(w), "o_dtype": str(call.o.dtype).replace("torch.", ""),
        "ms": ms, "ms_spread": spread(per_launch), "steps": steps, "warmup": warmup,
        "flops": flops, "tflops": tflops, "bytes": nbytes, "gbs": gbs,
        "gpu_launches_per_call": launches / steps,
        "l2": "flushed before every call (inputs fit in L2)" if flush is not None
              else "no flush: inputs larger than L2",
        "roofline": {"bound": bound, "achieved": tflops, "peak": peak, "unit": UNIT,
                     "frac": tflops / peak, "peak_source": note,
                     "hbm_frac": gbs / peaks["hbm_gbs"], "frac_of_fp32_ffma": tflops / ffma_peak,
                     "traffic": traffic},
        "clocks": clocks,
    }
    if oracle_seconds:
        rec["cpu_baseline"] = time_oracle_fwd_rows(x, w, max_seconds=oracle_seconds)
    del call, q, k, v, flush
    torch.cuda.empty_cache()
    return rec


def run_forward_workload(args, rank, world):
    """Forward-only measurement of one of the smaller workloads (a parity
    workload, timed on request): TFLOP/s of the forward, L2 flushed between
    launches when the inputs fit in L2."""
    import torch
    import torch.distributed as dist

    import attn_inputs
    import online_softmax_attention_gb300 as attn

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    w = attn_inputs.WORKLOADS[args.workload]
    x = attn_inputs.make_workload(w)
    flops = attention_flops(x["lengths_q"], x["lengths_k"], w.H, w.D, w.causal)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    cq = x["cu_seqlens_q"].to(dev) if x["cu_seqlens_q"] is not None else None
    ck = x["cu_seqlens_k"].to(dev) if x["cu_seqlens_k"] is not None else None
    out_dtype = torch.float32 if w.dtype == "bf16" else None
    call = attn.FwdCall(q, k, v, causal=w.causal, cu_seqlens_q=cq, cu_seqlens_k=ck,
                        out_dtype=out_dtype, kernel=args.kernel, num_splits=args.num_splits,
                        prune_threshold=args.prune_threshold)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if in_bytes < L2_BYTES else None
    stream = torch.cuda.current_stream()
    sync = dist.barrier if world > 1 else None
    per_launch, launches, clocks = time_forward_launches(call, stream, flush, args.steps, args.warmup,
                                                         local, sync)
    pruned_per_run = call.pruned_count() / (args.warmup + args.steps)
    ms = max_over_ranks(statistics.mean(per_launch), dev)
    unflushed = None
    if flush is not None:
        # the same launches back to back with the inputs left in L2, for reference
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for e0, e1 in evs:
            e0.record(stream)
            call.run(stream)
            e1.record(stream)
        torch.cuda.synchronize()
        unflushed = spread([a.elapsed_time(b) for a, b in evs])

    # end to end: host inputs in, o and lse out, through the same call
    pin = {n: x[n].contiguous().pin_memory() for n in ("q", "k", "v")}
    dev_in = {"q": q, "k": k, "v": v}
    o_h = torch.empty(call.o.shape, dtype=call.o.dtype).pin_memory()
    l_h = torch.empty(call.lse.shape, dtype=torch.float32).pin_memory()

    def e2e():
        for n, t in pin.items():
            dev_in[n].copy_(t, non_blocking=True)
        call.run(stream)
        o_h.copy_(call.o, non_blocking=True)
        l_h.copy_(call.lse, non_blocking=True)

    e2e()
    torch.cuda.synchronize()
    e_steps = max(2, min(args.steps, 10))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(e_steps):
        e2e()
    t1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1) / e_steps, dev)
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = o_h.numel() * o_h.element_size() + l_h.numel() * 4

    peaks = load_peaks()
    family = call.selected_kernel()
    achieved = flops / (ms * 1e-3) / 1e12
    peak, bound, note = fwd_peak(family, w, peaks, dev)
    nbytes = fwd_algorithmic_bytes(x["lengths_q"], x["lengths_k"], w.H, w.D, q.element_size(),
                                   v.element_size(), call.o.element_size())
    metric = f"attention fwd TFLOP/s ({w.note})"
    prune = {}
    if args.prune_threshold:
        # FLOPs stay those of the exact forward: the rate is exact-equivalent
        tiles = 0
        for lq_, lk_ in zip(x["lengths_q"], x["lengths_k"]):
            b = 128 if call.selected_kernel() == "tc" else 64
            tiles += -(-lq_ // b) * -(-lk_ // b) * w.H
        prune = {"prune_threshold": args.prune_threshold,
                 "pruned_fraction": pruned_per_run / tiles,
                 "flops": "of the exact forward (exact-equivalent rate)"}
        metric = f"attention fwd TFLOP/s, tile-pruned rho={args.prune_threshold} ({w.note})"
    traffic = None if (args.prune_threshold or args.num_splits or args.kernel != "auto") else \
        recorded_traffic("fwd:" + w.name, source_hash(fwd_kernel_sources(family, w.dtype)))
    line = {
        "metric": metric, "value": job_rate(flops, world, ms) / 1e12, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_label(w),
        "data": "synthetic",
        "step_ms": spread(per_launch), "step_ms_unflushed": unflushed,
        "config": {"workload": w.name, "kernel": family, "num_splits": call.num_splits(),
                   "tokens_q": int(sum(x["lengths_q"])), "tokens_k": int(sum(x["lengths_k"])),
                   "heads": w.H, "head_dim": w.D, "relation": "causal" if w.causal else "full",
                   "l2": "flushed before every launch (inputs fit in L2)" if flush is not None
                   else "no flush: inputs larger than L2",
                   "parallelism": f"replicas x{world}", **prune},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "traffic": traffic, "kernel": "fwd", "peak_source": note,
                     "bytes_per_launch": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
                     "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
        "e2e": {"value": job_rate(flops, world, e2e_ms) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle_fwd_rows(x, w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def time_oracle_csr_rows(x, w, max_seconds=15.0):
    """Time the oracle's CSR forward on random destination rows of the
    workload (their edges, scores and the source rows they read), adding rows
    until about `max_seconds` of CPU work; report edge-head pairs per second."""
    import numpy as np
    import torch

    import oracle
    rp = x["row_ptr"].numpy()
    col = x["col"].numpy()
    n_dst = len(rp) - 1
    rng = np.random.default_rng(0)
    spent, edges, rows_done, n = 0.0, 0, 0, 256
    while spent < max_seconds * 0.5:
        rows = rng.integers(0, n_dst, n)
        seg = [np.arange(rp[r], rp[r + 1]) for r in rows]
        eidx = np.concatenate(seg)
        srcs, remap = np.unique(col[eidx], return_inverse=True)
        sub_rp = np.concatenate([[0], np.cumsum([len(a) for a in seg])])
        kw = {}
        if x["scores"] is not None:
            kw["scores"] = x["scores"][torch.from_numpy(eidx)]
        else:
            kw["q"] = x["q"][torch.from_numpy(rows)]
            kw["k"] = x["k"][torch.from_numpy(srcs)]
        v = x["v"][torch.from_numpy(srcs)]
        t0 = time.perf_counter()
        oracle.csr_fwd(sub_rp, remap.astype(np.int32), v, **kw)
        spent += time.perf_counter() - t0
        edges += len(eidx) * w.H
        rows_done += n
        n = min(4 * n, 1 << 16)
    return {"value": edges / spent / 1e9, "unit": "Gedge/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{rows_done} random destination rows of the graph (all their edges, "
                      f"all heads), forward: {spent:.1f} s"}


def run_csr_workload(args, rank, world):
    """Attention over a CSR relation: edge-head pairs per second, with the
    gathered bytes against the HBM copy bandwidth."""
    import torch
    import torch.distributed as dist

    import attn_inputs
    import online_softmax_attention_gb300 as attn

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    w = attn_inputs.CSR_WORKLOADS[args.workload]
    x = attn_inputs.make_csr_workload(w)
    rp, col, v = x["row_ptr"].to(dev), x["col"].to(dev), x["v"].to(dev)
    n, E = len(x["row_ptr"]) - 1, x["col"].numel()
    kw = {"scores": x["scores"].to(dev)} if w.field_scores else \
        {"q": x["q"].to(dev), "k": x["k"].to(dev)}
    # rows taken along a Z-order curve through the points (part of the
    # relation's description, computed with the graph), or in index order
    order = x["row_order"].to(dev) if args.row_order == "curve" else None
    call = attn.CsrCall(rp, col, v, row_order=order, **kw)
    es = v.element_size()
    # bytes of one launch as the algorithm touches them: the relation, the
    # scores, one row of V (and of K) per edge and head, Q, O and lse
    gathered = 8 * (n + 1) + 4 * E + E * w.H * w.D * es + n * w.H * w.D * es + 4 * n * w.H
    gathered += 4 * E * w.H if w.field_scores else (E * w.H * w.D * es + n * w.H * w.D * es)
    compulsory = 8 * (n + 1) + 4 * E + v.numel() * es + n * w.H * w.D * es + 4 * n * w.H
    compulsory += 4 * E * w.H if w.field_scores else 2 * v.numel() * es
    in_bytes = sum(t.numel() * t.element_size() for t in [rp, col, v] + list(kw.values()))
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if in_bytes < L2_BYTES else None
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        call.run(stream)
    torch.cuda.synchronize()
    status = attn.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} ({attn.strerror(status)}) set during warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    n0 = attn.launch_count()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.start()
        for e0, e1 in evs:
            if flush is not None:
                flush.zero_()
            e0.record(stream)
            call.run(stream)
            e1.record(stream)
        torch.cuda.synchronize()
        clk.stop()
    if world > 1:
        dist.barrier()
    launches = attn.launch_count() - n0
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evs), dev)

    # end to end: the relation, scores / q, k and v in from pinned host memory, o and lse out
    host = {"row_ptr": x["row_ptr"], "col": x["col"], "v": x["v"]}
    devt = {"row_ptr": rp, "col": col, "v": v}
    if order is not None:
        host["row_order"] = x["row_order"]
        devt["row_order"] = order
    for name, t in kw.items():
        host[name] = x[name]
        devt[name] = t
    pin = {k_: t.contiguous().pin_memory() for k_, t in host.items()}
    o_h = torch.empty(call.o.shape, dtype=call.o.dtype).pin_memory()
    l_h = torch.empty(call.lse.shape, dtype=torch.float32).pin_memory()

    def e2e():
        for k_, t in pin.items():
            devt[k_].copy_(t, non_blocking=True)
        call.run(stream)
        o_h.copy_(call.o, non_blocking=True)
        l_h.copy_(call.lse, non_blocking=True)

    e2e()
    torch.cuda.synchronize()
    e_steps = max(2, min(args.steps, 10))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(e_steps):
        e2e()
    t1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1) / e_steps, dev)
    status = attn.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} ({attn.strerror(status)}) set in the timed region")

    peaks = load_peaks()
    csrc = "online_softmax_attention_gb300/csrc/"
    traffic = recorded_traffic(w.name, source_hash([csrc + "csr.cu", csrc + "common.cuh", csrc + "internal.h"]))
    rate = E * w.H * world / (ms * 1e-3) / 1e9
    achieved = gathered / (ms * 1e-3) / 1e9
    line = {
        "metric": f"attention over a CSR relation, Gedge/s ({w.note})", "value": rate,
        "unit": "Gedge/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_label(w),
        "data": "synthetic",
        "config": {"workload": w.name, "nodes": n, "edges": E, "avg_degree": E / max(1, n),
                   "heads": w.H, "head_dim": w.D,
                   "scores": "field" if w.field_scores else "dot-product",
                   "row_order": "Z-order curve through the points" if order is not None else "index order",
                   "bytes_gathered_per_launch": gathered, "bytes_compulsory_per_launch": compulsory,
                   "l2": "flushed before every launch (inputs fit in L2)" if flush is not None
                   else "no flush: inputs larger than L2",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "kernel": "csr_fwd",
                     "peak_source": f"HBM copy ({peaks['source']})",
                     "bytes": "gathered: one V (and K) row per edge and head",
                     "compulsory_gbs": compulsory / (ms * 1e-3) / 1e9,
                     "frac_compulsory": compulsory / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
        "e2e": {"value": E * w.H * world / (e2e_ms * 1e-3) / 1e9, "unit": "Gedge/s",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in pin.values()),
                "d2h_bytes_per_step": o_h.numel() * o_h.element_size() + l_h.numel() * 4,
                "ms_per_step": e2e_ms},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "cpu_baseline": None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle_csr_rows(x, w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args, rank, world):
    """Reference arm: the f64 CPU oracle on the host cores, bounded samples."""
    if rank != 0:
        return
    import attn_inputs
    w = attn_inputs.WORKLOADS[WORKLOAD]
    x = attn_inputs.make_workload(w)
    vals = []
    for _ in range(args.warmup):
        time_oracle_sample(x, w, max_seconds=4.0)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(time_oracle_sample(x, w, max_seconds=6.0))
    elapsed = time.perf_counter() - t0
    value = statistics.median(v["value"] for v in vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed * 1e3 / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "batch": 4, "seq_len": 8192,
                                            "heads": 32, "head_dim": 128, "relation": "causal"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": vals[0]["cores"],
                             "kind": "oracle", "sample": vals[0]["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=4,
                    help="sequences of N=8192 (4 = the benchmark workload; fewer for profiling)")
    ap.add_argument("--skip-e2e", action="store_true", help="profiling runs: no host-buffer leg")
    ap.add_argument("--no-workloads", action="store_true",
                    help="training workload: skip the forward-only records of the smaller configurations")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=(WORKLOAD,) + FWD_WORKLOADS + CSR_WORKLOADS,
                    help="the training workload (default), a forward-only workload, or a CSR one")
    ap.add_argument("--num-splits", type=int, default=0,
                    help="forward-only workloads: key splits (0 = library's choice)")
    ap.add_argument("--dq-mode", default="auto", choices=["auto", "fused", "separate"],
                    help="training workload: backward dq accumulated in the dK/dV kernel (fused) "
                         "or by its own deterministic kernel (separate); auto = separate")
    ap.add_argument("--row-order", default="curve", choices=["curve", "none"],
                    help="CSR workloads: rows taken along a Z-order curve through the points "
                         "(default) or in index order")
    ap.add_argument("--prune-threshold", type=float, default=0.0,
                    help="forward-only workloads, full relation: tile pruning rho (0 = exact)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.workload in CSR_WORKLOADS:
        run_csr_workload(args, rank, world)
        return
    if args.workload != WORKLOAD:
        run_forward_workload(args, rank, world)
        return

    import torch
    import torch.distributed as dist

    import attn_inputs
    import online_softmax_attention_gb300 as attn

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    w = attn_inputs.WORKLOADS[WORKLOAD]
    if args.batch != w.batch:
        import dataclasses
        w = dataclasses.replace(w, batch=args.batch)
    x = attn_inputs.make_workload(w)
    lq, lk = x["lengths_q"], x["lengths_k"]
    fwd_flops = attention_flops(lq, lk, w.H, w.D, w.causal)
    bwd_flops = 2.5 * fwd_flops
    step_flops = fwd_flops + bwd_flops

    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    cu = x["cu_seqlens_q"].to(dev) if x["cu_seqlens_q"] is not None else None
    fcall = attn.FwdCall(q, k, v, causal=True, cu_seqlens_q=cu, out_dtype=torch.float32,
                         kernel=args.kernel)
    bcall = attn.BwdCall(q, k, v, fcall.o, fcall.lse, dO, causal=True, cu_seqlens_q=cu,
                         kernel=args.kernel, dq_mode=args.dq_mode)
    dq_mode = bcall.selected_dq_mode()
    stream = torch.cuda.current_stream()
    stages = ["fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq"]

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fcall.run(stream)
        if ev is not None:
            ev[1].record(stream)
        bcall.preprocess(stream)
        if ev is not None:
            ev[2].record(stream)
        bcall.dkdv(stream)
        if ev is not None:
            ev[3].record(stream)
        bcall.dq_stage(stream)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = attn.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} ({attn.strerror(status)}) set during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    n0 = attn.launch_count()
    with ClockSampler(local) as clk:
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        clk.start()
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        end.record(stream)
        torch.cuda.synchronize()
        clk.stop()
    barrier()
    launches = attn.launch_count() - n0
    ms = start.elapsed_time(end) / args.steps
    stage_ms = {s: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j, s in enumerate(stages)}
    step_spread = spread([e[0].elapsed_time(e[4]) for e in evs])
    ms = max_over_ranks(ms, dev)
    status = attn.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    # end to end through the public API with host buffers.  The batch's
    # sequences are independent problems: each is copied in on one stream,
    # computed (forward + backward) on one of two compute streams (alternating,
    # so that the last wave of one sequence's kernels overlaps the next
    # sequence's first) and copied out on a fourth, so one sequence's copies
    # overlap its neighbours' computation.  Consecutive steps use two sets of
    # device buffers (slots), so that a step's copies in and its kernels need
    # not wait for the previous step's copies out: the host link, the
    # bottleneck here, then never idles between steps.
    pin = {n: x[n].contiguous().pin_memory() for n in ("q", "k", "v", "dO")}
    n_seq_b, len_b = w.batch, w.n_q
    T_, H_, D_ = q.shape

    def make_slot(dev_in):
        seqs_ = []
        for b_ in range(n_seq_b):
            sl = slice(b_ * len_b, (b_ + 1) * len_b)
            fb = attn.FwdCall(dev_in["q"][sl], dev_in["k"][sl], dev_in["v"][sl], causal=True,
                              out_dtype=torch.float32, kernel=args.kernel)
            bb = attn.BwdCall(dev_in["q"][sl], dev_in["k"][sl], dev_in["v"][sl], fb.o, fb.lse,
                              dev_in["dO"][sl], causal=True, kernel=args.kernel, dq_mode=args.dq_mode)
            seqs_.append((sl, fb, bb))
        evs_ = {k_: [torch.cuda.Event() for _ in seqs_] for k_ in ("in", "done", "out", "used")}
        for e_ in evs_["out"] + evs_["used"]:
            e_.record(stream)
        return {"dev_in": dev_in, "seqs": seqs_, "ev": evs_}

    slots = [make_slot({"q": q, "k": k, "v": v, "dO": dO})]
    if not args.skip_e2e:
        slots.append(make_slot({n: torch.empty_like(t) for n, t in (("q", q), ("k", k), ("v", v), ("dO", dO))}))
    outs_host = {"o": torch.empty((T_, H_, D_), dtype=torch.float32).pin_memory(),
                 "lse": torch.empty((n_seq_b, H_, len_b), dtype=torch.float32).pin_memory(),
                 "dq": torch.empty((T_, H_, D_), dtype=bcall.dq.dtype).pin_memory(),
                 "dk": torch.empty((T_, H_, D_), dtype=bcall.dk.dtype).pin_memory(),
                 "dv": torch.empty((T_, H_, D_), dtype=bcall.dv.dtype).pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in outs_host.values())
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    s_comp = [stream, torch.cuda.Stream(device=dev)]
    e2e_count = [0]

    def e2e_step():
        if args.skip_e2e:
            return
        slot = slots[e2e_count[0] % len(slots)]
        e2e_count[0] += 1
        seqs_, ev, dev_in = slot["seqs"], slot["ev"], slot["dev_in"]
        for i_, (sl, fb, bb) in enumerate(seqs_):
            s_in.wait_event(ev["used"][i_])  # this slot's previous kernels have read it
            with torch.cuda.stream(s_in):
                for n in ("q", "k", "v", "dO"):
                    dev_in[n][sl].copy_(pin[n][sl], non_blocking=True)
            ev["in"][i_].record(s_in)
        for i_, (sl, fb, bb) in enumerate(seqs_):
            cs = s_comp[i_ % 2]
            cs.wait_event(ev["in"][i_])
            cs.wait_event(ev["out"][i_])  # this slot's previous outputs were copied out
            fb.run(cs)
            bb.run(cs)
            ev["done"][i_].record(cs)
            ev["used"][i_].record(cs)
        for i_, (sl, fb, bb) in enumerate(seqs_):
            s_out.wait_event(ev["done"][i_])
            with torch.cuda.stream(s_out):
                outs_host["o"][sl].copy_(fb.o, non_blocking=True)
                outs_host["lse"][i_].copy_(fb.lse, non_blocking=True)
                outs_host["dq"][sl].copy_(bb.dq, non_blocking=True)
                outs_host["dk"][sl].copy_(bb.dk, non_blocking=True)
                outs_host["dv"][sl].copy_(bb.dv, non_blocking=True)
            ev["out"][i_].record(s_out)

    if not args.skip_e2e:
        # the per-sequence calls compute what the batched call did, bit for bit, in both slots
        lse_b = fcall.lse.cpu().view(H_, n_seq_b, len_b).permute(1, 0, 2)
        for _ in slots:
            for t_ in outs_host.values():
                t_.zero_()
            e2e_step()
            torch.cuda.synchronize()
            same = all(torch.equal(outs_host[n_], t_.cpu()) for n_, t_ in
                       (("o", fcall.o), ("dq", bcall.dq), ("dk", bcall.dk), ("dv", bcall.dv)))
            if not (same and torch.equal(outs_host["lse"], lse_b)):
                raise RuntimeError("end-to-end leg: per-sequence results differ from the batched call")
    # The same K steps as the device-timed leg, timed three times; the line
    # reports the median repetition (every repetition is listed beside it).  The
    # host link is shared with the machine's other GPUs, and one repetition can
    # catch a burst of someone else's traffic.
    e_steps = max(2, args.steps)
    e2e_reps = []
    for _ in range(3 if not args.skip_e2e else 1):
        barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(s_in)  # before the first copy in
        for _ in range(e_steps):
            e2e_step()
        t1.record(s_out)  # after the last copy out
        torch.cuda.synchronize()
        barrier()
        e2e_reps.append(max_over_ranks(t0.elapsed_time(t1) / e_steps, dev))
    e2e_ms = statistics.median(e2e_reps)
    status = attn.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} ({attn.strerror(status)}) set in the end-to-end leg")

    peaks = load_peaks()
    # algorithmic FLOPs per launch of each stage: fwd = S and PV contractions;
    # separate dq: dkdv = S (recompute), dP, dV, dK and dq = dQ only (its S / dP
    # recomputes are not algorithmic work); fused dq: dkdv = all five and the dq
    # stage is an HBM-bound conversion of the partial sums, as is the
    # preprocess (reads O f32 and dO bf16).
    if dq_mode == "fused":
        stage_flops = {"fwd": fwd_flops, "bwd_dkdv": 2.5 * fwd_flops}
    else:
        stage_flops = {"fwd": fwd_flops, "bwd_dkdv": 2.0 * fwd_flops, "bwd_dq": 0.5 * fwd_flops}
    dominant = max(stage_flops, key=lambda s: stage_ms[s])
    family = {"fwd": fcall.selected_kernel(), "bwd_dkdv": bcall.selected_kernel(),
              "bwd_dq": bcall.selected_kernel()}
    csrc = "online_softmax_attention_gb300/csrc/"
    shared = [csrc + "common.cuh", csrc + "internal.h"]
    tc_shared = shared + [csrc + "sm100.cuh"]
    kernel_files = {("fwd", "simt"): [csrc + "fwd_simt.cu"] + shared,
                    ("fwd", "tc"): [csrc + "fwd_tc.cu"] + tc_shared,
                    ("bwd_dkdv", "simt"): [csrc + "bwd_simt.cu"] + shared,
                    ("bwd_dq", "simt"): [csrc + "bwd_simt.cu"] + shared,
                    ("bwd_dkdv", "tc"): [csrc + "bwd_tc.cu"] + tc_shared,
                    ("bwd_dq", "tc"): [csrc + "bwd_tc.cu"] + tc_shared}
    using_tc = family[dominant] == "tc"
    achieved = stage_flops[dominant] / (stage_ms[dominant] * 1e-3) / 1e12
    region_s = ms * args.steps * 1e-3
    extra = {}
    if using_tc:
        # the burst peak for a timed region shorter than the seconds-long loop
        # that measured the sustained one; both fractions are printed
        sustained = region_s >= 4.0
        peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        bound, punit = "tensor", "TFLOP/s"
        peak_note = (f"bf16 dense, {'sustained' if sustained else 'burst'} ({peaks['source']}); "
                     f"timed region {region_s:.2f} s")
        extra = {"frac_of_burst": achieved / peaks["bf16_tflops"],
                 "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
    else:
        # FP32 FFMA: 152 SMs x 128 lanes x 2 FLOP x max SM clock
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        peak = sms * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
        bound, punit = "alu", "TFLOP/s"
        peak_note = f"FP32 FFMA: {sms} SMs x 128 lanes x 2 FLOP x {peaks['sm_max_mhz']:.0f} MHz"
    src = [p for p in kernel_files[(dominant, family[dominant])] if os.path.exists(os.path.join(ROOT, p))]
    tkey = dominant + ("_fused" if dominant == "bwd_dkdv" and dq_mode == "fused" else "")
    traffic = recorded_traffic(tkey, source_hash(src)) if src else None
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": punit,
                "frac": achieved / peak, "traffic": traffic, "kernel": dominant,
                "peak_source": peak_note, "flops_per_launch": stage_flops[dominant],
                "ms_per_launch": stage_ms[dominant],
                "algorithmic": "dK/dV: S recompute, dP, dV, dK = 2 x forward FLOPs" if dominant == "bwd_dkdv"
                else "see breakdown", **extra}

    fwd_tflops = fwd_flops / (stage_ms["fwd"] * 1e-3) / 1e12
    bwd_ms = stage_ms["bwd_preprocess"] + stage_ms["bwd_dkdv"] + stage_ms["bwd_dq"]
    bwd_tflops = bwd_flops / (bwd_ms * 1e-3) / 1e12
    value = job_rate(step_flops, world, ms) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD if w.batch == 4 else f"{WORKLOAD} (batch {w.batch})", "batch": w.batch, "seq_len": 8192, "heads": 32, "head_dim": 128,
                   "relation": "causal", "o_dtype": "f32", "grad_dtype": "bf16",
                   "kernels": family, "dq_mode": dq_mode,
                   "l2": "no flush: each input tensor is 268 MB, larger than the 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "step_ms": step_spread,
        "breakdown": {"fwd_ms": stage_ms["fwd"], "bwd_ms": bwd_ms,
                      "stage_ms": stage_ms, "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
                      "fwd_frac_of_bf16_peak": fwd_tflops / peaks["bf16_tflops"],
                      "bf16_peak_tflops": peaks["bf16_tflops"]},
        "roofline": roofline,
        "e2e": {"value": job_rate(step_flops, world, e2e_ms) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "ms_per_step_repetitions": e2e_reps, "steps_per_repetition": e_steps,
                "how": "per sequence: pinned host -> device copies, forward + backward, device -> "
                       "pinned host copies of o, lse, dq, dk, dv; copies on their own streams, "
                       "sequences alternating between two compute streams, so that copies and "
                       "kernel tails overlap the other sequences' computation; consecutive steps "
                       "alternate between two sets of device buffers"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if args.skip_e2e:
        line["e2e"] = None
    else:
        # what the host link allows: the step's bytes at the copy bandwidth
        # measured now (both directions at once), against the device step
        bw = copy_bandwidth(dev)
        line["e2e"]["copy_gbs"] = bw
        line["e2e"]["copy_floor_ms"] = (h2d + d2h) / (bw["both_gbs"] * 1e9) * 1e3
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle_sample(x, w)
    else:
        line["cpu_baseline"] = None
    if not args.no_workloads:
        # free the training workload's buffers first
        del fcall, bcall, slots, q, k, v, dO, outs_host, pin
        torch.cuda.empty_cache()
        oracle_s = 6.0 if (rank == 0 and world == 1 and not args.no_cpu_baseline) else 0.0
        line["workloads"] = {name: forward_record(name, dev, local, 20, 5, oracle_s)
                             for name in SUB_WORKLOADS}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
