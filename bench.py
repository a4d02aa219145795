#!/usr/bin/env python3
"""Throughput benchmark of the chunkwise gated delta rule forward pass.

One step = one full forward pass (gdr_chunk_fwd: the chunk-local stage and the
state recurrence) over the headline workload: B=1, T=4096, H=HV=12 heads,
K=V=128, C=64, bf16 q/k/v, fp32 gate and beta, q/k L2-normalised in the kernel,
output in the input dtype (bf16, as the optimisation script returns it) and an
fp32 final state. The same forward with fp32 output is timed beside it. Inputs
are seeded synthetic tensors already resident in HBM; the L2 cache is flushed
(a 512 MiB write) before every timed step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--out-dtype bf16|fp32]

With N > 1 (launched by torch.distributed.run) every rank runs the same
workload on its own GPU as a shard of 12 value heads of a 12N-head layer
(independent sequences, no collective on the data path): weak scaling. Rank 0
prints one JSON line. ``--impl reference`` times the float64 CPU oracle on the
host cores instead (rank 0 only). The default headline run at N = 1 also times
the other workloads' forwards the same way (device-resident inputs, L2 flushed,
CUDA events) and adds them to its line as ``other_workloads``
(``--skip-other-workloads`` leaves them out).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s for chunked gated-delta fwd (T=4096,H=12,K=V=128,C=64); % of roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# Algorithmic FLOPs per token per value head at C=64, K=V=128: decayed dots
# A_kk, A_qk (4CK), M^-1 applied to [exp(G)k | v] (2C(K+V)), W S, q S and
# k^T r (6KV), A_qk r (2CV) and the C x C inverse (~C^2/3).
FLOP_PER_TOKEN_HEAD = 181589


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--skip-other-workloads", action="store_true",
                    help="headline run only: leave out the timings of the other workloads")
    ap.add_argument("--out-dtype", choices=["bf16", "fp32"], default="bf16",
                    help="dtype of o in the timed forward (the other is timed beside it)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def workload(name):
    from chunkwise_gated_delta_gdr_gb300 import inputs as gin
    if name in gin.DECODE_WORKLOADS:
        return gin.DECODE_WORKLOADS[name]
    if name in gin.SSD_WORKLOADS:
        return gin.SSD_WORKLOADS[name]
    if name in gin.SEGMENTED_WORKLOADS:
        return gin.SEGMENTED_WORKLOADS[name]
    if name in gin.GENERAL_WORKLOADS:
        return gin.GENERAL_WORKLOADS[name]
    return gin.WORKLOADS[name or gin.HEADLINE]


def config_of(w, world, out_dtype="bf16"):
    return {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "HV": w.HV, "K": w.K, "V": w.V,
            "C": w.C, "gate": "scalar" if w.gate_mode == 0 else "per-key",
            "in_dtype": "bf16" if str(w.dtype).endswith("bfloat16") else "fp32",
            "out_dtype": out_dtype, "use_qk_l2norm": w.use_qk_l2norm,
            "initial_state": w.s0_std is not None, "l2_flush": "512MiB write before each step",
            "parallelism": f"{world} rank(s), value heads sharded, no collective",
            **({"segments": w.segments} if getattr(w, "segments", 1) > 1 else {})}


def algorithmic_bytes(w, out_bytes=4):
    """Compulsory HBM bytes of one forward: q, k (H heads), v, g, beta, o in its
    dtype, the fp32 final state and the fp32 initial state when there is one."""
    BT = w.B * w.T
    qk = 2 * BT * w.H * w.K * 2
    v = BT * w.HV * w.V * 2
    g = BT * w.HV * (w.K if w.gate_mode else 1) * 4
    beta = BT * w.HV * 4
    o = BT * w.HV * w.V * out_bytes
    state = w.B * w.HV * w.K * w.V * 4
    return qk + v + g + beta + o + state + (state if w.s0_std is not None else 0)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def source_hash(files=None):
    """Hash of the kernel sources (the named files under csrc/, else all of them)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunkwise_gated_delta_gdr_gb300", "csrc")
    paths = ([os.path.join(csrc, f) for f in sorted(files)] if files
             else sorted(glob.glob(os.path.join(csrc, "*"))))
    for f in paths:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(wname):
    """DRAM bytes per step from the committed ncu summary, if it was taken on
    the kernels as they are now (same hash of the source files the summary
    names, the files those kernels are built from); else None."""
    path = os.path.join(ROOT, "profiles", f"traffic_{wname}.md")
    try:
        text = open(path).read()
    except OSError:
        return None, None
    mh = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    ms = re.search(r"^sources:\s*(.+)$", text, re.M)
    files = ms.group(1).split() if ms else None
    try:
        current = source_hash(files)
    except OSError:
        return None, None
    if not mh or mh.group(1) != current:
        return None, None
    per = {}
    for m in re.finditer(r"^kernel\s+(\S+)\s+dram_bytes_per_launch:\s*([0-9.]+)", text, re.M):
        per[m.group(1)] = float(m.group(2))
    return (sum(per.values()) if per else None), per


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        try:
            import torch
            bus = getattr(torch.cuda.get_device_properties(device_index), "pci_bus_id", None)
        except Exception:
            bus = None
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "20"]
        if bus:
            cmd.insert(1, f"--id={bus}")
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def cpu_baseline(w, x, ssd=False):
    """The float64 oracle (as it stands) on the host cores, on the full workload."""
    import oracle
    ncpu = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    nseq = w.B * w.HV
    threads = max(1, min(ncpu, nseq))
    times = []
    for _ in range(2):
        t0 = time.perf_counter()
        if ssd:
            oracle.ssd_recurrent(x["q"], x["k"], x["v"], x["g"], x["s0"], scale=w.scale,
                                 use_qk_l2norm=w.use_qk_l2norm, nthreads=threads)
        else:
            oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"], scale=w.scale,
                             use_qk_l2norm=w.use_qk_l2norm, nthreads=threads)
        times.append(time.perf_counter() - t0)
        if times[-1] > 10:
            break
    t = min(times)
    return {"value": w.B * w.T / t, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"full workload ({w.B}x{w.T} tokens x {w.HV} heads), float64 token "
                      f"recurrence, OpenMP over {nseq} sequences, best of {len(times)}",
            "seconds": t}


def warm_l2_ms(step, stream, n):
    """Mean CUDA-event time of `n` back-to-back steps without the L2 flush
    (inputs and the workspace stay in L2 where they fit), outside the timed region."""
    import torch

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    step()
    for a, b in evs:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def run_reference(args, rank, world):
    """The float64 oracle, as it stands, timed on the host cores: OpenMP over
    all B x HV sequences of the workload, as many threads as cpu_baseline uses.
    A step is the whole workload when warm-up + timed steps fit about 90 s,
    else the first `ts` tokens of every sequence (all heads), sized to that
    budget; ms_per_step is the measured wall time of the step that ran, and
    the tokens/s are the tokens it processed over that time (the recurrence
    costs the same per token, so the rate is the full workload's)."""
    if rank != 0:
        return 0
    import oracle
    from chunkwise_gated_delta_gdr_gb300 import inputs as gin
    w = workload(args.workload)
    x = gin.make_inputs(w)
    ncpu = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    nseq = w.B * w.HV
    threads = max(1, min(ncpu, nseq))
    cut = lambda ts: {n: (t[:, :ts].contiguous() if (t is not None and n != "s0") else t)
                      for n, t in x.items()}

    def step(xs):
        oracle.recurrent(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"], xs["s0"],
                         scale=w.scale, use_qk_l2norm=w.use_qk_l2norm, nthreads=threads)

    # Calibrate on a short prefix of every sequence, then size the step.
    cal_ts = min(w.T, 256)
    t0 = time.perf_counter()
    step(cut(cal_ts))
    per_token = (time.perf_counter() - t0) / cal_ts
    budget = 90.0 / max(1, args.warmup + args.steps)
    ts = int(max(32, min(w.T, budget / per_token)))
    xs = x if ts == w.T else cut(ts)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        step(xs)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    per_step = statistics.mean(times)
    value = w.B * ts / per_step
    sample = ("whole workload" if ts == w.T else f"first {ts} of {w.T} tokens") + \
        (f" of all {nseq} (batch, head) sequences per step ({w.B}x{ts} tokens x {w.HV} heads), "
         f"float64 token recurrence, OpenMP over the sequences, {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, 1, "f64"),
            "full_workload_ms": per_step * 1e3 * (w.T / ts),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def timed(fn, stream, n, flush):
    """CUDA-event times (ms) of n calls of fn, each after an L2 flush that lies
    outside its events."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


OTHER_WORKLOADS = ("kda_gqa_t8192", "gdn_long_t65000", "kda_many_b64", "ssd_t4096_h12",
                   "gdn_h2_t65536", "decode_b64_h16", "gdn_c128_t4096_h12", "gdn_k64_t4096_h12")


def other_workloads(dev, stream, flush, hbm, steps=10, warmup=3):
    """The other workloads' forwards, timed as the headline is (device-resident
    inputs, L2 flushed before each call, CUDA events on the launching stream),
    so that their figures sit in the headline's JSON line: per workload the mean
    time per call, tokens/s and the fraction of the measured HBM copy rate for
    its compulsory bytes. A workload that fails reports its error instead."""
    import torch
    import chunkwise_gated_delta_gdr_gb300 as gdr
    from chunkwise_gated_delta_gdr_gb300 import inputs as gin
    res = {}
    for name in OTHER_WORKLOADS:
        try:
            w = workload(name)
            x = {n: (t.to(dev) if t is not None else None) for n, t in gin.make_inputs(w).items()}
            if name in gin.DECODE_WORKLOADS or name in gin.SSD_WORKLOADS:
                ssd = name in gin.SSD_WORKLOADS
                out = torch.empty(w.B, w.T, w.HV, w.V, dtype=torch.float32, device=dev)
                state = None if ssd else x["s0"].clone()

                def step():
                    if ssd:
                        gdr.ssd_chunk_fwd(x["q"], x["k"], x["v"], x["g"], None, chunk_size=w.C,
                                          scale=w.scale, use_qk_l2norm=w.use_qk_l2norm,
                                          out_dtype=torch.float32, output_final_state=False,
                                          stream=stream)
                    else:
                        gdr.recurrent_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], state,
                                          scale=w.scale, use_qk_l2norm=w.use_qk_l2norm,
                                          out=out, stream=stream)
                sbytes = 0 if ssd else 2 * w.B * w.HV * w.K * w.V * 4
                nbytes = sbytes + (2 * w.B * w.T * w.H * w.K * 2 + w.B * w.T * w.HV * w.V * 2 +
                                   2 * w.B * w.T * w.HV * 4 + w.B * w.T * w.HV * w.V * 4)
                odt = "fp32"
            else:
                segments = getattr(w, "segments", 1)
                dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16, gdr.GDR_BF16)
                nws = (gdr.chunk_fwd_segmented_workspace_size(dims, w.C, w.gate_mode, segments)
                       if segments > 1 else gdr.chunk_fwd_workspace_size(dims, w.C, w.gate_mode))
                ws = torch.empty(nws, dtype=torch.uint8, device=dev)
                out = torch.empty(w.B, w.T, w.HV, w.V, dtype=torch.bfloat16, device=dev)
                fin = torch.empty(w.B, w.HV, w.K, w.V, dtype=torch.float32, device=dev)

                def step():
                    if segments > 1:
                        gdr.chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"],
                                                segments=segments, chunk_size=w.C, scale=w.scale,
                                                use_qk_l2norm=w.use_qk_l2norm,
                                                out_dtype=torch.bfloat16, workspace=ws, out=out,
                                                final_state=fin, stream=stream)
                    else:
                        gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"],
                                      chunk_size=w.C, scale=w.scale, use_qk_l2norm=w.use_qk_l2norm,
                                      out_dtype=torch.bfloat16, workspace=ws, out=out,
                                      final_state=fin, stream=stream)
                nbytes = algorithmic_bytes(w, 2)
                odt = "bf16"
            for _ in range(warmup):
                flush.zero_()
                step()
            torch.cuda.synchronize()
            ms = statistics.mean(timed(step, stream, steps, flush))
            assert torch.isfinite(out.float()).all()
            res[name] = {"ms_per_step": ms, "tokens_per_s": w.B * w.T / (ms * 1e-3),
                         "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm,
                         "algorithmic_bytes_per_step": nbytes, "out_dtype": odt, "steps": steps}
            del x, out
        except Exception as e:   # reported, so that the headline line still prints
            res[name] = {"error": f"{type(e).__name__}: {e}"[:200]}
        torch.cuda.empty_cache()
    return res


def run_ours(args, rank, local_rank, world):
    import torch
    import chunkwise_gated_delta_gdr_gb300 as gdr
    from chunkwise_gated_delta_gdr_gb300 import inputs as gin
    from chunkwise_gated_delta_gdr_gb300 import shard

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    w = workload(args.workload)
    wr = gin.shrink(w, seed=w.seed + 1000 * rank)        # this rank's head shard
    x_cpu = gin.make_inputs(wr)
    x = {n: (t.to(dev) if t is not None else None) for n, t in x_cpu.items()}
    gate = w.gate_mode
    DT = {"bf16": torch.bfloat16, "fp32": torch.float32}
    CODE = {"bf16": gdr.GDR_BF16, "fp32": gdr.GDR_F32}
    main_dt = args.out_dtype
    other_dt = "fp32" if main_dt == "bf16" else "bf16"
    dims = {k_: gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16, CODE[k_])
            for k_ in DT}
    path = gdr.chunk_fwd_path(dims[main_dt], w.C, gate)
    # (one workspace serves both output dtypes: sized for the larger)
    ws = torch.empty(max(gdr.chunk_fwd_workspace_size(dims[k_], w.C, gate) for k_ in DT),
                     dtype=torch.uint8, device=dev)
    outs = {k_: torch.empty(w.B, w.T, w.HV, w.V, dtype=DT[k_], device=dev) for k_ in DT}
    fin = torch.empty(w.B, w.HV, w.K, w.V, dtype=torch.float32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    segments = getattr(w, "segments", 1)
    if segments > 1:
        seg_ws = torch.empty(max(gdr.chunk_fwd_segmented_workspace_size(dims[k_], w.C, gate,
                                                                        segments) for k_ in DT),
                             dtype=torch.uint8, device=dev)

    def step(dt=main_dt):
        # The call a user makes: gdr_chunk_fwd (or, for a segmented workload,
        # gdr_chunk_fwd_segmented).
        if segments > 1:
            gdr.chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"],
                                    segments=segments, chunk_size=w.C, scale=w.scale,
                                    use_qk_l2norm=w.use_qk_l2norm, out_dtype=DT[dt],
                                    workspace=seg_ws, out=outs[dt], final_state=fin,
                                    stream=stream)
            return
        gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"], chunk_size=w.C,
                      scale=w.scale, use_qk_l2norm=w.use_qk_l2norm, out_dtype=DT[dt],
                      workspace=ws, out=outs[dt], final_state=fin, stream=stream)

    def split_step(mid):
        # The two-launch form of the same forward (gdr_chunk_prepare +
        # gdr_chunk_recur), to time the chunk-local and recurrence kernels apart.
        gdr.chunk_prepare(x["q"], x["k"], x["v"], x["g"], x["beta"], workspace=ws,
                          chunk_size=w.C, scale=w.scale, use_qk_l2norm=w.use_qk_l2norm,
                          out_dtype=DT[main_dt], stream=stream)
        mid.record(stream)
        gdr.chunk_recur(x["q"], x["k"], x["s0"], workspace=ws, out=outs[main_dt],
                        final_state=fin, HV=w.HV, V=w.V, gate_mode=gate, chunk_size=w.C,
                        scale=w.scale, use_qk_l2norm=w.use_qk_l2norm, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
        step(other_dt)
    torch.cuda.synchronize()
    assert torch.isfinite(outs[main_dt].float()).all() and torch.isfinite(fin).all()
    assert gdr.stream_status(stream, seg_ws if segments > 1 else ws) == gdr.GDR_OK

    sampler = ClockSampler(local_rank)
    time.sleep(0.2)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    tot = timed(step, stream, args.steps, flush)
    if pg:
        pg.barrier()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    ms = shard.step_time_across_ranks(statistics.mean(tot), pg)

    # Outside the timed region: the same forward with the other output dtype,
    # the two-launch form split per kernel, and the warm-L2 figure.
    n_side = max(4, min(args.steps, 200))
    other = timed(lambda: step(other_dt), stream, n_side, flush)
    ms_other = shard.step_time_across_ranks(statistics.mean(other), pg)
    sevs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(n_side)]
    for a, m, b in sevs:
        flush.zero_()
        a.record(stream)
        split_step(m)
        b.record(stream)
    torch.cuda.synchronize()
    prep = [a.elapsed_time(m) for a, m, b in sevs]
    rec = [m.elapsed_time(b) for a, m, b in sevs]
    warm_ms = warm_l2_ms(step, stream, n_side)

    # End to end through the C ABI with host buffers: pinned inputs copied in,
    # o and the final state copied out, every step. Consecutive steps are
    # independent forward passes; they alternate between two streams (each
    # with its own device buffer and host outputs), so one step's copies
    # overlap another step's kernels, as a caller streaming batches would run.
    pin = {n: (t.pin_memory() if t is not None else None) for n, t in x_cpu.items()}
    E2E_STREAMS = 2
    out_h = [torch.empty(w.B, w.T, w.HV, w.V, dtype=DT[main_dt]).pin_memory()
             for _ in range(E2E_STREAMS)]
    fin_h = [torch.empty(w.B, w.HV, w.K, w.V, dtype=torch.float32).pin_memory()
             for _ in range(E2E_STREAMS)]
    streams = [torch.cuda.Stream(device=dev) for _ in range(E2E_STREAMS)]
    h2d = sum(t.numel() * t.element_size() for n, t in pin.items() if t is not None)
    d2h = out_h[0].numel() * out_h[0].element_size() + fin_h[0].numel() * 4
    e2e_steps = max(4, min(args.steps, 50))
    if segments > 1:
        # No host-buffer form of the segmented call: the inputs are copied into
        # per-stream device tensors, gdr_chunk_fwd_segmented runs, and o and the
        # final state are copied back, all on that stream.
        dbuf = [{n: torch.empty_like(t, device=dev) for n, t in pin.items() if t is not None}
                for _ in range(E2E_STREAMS)]
        dout = [torch.empty_like(outs[main_dt]) for _ in range(E2E_STREAMS)]
        dfin = [torch.empty_like(fin) for _ in range(E2E_STREAMS)]
        dws = [torch.empty_like(seg_ws) for _ in range(E2E_STREAMS)]
        method = f"H2D copies + gdr_chunk_fwd_segmented + D2H copies per step, {E2E_STREAMS} streams alternating"
    else:
        hbytes = gdr.chunk_fwd_host_buffer_size(dims[main_dt], w.C, gate, pin["s0"] is not None,
                                                True)
        hbuf = [torch.empty(hbytes, dtype=torch.uint8, device=dev) for _ in range(E2E_STREAMS)]
        method = f"gdr_chunk_fwd_host per step, {E2E_STREAMS} streams alternating"

    def e2e_step(i):
        j = i % E2E_STREAMS
        if segments > 1:
            d = dbuf[j]
            with torch.cuda.stream(streams[j]):
                for n, t in d.items():
                    t.copy_(pin[n], non_blocking=True)
                gdr.chunk_fwd_segmented(d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("s0"),
                                        segments=segments, chunk_size=w.C, scale=w.scale,
                                        use_qk_l2norm=w.use_qk_l2norm, out_dtype=DT[main_dt],
                                        workspace=dws[j], out=dout[j], final_state=dfin[j],
                                        stream=streams[j])
                out_h[j].copy_(dout[j], non_blocking=True)
                fin_h[j].copy_(dfin[j], non_blocking=True)
            return
        gdr.chunk_fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"], pin["s0"],
                           out=out_h[j], final_state=fin_h[j], device_buffer=hbuf[j],
                           chunk_size=w.C, scale=w.scale, use_qk_l2norm=w.use_qk_l2norm,
                           stream=streams[j])

    for i in range(2 * E2E_STREAMS):
        e2e_step(i)
    torch.cuda.synchronize()
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_a.record(stream)
    for s_ in streams:
        s_.wait_event(e_a)
    for i in range(e2e_steps):
        e2e_step(i)
    for s_ in streams:
        stream.wait_stream(s_)
    e_b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = shard.step_time_across_ranks(e_a.elapsed_time(e_b) / e2e_steps, pg)
    assert gdr.stream_status(stream, ws) == gdr.GDR_OK
    assert all(gdr.stream_status(s_, None) == gdr.GDR_OK for s_ in streams)

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0
    hbm, tflops, peak_kind = load_peaks()
    obytes = {"bf16": 2, "fp32": 4}
    bytes_alg = algorithmic_bytes(w, obytes[main_dt])
    bytes_other = algorithmic_bytes(w, obytes[other_dt])
    flops_alg = FLOP_PER_TOKEN_HEAD * w.B * w.T * w.HV
    achieved = bytes_alg / (ms * 1e-3) / 1e9
    traffic, traffic_per = recorded_traffic(w.name)
    # Kernels: the one-launch forward (fused_kernel: chunk producers, chains
    # and output items), or the chunk-local kernel and the recurrence
    # (chunk_tc_kernel, chain_kernel + output_kernel for the scalar gate;
    # chunk_kda_kernel, state_kda_tc_kernel for the per-key gate).
    if path == 0:
        ck, rk = "general_prep_kernel", "general_state_kernel"
    else:
        ck, rk = (("chunk_kda_kernel", "state_kda_tc_kernel") if gate
                  else ("chunk_tc_kernel", "chains+outputs (fused_kernel without the chunk stage, "
                                           "or chain_kernel+output_kernel)"))
    one_launch = path == 2 and segments == 1
    if one_launch:
        kernel_scope = ("fused_kernel (one cooperative launch: chunk producers, chains and "
                        "output items) after a memset of the chunk flags")
        launches = 1
        step_traffic = traffic
    elif segments > 1:
        kernel_scope = ("one gdr_chunk_fwd_segmented call: chunk-local kernel, 3 recurrence "
                        "launches (the last with the output items), identity and combine kernels")
        launches = 6
        step_traffic = None
    else:
        kernel_scope = f"one forward call: {ck} + {rk}"
        # Scalar gate on tensor cores: the chunk kernel, then the chains with the
        # output items in one launch when they fit on the SMs at once, else the
        # chain and output kernels.
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        launches = 2 if (gate or path == 0 or w.B * w.HV * 4 <= sms) else 3
        step_traffic = traffic
    tokens = world * w.B * w.T
    line = {
        "metric": METRIC, "value": tokens / (ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(w, world, main_dt),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": step_traffic, "scope": kernel_scope,
                     "algorithmic_bytes_per_step": bytes_alg, "peak_source": f"{peak_kind} hbm_gbs",
                     "tensor_tflops": flops_alg / (ms * 1e-3) / 1e12,
                     "tensor_frac_of_bf16_peak": flops_alg / (ms * 1e-3) / 1e12 / tflops},
        f"{other_dt}_output": {"ms_per_step": ms_other, "value": tokens / (ms_other * 1e-3),
                               "algorithmic_bytes_per_step": bytes_other,
                               "roofline_frac": bytes_other / (ms_other * 1e-3) / 1e9 / hbm,
                               "steps": n_side},
        "two_launch_form": {"chunk_local": {"kernel": ck, "ms": statistics.mean(prep),
                                            "traffic": (traffic_per or {}).get(ck)},
                            "recurrence": {"kernel": rk, "ms": statistics.mean(rec),
                                           "traffic": (traffic_per or {}).get(rk)},
                            **({"split_of": "the unsegmented forward (gdr_chunk_prepare + "
                                            "gdr_chunk_recur) on the same inputs"}
                               if segments > 1 else {})},
        "path": path,
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "method": method},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "wall_s_timed_loop": t_wall,
        "median_ms": statistics.median(tot),
        "warm_l2_ms": warm_ms,
    }
    line["cpu_baseline"] = cpu_baseline(w, x_cpu)
    if world == 1 and w.name == gin.HEADLINE and not args.skip_other_workloads:
        line["other_workloads"] = other_workloads(dev, stream, flush, hbm)
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def run_decode(args, rank, local_rank, world, kind="decode"):
    """The recurrent (decode) form on a decode workload: every step applies one
    token per sequence to states resident in HBM (read and written in place).
    kind "ssd": the chunkwise Mamba2 SSD forward on an SSD workload instead."""
    import torch
    import chunkwise_gated_delta_gdr_gb300 as gdr
    from chunkwise_gated_delta_gdr_gb300 import inputs as gin
    from chunkwise_gated_delta_gdr_gb300 import shard

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    w = workload(args.workload)
    wr = gin.shrink(w, seed=w.seed + 1000 * rank)
    x_cpu = gin.make_inputs(wr)
    x = {n: (t.to(dev) if t is not None else None) for n, t in x_cpu.items()}
    state = x["s0"].clone() if x["s0"] is not None else None
    out = torch.empty(w.B, w.T, w.HV, w.V, dtype=torch.float32, device=dev)
    last = {}
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call(q, k, v, g, beta):
        if kind == "ssd":
            last["o"], _ = gdr.ssd_chunk_fwd(q, k, v, g, None, chunk_size=w.C, scale=w.scale,
                                             use_qk_l2norm=w.use_qk_l2norm,
                                             out_dtype=torch.float32, output_final_state=False,
                                             stream=stream)
        else:
            gdr.recurrent_fwd(q, k, v, g, beta, state, scale=w.scale,
                              use_qk_l2norm=w.use_qk_l2norm, out=out, stream=stream)

    def step():
        call(x["q"], x["k"], x["v"], x["g"], x["beta"])

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    time.sleep(0.2)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    tot = [a.elapsed_time(b) for a, b in evs]
    ms = shard.step_time_across_ranks(statistics.mean(tot), pg)
    warm_ms = warm_l2_ms(step, stream, max(4, min(args.steps, 200)))
    if kind == "ssd":
        assert torch.isfinite(last["o"]).all()
    else:
        assert torch.isfinite(out).all() and torch.isfinite(state).all()

    # End to end: the token inputs come from pinned host memory and o goes back
    # every step; the states stay resident on the device (as in decoding).
    names = ("q", "k", "v", "g", "beta")
    pin = {n: x_cpu[n].pin_memory() for n in names}
    dbuf = {n: torch.empty_like(x[n]) for n in names}
    out_h = torch.empty(w.B, w.T, w.HV, w.V, dtype=torch.float32).pin_memory()
    h2d = sum(pin[n].numel() * pin[n].element_size() for n in names)
    d2h = out_h.numel() * 4
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(3, min(args.steps, 200))
    e_a.record(stream)
    for _ in range(n_e2e):
        for n in names:
            dbuf[n].copy_(pin[n], non_blocking=True)
        call(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["g"], dbuf["beta"])
        out_h.copy_(last["o"] if kind == "ssd" else out, non_blocking=True)
    e_b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = shard.step_time_across_ranks(e_a.elapsed_time(e_b) / n_e2e, pg)
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0
    hbm, _, peak_kind = load_peaks()
    if kind == "ssd":
        # The SSD forward runs the launches of gdr_chunk_fwd: one cooperative
        # launch when the chains fit beside the producers, else the chunk kernel
        # and the chains with the output items (or chain and output kernels).
        dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16, gdr.GDR_F32)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        if gdr.chunk_fwd_path(dims, w.C, 0) == 2:
            launches, scope = 1, "one gdr_ssd_chunk_fwd call: fused_kernel (one cooperative launch)"
        else:
            launches = 2 if w.B * w.HV * 4 <= sms else 3
            scope = "one gdr_ssd_chunk_fwd call: chunk_tc_kernel + chains and outputs"
    else:
        launches, scope = 1, "one gdr_recurrent_fwd call (one decode kernel)"
    sbytes = 0 if kind == "ssd" else 2 * w.B * w.HV * w.K * w.V * 4   # state read + write
    io = (2 * w.B * w.T * w.H * w.K * 2 + w.B * w.T * w.HV * w.V * 2 + 2 * w.B * w.T * w.HV * 4 +
          w.B * w.T * w.HV * w.V * 4)
    bytes_alg = sbytes + io
    achieved = bytes_alg / (ms * 1e-3) / 1e9
    tokens = world * w.B * w.T
    line = {
        "metric": (f"tokens/s of the chunkwise SSD forward ({w.name}); % of HBM roofline"
                   if kind == "ssd" else
                   f"tokens/s of the recurrent decode step ({w.name}); % of HBM roofline"),
        "value": tokens / (ms * 1e-3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "HV": w.HV, "K": w.K,
                   "V": w.V, "gate": "scalar", "in_dtype": "bf16", "out_dtype": "fp32",
                   "state": "none" if kind == "ssd" else "fp32 in place",
                   "l2_flush": "512MiB write before each step",
                   "parallelism": f"{world} rank(s), value heads sharded, no collective"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": None,
                     "scope": scope,
                     "algorithmic_bytes_per_step": bytes_alg, "peak_source": f"{peak_kind} hbm_gbs"},
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "median_ms": statistics.median(tot),
        "warm_l2_ms": warm_ms,
    }
    line["cpu_baseline"] = cpu_baseline(w, x_cpu, ssd=kind == "ssd")
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    from chunkwise_gated_delta_gdr_gb300 import inputs as gin
    if args.workload in gin.DECODE_WORKLOADS:
        return run_decode(args, rank, local_rank, world)
    if args.workload in gin.SSD_WORKLOADS:
        return run_decode(args, rank, local_rank, world, kind="ssd")
    return run_ours(args, rank, local_rank, world)


if __name__ == "__main__":
    sys.exit(main())
