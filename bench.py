#!/usr/bin/env python3
"""Benchmark of the selective-scan hot path on B300.

One step = one ssm_scan_fwd over the Mamba-1.4B layer workload with its fused front end
(batch 8, d_inner 4096, d_state 16, L 2048, bf16 in/out, fp32 state): causal conv1d + SiLU,
softplus step, zero-order-hold discretisation, scan, C readout, D skip and SiLU gate, all in one
kernel launch.  Inputs are seeded synthetic tensors resident in HBM before the timed region.

Prints ONE JSON line (rank 0).  Keys beyond the base contract:
  roofline      dominant kernel vs the binding one of three roofs, each algorithmic work per launch /
                CUDA-event launch time: FP32 lane ops (148 SMs x 128 lanes x max SM clock), MUFU
                transcendentals (148 SMs x measured ex2 rate/clk x max SM clock), HBM bytes (measured
                copy bandwidth); all three are listed under "terms"
  hbm           the same launch against the measured HBM copy bandwidth
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the workload, host cores
  e2e           the same metric through the public API with pinned host buffers, copies included
  decode        the constant-state decode workload (ssm_state_update, 64 layers x 128 tokens)

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl b300|reference]
Under torchrun (N > 1) every rank runs its own batch (weak scaling, no data-path collective); the
reported value is the elements of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

WORKLOAD = "mamba1.4b_conv"
METRIC = "scan elems/s (B*D*L*N)"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
MAX_SM_MHZ = 2032.0
FP32_LANES_PER_SM = 128   # FP32 FMA lanes per SM (4 sub-partitions x 32)
E2E_TWO_UPLOAD_STREAMS = os.environ.get("SSM_BENCH_E2E_UPLOAD_STREAMS", "2") != "1"


# ---------------------------------------------------------------------------------------------
# accounting (per unit = one (b, d, t) of the scan)
# ---------------------------------------------------------------------------------------------
def scan_bytes(cfg) -> int:
    """Algorithmic HBM bytes of one scan launch: u/x, delta, z read and y written once per (b, d, t),
    B and C once per (b, n, t), per-channel parameters once, final state written once."""
    e = 2 if cfg.dtype == "bf16" else 4
    bdl = cfg.batch * cfg.dim * cfg.seqlen
    per_bdl = e * (2 + (1 if cfg.has_z else 0) + 1)
    bc = 2 * cfg.batch * cfg.dstate * cfg.seqlen * e
    params = 4 * cfg.dim * (cfg.dstate + 2 + (5 if cfg.conv else 0))
    state = 4 * cfg.batch * cfg.dim * cfg.dstate
    return bdl * per_bdl + bc + params + state


def scan_mufu_ops(cfg) -> int:
    """Transcendental operations the scan requires per (b, d, t): N exponentials for Abar, softplus
    (exp + log), the gate's sigmoid (exp + reciprocal) and, with the fused conv, its SiLU sigmoid
    (exp + reciprocal)."""
    per = cfg.dstate + 2 + (2 if cfg.has_z else 0) + (2 if cfg.conv else 0)
    return per * cfg.batch * cfg.dim * cfg.seqlen


def scan_fp32_ops(cfg) -> int:
    """FP32-pipe lane operations the recurrence needs per element (b, d, t, n), counting a fused
    multiply-add as one: the exponent argument dt*A; with zero-order hold the input term v*(-1/A)*B (two
    products), the update Abar*(h - g) + g (a difference and an FMA) and the readout FMA, 6 in all; with
    the simplified B*dt*v (dt*v shared by the N states), one product, one FMA and the readout FMA, 4.
    The per-(b, d, t) work (softplus, conv, gate) is not counted."""
    return (6 if cfg.zoh else 4) * cfg.elements


# dram__bytes_read.sum + dram__bytes_write.sum of one final-pass launch of the scan kernel on each
# workload, from the ncu capture summarised under profiles/, keyed by the hash of the kernel sources it
# was taken on: after any change to those sources the figure no longer applies and is reported as null.
KERNEL_SOURCES = ("scan_p16.cuh", "ssm_device.cuh", "ssm_internal.h", "abi.cu")
TRAFFIC = {"mamba1.4b_conv": (405801472 + 113594880, "e20da626d4c56ef4")}


def hold_gpu(us: float = 200.0) -> None:
    """Queue a short device-side sleep, so that the host has enqueued a step's launches (argument checks,
    tensor maps, the launch calls) before the GPU reaches the step's start event: the CUDA events then time
    the device work, not the host's launch latency (the end-to-end leg times the host path)."""
    torch.cuda._sleep(int(us * 2000))  # ~2 GHz SM clock: about `us` microseconds


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "selective_state_space_156_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(workload: str, override):
    if override is not None:
        return override
    got = TRAFFIC.get(workload)
    return got[0] if got and got[1] == kernel_source_hash() else None


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return json.load(open(p))
        except Exception:
            pass
    return {}


def mufu_rate_per_clk(device_ok: bool) -> tuple:
    """ex2 results per clock per SM: measured by bench_peaks.cu when it builds and runs, else 32 (the
    rate measured on the B300s)."""
    if device_ok:
        exe = os.path.join(ROOT, "bench_peaks")
        src = os.path.join(ROOT, "bench_peaks.cu")
        try:
            if not os.path.exists(exe) or os.path.getmtime(exe) < os.path.getmtime(src):
                subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe, src],
                               check=True, capture_output=True, timeout=300)
            out = subprocess.run([exe], capture_output=True, text=True, timeout=120).stdout.strip().splitlines()[-1]
            j = json.loads(out)
            return float(j["per_clk_per_sm"]["ex2"]), j
        except Exception as e:  # keep the benchmark running; say where the number came from
            return 32.0, {"error": str(e)}
    return 32.0, {}


# ---------------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        self.t0 = time.time()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self) -> dict:
        t1 = getattr(self, "t1", time.time())
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if self.t0 - 0.05 <= ts <= t1 + 0.05] or [p for _, p in rows]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        mhz = [float(p[1]) for p in inside if p[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in inside:
            for name, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": float(inside[0][2]) if inside[0][2].replace(".", "").isdigit() else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max((float(p[3]) for p in inside if p[3].replace(".", "").isdigit()), default=None)}


# ---------------------------------------------------------------------------------------------
# distributed plumbing (timing only: barrier + max over ranks, no data-path collective)
# ---------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_batches(total_ranks: int, rank: int, per_rank_batch: int):
    """Weak scaling: rank r owns global batch rows [r * per_rank_batch, (r + 1) * per_rank_batch)."""
    if not 0 <= rank < total_ranks:
        raise ValueError(f"rank {rank} outside [0, {total_ranks})")
    return range(rank * per_rank_batch, (rank + 1) * per_rank_batch)


def rank_inputs(cfg, rank: int) -> dict:
    """Rank r's shard of the global batch: its own batch rows (u/x, delta, z, B, C drawn from a seed of
    its own) and the one layer's parameters every rank shares (A, D skip, dt bias, conv filter).  Rows
    are independent recurrences, so the shards need no exchange."""
    return workloads.make_scan_inputs(cfg, seed=cfg.seed + 7919 * rank, params_seed=cfg.seed)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time, on every rank (a collective on the timing only, never on data)."""
    if world == 1:
        return x
    on_gpu = torch.distributed.get_backend() == "nccl"
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: int, world: int, ms_slowest: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank / (ms_slowest * 1e-3)


def config_dict(cfg, world: int) -> dict:
    return {"workload": f"{cfg.name}: batch={cfg.batch} d_inner={cfg.dim} d_state={cfg.dstate} "
                        f"L={cfg.seqlen} {cfg.dtype} I/O, fp32 state"
                        + (", fused conv1d(k=4)+SiLU" if cfg.conv else "")
                        + (", ZOH" if cfg.zoh else ", B*dt") + (", D skip" if cfg.has_D else "")
                        + (", SiLU(z) gate" if cfg.has_z else ""),
            "global_batch": cfg.batch * world, "seq_len": cfg.seqlen,
            "parallelism": f"replicas x{world} (batch shards, no collective)",
            "l2": f"256 MB buffer written between timed steps, outside the events; inputs "
                  f"{scan_bytes(cfg) / 1e6:.0f} MB"}


# ---------------------------------------------------------------------------------------------
# CPU baseline (the oracle as it stands, bounded sample, host cores)
# ---------------------------------------------------------------------------------------------
def oracle_rate(d: dict, target_s: float, seed: int = 0):
    """Runs the fp64 oracle on a growing sample of (b, d) rows until one run takes >= target_s/4, then
    once more sized for about target_s.  Returns (elements/s, threads, rows, seconds)."""
    import numpy as np
    import oracle
    Bsz, D, L = d["u"].shape
    N = d["A"].shape[1]
    rng = np.random.default_rng(seed)
    allrows = [(int(b), int(c)) for b, c in zip(rng.integers(0, Bsz, 1 << 16), rng.integers(0, D, 1 << 16))]
    R = 16
    while True:
        t = time.time()
        _, _, nt = oracle.scan(d, rows=allrows[:R])
        dt = time.time() - t
        if dt >= target_s / 4 or R >= len(allrows):
            break
        R = min(len(allrows), R * 4)
    R2 = max(1, min(len(allrows), int(R * target_s / max(dt, 1e-6))))
    t = time.time()
    _, _, nt = oracle.scan(d, rows=allrows[:R2])
    dt = time.time() - t
    return R2 * L * N / dt, nt, R2, dt


# ---------------------------------------------------------------------------------------------
# the b300 arm
# ---------------------------------------------------------------------------------------------
def run_b300(args, rank, world, local):
    import selective_state_space_156_b300 as ssm
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.backward_only:  # the training step alone (profiling runs)
        cfg = workloads.SCAN_CONFIGS[args.workload]
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in rank_inputs(cfg, rank).items()}
        hbm_peak = measured_peaks().get("hbm_gbs") or FALLBACK_HBM_GBS
        out = run_backward(ssm, dev, cfg, g, hbm_peak, world, steps=max(args.steps, 1))
        if rank == 0:
            print(json.dumps({"backward": out}), flush=True)
        return
    if args.ssd_only:  # the Mamba-2 (SSD) layer alone (profiling runs)
        pk = measured_peaks()
        ssd = run_ssd(ssm, dev, pk.get("hbm_gbs") or FALLBACK_HBM_GBS, pk.get("bf16_tflops") or FALLBACK_BF16_TFLOPS,
                      world, steps=max(args.steps, 1))
        if rank == 0:
            print(json.dumps({"ssd": ssd}), flush=True)
        return
    if args.decode_only:  # the decode workload alone (profiling runs; smaller with --decode-layers/steps)
        hbm_peak = measured_peaks().get("hbm_gbs") or FALLBACK_HBM_GBS
        decode = run_decode(ssm, dev, hbm_peak, world, steps=args.decode_steps, nlayers=args.decode_layers)
        if rank == 0:
            print(json.dumps({"decode": decode}), flush=True)
        return
    cfg = workloads.SCAN_CONFIGS[args.workload]
    cpu_inputs = rank_inputs(cfg, rank)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in cpu_inputs.items()}
    y = torch.empty_like(g["u"])
    h_out = torch.empty((cfg.batch, cfg.dim, cfg.dstate), dtype=torch.float32, device=dev)
    nws = ssm.ssm_scan_workspace_size(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"],
                                      delta_bias=g["delta_bias"], z=g["z"], conv_w=g["conv_w"], conv_b=g["conv_b"],
                                      h_out=h_out, y=y)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)
    launches_per_step = 2 if nws > 0 else 1

    def step():
        ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], Dskip=g["Dskip"], delta_bias=g["delta_bias"],
                         z=g["z"], conv_w=g["conv_w"], conv_b=g["conv_b"], h_out=h_out, y=y, workspace=ws)

    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        wall0 = time.time()
        hold_gpu(2000.0)                  # the host runs ahead of the queue from the first step on
        for i in range(K):
            flush.zero_()                 # L2 flush between timed steps, outside the events
            ev0[i].record(stream)
            step()
            ev1[i].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        wall = time.time() - wall0
        clk.mark_end()
    times = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    ms_local = statistics.fmean(times)
    ms = max_over_ranks(ms_local, world)
    elements = cfg.elements
    value = aggregate_rate(elements, world, ms)

    # --- end to end through the public API with pinned host buffers ---
    # Every step uploads its inputs from pinned host memory, runs the scan and reads y back.  Steps are
    # pipelined over three streams and two sets of device buffers: the upload of step i + 1 overlaps the
    # scan of step i and the read-back of step i - 1 (the two copy directions use separate engines).
    # The serial form (upload, scan, read-back, one after the other) is reported beside it.
    e2e = None
    if not args.no_e2e:
        names = ["u", "delta", "z", "Bm", "Cm", "A", "Dskip", "delta_bias", "conv_w", "conv_b"]
        host = {k: cpu_inputs[k].pin_memory() for k in names}
        devb = [{k: torch.empty_like(host[k], device=dev) for k in names} for _ in range(2)]
        ybuf = [torch.empty_like(y) for _ in range(2)]
        y_host = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = y_host[0].numel() * y_host[0].element_size()
        s_in, s_in2, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(4))
        up_done = [torch.cuda.Event() for _ in range(2)]
        up_done2 = [torch.cuda.Event() for _ in range(2)]
        # the uploads of a step go out on two streams (two copy engines), in two halves of similar size
        halves = (["u", "Bm", "Cm", "A", "Dskip"], ["delta", "z", "delta_bias", "conv_w", "conv_b"])
        if not E2E_TWO_UPLOAD_STREAMS:
            halves = (names, [])
        run_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        for ev in run_done + out_done:
            ev.record(stream)

        def e2e_step(i):
            k = i % 2
            for st_, evs, part in ((s_in, up_done, halves[0]), (s_in2, up_done2, halves[1])):
                with torch.cuda.stream(st_):
                    st_.wait_event(run_done[k])       # the scan that last read buffer k is done
                    for n in part:
                        devb[k][n].copy_(host[n], non_blocking=True)
                    evs[k].record(st_)
            with torch.cuda.stream(s_run):
                s_run.wait_event(up_done[k])
                s_run.wait_event(up_done2[k])
                s_run.wait_event(out_done[k])         # y buffer k has been read back
                b_ = devb[k]
                ssm.ssm_scan_fwd(b_["u"], b_["delta"], b_["A"], b_["Bm"], b_["Cm"], Dskip=b_["Dskip"],
                                 delta_bias=b_["delta_bias"], z=b_["z"], conv_w=b_["conv_w"], conv_b=b_["conv_b"],
                                 y=ybuf[k], workspace=ws, stream=s_run)
                run_done[k].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(run_done[k])
                y_host[k].copy_(ybuf[k], non_blocking=True)
                out_done[k].record(s_out)

        def serial_step():
            b_ = devb[0]
            for n in names:
                b_[n].copy_(host[n], non_blocking=True)
            ssm.ssm_scan_fwd(b_["u"], b_["delta"], b_["A"], b_["Bm"], b_["Cm"], Dskip=b_["Dskip"],
                             delta_bias=b_["delta_bias"], z=b_["z"], conv_w=b_["conv_w"], conv_b=b_["conv_b"],
                             y=ybuf[0], workspace=ws)
            y_host[0].copy_(ybuf[0], non_blocking=True)

        for i in range(4):
            e2e_step(i)
        serial_step()
        torch.cuda.synchronize()
        E = max(3, min(args.e2e_steps, K))
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        t0.record(s_in)
        for i in range(E):
            e2e_step(i)
        s_in.wait_event(out_done[(E - 1) % 2])
        s_in.wait_event(out_done[E % 2])
        t1.record(s_in)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(t0.elapsed_time(t1) / E, world)
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        for _ in range(E):
            serial_step()
        b_.record(stream)
        torch.cuda.synchronize()
        serial_ms = max_over_ranks(a_.elapsed_time(b_) / E, world)
        e2e = {"value": aggregate_rate(elements, world, e2e_ms), "unit": "elem/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E,
               "h2d_gbs": h2d / (e2e_ms * 1e-3) / 1e9,
               "pipelined": f"{'2 upload streams' if E2E_TWO_UPLOAD_STREAMS else '1 upload stream'}, scan stream, "
                            "read-back stream, 2 buffer sets",
               "serial_ms_per_step": serial_ms, "serial_value": aggregate_rate(elements, world, serial_ms)}

    # --- roofline of the dominant (only) kernel ---
    peaks = measured_peaks()
    hbm_peak = peaks.get("hbm_gbs")
    hbm_src = "measured" if hbm_peak else "fallback"
    hbm_peak = hbm_peak or FALLBACK_HBM_GBS
    rate_clk, probe = mufu_rate_per_clk(not args.no_peaks) if rank == 0 else (32.0, {})
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mufu_peak = sms * rate_clk * MAX_SM_MHZ * 1e6           # ex2-class ops / s
    fp32_peak = sms * FP32_LANES_PER_SM * MAX_SM_MHZ * 1e6  # FP32 lane operations / s
    mufu_ops = scan_mufu_ops(cfg)
    fp32_ops = scan_fp32_ops(cfg)
    nbytes = scan_bytes(cfg)
    t_s = ms * 1e-3
    # the three roofs of the launch; the one with the longest ideal time binds
    terms = {
        "fp32": {"ideal_us": fp32_ops / fp32_peak * 1e6, "ops_per_launch": fp32_ops, "achieved": fp32_ops / t_s / 1e12,
                 "peak": fp32_peak / 1e12, "unit": "TFLOP/s (FP32 lane ops)",
                 "peak_source": f"derived: {sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x {MAX_SM_MHZ:.0f} MHz"},
        "mufu": {"ideal_us": mufu_ops / mufu_peak * 1e6, "ops_per_launch": mufu_ops, "achieved": mufu_ops / t_s / 1e12,
                 "peak": mufu_peak / 1e12, "unit": "Tmufu/s",
                 "peak_source": f"derived: {sms} SMs x {rate_clk:.1f} ex2/clk/SM (bench_peaks.cu) x {MAX_SM_MHZ:.0f} MHz"},
        "hbm": {"ideal_us": nbytes / (hbm_peak * 1e9) * 1e6, "bytes_per_launch": nbytes, "achieved": nbytes / t_s / 1e9,
                "peak": hbm_peak, "unit": "GB/s", "peak_source": f"{hbm_src} (MEASURED_PEAKS.json hbm_gbs)"},
    }
    bind = max(terms, key=lambda k: terms[k]["ideal_us"])
    tb = terms[bind]
    roof = {"bound": "hbm" if bind == "hbm" else "alu", "pipe": bind, "achieved": tb["achieved"], "peak": tb["peak"],
            "unit": tb["unit"], "frac": tb["achieved"] / tb["peak"], "traffic": traffic_for(args.workload, args.traffic),
            "kernel_source_hash": kernel_source_hash(),
            "peak_source": tb["peak_source"], "kernel": "scan_p16_kernel (final pass)",
            "terms": {k: {kk: vv for kk, vv in v.items() if kk != "peak_source"} | {"frac": v["achieved"] / v["peak"]}
                      for k, v in terms.items()}}
    hbm = {"achieved_gbs": nbytes / t_s / 1e9, "peak_gbs": hbm_peak, "frac": nbytes / t_s / 1e9 / hbm_peak,
           "bytes_per_launch": nbytes, "peak_source": hbm_src}

    # --- the other scan workloads of the suite (not the headline) ---
    others = None
    if not args.no_configs:
        others = run_other_configs(ssm, dev, args.workload, hbm_peak, fp32_peak, mufu_peak, world)

    # --- a training step: forward keeping every state, then the backward pass ---
    backward = None
    if not args.no_backward:
        backward = run_backward(ssm, dev, cfg, g, hbm_peak, world)

    # --- decode workload (ssm_state_update) ---
    decode = None
    if not args.no_decode:
        decode = run_decode(ssm, dev, hbm_peak, world, steps=args.decode_steps, nlayers=args.decode_layers)

    # --- Mamba-2 (SSD) layer on the tensor cores ---
    ssd = None
    if not args.no_ssd:
        pk = measured_peaks()
        ssd = run_ssd(ssm, dev, hbm_peak, pk.get("bf16_tflops") or FALLBACK_BF16_TFLOPS, world)

    # --- CPU baseline: oracle on host cores, rank 0 at N = 1 only ---
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        rate, nt, R, secs = oracle_rate(cpu_inputs, args.cpu_seconds)
        cpu = {"value": rate, "unit": "elem/s", "cores": nt, "kind": "oracle",
               "sample": f"{R} random (b, d) rows of {cfg.batch * cfg.dim}, full L={cfg.seqlen}, N={cfg.dstate} "
                         f"({secs:.1f} s, fp64 C, one thread per row)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "elem/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_dict(cfg, world),
            "gpu_launches": K * launches_per_step,
            "roofline": roof, "hbm": hbm, "cpu_baseline": cpu, "e2e": e2e, "decode": decode, "backward": backward,
            "ssd": ssd,
            "other_workloads": others,
            "clocks": clk.summary(), "wall_s_timed_region": wall, "mufu_probe": probe,
            "ms_per_step_min": min(times), "ms_per_step_median": statistics.median(times),
        }
        print(json.dumps(line), flush=True)


def run_decode(ssm, dev, hbm_peak, world, steps=None, nlayers=None):
    """64 layers x 128 tokens of ssm_state_update, layer-major per token, replayed as one CUDA graph per
    token.  Every layer keeps its own fp32 state cache (5.4 GB in total); per-token inputs come from a
    pool of 64 sets (512 MB), so neither states nor inputs can stay in L2 between uses."""
    cfg = workloads.DECODE_CONFIG
    P = 64
    steps = steps or cfg.steps
    nl = nlayers or cfg.layers
    pool = workloads.make_decode_pool(cfg, P, device=dev)
    layers = [workloads.make_decode_layer(cfg, l, device=dev) for l in range(nl)]
    y = torch.empty((cfg.batch, cfg.dim), dtype=torch.bfloat16, device=dev)

    def token(step):
        for l in range(nl):
            k = workloads.decode_pool_index(l, step, P)
            L_ = layers[l]
            ssm.ssm_state_update(L_["state"], pool["u"][k], pool["delta"][k], L_["A"], pool["Bm"][k], pool["Cm"][k],
                                 Dskip=L_["Dskip"], delta_bias=L_["delta_bias"], z=pool["z"][k], y=y)

    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    graphs = []
    with torch.cuda.stream(s):
        token(0)  # warm-up outside capture
        for gi in range(P):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=s):
                token(gi)
            graphs.append(gr)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for st in range(steps):
        graphs[st % P].replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    ms = max_over_ranks(ms, world)
    state_bytes = cfg.batch * cfg.dim * cfg.dstate * 4
    per_call = 2 * state_bytes + 3 * cfg.batch * cfg.dim * 2 + 2 * cfg.batch * cfg.dstate * 2 + \
        cfg.batch * cfg.dim * 2 + cfg.dim * (cfg.dstate + 2) * 4
    calls = steps * nl
    gbs = per_call * calls / (ms * 1e-3) / 1e9
    return {"workload": f"{cfg.name}: batch={cfg.batch} d_inner={cfg.dim} d_state={cfg.dstate} x {nl} layers "
                        f"x {steps} tokens, bf16 I/O, fp32 state cache updated in place",
            "tokens_per_s": world * cfg.batch * steps / (ms * 1e-3), "ms_total": ms,
            "us_per_layer_call": ms * 1e3 / calls, "state_cache_gbs": 2 * state_bytes * calls / (ms * 1e-3) / 1e9,
            "hbm_gbs": gbs, "hbm_frac": gbs / hbm_peak, "bytes_per_call": per_call, "launch": "CUDA graph per token"}


def run_other_configs(ssm, dev, skip: str, hbm_peak: float, fp32_peak: float, mufu_peak: float, world: int,
                      steps: int = 20) -> dict:
    """Every other scan workload of the suite, timed like the headline (L2 flushed between steps, CUDA
    events, mean of `steps`): time, elements/s and the three roofline fractions.  The long sequence runs
    as one call with the L split and, as it is also used, as 32 chained calls of 2048 steps."""
    out = {}
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for name, cfg in workloads.SCAN_CONFIGS.items():
        if name == skip:
            continue
        d = workloads.make_scan_inputs(cfg)
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        y = torch.empty_like(g["u"])
        h = torch.empty((cfg.batch, cfg.dim, cfg.dstate), dtype=torch.float32, device=dev)
        kw = dict(Dskip=g["Dskip"], delta_bias=g["delta_bias"], z=g["z"], conv_w=g["conv_w"], conv_b=g["conv_b"],
                  zoh=cfg.zoh)
        ws = ssm.ssm_scan_workspace_size(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], h_out=h, y=y, **kw)
        wsb = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
        variants = {"one call": lambda: ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], y=y, h_out=h,
                                                          workspace=wsb, **kw)}
        if cfg.chunk:
            pieces = [{k: g[k][..., a:a + cfg.chunk].contiguous() for k in ("u", "delta", "z", "Bm", "Cm")}
                      for a in range(0, cfg.seqlen, cfg.chunk)]
            yp = torch.empty_like(pieces[0]["u"])
            p0 = pieces[0]
            wsc = ssm.ssm_scan_workspace_size(p0["u"], p0["delta"], g["A"], p0["Bm"], p0["Cm"], h0=h, h_out=h, y=yp,
                                              **dict(kw, z=p0["z"]))
            wsc = torch.empty(max(wsc, 1), dtype=torch.uint8, device=dev)

            def chained():
                h.zero_()
                for pc in pieces:
                    ssm.ssm_scan_fwd(pc["u"], pc["delta"], g["A"], pc["Bm"], pc["Cm"], h0=h, h_out=h, y=yp,
                                     workspace=wsc, **dict(kw, z=pc["z"]))
            variants[f"{cfg.seqlen // cfg.chunk} chained calls"] = chained
            # the same chain captured once as a CUDA graph: the calls' host work (argument checks, tensor
            # maps, launches) leaves the timed path, as in a serving loop that replays a captured prefill
            chained()
            torch.cuda.synchronize()
            cs = torch.cuda.Stream(device=dev)
            cs.wait_stream(torch.cuda.current_stream())
            gchain = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gchain, stream=cs):
                chained()
            torch.cuda.current_stream().wait_stream(cs)
            variants[f"{cfg.seqlen // cfg.chunk} chained calls, CUDA graph"] = gchain.replay
        res = {}
        for vname, fn in variants.items():
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(steps):
                hold_gpu()
                flush.zero_()
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record()
                fn()
                b_.record()
                torch.cuda.synchronize()
                ts.append(a_.elapsed_time(b_))
            ms = max_over_ranks(statistics.fmean(ts), world)
            t_s = ms * 1e-3
            res[vname] = {"ms": ms, "value": aggregate_rate(cfg.elements, world, ms),
                          "fp32_frac": scan_fp32_ops(cfg) / t_s / fp32_peak,
                          "mufu_frac": scan_mufu_ops(cfg) / t_s / mufu_peak,
                          "hbm_frac": scan_bytes(cfg) / t_s / 1e9 / hbm_peak}
        out[f"{name}: batch={cfg.batch} d_inner={cfg.dim} d_state={cfg.dstate} L={cfg.seqlen} {cfg.dtype}"] = res
        del g, d
    return out


def run_ssd(ssm, dev, hbm_peak, tensor_peak, world, steps=20):
    """The Mamba-2 (SSD) layer on the tensor cores: 8 x 80 heads x 64 channels x 128 states x 2048 steps,
    bf16, one group.  Inputs per rank are drawn from the rank's seed; a 256 MB buffer is written between
    timed launches (outside the events) so that every launch reads its inputs from HBM.  Roofline terms:
    the chunked algorithm's dense products (per 128-step chunk and head: C B^T, C S, M X and the state
    increment, without the hi/lo repeats the kernel adds for precision) against the measured bf16 tensor
    peak, and the bytes it must move (x, dt, B, C in; y out) against the measured HBM bandwidth."""
    cfg = workloads.SSD_CONFIGS["mamba2_2.7b"]
    rank = int(os.environ.get("RANK", "0"))
    d = workloads.make_ssd_inputs(cfg, seed=cfg.seed + 7919 * rank)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    y = torch.empty_like(g["x"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call():
        ssm.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["Bm"], g["Cm"], nheads=cfg.nheads, ngroups=cfg.ngroups,
                         Dskip=g["Dskip"], dt_bias=g["dt_bias"], y=y)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        hold_gpu()
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = max_over_ranks(statistics.median(times), world)
    flags = ssm.ssm_device_error()
    Bsz, D, L = g["x"].shape
    H, G, P, N, Q = cfg.nheads, cfg.ngroups, cfg.headdim, cfg.dstate, 128
    chunks = (L + Q - 1) // Q
    flops = 2.0 * Bsz * H * chunks * (Q * Q * N + Q * N * P + Q * Q * P + N * Q * P)
    byts = 2 * Bsz * D * L * 2 + Bsz * H * L * 2 + 2 * Bsz * G * L * N * 2
    t_tensor = flops / (tensor_peak * 1e12) * 1e3
    t_hbm = byts / (hbm_peak * 1e9) * 1e3
    return {"workload": f"{cfg.name}: batch {Bsz}, {H} heads x {P}, d_state {N}, {G} group, L {L}, bf16 "
                        "(ssd_scan_fwd, chunks of 128 on tcgen05)",
            "ms": ms, "ms_min": min(times), "elements_per_s": world * Bsz * D * L * N / (ms * 1e-3),
            "tokens_per_s": world * Bsz * L / (ms * 1e-3),
            "tensor_tflops": flops / (ms * 1e-3) / 1e12, "tensor_peak_tflops": tensor_peak,
            "tensor_frac": t_tensor / ms, "hbm_gbs": byts / (ms * 1e-3) / 1e9, "hbm_peak_gbs": hbm_peak,
            "hbm_frac": t_hbm / ms, "roofline_frac": max(t_tensor, t_hbm) / ms,
            "bound": "tensor" if t_tensor >= t_hbm else "hbm",
            "flops_per_launch": flops, "bytes_per_launch": byts, "steps": steps, "device_error_flags": flags,
            "peaks": "of measured (MEASURED_PEAKS.json: bf16 burst, HBM copy)"}


def run_backward(ssm, dev, cfg, g, hbm_peak, world, steps=5):
    """A training step of the layer: the forward that keeps a state checkpoint every 8 steps (h_ckpt,
    (B, ceil(L/8), D, N) fp32), then ssm_scan_bwd, which recomputes each 8-step group's states from the
    checkpoint before it.  Reported beside the forward-only headline, with the HBM bytes each launch must
    move at least."""
    Bsz, D, L = g["u"].shape
    N = g["A"].shape[1]
    nck = ssm.ckpt_count(L)
    h_ckpt = torch.empty((Bsz, nck, D, N), dtype=torch.float32, device=dev)
    gen = torch.Generator(device=dev).manual_seed(17)
    dy = torch.randn((Bsz, D, L), generator=gen, device=dev).to(g["u"].dtype)
    kw = dict(Dskip=g["Dskip"], delta_bias=g["delta_bias"], z=g["z"], conv_w=g["conv_w"], conv_b=g["conv_b"])
    y = torch.empty_like(g["u"])

    def fwd():
        ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], y=y, h_ckpt=h_ckpt, **kw)

    def bwd():
        return ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["Bm"], g["Cm"], dy, h_ckpt, **kw)

    for _ in range(2):
        fwd()
        bwd()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record()
        fwd()
        ev[i][1].record()
        bwd()
        ev[i][2].record()
    torch.cuda.synchronize()
    t_f = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    t_b = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    t_f, t_b = max_over_ranks(t_f, world), max_over_ranks(t_b, world)
    e = g["u"].element_size()
    bdl = Bsz * D * L
    ckpt_bytes = Bsz * D * nck * N * 4
    fwd_bytes = bdl * e * 4 + ckpt_bytes                        # u, delta, z in; y out; checkpoints out
    bwd_bytes = bdl * e * 7 + ckpt_bytes + 2 * Bsz * N * L * 4  # u, delta, z, dy in; du, ddelta, dz out; checkpoints
    return {"workload": f"{cfg.name}: forward keeping a state checkpoint every 8 steps (h_ckpt) + ssm_scan_bwd "
                        f"recomputing the states in between",
            "ms_forward_ckpt": t_f, "ms_backward": t_b, "ms_train_step": t_f + t_b,
            "elements_per_s_train_step": world * bdl * N / ((t_f + t_b) * 1e-3),
            "forward_hbm_gbs": fwd_bytes / (t_f * 1e-3) / 1e9, "forward_hbm_frac": fwd_bytes / (t_f * 1e-3) / 1e9 / hbm_peak,
            "backward_hbm_gbs": bwd_bytes / (t_b * 1e-3) / 1e9,
            "backward_hbm_frac": bwd_bytes / (t_b * 1e-3) / 1e9 / hbm_peak,
            "bytes_forward": fwd_bytes, "bytes_backward": bwd_bytes, "checkpoint_bytes": ckpt_bytes, "steps": steps}


# ---------------------------------------------------------------------------------------------
# the reference arm: the oracle as it stands, on the host cores
# ---------------------------------------------------------------------------------------------
def run_reference(args, rank, world):
    if rank != 0:
        return
    cfg = workloads.SCAN_CONFIGS[args.workload]
    d = rank_inputs(cfg, 0)
    budget = 150.0  # seconds for the whole --steps K --warmup W run
    rate0, nt, R0, secs0 = oracle_rate(d, 2.0)
    per_step_s = min(5.0, budget / max(1, args.steps + args.warmup))
    rows = max(1, int(rate0 * per_step_s / (cfg.seqlen * cfg.dstate)))
    import numpy as np
    import oracle
    rng = np.random.default_rng(1)
    R = cfg.batch * cfg.dim
    sample = [(int(i // cfg.dim), int(i % cfg.dim)) for i in rng.choice(R, min(rows, R), replace=False)]
    for _ in range(args.warmup):
        oracle.scan(d, rows=sample)
    t = time.time()
    for _ in range(args.steps):
        _, _, nt = oracle.scan(d, rows=sample)
    secs = time.time() - t
    elems = len(sample) * cfg.seqlen * cfg.dstate * args.steps
    value = elems / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "elem/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(cfg, 1),
            "cpu_baseline": {"value": value, "unit": "elem/s", "cores": nt, "kind": "oracle",
                             "sample": f"{len(sample)} random (b, d) rows per step of {R}, full L={cfg.seqlen}"},
            "e2e": {"value": value, "unit": "elem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["b300", "reference"], default="b300")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(workloads.SCAN_CONFIGS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch from an ncu capture of this kernel (reported as is)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip the training-step (backward) measurement")
    ap.add_argument("--no-configs", action="store_true", help="skip timing the other scan workloads")
    ap.add_argument("--backward-only", action="store_true", help="run only the training-step measurement")
    ap.add_argument("--decode-only", action="store_true", help="run only the decode workload")
    ap.add_argument("--no-ssd", action="store_true", help="skip the Mamba-2 (SSD) layer")
    ap.add_argument("--ssd-only", action="store_true", help="run only the Mamba-2 (SSD) layer")
    ap.add_argument("--decode-layers", type=int, default=None, help="decode layers (default 64)")
    ap.add_argument("--decode-steps", type=int, default=None, help="decode tokens (default 128)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-peaks", action="store_true", help="skip the bench_peaks.cu MUFU-rate probe")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        run_b300(args, rank, world, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
