#!/usr/bin/env python
"""Throughput of the fused exact-attention hot path on one (or N) GB300.

One step = the whole path on one synthetic batch: fa_fwd (O, LSE; with the
tail of its schedule split and merged by a second kernel when the last wave of
CTAs is partly filled) then the three backward stages (preprocess, recompute
main kernel, dQ convert), bf16,
B=2 H=16 N=4096 d=128, non-causal, inputs i.i.d. N(0,1) rounded to bf16.
FLOPs per step: 4*B*H*N^2*d (forward) + 2.5x that (backward).

Arms:
  default           our CUDA kernels through the C ABI; prints one JSON line.
  --impl reference  the fp64 CPU oracle on the host cores, on a bounded sample
                    of the same workload (a strip of query rows of one head).

Timing: W untimed warm-up steps, then exactly K steps between a barrier and a
device synchronize. L2 is flushed (256 MiB write) before every step; each step
is timed with CUDA events on the launching stream, and so is every kernel
launch of the dominant kernel. Under torchrun each rank runs its own batch
(weak scaling, no collective on the data path); rank 0 reports the max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s on 1 GB300 (bf16) and % of tensor-core peak"
B, H, N, D = 2, 16, 4096, 128
WORKLOAD = f"fwd+bwd bf16 B={B} H={H} N={N} d={D} non-causal"
FWD_FLOPS = 4.0 * B * H * N * N * D
BWD_FLOPS = 2.5 * FWD_FLOPS
STEP_FLOPS = FWD_FLOPS + BWD_FLOPS
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "bwd_main_traffic.txt")
BWD_SOURCE = os.path.join(ROOT, "exact_attention_30_gb300", "csrc", "attn_bwd_bf16.cu")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="fa", choices=["fa", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--heads", type=int, default=None,
                   help="override H (smaller profiling captures); the JSON line names the change")
    p.add_argument("--op", default="attention", choices=["attention", "softmax", "decode", "minilab"],
                   help="softmax: time the fused row softmax on the B*H*N x N score matrix of "
                        "the shape; decode: time KV-cache decode on --decode-workload (both "
                        "HBM-bound; not the headline line)")
    p.add_argument("--decode-workload", default="decode_bf16_8x32x1x32768x128",
                   help="named decode workload for --op decode")
    p.add_argument("--decode-shape", type=int, nargs=5, metavar=("B", "H", "NQ", "NK", "D"),
                   default=None, help="another decode shape (profiling captures); the JSON line names it")
    p.add_argument("--dtype", default="bf16", choices=["bf16", "f32"],
                   help="element type for --op softmax")
    p.add_argument("--varlen", action="store_true",
                   help="packed variable-length batch: 16 sequences of seeded lengths in [512, 8192], "
                        "H=16, d=128, fwd+bwd (with --causal: causal); not the headline line")
    p.add_argument("--causal", action="store_true",
                   help="causal attention (FLOPs counted as half of the full count, the usual "
                        "convention; the JSON line names it)")
    p.add_argument("--shape", type=int, nargs=4, metavar=("B", "H", "N", "D"), default=None,
                   help="another [B,H,N,d] shape (the JSON line names it); the default is the "
                        "headline shape")
    args = p.parse_args()
    global B, H, N, D, WORKLOAD, FWD_FLOPS, BWD_FLOPS, STEP_FLOPS
    if args.shape is not None:
        B, H, N, D = args.shape
    if args.heads is not None:
        H = args.heads
    WORKLOAD = f"fwd+bwd bf16 B={B} H={H} N={N} d={D} " + ("causal" if args.causal else "non-causal")
    FWD_FLOPS = 4.0 * B * H * N * N * D * (0.5 if args.causal else 1.0)
    BWD_FLOPS = 2.5 * FWD_FLOPS
    STEP_FLOPS = FWD_FLOPS + BWD_FLOPS
    return args


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a per-rank float over the process group (identity when not distributed).

    Rank 0 reports step times this way: the job is as slow as its slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, flops_per_rank_step: float, ms_per_step_max: float) -> float:
    """Whole-job TFLOP/s: every rank processes its own batch (weak scaling)."""
    return world * flops_per_rank_step / (ms_per_step_max * 1e-3) / 1e12


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "hbm_gbs": float(pk["hbm_gbs"])}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS, bf16_tflops_sustained=1700.0), "fallback"


# A timed region counts as "sustained" (the power-capped GEMM loop's figure)
# only when it lasted at least this long and the clock sampler saw the power
# cap active; anything shorter is a burst, compared with the burst GEMM.
SUSTAINED_MIN_SECONDS = 2.0


def bf16_peak(peaks, src, clocks, timed_seconds):
    """(peak TFLOP/s, label) for a tensor-bound kernel timed over `timed_seconds`."""
    capped = bool(clocks) and "sw_power_cap" in (clocks.get("reasons") or [])
    if capped and timed_seconds >= SUSTAINED_MIN_SECONDS:
        return peaks["bf16_tflops_sustained"], f"{src} bf16 sustained (timed {timed_seconds:.1f} s under sw_power_cap)"
    why = "no power cap sampled" if not capped else f"timed region {timed_seconds:.2f} s < {SUSTAINED_MIN_SECONDS} s"
    return peaks["bf16_tflops"], f"{src} bf16 burst ({why})"


def fwd_kernel_name(B, H, N, D, sms):
    """The forward kernel a bf16 fixed-length problem runs on, on a GPU with
    `sms` SMs, by the routing rule fa.h documents for fa_fwd_plan: d = 64
    and B*H*ceil(N/512) >= 3/4 of the SMs take the four-query-tile kernel."""
    if D == 64 and 4 * B * H * (-(-N // 512)) >= 3 * sms:
        return "fwd_bf16_q4_kernel"
    return f"fwd_bf16_kernel<{D}>"


def read_traffic():
    """DRAM bytes per launch of the backward main kernel from the committed ncu
    summary, or None when the kernel source changed since it was captured."""
    try:
        fields = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 2 and not line.startswith("#"):
                    fields[parts[0]] = parts[1]
        with open(BWD_SOURCE, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if fields.get("source_sha256") != sha:
            return None
        return float(fields["dram_bytes_per_launch_full_size"])
    except Exception:
        return None


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, uuid: str | None):
        self.proc = None
        self.path = os.path.join("/tmp", f"fa_bench_clocks_{os.getpid()}.csv")
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t_start = None

    def wait_first_sample(self, timeout=3.0):
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < timeout:
            if os.path.getsize(self.path) > 0:
                return
            time.sleep(0.05)

    def mark(self):
        self.t_mark = os.path.getsize(self.path) if self.proc is not None else 0

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            f.seek(self.t_mark)
            lines = [ln.strip() for ln in f if ln.strip()]
        os.remove(self.path)
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------- oracle arm
def oracle_step_rows(q64, k64, v64, do64, scale, rows):
    """fwd + bwd of the oracle restricted to a strip of query rows of one head.

    The backward is a sum over query rows, so a strip gives exact dQ rows and
    that strip's exact contribution to dK and dV."""
    from oracle import attention_bwd, attention_fwd
    qs, dos = q64[rows], do64[rows]
    attention_fwd(qs, k64, v64, scale)
    attention_bwd(qs, k64, v64, dos, scale)
    return len(rows) * N * D * (4.0 + 10.0)  # fwd 4*R*N*d + bwd 2.5x


def oracle_sample_inputs(seed=0):
    import numpy as np
    import torch

    from exact_attention_30_gb300.inputs import random_qkv
    q, k, v, do = random_qkv(1, 1, N, D, torch.bfloat16, seed=seed)
    f = lambda t: t[0, 0].to(torch.float64).numpy()
    return f(q), f(k), f(v), f(do), np.float32(1 / math.sqrt(D))


def blas_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            try:
                return int(os.environ[var])
            except ValueError:
                pass
    return os.cpu_count()


def cpu_baseline_causal(seconds: float):
    """The oracle, causal, on whole seeded heads of the workload's shape (the
    causal mask needs every row's index, so no strips); FLOPs counted as half
    of the full count, like the GPU line."""
    from oracle import attention_bwd, attention_fwd
    flops, heads = 0.0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or heads == 0:
        q64, k64, v64, do64, scale = oracle_sample_inputs(seed=heads)
        attention_fwd(q64, k64, v64, scale, causal=True)
        attention_bwd(q64, k64, v64, do64, scale, causal=True)
        flops += 0.5 * N * N * D * (4.0 + 10.0)
        heads += 1
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"fp64 numpy oracle, causal fwd+bwd of {heads} seeded head(s) of N={N}, d={D}, "
                      f"{dt:.1f} s (input generation included)"}


def cpu_baseline(seconds: float):
    """Time the oracle on the host cores for about `seconds`: fwd+bwd of
    256-row query strips of successive seeded heads of the workload's shape."""
    flops, rows_done, heads = 0.0, 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        q64, k64, v64, do64, scale = oracle_sample_inputs(seed=heads)
        heads += 1
        for r0 in range(0, N, 256):
            if time.perf_counter() - t0 >= seconds:
                break
            rows = list(range(r0, min(r0 + 256, N)))
            flops += oracle_step_rows(q64, k64, v64, do64, scale, rows)
            rows_done += len(rows)
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"fp64 numpy oracle, fwd+bwd of {rows_done} query rows (256-row strips over "
                      f"{heads} seeded head(s) of N={N}, d={D}) against all {N} keys, {dt:.1f} s "
                      f"(input generation included)"}


def parity_sample(q_h, k_h, v_h, do_h, o, lse, dq, scale):
    """Part of the CPU-baseline leg: the fp64 oracle on sampled query rows of
    the bench's own inputs, against the GPU's O, LSE and dQ of the timed step
    (dQ rows are row-local, so a strip of rows is exact; dK and dV, sums over
    every query, are left to the parity tests). Errors: max |gpu - ref| /
    max |ref| over the checked rows for O and dQ, max |gpu - ref| for LSE."""
    import numpy as np

    from oracle import attention_bwd, attention_fwd_rows
    rows = sorted(set(np.linspace(0, N - 1, 33).astype(int).tolist()))
    heads = [(0, 0), (B - 1, H - 1)]
    err = {"O": 0.0, "LSE": 0.0, "dQ": 0.0}
    o_h, l_h, dq_h = o.float().cpu(), lse.cpu(), dq.float().cpu()
    for b, h in heads:
        f = lambda t: t[b, h].double().numpy()
        Q, K, V, dO = f(q_h), f(k_h), f(v_h), f(do_h)
        O, LSE = attention_fwd_rows(Q, K, V, scale, rows)
        dQ = attention_bwd(Q[rows], K, V, dO[rows], scale)[0]
        go, gl, gdq = o_h[b, h][rows].double().numpy(), l_h[b, h][rows].double().numpy(), dq_h[b, h][rows].double().numpy()
        err["O"] = max(err["O"], float(np.abs(go - O).max() / np.abs(O).max()))
        err["LSE"] = max(err["LSE"], float(np.abs(gl - LSE).max()))
        err["dQ"] = max(err["dQ"], float(np.abs(gdq - dQ).max() / np.abs(dQ).max()))
    tol = {"O": 2e-2, "LSE": 1e-3, "dQ": 5e-2}
    return {"checked": f"O, LSE and dQ of {len(rows)} query rows in heads {heads} of the bench inputs",
            "max_err": err, "tol": tol, "pass": all(err[k] <= tol[k] for k in tol)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    q64, k64, v64, do64, scale = oracle_sample_inputs()
    # size the strip so that the whole run stays within about two minutes
    t0 = time.perf_counter()
    oracle_step_rows(q64, k64, v64, do64, scale, list(range(64)))
    t64 = time.perf_counter() - t0
    budget = 120.0 / max(1, args.steps + args.warmup)
    R = int(max(8, min(N, 64 * budget / max(t64, 1e-6))))
    R = 1 << int(math.log2(R))
    for i in range(args.warmup):
        oracle_step_rows(q64, k64, v64, do64, scale, list(range(R)))
    times, flops = [], 0.0
    for i in range(args.steps):
        r0 = (i * R) % N
        rows = [(r0 + t) % N for t in range(R)]
        t0 = time.perf_counter()
        flops = oracle_step_rows(q64, k64, v64, do64, scale, rows)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms * 1e-3) / 1e12
    sample = (f"per step: fp64 numpy oracle fwd+bwd of {R} query rows of one head "
              f"(N={N}, d={D}) against all keys")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "d": D,
                   "sample_rows_per_step": R, "flops_per_step_sample": flops},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import exact_attention_30_gb300 as fa
    from exact_attention_30_gb300.inputs import random_qkv

    fa.load_library()
    stream = torch.cuda.current_stream(dev)
    scale = 1 / math.sqrt(D)
    q_h, k_h, v_h, do_h = random_qkv(B, H, N, D, torch.bfloat16, seed=rank)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, D), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    causal = bool(args.causal)
    # the forward's scratch for splitting a partly filled last wave (none when
    # nothing is split); the step then launches the merge kernel as well
    fws_bytes = fa.fa_fwd_workspace_bytes(B, H, N, D, causal=causal)
    fws = torch.empty(fws_bytes, dtype=torch.uint8, device=dev) if fws_bytes else None
    launches_per_step = 4 + (1 if fws_bytes else 0)

    def bwd_stage(stage):
        fa.fa_bwd_stage(stage, q, k, v, o, do, lse, scale, workspace=ws, dq=dq, dk=dk, dv=dv,
                        causal=causal)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fa_fwd(q, k, v, scale, out=o, lse=lse, causal=causal, workspace=fws)
        if ev is not None:
            ev[1].record(stream)
        bwd_stage(fa.FA_BWD_PREPROCESS)
        if ev is not None:
            ev[2].record(stream)
        bwd_stage(fa.FA_BWD_MAIN)
        if ev is not None:
            ev[3].record(stream)
        bwd_stage(fa.FA_BWD_DQ_CONVERT)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_check_device_status(dev) != fa.FA_OK:
        raise RuntimeError("device status not OK after warm-up")

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(dev.index, uuid) if rank == 0 else None
    if sampler:
        sampler.wait_first_sample()
        sampler.mark()

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        step(events[i])
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    status = fa.fa_check_device_status(dev)
    if status != fa.FA_OK:
        raise RuntimeError(f"device status {fa.fa_status_string(status)}")

    step_ms = [e[0].elapsed_time(e[4]) for e in events]
    fwd_ms = [e[0].elapsed_time(e[1]) for e in events]
    pre_ms = [e[1].elapsed_time(e[2]) for e in events]
    main_ms = [e[2].elapsed_time(e[3]) for e in events]
    conv_ms = [e[3].elapsed_time(e[4]) for e in events]
    ms_per_step = max_over_ranks(sum(step_ms) / len(step_ms), dev)

    # End to end through the public API with pinned host buffers: every step
    # copies its four inputs host -> device, runs fa_fwd + fa_bwd, and copies
    # dQ, dK, dV device -> host. Steps are pipelined over two buffer sets and
    # three streams (inputs in, compute, results out), so step i+1's inputs
    # and step i-1's results move while step i computes; the timed region runs
    # from the first input copy to the last result copy.
    pin = lambda t: t.pin_memory()
    host_in = [tuple(pin(t.clone()) for t in (q_h, k_h, v_h, do_h)) for _ in range(2)]
    host_out = [tuple(torch.empty(q_h.shape, dtype=q_h.dtype).pin_memory() for _ in range(3))
                for _ in range(2)]
    dev_in = [(q, k, v, do)] + [tuple(torch.empty_like(t) for t in (q, k, v, do))]
    dev_o = [(o, lse)] + [(torch.empty_like(o), torch.empty_like(lse))]
    dev_out = [(dq, dk, dv)] + [tuple(torch.empty_like(t) for t in (dq, dk, dv))]
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ws2 = [ws, torch.empty_like(ws)]
    e2e_steps = max(3, args.steps)  # the same K steps as the device-timed loop

    def e2e_run(n):
        done_cmp = [None, None]   # compute of the last step that used each buffer set
        done_out = [None, None]   # result copy of the last step that used each set
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_in):
                if done_cmp[b] is not None:
                    s_in.wait_event(done_cmp[b])
                for dst, src in zip(dev_in[b], host_in[b]):
                    dst.copy_(src, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in)
                if done_out[b] is not None:
                    s_cmp.wait_event(done_out[b])  # dQ/dK/dV of set b were copied out
                qq, kk, vv, dd = dev_in[b]
                oo, ll = dev_o[b]
                g1, g2, g3 = dev_out[b]
                fa.fa_fwd(qq, kk, vv, scale, out=oo, lse=ll, causal=causal, workspace=fws)
                fa.fa_bwd(qq, kk, vv, oo, dd, ll, scale, workspace=ws2[b], dq=g1, dk=g2, dv=g3,
                          causal=causal)
                done_cmp[b] = torch.cuda.Event()
                done_cmp[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_cmp[b])
                for dst, src in zip(host_out[b], dev_out[b]):
                    dst.copy_(src, non_blocking=True)
                done_out[b] = torch.cuda.Event()
                done_out[b].record(s_out)

    e2e_run(3)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_event(e0)
    s_out.wait_event(e0)
    e2e_run(e2e_steps)
    s_in.wait_stream(s_out)
    s_in.wait_stream(s_cmp)
    e1.record(s_in)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    nbytes = q_h.numel() * q_h.element_size()

    if rank != 0:
        torch.distributed.destroy_process_group()
        return 0

    peaks, peak_src = read_peaks()
    # The denominator is the burst bf16 figure (a GEMM timed alone) unless the
    # timed loop ran for seconds under the power cap; the other figure is
    # reported beside it.
    peak, peak_label = bf16_peak(peaks, peak_src, clocks, wall)
    burst, sustained = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    mean = lambda xs: sum(xs) / len(xs)
    main_avg = mean(main_ms)
    achieved = BWD_FLOPS / (main_avg * 1e-3) / 1e12
    traffic = read_traffic() if (B, H, N, D) == (2, 16, 4096, 128) and not causal else None
    fwd_avg = mean(fwd_ms)
    value = job_throughput(world, STEP_FLOPS, ms_per_step)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "d": D,
                   "flops_per_step": STEP_FLOPS,
                   "l2": "flushed before every step (256 MiB write, outside the per-step events)",
                   "parallelism": f"replicas x{world}, independent batches, no collective"},
        "roofline": {"kernel": f"bwd_main_kernel<{D}, {'true' if causal else 'false'}>",
                     "bound": "tensor", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": peak_label,
                     "frac_of_burst_peak": achieved / burst, "burst_peak": burst,
                     "frac_of_sustained_peak": achieved / sustained, "sustained_peak": sustained,
                     "timed_region_s": wall,
                     "algorithmic_flops_per_launch": BWD_FLOPS},
        "components": {
            "fwd": {"kernel": fwd_kernel_name(B, H, N, D, torch.cuda.get_device_properties(dev).multi_processor_count) + (" + fwd_tail_merge_kernel" if fws_bytes else ""),
                    "ms": fwd_avg,
                    "tflops": FWD_FLOPS / (fwd_avg * 1e-3) / 1e12,
                    "frac_of_peak": FWD_FLOPS / (fwd_avg * 1e-3) / 1e12 / peak,
                    "frac_of_burst_peak": FWD_FLOPS / (fwd_avg * 1e-3) / 1e12 / burst,
                    "frac_of_sustained_peak": FWD_FLOPS / (fwd_avg * 1e-3) / 1e12 / sustained},
            "bwd_preprocess": {"ms": mean(pre_ms)},
            "bwd_main": {"ms": main_avg, "tflops": achieved, "frac_of_peak": achieved / peak,
                         "frac_of_burst_peak": achieved / burst,
                         "frac_of_sustained_peak": achieved / sustained},
            "bwd_dq_convert": {"ms": mean(conv_ms)},
            "bwd_total": {"ms": mean(pre_ms) + main_avg + mean(conv_ms),
                          "tflops": BWD_FLOPS / ((mean(pre_ms) + main_avg + mean(conv_ms)) * 1e-3) / 1e12},
            "step_ms_median": statistics.median(step_ms),
            "wall_ms_per_step_incl_flush": 1e3 * wall / args.steps,
        },
        "e2e": {"value": job_throughput(world, STEP_FLOPS, e2e_ms), "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "pipelined": "2 buffer sets, input/compute/result streams",
                "h2d_bytes_per_step": 4 * nbytes,
                "d2h_bytes_per_step": 3 * nbytes},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if causal:
        line["config"]["flop_count"] = "causal: half of 4*B*H*N^2*d forward, 2.5x that backward"
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = (cpu_baseline_causal if causal else cpu_baseline)(args.cpu_seconds)
        if not causal:
            line["cpu_baseline"]["parity_sample"] = parity_sample(q_h, k_h, v_h, do_h, o, lse, dq, scale)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_softmax(args):
    """Fused row softmax over the B*H*N x N score matrix of standard attention."""
    import torch

    import exact_attention_30_gb300 as fa

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.load_library()
    dtype = torch.bfloat16 if args.dtype == "bf16" else torch.float32
    rows, cols = B * H * N, N
    g = torch.Generator().manual_seed(0)
    x = (torch.randn(rows, cols, generator=g, dtype=torch.float32) * 4).to(dtype).to(dev)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        fa.fa_softmax_rows(x, scale=1.0, out=y)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for e0, e1 in ev:
        e0.record(stream)
        fa.fa_softmax_rows(x, scale=1.0, out=y)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    nbytes = 2 * x.numel() * x.element_size()
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, src = read_peaks()
    line = {
        "metric": "fused row softmax GB/s (HBM-bound)", "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
        "data": "synthetic",
        "config": {"workload": f"row softmax of the {rows} x {cols} score matrix "
                               f"(B={B} H={H} N={N}), {args.dtype} in and out",
                   "l2": "input and output each larger than L2"},
        "roofline": {"kernel": "softmax_warp_kernel" if cols <= 2048 else "softmax_block_kernel",
                     "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": f"{src} copy bandwidth",
                     "algorithmic_bytes_per_launch": nbytes},
        "gpu_launches": args.steps,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_softmax(args.cpu_seconds, cols, args.dtype)
    print(json.dumps(line), flush=True)
    return 0


def cpu_baseline_softmax(seconds: float, cols: int, dtype: str):
    """The oracle's row softmax (fp64) on seeded blocks of 256 rows of the same
    width; bytes counted as the GPU line counts them (each row read and written
    once in the line's dtype)."""
    import numpy as np
    import torch

    from oracle import row_softmax
    es = 2 if dtype == "bf16" else 4
    rows_done, blk = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or blk == 0:
        g = torch.Generator().manual_seed(blk)
        x = (torch.randn(256, cols, generator=g, dtype=torch.float32) * 4)
        row_softmax(x.to(torch.float64).numpy())
        rows_done += 256
        blk += 1
    dt = time.perf_counter() - t0
    return {"value": rows_done * cols * 2 * es / dt / 1e9, "unit": "GB/s", "cores": blas_threads(),
            "kind": "oracle", "sample": f"fp64 numpy oracle row softmax of {rows_done} rows x {cols} "
                                        f"columns, {dt:.1f} s (input generation included)"}


def cpu_baseline_decode(seconds: float, w):
    """The oracle (the plain definition over all cached keys) on seeded single
    heads of the decode workload's shape; bytes counted like the GPU line (K
    and V of each head once)."""
    import torch

    from exact_attention_30_gb300.inputs import random_qkv
    from oracle import attention_fwd
    heads = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or heads == 0:
        q, k, v, _ = random_qkv(1, 1, w.Nq, w.d, torch.bfloat16, seed=heads, with_do=False,
                                big_key_every=64, n_k=w.Nk)
        f = lambda t: t[0, 0].to(torch.float64).numpy()
        attention_fwd(f(q), f(k), f(v), w.scale)
        heads += 1
    dt = time.perf_counter() - t0
    return {"value": heads * 4.0 * w.Nk * w.d / dt / 1e9, "unit": "GB/s", "cores": blas_threads(),
            "kind": "oracle", "sample": f"fp64 numpy oracle decode of {heads} seeded head(s) "
                                        f"(Nq={w.Nq}, Nk={w.Nk}, d={w.d}), {dt:.1f} s (input generation included)"}


def run_decode(args):
    """KV-cache decode (fa_decode: split kernel + combine kernel) on a named workload."""
    import torch

    import exact_attention_30_gb300 as fa
    from exact_attention_30_gb300.inputs import DECODE_WORKLOADS, decode_inputs

    w = DECODE_WORKLOADS[args.decode_workload]
    if args.decode_shape is not None:
        from exact_attention_30_gb300.inputs import DecodeWorkload
        b_, h_, nq_, nk_, d_ = args.decode_shape
        w = DecodeWorkload(f"decode_bf16_{b_}x{h_}x{nq_}x{nk_}x{d_}", b_, h_, nq_, nk_, d_)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.load_library()
    q, k, v = (t.to(dev) for t in decode_inputs(w, seed=0))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    ws = torch.empty(fa.fa_decode_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d), dtype=torch.uint8,
                     device=dev)
    splits, kps = fa.fa_decode_plan(w.B, w.H, w.Nq, w.Nk, w.d)
    stream = torch.cuda.current_stream(dev)
    call = lambda: fa.fa_decode(q, k, v, w.scale, out=o, lse=lse, workspace=ws)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for e0, e1 in ev:
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    nbytes = w.hbm_bytes()
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, src = read_peaks()
    line = {
        "metric": "KV-cache decode GB/s (HBM-bound)", "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: B={w.B} H={w.H} Nq={w.Nq} Nk={w.Nk} d={w.d}, "
                               f"{splits} key ranges of {kps}",
                   "l2": "K and V larger than L2 (no flush)",
                   "tflops": w.flops() / (ms * 1e-3) / 1e12},
        "roofline": {"kernel": "decode_split_kernel + decode_combine_kernel (one fa_decode call)",
                     "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": f"{src} copy bandwidth",
                     "algorithmic_bytes_per_launch": nbytes},
        # every fa_decode call launches two kernels: the split kernel and the combine kernel
        "gpu_launches": 2 * args.steps,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(args.cpu_seconds, w)
    print(json.dumps(line), flush=True)
    return 0


def varlen_lengths(n=16, lo=512, hi=8192, seed=0):
    """Seeded sequence lengths of the variable-length workload."""
    import numpy as np
    return [int(x) for x in np.random.default_rng(seed).integers(lo, hi + 1, size=n)]


def run_varlen(args):
    """fa_fwd_varlen + fa_bwd_varlen on a packed batch of mixed lengths."""
    import torch

    import exact_attention_30_gb300 as fa
    from exact_attention_30_gb300.inputs import random_varlen

    lens = varlen_lengths()
    Hh, Dd = 16, 128
    causal = bool(args.causal)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.load_library()
    q, k, v, do, cu = (t.to(dev) for t in random_varlen(lens, Hh, Dd, torch.bfloat16, seed=0))
    maxlen = max(lens)
    scale = 1 / math.sqrt(Dd)
    stream = torch.cuda.current_stream(dev)
    ws = torch.empty(fa.fa_bwd_varlen_workspace_bytes(len(lens), Hh, q.shape[0], maxlen, Dd),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        o, lse = fa.fa_fwd_varlen(q, k, v, cu, maxlen, scale, causal=causal)
        if ev is not None:
            ev[1].record(stream)
        fa.fa_bwd_varlen(q, k, v, o, do, lse, cu, maxlen, scale, causal=causal, workspace=ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for e in ev:
        flush.zero_()
        step(e)
    torch.cuda.synchronize(dev)
    if fa.fa_check_device_status(dev) != fa.FA_OK:
        raise RuntimeError("device status not OK")
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / len(ev)
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / len(ev)
    f = 0.5 if causal else 1.0
    fwd_flops = sum(4.0 * Hh * n * n * Dd for n in lens) * f
    step_flops = fwd_flops * 3.5
    value = step_flops / ((fwd_ms + bwd_ms) * 1e-3) / 1e12
    peaks, src = read_peaks()
    vpeak, vlabel = bf16_peak(peaks, src, None, (fwd_ms + bwd_ms) * 1e-3 * args.steps)
    line = {
        "metric": "variable-length attention fwd/bwd TFLOP/s (bf16)", "value": value, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": fwd_ms + bwd_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"packed batch of {len(lens)} sequences, lengths {lens} (seeded), "
                               f"H={Hh}, d={Dd}, {'causal' if causal else 'non-causal'}",
                   "total_rows": int(q.shape[0]), "flops_per_step": step_flops,
                   "flop_count": "sum over sequences of 4*H*n^2*d forward (half if causal), 2.5x backward",
                   "l2": "flushed before every step"},
        "components": {"fwd": {"ms": fwd_ms, "tflops": fwd_flops / (fwd_ms * 1e-3) / 1e12},
                       "bwd": {"ms": bwd_ms, "tflops": 2.5 * fwd_flops / (bwd_ms * 1e-3) / 1e12}},
        "roofline": {"kernel": "fwd_bf16_kernel + bwd stages (one step)", "bound": "tensor",
                     "achieved": value, "peak": vpeak, "unit": "TFLOP/s",
                     "frac": value / vpeak, "traffic": None,
                     "peak_source": vlabel,
                     "frac_of_burst_peak": value / peaks["bf16_tflops"], "burst_peak": peaks["bf16_tflops"],
                     "frac_of_sustained_peak": value / peaks["bf16_tflops_sustained"]},
        "gpu_launches": 4 * args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_minilab(args):
    """The mini-lab configuration (fp32, B=H=1, N=16, d=8): the forward's
    latency per call. Device time between CUDA events around each call, and
    end to end through the public API with the 1.5 KB of inputs copied in from
    pinned host memory and O, LSE read back every call."""
    import numpy as np
    import torch

    import exact_attention_30_gb300 as fa
    from exact_attention_30_gb300.inputs import minilab_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.load_library()
    q64, k64, v64 = minilab_inputs()
    to_host = lambda a: torch.from_numpy(a.astype(np.float32)).reshape(1, 1, 16, 8).pin_memory()
    qh, kh, vh = to_host(q64), to_host(k64), to_host(v64)
    q, k, v = (t.to(dev) for t in (qh, kh, vh))
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 16), dtype=torch.float32, device=dev)
    oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    scale = 1 / math.sqrt(8)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        fa.fa_fwd(q, k, v, scale, out=o, lse=lse)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for e0, e1 in ev:
        e0.record(stream)
        fa.fa_fwd(q, k, v, scale, out=o, lse=lse)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    us = sorted(1e3 * a.elapsed_time(b) for a, b in ev)  # isolated calls: host submission included
    # device time per call: 100 calls captured in a CUDA graph (no host work
    # between them), the graph replayed args.steps // 100 times
    per_graph = 100
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for _ in range(per_graph):
                fa.fa_fwd(q, k, v, scale, out=o, lse=lse)
    stream.wait_stream(side)
    graph.replay()
    torch.cuda.synchronize(dev)
    replays = max(1, args.steps // per_graph)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(replays):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    mean_us = 1e3 * e0.elapsed_time(e1) / (replays * per_graph)  # mean over the replayed calls
    # end to end: copy in, forward, read O and LSE back, every call
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        for dst, src in ((q, qh), (k, kh), (v, vh)):
            dst.copy_(src, non_blocking=True)
        fa.fa_fwd(q, k, v, scale, out=o, lse=lse)
        oh.copy_(o, non_blocking=True)
        lh.copy_(lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_us = 1e3 * e0.elapsed_time(e1) / args.steps
    line = {
        "metric": "mini-lab fp32 forward device time per call (calls replayed from a CUDA graph)",
        "value": mean_us, "unit": "us",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_us * 1e-3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "fp32 forward B=1 H=1 N=16 d=8 (default_rng(0) inputs)",
                   "isolated_call_us": {"median": us[len(us) // 2], "p10": us[len(us) // 10],
                                        "p90": us[(9 * len(us)) // 10],
                                        "note": "CUDA events around one call on an idle stream, "
                                                "host submission included"},
                   "l2": "not flushed (1.5 KB of inputs)"},
        "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": 3 * qh.numel() * 4,
                "d2h_bytes_per_step": (oh.numel() + lh.numel()) * 4},
        # one forward kernel per call: the isolated calls, the graph-replayed
        # calls and the end-to-end calls are all timed
        "gpu_launches": args.steps + replays * per_graph + args.steps,
        "launches_timed": {"isolated": args.steps, "graph_replayed": replays * per_graph,
                           "end_to_end": args.steps},
    }
    if not args.no_cpu_baseline:
        from oracle import attention_fwd  # the baseline leg may run the oracle
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < min(args.cpu_seconds, 2.0):
            O_ref, L_ref = attention_fwd(q64, k64, v64, scale)
            n += 1
        cpu_us = 1e6 * (time.perf_counter() - t0) / n
        # the last end-to-end call's O and LSE (already in host memory) against
        # the oracle's result of the same problem, at the fp32 tolerance
        err = max(float(np.abs(oh.reshape(16, 8).numpy() - O_ref).max()),
                  float(np.abs(lh.reshape(16).numpy() - L_ref).max()))
        if not err <= 1e-5:
            raise RuntimeError(f"mini-lab forward differs from the oracle by {err:.3g} (> 1e-5)")
        line["cpu_baseline"] = {"value": cpu_us, "unit": "us", "cores": 1, "kind": "oracle",
                                "sample": f"fp64 numpy oracle forward of the same 16 x 8 problem, {n} calls",
                                "max_abs_diff_vs_gpu": err}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.op == "softmax":
        return run_softmax(args)
    if args.op == "minilab":
        return run_minilab(args)
    if args.varlen:
        return run_varlen(args)
    if args.op == "decode":
        return run_decode(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
