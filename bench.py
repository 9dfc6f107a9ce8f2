"""Benchmark: bf16 forward attention on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long128k|self8k|cross4k32k|stress16381|tiny|decode32k|causal8k|
                                gqa8k|varlen16|short77]

Workload (default): long-context self-attention, BSHD, B=1, H=8,
Sq=Sk=131072, d=128, bf16 Q/K/V ~ N(0,1) from a fixed seed, scale 1/sqrt(128),
RTNA output rounding: the largest single-GPU shape. One step = one call of the
fused kernel per output rounding mode of the workload over the same inputs
(self8k runs RTNE, RTNA and RTZ). Metric: TFLOP/s counted as 4*B*H*Sq*Sk*d per
call, and the fraction of the measured dense bf16 peak. Inputs (768 MiB) exceed
the 129 MB L2; L2 is not flushed between steps. Besides the K timed steps, at
least 100 further launches are timed one by one for the launch-time
distribution (median, p5, p95).

--impl reference times the fp64 CPU oracle (test infrastructure) on the host cores
on a bounded sample of the same workload, in the same unit.
With N > 1 every rank runs its own copy of the workload on its own GPU (weak
scaling, no data exchange); rank 0 prints the max-over-ranks timing. Ranks come
from torchrun (RANK / WORLD_SIZE / LOCAL_RANK in the environment) or, when those
are unset, from N processes that bench.py starts itself (rendezvous on
127.0.0.1).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# Pin the BLAS thread count before numpy loads, so the CPU baseline states the
# number of threads it actually used.
_CPU_THREADS = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_CPU_THREADS))
os.environ.setdefault("OMP_NUM_THREADS", str(_CPU_THREADS))

import numpy as np  # noqa: E402
import torch  # noqa: E402


def _blas_threads() -> int:
    """Threads the oracle's BLAS runs with: as the BLAS reports it where
    threadpoolctl is installed, else the environment setting above (which a
    caller may have preset)."""
    try:
        from threadpoolctl import threadpool_info

        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:  # noqa: BLE001 - optional dependency
        pass
    return int(os.environ.get("OPENBLAS_NUM_THREADS", _CPU_THREADS))

METRIC = "attention fwd TFLOP/s (4·B·H·Sq·Sk·d) and % of GB300 dense bf16 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
L2_BYTES = 129e6


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = ("bf16_forward_attention_gb300/csrc/attn_fwd_kernel.cuh",
                  "bf16_forward_attention_gb300/csrc/ptx.cuh",
                  "bf16_forward_attention_gb300/csrc/attn_fwd.cu",
                  "bf16_forward_attention_gb300/csrc/splitkv_combine.cuh")


def roofline_of(flops: float, io_bytes: float, launch_s: float, peaks: dict, sustained: bool):
    """(bound, achieved, peak, unit) of one launch. The bound is the roofline that
    caps the workload's arithmetic intensity (counted flops per algorithmic byte):
    below the ridge (dense bf16 peak / HBM bandwidth) it is HBM, reported in GB/s
    of algorithmic bytes; above it, the tensor pipe, in counted TFLOP/s."""
    tflops = float(peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"])
    gbs = float(peaks["hbm_gbs"])
    ridge = tflops * 1e12 / (gbs * 1e9)
    if flops / io_bytes < ridge:
        return "hbm", io_bytes / launch_s / 1e9, gbs, "GB/s"
    return "tensor", flops / launch_s / 1e12, tflops, "TFLOP/s"


def kernel_sources_hash() -> str:
    """sha256 (16 hex) of the kernel sources with comments and whitespace removed,
    so that only a change that can alter the compiled kernel makes it differ."""
    import hashlib
    import re

    code = []
    for p in KERNEL_SOURCES:
        text = open(os.path.join(ROOT, p)).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        code.append(" ".join(text.split()))
    return hashlib.sha256("\n".join(code).encode()).hexdigest()[:16]


def _recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu record, if it was taken on
    the current kernel code (else None: the counters are stale)."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["attn_fwd_kernel"][workload]
        h = kernel_sources_hash()
    except (OSError, KeyError, ValueError):
        return None
    return float(rec["dram_bytes_per_launch"]) if rec.get("sources_sha256_16") == h else None


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _free_port() -> int:
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _replica_entry(rank: int, world: int, port: int, target, target_args):
    """One replica rank: the environment torchrun would have set, then target."""
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    rc = target(*target_args)
    sys.stdout.flush()
    if rc:
        raise SystemExit(rc)


def run_replicas(world: int, target, target_args=()) -> int:
    """Starts `world` processes (spawned, so none inherits a CUDA context), rank r
    on GPU r, each calling target(*target_args) with the torchrun environment set.
    Returns 0 if every rank exited 0, else 1."""
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_replica_entry, args=(r, world, port, target, target_args))
             for r in range(world)]
    for pr in procs:
        pr.start()
    # A rank that fails would leave the others waiting at a barrier: end them.
    while any(pr.is_alive() for pr in procs):
        if any(pr.exitcode not in (None, 0) for pr in procs):
            for pr in procs:
                if pr.is_alive():
                    pr.terminate()
            break
        time.sleep(0.2)
    for pr in procs:
        pr.join()
    return 0 if all(pr.exitcode == 0 for pr in procs) else 1


def max_over_ranks(x: float, dist, device=None) -> float:
    """Max of a per-rank float over the process group (the job is as slow as its
    slowest rank). Works with NCCL (device tensor) and gloo (CPU tensor)."""
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons every 200 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                stamp, frac = (parts[0].split(".") + ["0"])[:2]
                ts = time.mktime(time.strptime(stamp, "%Y/%m/%d %H:%M:%S")) + float("0." + frac)
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        reasons = sorted({n for r in use for n, v in zip(self.REASONS, r[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": reasons, "samples": len(use),
                "window": "timed region" if inside else "whole run (timed region shorter than a sample)"}


def _cpu_sample(w, q, k, v, budget_s: float):
    """The oracle on host cores: whole row blocks of successive heads until the
    time budget is used. Returns (flops counted, seconds, rows)."""
    from oracle import attention_rows_fp64, bf16_bits_to_f64, to_bhsd
    from bf16_forward_attention_gb300 import inputs

    scale = inputs.default_scale()
    if w.seqlens:
        return _cpu_sample_varlen(w, q, k, v, budget_s, scale)
    qb, kb, vb = (to_bhsd(t.view(torch.int16).numpy(), w.layout) for t in (q, k, v))
    rows_done, pairs, t_used, i = 0, 0, 0.0, 0
    block = 256
    group = w.H // w.kv_heads
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    while t_used < budget_s:
        b, h = heads[i % len(heads)]
        r0 = ((i // len(heads)) * block) % w.Sq
        rows = np.arange(r0, min(w.Sq, r0 + block))
        kh, vh = bf16_bits_to_f64(kb[b, h // group]), bf16_bits_to_f64(vb[b, h // group])
        qh = bf16_bits_to_f64(qb[b, h])
        t0 = time.perf_counter()
        attention_rows_fp64(qh, kh, vh, scale, rows, causal=w.causal)
        t_used += time.perf_counter() - t0
        rows_done += rows.size
        pairs += (int(np.clip(rows + (w.Sk - w.Sq) + 1, 0, w.Sk).sum()) if w.causal
                  else rows.size * w.Sk)
        i += 1
    return 4.0 * pairs * w.D, t_used, rows_done


def _cpu_sample_varlen(w, q, k, v, budget_s, scale):
    """The oracle on a packed variable-length batch: blocks of rows of successive
    (sequence, head) pairs, each against its sequence's keys."""
    from oracle import attention_rows_fp64, bf16_bits_to_f64

    cq, ck = w.cu_seqlens
    qn, kn, vn = (t.view(torch.int16).numpy() for t in (q, k, v))
    group = w.H // w.kv_heads
    items = [(b, h) for b in range(w.B) for h in range(w.H) if cq[b + 1] > cq[b] and ck[b + 1] > ck[b]]
    rows_done, pairs, t_used, i = 0, 0, 0.0, 0
    while t_used < budget_s:
        b, h = items[i % len(items)]
        sq, sk = int(cq[b + 1] - cq[b]), int(ck[b + 1] - ck[b])
        r0 = ((i // len(items)) * 256) % sq
        rows = np.arange(r0, min(sq, r0 + 256))
        qh = bf16_bits_to_f64(qn[cq[b]:cq[b + 1], h])
        kh = bf16_bits_to_f64(kn[ck[b]:ck[b + 1], h // group])
        vh = bf16_bits_to_f64(vn[ck[b]:ck[b + 1], h // group])
        t0 = time.perf_counter()
        attention_rows_fp64(qh, kh, vh, scale, rows, causal=w.causal)
        t_used += time.perf_counter() - t0
        rows_done += rows.size
        pairs += (int(np.clip(rows + (sk - sq) + 1, 0, sk).sum()) if w.causal else rows.size * sk)
        i += 1
    return 4.0 * pairs * w.D, t_used, rows_done


def _env_record(dev):
    """Versions and GPU state the numbers were taken with."""
    import subprocess

    def run(cmd):
        try:
            return subprocess.run(cmd, capture_output=True, text=True, timeout=20,
                                  cwd=ROOT).stdout.strip() or None
        except (OSError, subprocess.SubprocessError):
            return None

    props = torch.cuda.get_device_properties(dev)
    nvcc = run(["nvcc", "--version"])
    return {
        "git": run(["git", "rev-parse", "--short", "HEAD"]),
        "torch": torch.__version__, "cuda_runtime": torch.version.cuda,
        "nvcc": nvcc.splitlines()[-1] if nvcc else None,
        "driver": run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                       "-i", str(dev.index or 0)]),
        "sm_count": props.multi_processor_count,
        "compute_capability": f"{props.major}.{props.minor}",
        "kernel_code_hash": kernel_sources_hash(),
    }


def _keys_seen(w):
    return f"its visible keys of {w.Sk} (causal)" if w.causal else f"all {w.Sk} keys"


def _config(w, world):
    big = 3 * 2 * w.B * w.H * max(w.Sq, w.Sk) * w.D > L2_BYTES
    if w.seqlens:
        lens = [a for a, _ in w.seqlens]
        return {"workload": f"{w.name}: variable-length self-attention fwd, packed tokens "
                            f"(token, head, d), {w.B} sequences of {min(lens)}..{max(lens)} tokens "
                            f"({sum(lens)} in all), H={w.H}, d={w.D}"
                            + (", causal mask" if w.causal else "")
                            + f", rounding {'/'.join(m.upper() for m in w.roundings)}",
                "layout": "packed", "B": w.B, "H": w.H, "H_kv": w.kv_heads, "d": w.D,
                "seqlens": lens, "causal": w.causal, "roundings": list(w.roundings),
                "calls_per_step": len(w.roundings), "qk_dist": f"N(0,{w.qk_std:g}^2)",
                "v_dist": "N(0,1)", "seed": w.seed,
                "l2": "inputs larger than L2 (not flushed)",
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    return {"workload": f"{w.name}: {'self' if w.Sq == w.Sk else 'cross'}-attention fwd, "
                        f"{w.layout.upper()}, B={w.B}, H={w.H}, Sq={w.Sq}, Sk={w.Sk}, d={w.D}, "
                        + (f"{w.kv_heads} key/value heads, " if w.kv_heads != w.H else "")
                        + ("causal mask, " if w.causal else "")
                        + f"rounding {'/'.join(m.upper() for m in w.roundings)}",
            "layout": w.layout, "B": w.B, "H": w.H, "Sq": w.Sq, "Sk": w.Sk, "d": w.D,
            "H_kv": w.kv_heads, "causal": w.causal,
            "roundings": list(w.roundings), "calls_per_step": len(w.roundings),
            "qk_dist": f"N(0,{w.qk_std:g}^2)", "v_dist": "N(0,1)" if w.v_dist == "normal" else "U(-1,1)",
            "specials": w.specials, "seed": w.seed,
            "l2": "inputs larger than L2 (not flushed)" if big else "inputs fit in L2 (not flushed)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args, w):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    from bf16_forward_attention_gb300 import inputs

    q, k, v = inputs.make_qkv(w)
    # Each step is a bounded sample of the workload; the whole run stays near
    # 150 s of CPU work whatever --steps and --warmup are.
    n = max(1, args.warmup + args.steps)
    step_s = args.ref_step_seconds if args.ref_step_seconds else min(10.0, max(0.5, 150.0 / n))
    done = []
    for i in range(args.warmup + args.steps):
        f, t, rows = _cpu_sample(w, q, k, v, budget_s=step_s)
        if i >= args.warmup:
            done.append((f, t, rows))
    t_total = sum(t for _, t, _ in done)
    value = sum(f for f, _, _ in done) / t_total / 1e12
    rows = sum(r for _, _, r in done)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / max(1, len(done)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
                         "sample": f"{rows} query rows of the workload, each against {_keys_seen(w)} "
                                   f"(~{step_s:.2g} s of fp64 CPU work per step)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    world, rank, local = _dist()
    import bf16_forward_attention_gb300 as attn
    from bf16_forward_attention_gb300 import inputs

    attn.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    q_h, k_h, v_h = inputs.make_qkv(w)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    outs = {m: torch.empty_like(q) for m in w.roundings}
    stream = torch.cuda.current_stream(dev)
    flops_call = float(w.flops)
    splits, workspace = 1, None
    if w.splitkv:
        splits = attn.splitkv_num_splits(w.B, w.H, w.Sq, w.Sk)
        workspace = torch.empty(max(16, attn.splitkv_workspace_bytes(w.B, w.H, w.Sq, w.Sk, splits)),
                                dtype=torch.uint8, device=dev)
    launches_per_call = 2 if splits > 1 else 1
    split_tail = args.split_tail and splits == 1 and not w.causal and not w.seqlens
    if split_tail:
        # The full waves and the pairs are separate launches (one of them when
        # the call is a single partial wave of pairs, or has no pairs).
        pairs = attn.split_tail_items(w.B, w.H, w.Sq, w.Sk)
        if pairs < 0:
            raise attn.AttnError(pairs, attn.status_str(pairs))
        n_items = w.B * w.H * -(-w.Sq // 256)
        launches_per_call = 2 if 0 < pairs < n_items else 1

    cu_dev = None
    if w.seqlens:
        cu_dev = tuple(torch.from_numpy(a).to(dev) for a in w.cu_seqlens)
        max_sq = max(a for a, _ in w.seqlens)

    def call(qq, kk, vv, m, out=None, cu=None):
        if w.seqlens:
            cqd, ckd = cu if cu is not None else cu_dev
            return attn.attn_fwd_varlen(qq, kk, vv, cqd, ckd, max_sq, causal=w.causal, rounding=m,
                                        out=out)
        if splits > 1:
            return attn.attn_fwd_splitkv(qq, kk, vv, num_splits=splits, layout=w.layout,
                                         rounding=m, out=out, workspace=workspace)
        if w.causal or w.kv_heads != w.H or split_tail:
            return attn.attn_fwd_ex(qq, kk, vv, causal=w.causal, layout=w.layout, rounding=m,
                                    out=out, split_tail=split_tail)
        return attn.attn_fwd(qq, kk, vv, layout=w.layout, rounding=m, out=out)

    def step():
        for m in w.roundings:
            call(q, k, v, m, outs[m])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if attn.attn_fwd_last_error() != attn.ATTN_OK:
        raise RuntimeError("a device-side wait timed out during warm-up")

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
        time.sleep(0.6)  # nvidia-smi takes a moment to start sampling
    n_calls = args.steps * len(w.roundings)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_calls)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.mark("t0")
    t_start.record(stream)
    i = 0
    for _ in range(args.steps):
        for m in w.roundings:
            ev[i][0].record(stream)
            call(q, k, v, m, outs[m])
            ev[i][1].record(stream)
            i += 1
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark("t1")
    if dist:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    if dist:
        elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    launch_ms = sorted(a.elapsed_time(b) for a, b in ev)
    clocks = sampler.stop() if rank == 0 else None
    if attn.attn_fwd_last_error() != attn.ATTN_OK:
        raise RuntimeError("a device-side wait timed out in the timed region")

    if rank != 0:
        dist.destroy_process_group()
        return 0

    # Launch-time distribution: the timed launches, plus single launches timed one
    # by one until there are at least --dist-launches of them (outside the timed
    # region; value and roofline use the timed region only).
    dist_ms = list(launch_ms)
    extra = max(0, args.dist_launches - len(dist_ms))
    if extra:
        evx = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(extra)]
        for i in range(extra):
            m = w.roundings[i % len(w.roundings)]
            evx[i][0].record(stream)
            call(q, k, v, m, outs[m])
            evx[i][1].record(stream)
        torch.cuda.synchronize(dev)
        dist_ms += [a.elapsed_time(b) for a, b in evx]
        if attn.attn_fwd_last_error() != attn.ATTN_OK:
            raise RuntimeError("a device-side wait timed out in the distribution launches")
    dist_ms.sort()

    # End to end through the public API, everything inside the timed region:
    # attn_fwd_host (attn_fwd_varlen_host for a packed batch), the C ABI's
    # host-buffer entries (pinned host inputs in, pinned host output back, the
    # copies overlapped with the kernels in chunks); one call per mode, each with
    # its own stream and workspace, each uploading its own copy of the inputs.
    # Split-KV workloads: the inputs go up once, then one device call per mode,
    # each result read back.
    qp, kp, vp = (t.pin_memory() for t in (q_h, k_h, v_h))
    host_out = {m: torch.empty(q_h.shape, dtype=torch.bfloat16).pin_memory() for m in w.roundings}
    in_bytes = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h))
    cu_pinned = tuple(torch.from_numpy(a).pin_memory() for a in w.cu_seqlens) if w.seqlens else ()
    host_api = splits == 1

    if host_api and w.seqlens:
        cu_host = tuple(torch.from_numpy(a) for a in w.cu_seqlens)
        ws_bytes = attn.load_library().attn_fwd_varlen_host_workspace_bytes(
            w.B, w.H, w.kv_heads, q_h.shape[0], k_h.shape[0], w.D)
        e2e_ws = [torch.empty(ws_bytes, dtype=torch.uint8, device=dev) for _ in w.roundings]
        e2e_streams = [torch.cuda.Stream(dev) for _ in w.roundings]
        h2d_bytes = (in_bytes + sum(t.numel() * 4 for t in cu_host)) * len(w.roundings)

        def e2e_step():
            for i, m in enumerate(w.roundings):
                with torch.cuda.stream(e2e_streams[i]):
                    attn.attn_fwd_varlen_host(qp, kp, vp, *cu_host, causal=w.causal, rounding=m,
                                              out=host_out[m], workspace=e2e_ws[i], device=dev)
    elif host_api:
        ws_bytes = attn.host_workspace_bytes(w.B, w.H, w.kv_heads, w.Sq, w.Sk, w.D)
        e2e_ws = [torch.empty(ws_bytes, dtype=torch.uint8, device=dev) for _ in w.roundings]
        e2e_streams = [torch.cuda.Stream(dev) for _ in w.roundings]
        h2d_bytes = in_bytes * len(w.roundings)

        def e2e_step():
            for i, m in enumerate(w.roundings):
                with torch.cuda.stream(e2e_streams[i]):
                    attn.attn_fwd_host(qp, kp, vp, causal=w.causal, layout=w.layout, rounding=m,
                                       out=host_out[m], workspace=e2e_ws[i], device=dev)
    else:
        e2e_streams = []
        h2d_bytes = in_bytes + sum(t.numel() * t.element_size() for t in cu_pinned)

        def e2e_step():
            qd, kd, vd = (t.to(dev, non_blocking=True) for t in (qp, kp, vp))
            cu = tuple(t.to(dev, non_blocking=True) for t in cu_pinned) or None
            for m in w.roundings:
                host_out[m].copy_(call(qd, kd, vd, m, cu=cu), non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    e_steps = max(3, min(10, args.steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s_ in e2e_streams:
        s_.wait_event(e0)
    for _ in range(e_steps):
        e2e_step()
    for s_ in e2e_streams:
        stream.wait_stream(s_)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = e0.elapsed_time(e1) / e_steps
    e2e = {"value": flops_call * len(w.roundings) / (e_ms * 1e-3) / 1e12, "unit": UNIT,
           "ms_per_step": e_ms,
           "api": (("attn_fwd_varlen_host" if w.seqlens else "attn_fwd_host") + " (host buffers)")
                  if host_api else "device buffers + copies",
           "h2d_bytes_per_step": h2d_bytes,
           "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_out.values())}

    peaks, peak_src = _peaks()
    timed_s = elapsed_ms * 1e-3
    sustained = timed_s >= 1.0
    peak = float(peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"])
    avg_launch_ms = sum(launch_ms) / len(launch_ms)
    tflops_launch = flops_call / (avg_launch_ms * 1e-3) / 1e12
    bound, achieved, roof_peak, roof_unit = roofline_of(flops_call, w.io_bytes, avg_launch_ms * 1e-3,
                                                        peaks, sustained)
    value = world * flops_call * n_calls / timed_s / 1e12

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        f, t, rows = _cpu_sample(w, q_h, k_h, v_h, budget_s=args.cpu_seconds)
        cpu = {"value": f / t / 1e12, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
               "sample": f"{rows} query rows of the workload, each against {_keys_seen(w)} "
                         f"({t:.1f} s of fp64 CPU work)"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _config(w, world),
        "pct_of_dense_bf16_peak": 100.0 * tflops_launch / peak,
        "launch_ms": {"median": dist_ms[len(dist_ms) // 2],
                      "p5": dist_ms[int(0.05 * (len(dist_ms) - 1))],
                      "p95": dist_ms[int(0.95 * (len(dist_ms) - 1))], "n": len(dist_ms),
                      "timed_region_mean": avg_launch_ms, "timed_region_n": len(launch_ms)},
        "roofline": {"bound": bound, "achieved": achieved, "peak": roof_peak, "unit": roof_unit,
                     "frac": achieved / roof_peak,
                     "traffic": (args.traffic if args.traffic is not None else
                                 _recorded_traffic(w.name + ("+split_tail" if split_tail else ""))),
                     "peak_kind": (f"{'sustained' if sustained else 'burst'} dense bf16 ({peak_src})"
                                   if bound == "tensor" else f"HBM copy bandwidth ({peak_src})"),
                     "algorithmic_bytes": w.io_bytes,
                     "kernel": "attn_fwd_kernel" + (" + attn_splitkv_combine" if splits > 1 else ""),
                     "note": (("achieved counts 4*d per visible (query, key) pair and head "
                               f"({w.visible_pairs} pairs per head under the causal mask) per launch"
                               if w.causal else "achieved counts 4*B*H*Sq*Sk*d per launch")
                              + "; the kernel also runs the P_lo*V product, 1.5x the counted tensor "
                                "work") if bound == "tensor" else
                             ("achieved counts the algorithmic bytes per launch (Q, K, V read once, O "
                              "written once); the workload's counted flops per byte are below the "
                              "ridge of the dense bf16 peak over HBM bandwidth")},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": n_calls * launches_per_call,
        "splits": splits,
        "split_tail": split_tail,
        "clocks": clocks,
        "gpu": torch.cuda.get_device_name(dev),
        "env": _env_record(dev),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="long128k")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=None,
                    help="fp64 CPU seconds per reference step (default: a 150 s budget for "
                         "the whole run over warmup + steps, 0.5..10 s per step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dist-launches", type=int, default=100,
                    help="launches timed one by one, after the timed steps, for the launch-time "
                         "distribution (at least the timed launches are used if more)")
    ap.add_argument("--split-tail", action="store_true",
                    help="run the device calls with ATTN_FLAG_SPLIT_TAIL (the last, partial wave "
                         "on pairs of CTAs; an item's bits then depend on the size of the call)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the kernel, from an ncu capture")
    args = ap.parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # No launcher: start the replica ranks here (one process per GPU).
        return run_replicas(args.gpus, main, (argv if argv is not None else sys.argv[1:],))
    if args.impl == "ours" and args.warmup < 3:
        args.warmup = 3
    from bf16_forward_attention_gb300 import inputs

    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
