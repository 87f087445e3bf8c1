#!/usr/bin/env python3
"""Benchmark: exact ring attention (bf16, causal, striped, GQA) on B300.

One step = one ra_forward over the whole workload (every query shard folds
every key/value shard in ring order).  Default workload: B=1, 32 query heads
sharing 8 KV heads, S = 131072 tokens in N = 16 striped shards of 8192, D = 128,
causal.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and a
device synchronise, each step bracketed by CUDA events on the launching
stream; the inputs (1.5 GiB) are larger than L2, so no flush is needed.
Multi-GPU: every rank runs its own replica of the workload (the path needs no
exchange on one GPU per ring); value = FLOPs of all ranks / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s & tokens/s (bf16, causal-adj) at S=128K; % of BF16 tensor peak"
def kernel_name(wl, sm_count=148, l2_bytes=126 * 10**6):
    """The tensor-core forward instantiation ra_forward runs on the workload:
    fwd_kernel<D, LOG, SELFTEST, RAGGED, MODE>, MODE the stream-K variant for
    non-causal problems with one to two work items per SM (items: pairs of
    query tiles, by head pairs when the GQA group is even), else the ring
    entered at block N-1 when the key/value blocks of the query shards the
    grid holds at once exceed the L2 (not for contiguous causal shards), else
    the ring order."""
    Sb = wl.S // wl.N
    nt = (Sb + 127) // 128
    g = wl.Hq // wl.Hkv
    per_shard = g // 2 if g % 2 == 0 else g
    per = per_shard * wl.N * (nt if g % 2 == 0 else (nt + 1) // 2)
    items = wl.B * wl.Hkv * per
    streamk = (not wl.causal) and sm_count <= items < 2 * sm_count
    ragged = "true" if Sb % 128 else "false"
    grid = min(items, sm_count)
    shards = min(wl.N, -(-grid // per_shard))
    from_last = (not (wl.causal and int(wl.striped) == 0) and wl.N > 1
                 and shards * 4 * Sb * wl.D > l2_bytes)
    mode = "kModeStreamK" if streamk else ("kModeRingFromLast" if from_last else "kModeRing")
    return f"ra::tc::fwd_kernel<{wl.D}, false, false, {ragged}, {mode}>"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="gqa_128k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ring", action="store_true",
                    help="run the workload as a real ring over the job's ranks (shard r on "
                         "rank r, K/V blocks passed between ranks); strong scaling")
    ap.add_argument("--cpu-configs", action="store_true",
                    help="time the float64 oracle in full on the four smallest workloads on all host cores, "
                         "comparing every row with the library's output; one JSON line each")
    ap.add_argument("--op", default="forward",
                    choices=["forward", "backward", "merge", "stripe", "f32", "ulysses"],
                    help="forward: the ring-attention step (default); backward: ra_backward "
                         "(dq, dk, dv) on the workload; merge / stripe: the HBM-bound helpers "
                         "on the workload's output / query tensors; f32: the fp32 SIMT path on "
                         "the workload")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms: float, device=None) -> float:
    """Largest timed duration over all ranks (no-op without a process group).

    Replicas run independently; this reduction and the barriers around the
    timed region are the only cross-rank communication of the bench."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world: int, work_per_step: float, steps: int, max_ms: float) -> float:
    """Whole-job rate: the work of all replicas over the slowest rank's time
    (work units per second)."""
    return world * work_per_step * steps / (max_ms * 1e-3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in ("exact_long_context_order_b300/csrc/ra_tc.cu",
                "exact_long_context_order_b300/csrc/ptx.cuh",
                "exact_long_context_order_b300/csrc/schedule.cuh",
                "exact_long_context_order_b300/csrc/waits.cuh",
                "exact_long_context_order_b300/csrc/tmap.h"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name):
    """DRAM bytes per launch of the forward kernel on this workload, from a
    committed ncu summary line
        traffic_bytes_per_launch[<workload name>]: <bytes> (kernel source <hash>)
    if one was taken on the current kernel source (else None)."""
    pat = re.compile(r"traffic_bytes_per_launch\[([^\]]+)\]:\s*([0-9.eE+]+)\s*"
                     r"\(kernel source ([0-9a-f]+)\)")
    pdir = os.path.join(ROOT, "profiles")
    for fn in sorted(os.listdir(pdir)) if os.path.isdir(pdir) else []:
        if not fn.endswith(".md"):
            continue
        for m in pat.finditer(open(os.path.join(pdir, fn)).read()):
            if m.group(1) == workload_name and m.group(3) == kernel_source_hash():
                return float(m.group(2))
    return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        self.dev = device_index

    def start(self):
        import tempfile
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            ident = str(self.dev)
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={ident}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:7]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        load = [r for r in rows if r[2] > 200.0] or rows  # samples under load (power)
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in load for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": float(np.median([r[0] for r in load])),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": max(r[2] for r in rows)}


# ---------------------------------------------------------------- CPU oracle sample
def cpu_oracle_sample(wl, seconds):
    """Times the float64 oracle on a bounded, stratified sample of the
    workload's query rows (each against every key it sees)."""
    import oracle
    import ragen
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from helpers import sample_rows
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        threads = os.cpu_count()
    B, Hq, Hkv, S, N, D = wl.B, wl.Hq, wl.Hkv, wl.S, wl.N, wl.D
    g = Hq // Hkv
    pos = oracle.positions(S, N, wl.striped)
    rows = sample_rows(wl.seed + 7, B, Hq, S, N, 4096)
    rng = np.random.default_rng(0)
    rng.shuffle(rows)
    flops = 0.0
    done = 0
    t_total = 0.0
    kv_cache = {}
    scale = 1.0 / math.sqrt(D)
    kept_rows, kept_o, kept_l = [], [], []
    for c0 in range(0, len(rows), 32):
        if t_total >= seconds:
            break
        chunk = rows[c0:c0 + 32]
        # group by kv head; inputs are regenerated outside the timed part
        by = {}
        for (b, h, p) in chunk:
            by.setdefault((b, h // g), []).append((b, h, p))
        for (b, kvh), rr in by.items():
            if (b, kvh) not in kv_cache:
                if len(kv_cache) * S * D * 16 > (8 << 30):
                    kv_cache.clear()
                base = (b * Hkv + kvh) * S * D
                kk = oracle.bf16_bits_to_f64(ragen.normal_bf16(wl.seed, ragen.TENSOR_K, S * D, start=base))
                vv = oracle.bf16_bits_to_f64(ragen.normal_bf16(wl.seed, ragen.TENSOR_V, S * D, start=base))
                kv_cache[(b, kvh)] = (kk.reshape(S, D), vv.reshape(S, D))
            kk, vv = kv_cache[(b, kvh)]
            qidx = [(bb * Hq + hh) * S + pp for (bb, hh, pp) in rr]
            qq = oracle.bf16_bits_to_f64(ragen.normal_bf16_rows(wl.seed, ragen.TENSOR_Q, qidx, D))
            qpos = pos[[pp for (_, _, pp) in rr]]
            t0 = time.perf_counter()
            o, l = oracle.attend_rows(qq, qpos, kk, vv, pos, wl.causal, scale)
            t_total += time.perf_counter() - t0
            kept_rows += rr
            kept_o.append(o)
            kept_l.append(l)
            vis = (qpos + 1) if wl.causal else np.full(len(rr), S)
            flops += float(4.0 * D * vis.sum())
            done += len(rr)
    return {"flops": flops, "seconds": t_total, "rows": done, "threads": threads,
            "sample_rows": kept_rows,
            "o": np.concatenate(kept_o) if kept_o else np.zeros((0, D)),
            "lse": np.concatenate(kept_l) if kept_l else np.zeros(0)}


def parity_block(r, out, lse, wl):
    """Compares the device output on the rows the CPU-baseline sample
    computed with the oracle (outside the timed region)."""
    import torch
    rows = r["sample_rows"]
    if not rows:
        return None
    idx = torch.tensor([(b * wl.Hq + h) * wl.S + p for (b, h, p) in rows], device=out.device)
    got_o = out.view(-1, wl.D)[idx].double().cpu().numpy()
    got_l = lse.view(-1)[idx].double().cpu().numpy()
    d = np.abs(got_o - r["o"])
    return {"max_abs": float(d.max()), "mean_abs": float(d.mean()),
            "lse_max_abs": float(np.abs(got_l - r["lse"]).max()), "rows": len(rows),
            "tol": {"max_abs": 2e-2, "mean_abs": 2e-3, "lse_max_abs": 2e-3},
            "rows_from": "the cpu_baseline sample (stratified over heads and shards)"}


def main_config(wl, world):
    """The `config` object of the forward bench line (both arms)."""
    return dict(wl.describe(), parallelism=f"replicas{world}",
                l2="inputs larger than L2 (no flush)",
                flops_per_step=wl.flops(), flops_exact_per_step=wl.flops_exact())


def reference_arm(args, wl):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    steps_t = []
    tot_flops = 0.0
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))  # whole run within minutes
    for s in range(args.warmup + args.steps):
        r = cpu_oracle_sample(wl, per_step)
        if s >= args.warmup:
            steps_t.append(r["seconds"])
            tot_flops += r["flops"]
            rows, threads = r["rows"], r["threads"]
    t = sum(steps_t)
    value = tot_flops / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": main_config(wl, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"float64 NumPy oracle (plain softmax attention per row) on "
                                   f"{rows} stratified query rows per step of {wl.name}, each "
                                   f"against all keys it sees; FLOPs = 4*D*visible keys"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0



# ---------------------------------------------------------------- full oracle on the small workloads
CPU_CONFIGS = ("toy_f32", "noncausal_8k", "causal_32k_contig", "causal_32k_striped")


def _oracle_slice(task):
    """One (batch, query head) slice of a workload through the float64 oracle
    (plain full attention, every row), in a spawned worker with one BLAS
    thread, compared with the device's output for that slice.  Returns
    (oracle seconds, max-abs, sum-abs, elements, lse max-abs)."""
    name, b, h, got_o, got_l = task
    import oracle
    import ragen
    wl = ragen.WORKLOADS[name]
    S, D, N = wl.S, wl.D, wl.N
    g = wl.Hq // wl.Hkv

    def slab(tid, H, hh):
        n, start = S * D, (b * H + hh) * S * D
        if wl.dtype == "bf16":
            x = oracle.bf16_bits_to_f64(ragen.normal_bf16(wl.seed, tid, n, start=start))
        else:
            x = ragen.normal_f32(wl.seed, tid, n, start=start).astype(np.float64)
        return oracle.to_token_order(x.reshape(S, D), N, wl.striped)[None, None]

    q = slab(ragen.TENSOR_Q, wl.Hq, h)
    k = slab(ragen.TENSOR_K, wl.Hkv, h // g)
    v = slab(ragen.TENSOR_V, wl.Hkv, h // g)
    t0 = time.perf_counter()
    o, lse = oracle.full_attention(q, k, v, wl.causal)
    dt = time.perf_counter() - t0
    o = oracle.to_shard_major(o[0, 0], N, wl.striped)
    lse = oracle.to_shard_major(lse[0, 0][:, None], N, wl.striped)[:, 0]
    if wl.dtype == "bf16":
        got = oracle.bf16_bits_to_f64(got_o.view(np.uint16))
    else:
        got = got_o.astype(np.float64)
    d = np.abs(got - o)
    return dt, float(d.max()), float(d.sum()), int(d.size), float(np.abs(got_l - lse).max())


def cpu_configs_arm(args):
    """The float64 oracle in full (every query row) on the four smallest workloads, on all
    host cores (one spawned worker per core, each over whole (batch, head)
    slices), each compared row by row with the library's output for the same
    inputs.  Prints one JSON line per workload."""
    import multiprocessing as mp

    import torch

    import exact_long_context_order_b300 as ra
    import ragen
    if not torch.cuda.is_available():
        raise SystemExit("--cpu-configs compares with the GPU output and needs a CUDA device")
    torch.cuda.set_device(0)
    ra.lib()
    cores = len(os.sched_getaffinity(0))
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"  # the workers' BLAS: one thread each, one worker per core
    ctx = mp.get_context("spawn")
    cpu_model = ""
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                cpu_model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    with ctx.Pool(cores) as pool:
        pool.map(abs, range(cores))  # start every worker before timing
        for name in CPU_CONFIGS:
            wl = ragen.WORKLOADS[name]
            qs, kvs = wl.shapes()
            dev = []
            for tid, shape in ((ragen.TENSOR_Q, qs), (ragen.TENSOR_K, kvs),
                               (ragen.TENSOR_V, kvs)):
                if wl.dtype == "bf16":
                    x = ragen.normal_bf16(wl.seed, tid, int(np.prod(shape))).reshape(shape)
                    dev.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16))
                else:
                    x = ragen.normal_f32(wl.seed, tid, int(np.prod(shape))).reshape(shape)
                    dev.append(torch.from_numpy(x).cuda())
            out, lse = ra.forward(*dev, wl.N, causal=wl.causal, striped=wl.striped)
            ra.check()
            o_h = (out.view(torch.int16) if wl.dtype == "bf16" else out).cpu().numpy()
            l_h = lse.double().cpu().numpy()
            tasks = [(name, b, h, o_h[b, h], l_h[b, h]) for b in range(wl.B)
                     for h in range(wl.Hq)]
            t0 = time.perf_counter()
            res = pool.map(_oracle_slice, tasks, chunksize=1)
            wall = time.perf_counter() - t0
            n_el = sum(r[3] for r in res)
            line = {
                "cpu_oracle_full": wl.name, "value": wl.flops() / wall / 1e12, "unit": "TFLOP/s",
                "cores": cores, "cpu_model": cpu_model, "wall_s": wall,
                "oracle_cpu_s": sum(r[0] for r in res), "config": wl.describe(),
                "how": "float64 NumPy oracle (oracle.full_attention, every row) per (batch, "
                       "head) slice in spawned workers, one per core, one BLAS thread each; "
                       "value = the metric's FLOPs (4*B*Hq*S^2*D, halved if causal) / wall "
                       "time of all slices",
                "parity": {"rows": wl.B * wl.Hq * wl.S, "max_abs": max(r[1] for r in res),
                           "mean_abs": sum(r[2] for r in res) / n_el,
                           "lse_max_abs": max(r[4] for r in res),
                           "against": "the library's forward (ra_forward) on the same inputs"},
            }
            print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- helper kernels
def aux_arm(args, wl):
    """Times ra_merge / ra_stripe (HBM-bound) or the fp32 SIMT forward."""
    import torch
    import exact_long_context_order_b300 as ra
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    ra.lib()
    stream = torch.cuda.current_stream()
    qs, _ = wl.shapes()
    rows = qs[0] * qs[1] * qs[2]
    D = qs[3]
    peaks, peak_src = load_peaks()
    gen = torch.Generator(device="cuda").manual_seed(wl.seed)
    if args.op == "merge":
        oa = torch.randn((rows, D), device="cuda", generator=gen).to(torch.bfloat16)
        ob = torch.randn((rows, D), device="cuda", generator=gen).to(torch.bfloat16)
        la = torch.randn((rows,), device="cuda", generator=gen)
        lb = torch.randn((rows,), device="cuda", generator=gen)
        bytes_per = rows * (3 * D * 2 + 3 * 4)  # read a, b, lse_a, lse_b; write a, lse_a

        def step():
            ra.merge(oa, la, ob, lb, stream=stream)
        name, bound_unit = "ra::aux::merge_kernel<bf16>", "GB/s"
    elif args.op == "ulysses":
        B, H, S, D = qs
        x = torch.randn((wl.N, B, H, S // wl.N, D), device="cuda", generator=gen).to(torch.bfloat16)
        y = torch.empty((wl.N, B, H // wl.N, S, D), dtype=torch.bfloat16, device="cuda")
        bytes_per = 2 * x.numel() * 2

        def step():
            ra.ulysses_exchange(x, wl.N, out=y, stream=stream)
        name, bound_unit = "ra::aux::ulysses_chunks_kernel<uint4>", "GB/s"
    elif args.op == "stripe":
        x = torch.randn(qs, device="cuda", generator=gen).to(torch.bfloat16)
        y = torch.empty_like(x)
        bytes_per = 2 * x.numel() * 2

        def step():
            ra.stripe(x, wl.N, out=y, stream=stream)
        name, bound_unit = "ra::aux::stripe_kernel<uint4>", "GB/s"
    else:
        import ragen
        # the fp32 path runs the fp32 workload unless another one was asked for
        # (then on fp32 copies of that workload's shapes)
        toy = ragen.WORKLOADS["toy_f32"] if args.workload == "gqa_128k" else wl
        qs2, kvs2 = toy.shapes()
        q = torch.randn(qs2, device="cuda", generator=gen)
        k = torch.randn(kvs2, device="cuda", generator=gen)
        v = torch.randn(kvs2, device="cuda", generator=gen)
        out = torch.empty_like(q)
        lse = torch.empty(qs2[:3], device="cuda")
        bytes_per = None
        flops = toy.flops()

        def step():
            ra.forward(q, k, v, toy.N, causal=toy.causal, striped=toy.striped, out=out, lse=lse,
                       stream=stream)
        name, bound_unit = "ra::simt::fwd_kernel<float>", "GFLOP/s"
        wl = toy
    for _ in range(args.warmup):
        step()
    ra.check(stream)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    if bytes_per is not None:
        value = bytes_per / (ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "achieved": value, "peak": peak, "unit": "GB/s",
                "frac": value / peak, "traffic": None, "kernel": name,
                "peak_source": f"{peak_src} hbm_gbs"}
        metric = f"{args.op} HBM throughput (GB/s) on {wl.name} tensors"
    else:
        value = flops / (ms * 1e-3) / 1e9
        # fp32 FMA peak from unit counts and the maximum clock: 148 SMs x 128
        # fp32 lanes x 2 FLOP per FMA x 2032 MHz
        alu_peak = 148 * 128 * 2 * 2.032e9 / 1e9
        roof = {"bound": "alu", "achieved": value, "peak": alu_peak, "unit": "GFLOP/s",
                "frac": value / alu_peak, "traffic": None, "kernel": name,
                "peak_source": "derived: 148 SMs x 128 fp32 lanes x 2 FLOP x 2032 MHz"}
        metric = f"fp32 SIMT forward GFLOP/s on {wl.name}"
    line = {"metric": metric, "value": value, "unit": bound_unit, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if args.op != "f32" else "f32", "data": "synthetic",
            "config": dict(wl.describe(), op=args.op), "gpu_launches": args.steps,
            "roofline": roof}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0

def backward_arm(args, wl):
    """Times ra_backward (delta, then the dq and dk/dv kernels) on the
    workload.  FLOPs follow the usual convention of 2.5 times the forward's
    (five tile GEMMs per visible tile pair against the forward's two); the
    two-kernel design executes seven, which the line also reports."""
    import torch
    import ragen
    import exact_long_context_order_b300 as ra
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    ra.lib()
    if wl.dtype != "bf16":
        raise SystemExit("the backward bench runs bf16 workloads")
    qs, kvs = wl.shapes()
    dev = []
    for tid, shape in ((ragen.TENSOR_Q, qs), (ragen.TENSOR_K, kvs), (ragen.TENSOR_V, kvs),
                       (ragen.TENSOR_DO, qs)):
        h = torch.empty(shape, dtype=torch.int16, pin_memory=True)
        ragen.normal_bf16(wl.seed, tid, h.numel(), out=h.numpy().reshape(-1).view(np.uint16))
        dev.append(h.to("cuda").view(torch.bfloat16))
    q, k, v, dout = dev
    stream = torch.cuda.current_stream()
    out, lse = ra.forward(q, k, v, wl.N, causal=wl.causal, striped=wl.striped, stream=stream)
    rc, need = ra.ra_backward_workspace(wl.B, wl.Hq, wl.S, wl.D)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def step():
        return ra.backward(q, k, v, out, lse, dout, wl.N, causal=wl.causal, striped=wl.striped,
                           workspace=ws, stream=stream)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):  # after the sampler's pause (see the forward arm)
        step()
    ra.check(stream)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s_ in range(args.steps):
        ev[s_][0].record(stream)
        step()
        ev[s_][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    rc = ra.ra_check(ra._stream_handle(stream))
    if rc != ra.RA_OK:
        raise SystemExit(f"device status after timed region: {ra.ra_strerror(rc)}")
    ms = t0.elapsed_time(t1) / args.steps
    call_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    flops = 2.5 * wl.flops()
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    peak_sus = float(peaks.get("bf16_tflops_sustained", peak))
    value = flops / (ms * 1e-3) / 1e12
    achieved = flops / (call_ms * 1e-3) / 1e12
    line = {
        "metric": "attention backward TFLOP/s (bf16, causal-adj, 2.5x forward FLOPs)",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(wl.describe(), op="backward", l2="inputs larger than L2 (no flush)",
                       flops_per_step=flops, executed_gemm_flops_per_step=3.5 * wl.flops()),
        "gpu_launches": 3 * args.steps,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "ra_backward: delta, ra::tcb::dq_kernel, ra::tcb::dkv_kernel",
                     "peak_source": f"{peak_src} bf16_tflops (burst)",
                     "frac_of_sustained": achieved / peak_sus,
                     "executed_frac": 1.4 * achieved / peak},
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- true ring across ranks
def ring_arm(args, wl):
    """The workload as a real ring over the ranks of this job (--ring): rank r
    holds shard r of N = world size (the workload's layout), and each step is
    ring_attention -- N calls of ra_ring_step, with each K/V block passed to
    the next rank (NCCL send/recv between GPUs) while the current one is
    folded.  With --op backward a step is a training step: the forward ring,
    then ring_attention_backward (N calls of ra_ring_step_backward, each
    block's dk/dv accumulators passed on with it), FLOPs 3.5 times the
    forward's (the forward plus the backward's usual 2.5).  The total problem
    is fixed as ranks are added (strong scaling); value = the step's FLOPs /
    the slowest rank's time."""
    import torch
    import torch.distributed as dist
    import exact_long_context_order_b300 as ra
    import ragen
    from exact_long_context_order_b300.ring import ring_attention, ring_attention_backward
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if not dist.is_initialized():
        dist.init_process_group("nccl" if world > 1 else "gloo",
                                device_id=torch.device("cuda", local) if world > 1 else None,
                                init_method=None if world > 1 else "tcp://127.0.0.1:" +
                                str(os.environ.get("MASTER_PORT", "29512")),
                                rank=rank, world_size=world)
    ra.lib()
    if wl.dtype != "bf16" or wl.S % world:
        raise SystemExit("--ring runs bf16 workloads whose S is a multiple of the rank count")
    Sb = wl.S // world
    # this rank's shard of q, k, v: i.i.d. N(0, 1) from the generator, drawn at
    # the shard's own counter range of each (batch, head) slice
    def shard(tid, H):
        h = torch.empty((wl.B, H, Sb, wl.D), dtype=torch.int16, pin_memory=True)
        flat = h.numpy().reshape(wl.B * H, Sb * wl.D)
        for bh in range(wl.B * H):
            ragen.normal_bf16(wl.seed, tid, Sb * wl.D, start=(bh * wl.S + rank * Sb) * wl.D,
                              out=flat[bh].view(np.uint16))
        return h.to("cuda").view(torch.bfloat16)
    q, k, v = shard(ragen.TENSOR_Q, wl.Hq), shard(ragen.TENSOR_K, wl.Hkv), shard(ragen.TENSOR_V,
                                                                                  wl.Hkv)
    out = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.Hq, Sb), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    train = args.op == "backward"
    dout = shard(ragen.TENSOR_DO, wl.Hq) if train else None

    def step():
        ring_attention(q, k, v, causal=wl.causal, layout=int(wl.striped), out=out, lse=lse)
        if train:
            ring_attention_backward(q, k, v, out, lse, dout, causal=wl.causal,
                                    layout=int(wl.striped))

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):  # after the sampler's pause (see the forward arm)
        step()
    ra.check(stream)
    dist.barrier()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop()
    rc = ra.ra_check(ra._stream_handle(stream))
    if rc != ra.RA_OK:
        raise SystemExit(f"device status after timed region: {ra.ra_strerror(rc)}")
    t_max = max_over_ranks(a.elapsed_time(b), device="cuda")
    step_flops = (3.5 if train else 1.0) * wl.flops()
    value = step_flops * args.steps / (t_max * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    if rank == 0:
        line = {
            "metric": ("attention training step TFLOP/s (bf16, forward + backward, 3.5x the "
                       "forward's FLOPs)") if train else METRIC,
            "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max / args.steps,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": dict(wl.describe(), parallelism=f"ring{world}", ring_devices=world,
                           tokens_per_rank=Sb, l2="inputs larger than L2 (no flush)",
                           flops_per_step=step_flops, op="backward" if train else "forward"),
            "tokens_per_s": wl.B * wl.S * args.steps / (t_max * 1e-3),
            "frac_of_bf16_peak": value / world / float(peaks["bf16_tflops"]),
            # per rank and ring step: the forward kernel; in training also the
            # delta kernel (first step), the dq and the dk/dv kernels
            "gpu_launches": args.steps * world * (world * 3 + 1 if train else world),
            "clocks": clk, "e2e": None,
            "how": "ring_attention per step: N ra_ring_step calls per rank, K/V blocks sent to "
                   "the next rank while the current block is folded" +
                   ("; then ring_attention_backward: N ra_ring_step_backward calls per rank, "
                    "each block's fp32 dk/dv accumulators sent on with it" if train else ""),
        }
        print(json.dumps(line), flush=True)
    dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------- our arm
def main():
    args = parse()
    import ragen
    wl = ragen.WORKLOADS[args.workload]
    if args.cpu_configs:
        return cpu_configs_arm(args)
    if args.impl == "reference":
        return reference_arm(args, wl)
    if args.ring:
        return ring_arm(args, wl)
    if args.op == "backward":
        return backward_arm(args, wl)
    if args.op != "forward":
        return aux_arm(args, wl)

    import torch
    import torch.distributed as dist
    import exact_long_context_order_b300 as ra

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    ra.lib()  # fail loudly if the library is missing
    props = torch.cuda.get_device_properties(local)

    dtype = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    qs, kvs = wl.shapes()
    # inputs: generated on the host (same generator as the tests), pinned
    hosts = []
    for tid, shape in ((ragen.TENSOR_Q, qs), (ragen.TENSOR_K, kvs), (ragen.TENSOR_V, kvs)):
        h = torch.empty(shape, dtype=torch.int16 if wl.dtype == "bf16" else torch.float32,
                        pin_memory=True)
        flat = h.numpy().reshape(-1)
        if wl.dtype == "bf16":
            ragen.normal_bf16(wl.seed, tid, h.numel(), out=flat.view(np.uint16))
        else:
            ragen.normal_f32(wl.seed, tid, h.numel(), out=flat)
        hosts.append(h)
    dev = [h.to("cuda").view(dtype) for h in hosts]
    q, k, v = dev
    out = torch.empty_like(q)
    lse = torch.empty(qs[:3], dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    flops = wl.flops()
    tokens = wl.B * wl.S

    def step():
        ra.forward(q, k, v, wl.N, causal=wl.causal, striped=wl.striped, out=out, lse=lse,
                   stream=stream)

    # ------------------------------------------------ device-resident timed region
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    # the warm-up runs after the sampler's start-up pause, so that the timed
    # steps do not begin on clocks that ramped down while the GPU was idle
    for _ in range(args.warmup):
        step()
    ra.check(stream)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        ev[s][0].record(stream)
        step()
        ev[s][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    rc = ra.ra_check(ra._stream_handle(stream))
    if rc != ra.RA_OK:
        raise SystemExit(f"device status after timed region: {ra.ra_strerror(rc)}")
    total_ms = t_start.elapsed_time(t_end)
    per_launch_ms = [a.elapsed_time(b) for a, b in ev]
    launch_avg_ms = float(np.mean(per_launch_ms))
    t_max = max_over_ranks(total_ms, device="cuda")
    value = aggregate_rate(world, flops, args.steps, t_max) / 1e12
    tok_s = aggregate_rate(world, tokens, args.steps, t_max)

    # ------------------------------------------------ end to end: host buffers through the C ABI
    # ra_forward_host per step: H2D copies of q, k, v, the forward, D2H of out
    # and lse, pipelined inside the call over chunks of KV-head groups.  Steps
    # also alternate between two streams with two device staging sets, so one
    # step's copies may overlap the other's kernel.
    e2e = None
    if not args.no_e2e:
        hdt = torch.int16 if wl.dtype == "bf16" else torch.float32
        outs_h = [torch.empty(qs, dtype=hdt, pin_memory=True) for _ in range(2)]
        lses_h = [torch.empty(qs[:3], dtype=torch.float32, pin_memory=True) for _ in range(2)]
        stage = [(torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                  torch.empty_like(q), torch.empty(qs[:3], dtype=torch.float32, device="cuda"))
                 for _ in range(2)]
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        h2d = sum(h.numel() * h.element_size() for h in hosts)
        d2h = outs_h[0].numel() * outs_h[0].element_size() + lses_h[0].numel() * 4
        dt = ra.RA_BF16 if wl.dtype == "bf16" else ra.RA_F32
        P = ra._ptr

        def e2e_step(i):
            sq, sk, sv, so, sl = stage[i % 2]
            rc_ = ra.ra_forward_host(P(hosts[0]), P(hosts[1]), P(hosts[2]), P(outs_h[i % 2]),
                                     P(lses_h[i % 2]), P(sq), P(sk), P(sv), P(so), P(sl), wl.B,
                                     wl.Hq, wl.Hkv, wl.S, wl.D, wl.N, int(wl.causal),
                                     int(wl.striped), 0.0, dt, ra._stream_handle(streams[i % 2]))
            if rc_ != ra.RA_OK:
                raise SystemExit(ra.ra_strerror(rc_))

        e2e_step(0)
        e2e_step(1)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        main = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        for st_ in streams:
            st_.wait_stream(main)
        for i in range(args.steps):
            e2e_step(i)
        for st_ in streams:
            main.wait_stream(st_)
        b.record(main)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(a.elapsed_time(b), device="cuda")
        e2e = {"value": aggregate_rate(world, flops, args.steps, e_ms) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms / args.steps,
               "how": "ra_forward_host per step (each call pipelines 8 chunks of KV-head "
                      "groups: copies in, forward, copies out); two caller streams and "
                      "staging sets alternate between steps"}
        # the e2e outputs must equal the device-resident run (same inputs)
        for oh in outs_h:
            if not torch.equal(oh.to("cuda").view(dtype), out):
                raise SystemExit("end-to-end output differs from the device-resident output")

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    peak_sus = float(peaks.get("bf16_tflops_sustained", peak))
    achieved = flops / (launch_avg_ms * 1e-3) / 1e12
    traffic = profiled_traffic(wl.name)
    # exponentials the softmax evaluates: one per visible (query, key) pair
    pairs = wl.B * wl.Hq * (wl.S * (wl.S + 1) / 2 if wl.causal else wl.S * wl.S)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": main_config(wl, world),
        "tokens_per_s": tok_s,
        "frac_of_bf16_peak": value / world / peak,
        "gpu_launches": args.steps,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": kernel_name(wl, props.multi_processor_count, props.L2_cache_size),
                     "peak_source": f"{peak_src} bf16_tflops (burst)",
                     "frac_of_sustained": achieved / peak_sus,
                     "launch_ms_mean": launch_avg_ms,
                     "launch_ms_median": float(np.median(per_launch_ms)),
                     "exp_per_s": pairs / (launch_avg_ms * 1e-3),
                     "hbm_gbs": (traffic / (launch_avg_ms * 1e-3) / 1e9) if traffic else None,
                     "hbm_frac": (traffic / (launch_avg_ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"]))
                     if traffic else None},
        "clocks": clk,
        "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline:
        r = cpu_oracle_sample(wl, args.cpu_seconds)
        line["parity"] = parity_block(r, out, lse, wl)
        cpu_rate = r["flops"] / r["seconds"]
        line["cpu_baseline"] = {
            "value": cpu_rate / 1e12, "unit": "TFLOP/s", "cores": r["threads"],
            "kind": "oracle",
            "sample": f"float64 NumPy oracle (plain softmax attention per row) on {r['rows']} "
                      f"stratified query rows of {wl.name}, each against all keys it sees; "
                      f"FLOPs = 4*D*visible keys; {r['seconds']:.1f} s of CPU time",
            "seconds_per_row": r["seconds"] / max(1, r["rows"]),
            # labelled extrapolation: the whole step's metric FLOPs at the
            # sample's rate (rows differ in cost; the sample is stratified)
            "extrapolated_step_s": flops / cpu_rate}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
