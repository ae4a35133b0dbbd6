#!/usr/bin/env python
"""Benchmark of the Q2_K decode projection on GB300.

Headline workload: the m=1 Q2_K GEMV with bf16 activations at
N = K = 16384 (88,080,384 weight bytes), one C-ABI call per step.  The
metric is weight-stream GB/s (and us per call); the roofline fraction is
against the measured HBM copy bandwidth in MEASURED_PEAKS.json.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--all]

* Steps are timed in CUDA graphs of up to 100 C-ABI calls, with CUDA events
  on the launching stream, bracketed by a barrier and synchronize.
* L2 is defeated by cycling R weight copies with R x bytes >= 3 x L2.
* Clocks and throttle reasons are sampled with nvidia-smi during the timed
  region.
* e2e repeats the metric with host buffers: each step copies the weights
  and x from pinned host memory, calls the C ABI, and reads y back.
* cpu_baseline times the CPU oracle on a bounded sample, on one host thread and
  on every host core (threads over output rows; the line's value).
* --impl reference times the CPU oracle on the same workload on every host
  core (rank 0 only).
* --ncu-case [mv|mt|gemm|small|q3k|mmq|moe] runs a few untimed calls for a profiler
  capture and prints no JSON line: mv = the headline kernel (bf16 GEMV) and
  the q8_1 MMVQ at m=1 on the headline shape; mt = the same shape at m=8
  (the tensor-core MMVQ); gemm = the dense bf16 GEMM at m=64 and m=256,
  N=K=16384; small = one call of every other kernel at the configurations'
  shapes; q3k = the Q3_K MMVQ at m=1 and 2; mmq = the Q2_K matmul for many
  tokens at m=64 and m=256, N=K=16384; moe = the MoE step on 8 experts.
* After the headline (one GPU, --steps 1000 or more) every configuration of
  the sweep is timed with 300 calls each and added to the JSON line as
  configs_measured, with its own clock record (--no-configs skips it).  --all times them with 2000
  calls each and prints one JSON object per configuration to stderr (and to
  the file --all-out names).
With torchrun (N > 1) every rank runs an independent replica (the path is
replicated, not sharded); value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

# the headline metric: weight-stream GB/s of the m=1 Q2_K GEMV at N=K=16384
METRIC = "Q2_K GEMV weight GB/s at m=1 (fraction of ~8 TB/s HBM); µs per decode projection"
N_HEAD = K_HEAD = 16384
W_BYTES_HEAD = N_HEAD * (K_HEAD // 256) * 84
ALG_BYTES_HEAD = W_BYTES_HEAD + 2 * K_HEAD + 4 * N_HEAD  # weights + bf16 x + fp32 y
FALLBACK_HBM_GBS = 6800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1931.4)), "measured"
    return FALLBACK_HBM_GBS, 1900.0, "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    for f in ("q2k_m1.cu", "q2k_slice.cuh", "q2k_common.cuh"):
        h.update(open(os.path.join(ROOT, "mmvq_q2_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic():
    """DRAM bytes per launch of the headline kernel from the committed ncu
    summary, or None when the kernel source changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_source_sha") != kernel_source_sha():
        return None
    return d.get("dram_bytes_per_launch")


# ---- distributed plumbing (host logic, covered by gloo tests) --------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(elapsed_s: float, units: float, group=None):
    """(max elapsed over ranks, sum of units over ranks)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---- clocks -------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---- timing helpers -----------------------------------------------------------------

def graph_time(launch, steps: int, warmup: int, batch: int = 100):
    """Time exactly `steps` calls of launch(i) replayed from CUDA graphs of
    up to `batch` calls; returns (elapsed seconds, calls timed)."""
    import torch
    stream = torch.cuda.Stream()
    for i in range(3):  # eager warm-up (per-kernel attributes, lazy module load)
        with torch.cuda.stream(stream):
            launch(i)
    torch.cuda.synchronize()

    def capture(n, offset):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                launch(offset + i)
        return g

    b = min(batch, max(1, steps))
    g_main = capture(b, 0)
    tail = steps % b
    g_tail = capture(tail, b) if tail else None
    w_reps = max(1, (warmup + b - 1) // b)
    for _ in range(w_reps):
        g_main.replay()
    torch.cuda.synchronize()
    barrier()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps // b):
            g_main.replay()
        if g_tail is not None:
            g_tail.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier()
    return start.elapsed_time(end) / 1e3, steps


def copies_for(nbytes: int, l2: int) -> int:
    return max(1, -(-3 * l2 // max(1, nbytes)))


# ---- our arm ---------------------------------------------------------------------------

def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from mmvq_q2_gb300 import build as b
    b.build()
    import mmvq_q2_gb300 as q
    L = q.lib()
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 1024 * 1024))
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    hbm, _, peak_src = peaks()

    # headline workload
    W = synth.q2k_matrix(0, "sweep.W16384", N_HEAD, K_HEAD)
    x = synth.bf16_normal(0, "sweep.x1", (1, K_HEAD))
    R = copies_for(W.nbytes, l2)
    Wd0 = torch.from_numpy(W).cuda()
    Ws = [Wd0] + [Wd0.clone() for _ in range(R - 1)]
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    yd = torch.empty((1, N_HEAD), dtype=torch.float32, device="cuda")
    fn = L.q2k_gemv_bf16
    wp = [ctypes.c_void_p(w.data_ptr()) for w in Ws]
    xp, yp = ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(yd.data_ptr())

    def launch(i):
        st = fn(wp[i % R], N_HEAD, K_HEAD, xp, 1, K_HEAD, yp, N_HEAD,
                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        if st != 0:
            raise RuntimeError(f"q2k_gemv_bf16 status {st}")

    clocks = ClockSampler(gpu_id)
    clocks.start()
    elapsed, n = graph_time(launch, args.steps, args.warmup)
    ck = clocks.stop()
    t_call = elapsed / n
    tot_t, tot_bytes = aggregate(elapsed, float(n) * W_BYTES_HEAD)
    value = tot_bytes / tot_t / 1e9
    achieved = ALG_BYTES_HEAD / t_call / 1e9

    # e2e through the C ABI with host buffers
    Wh = torch.from_numpy(W).pin_memory()
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    yh = torch.empty((1, N_HEAD), dtype=torch.float32).pin_memory()
    Wdev = torch.empty_like(Wd0)
    xdev = torch.empty((1, K_HEAD), dtype=torch.int16, device="cuda")
    e_steps = min(args.steps, 200)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(max(3, min(args.warmup, 10)) + e_steps):
            if i == max(3, min(args.warmup, 10)):
                torch.cuda.synchronize()
                barrier()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(s)
            Wdev.copy_(Wh, non_blocking=True)
            xdev.copy_(xh, non_blocking=True)
            st = fn(ctypes.c_void_p(Wdev.data_ptr()), N_HEAD, K_HEAD, ctypes.c_void_p(xdev.data_ptr()), 1, K_HEAD,
                    yp, N_HEAD, ctypes.c_void_p(s.cuda_stream))
            if st != 0:
                raise RuntimeError(f"q2k_gemv_bf16 status {st}")
            yh.copy_(yd, non_blocking=True)
        e1.record(s)
    torch.cuda.synchronize()
    barrier()
    e_el, e_bytes = aggregate(e0.elapsed_time(e1) / 1e3, float(e_steps) * W_BYTES_HEAD)
    e2e = {"value": e_bytes / e_el / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": int(W.nbytes + x.nbytes), "d2h_bytes_per_step": int(yh.numel() * 4),
           "us_per_step": e_el / e_steps * 1e6}

    # parity spot check of the timed output against the oracle (sampled rows)
    import oracle
    rows = np.arange(0, N_HEAD, 1021)
    ref = oracle.matvec(np.ascontiguousarray(W[rows]), len(rows), K_HEAD,
                        synth.bf16_bits_to_f32(x).astype(np.float64))
    got = yd.cpu().numpy()[0, rows]
    parity_err = float(np.max(np.abs(got - ref[0])) / np.linalg.norm(ref[0]))

    line = None
    if rank == 0:
        cpu = cpu_baseline(W, x) if ws == 1 else None
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_call * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int32 dot + f32 (Q2_K weights, bf16 activations)", "data": "synthetic",
            "config": {"workload": "q2k_gemv_bf16 m=1 N=K=16384 (Q2_K weights, bf16 x, f32 y)",
                       "weight_bytes": W_BYTES_HEAD, "l2": f"{R} rotating weight copies ({R * W.nbytes >> 20} MiB > 3x L2)",
                       "graph_batch": 100, "parallelism": f"replicas x{ws}"},
            "us_per_call": t_call * 1e6,
            "tokens_per_s": 1.0 / t_call,
            "frac_of_hbm_roofline_time": (ALG_BYTES_HEAD / (hbm * 1e9)) / t_call,
            "clocks": ck,
            "e2e": e2e,
            "gpu_launches": n,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": committed_traffic(),
                         "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                         "algorithmic_bytes_per_launch": ALG_BYTES_HEAD},
            "parity_max_rel_err_sampled": parity_err,
            "cpu_baseline": cpu,
        }
    if args.all or (ws == 1 and not args.no_configs and args.steps >= 1000):
        # every configuration, timed in this run after the headline (fewer
        # calls each unless --all); clocks sampled across it.  Short runs
        # (profiler captures) leave it out, so their launches are the
        # headline's alone.
        scale = 1.0 if args.all else 0.15
        sampler = ClockSampler(gpu_id)
        sampler.start()
        try:
            recs, err = sweep(q, L, l2, hbm, rank, args.all_out, scale=scale), None
        except Exception as ex:  # the headline line goes out whatever happens here
            recs, err = [], f"{type(ex).__name__}: {ex}"
        ck2 = sampler.stop()
        if line is not None:
            line["configs_measured"] = {
                "what": "every configuration of the sweep, timed in this process after the headline: CUDA graphs "
                        "of C-ABI calls, weights cycled past L2, us per call and fraction of the measured HBM peak",
                "calls_per_config": f"{max(100, int(2000 * scale))} (graphs of 100)",
                "clocks": ck2,
                "rows": {r["config"]: {"us_per_call": round(r["us_per_call"], 3), "frac_hbm": round(r["frac_hbm"], 4)}
                         for r in recs},
            }
            if err:
                line["configs_measured"]["error"] = err
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line


def host_cores() -> int:
    """Cores this process may run on (nproc)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_matvec_threads(W, xf, threads: int):
    """The oracle's matvec over the rows of W, split into `threads`
    contiguous row ranges run side by side (each range is one unchanged
    oracle call; the C call releases the GIL).  Returns y [m, rows]."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    n = W.shape[0]
    bounds = np.linspace(0, n, threads + 1).astype(int)
    parts = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]

    def one(ab):
        a, b = ab
        return oracle.matvec(np.ascontiguousarray(W[a:b]), b - a, K_HEAD, xf)

    if len(parts) == 1:
        return one(parts[0])
    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        return np.concatenate(list(ex.map(one, parts)), axis=1)


def cpu_baseline(W, x, budget_s: float = 10.0):
    """The oracle on a bounded sample of the headline workload, on one host
    thread and on every host core (threads over output rows): rows of W until
    about budget_s seconds of single-thread CPU work.  The all-cores figure
    is the line's value; `cores` is the threads it used, `host_cores` nproc."""
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    oracle_matvec_threads(W[:8], xf, 1)  # loads the oracle library
    rows = 64
    t0 = time.perf_counter()
    oracle_matvec_threads(W[:rows], xf, 1)
    t_row = (time.perf_counter() - t0) / rows
    n = int(min(N_HEAD, max(rows, budget_s / max(t_row, 1e-9))))
    t0 = time.perf_counter()
    y1 = oracle_matvec_threads(W[:n], xf, 1)
    dt1 = time.perf_counter() - t0
    nc = host_cores()
    t0 = time.perf_counter()
    yn = oracle_matvec_threads(W[:n], xf, nc)
    dtn = time.perf_counter() - t0
    assert np.array_equal(y1, yn)  # the row split leaves every row's arithmetic as it was
    gb = n * (K_HEAD // 256) * 84 / 1e9
    return {"value": gb / dtn, "unit": "GB/s", "cores": nc, "host_cores": nc, "kind": "oracle",
            "sample": f"first {n} of {N_HEAD} rows of the N=K=16384 m=1 workload, {nc} threads over rows "
                      f"({dtn:.2f} s)",
            "single_thread": {"value": gb / dt1, "unit": "GB/s", "threads": 1, "seconds": dt1}}


# ---- sweep over every configuration (--all) ------------------------------------------------

def sweep(q, L, l2, hbm, rank, all_out=None, scale=1.0):
    """Time every configuration of the sweep (graphs of C-ABI calls, weights
    cycled past L2); scale < 1 times fewer calls per configuration.  Returns
    the records."""
    import torch
    out = []

    def gt(launch, steps, warmup):
        return graph_time(launch, max(100, int(steps * scale)), max(10, int(warmup * scale)))

    def rec(name, t_call, nbytes, m, extra=None):
        d = {"config": name, "us_per_call": t_call * 1e6, "bytes_per_call": int(nbytes),
             "GBps": nbytes / t_call / 1e9, "frac_hbm": nbytes / t_call / 1e9 / hbm,
             "tokens_per_s": m / t_call}
        if extra:
            d.update(extra)
        out.append(d)
        print(json.dumps(d), file=sys.stderr, flush=True)

    cur = lambda: ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)  # noqa: E731
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    def check(st, name):
        if st != 0:
            raise RuntimeError(f"{name} status {st}")

    # cfg0 and cfg4: Q2_K GEMV / MMVQ
    shapes = [(512, 4096, (1,))] + [(n, n, (1, 2, 4, 8)) for n in (4096, 8192, 16384)]
    for N, K, ms in shapes:
        W = synth.q2k_matrix(0, f"sweep.W{N}x{K}", N, K)
        R = copies_for(W.nbytes, l2)
        W0 = torch.from_numpy(W).cuda()
        Ws = [W0] + [W0.clone() for _ in range(R - 1)]
        wp = [P(w) for w in Ws]
        for m in ms:
            x = synth.bf16_normal(0, f"sweep.x{m}.{K}", (m, K))
            xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
            xq = q.q8_1_quantize_rows(xd)
            y = torch.empty((m, N), dtype=torch.float32, device="cuda")
            nb = W.nbytes
            el, n = gt(lambda i: check(L.q2k_gemv_bf16(wp[i % R], N, K, P(xd), m, K, P(y), N, cur()), "gemv"),
                               2000, 100)
            rec(f"gemv_bf16 N={N} K={K} m={m}", el / n, nb + 2 * m * K + 4 * m * N, m)
            el, n = gt(lambda i: check(L.q2k_mmvq_q8_1(wp[i % R], N, K, P(xq), m, P(y), N, cur()), "mmvq"),
                               2000, 100)
            rec(f"mmvq_q8_1 N={N} K={K} m={m}", el / n, nb + xq.numel() + 4 * m * N, m)
        del Ws, W0
        torch.cuda.empty_cache()

    # cfg2: pair (q8_1 quantise + one launch for both)
    K = 4096
    Wa = synth.q2k_matrix(0, "cfg2.wq_a", 1024, K)
    Wb = synth.q2k_matrix(0, "cfg2.wkv", 512, K)
    R = copies_for(Wa.nbytes + Wb.nbytes, l2)
    Was = [torch.from_numpy(Wa).cuda() for _ in range(R)]
    Wbs = [torch.from_numpy(Wb).cuda() for _ in range(R)]
    for m in (1, 4, 8):
        x = synth.bf16_normal(0, f"cfg2.x{m}", (m, K))
        xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        xq = torch.empty((m, q.q8_1_row_bytes(K)), dtype=torch.uint8, device="cuda")
        ya = torch.empty((m, 1024), dtype=torch.float32, device="cuda")
        yb = torch.empty((m, 512), dtype=torch.float32, device="cuda")

        def pair(i):
            check(L.q8_1_quantize_rows(P(xd), m, K, K, P(xq), cur()), "q8")
            check(L.q2k_mmvq_pair(P(Was[i % R]), 1024, P(ya), P(Wbs[i % R]), 512, P(yb), K, P(xq), m, cur()), "pair")
        el, n = gt(pair, 2000, 100)
        rec(f"pair (q8_1 + wq_a/wkv) m={m}", el / n, Wa.nbytes + Wb.nbytes + xq.numel() + 2 * m * K + 4 * m * 1536, m)
        # the same as one call from bf16 (the q8_1 encoding inside the pair launch for m = 1)
        def pair_bf16(i):
            check(L.q2k_mmvq_pair_bf16(P(Was[i % R]), 1024, P(ya), P(Wbs[i % R]), 512, P(yb), K, P(xd), m, P(xq),
                                       cur()), "pair_bf16")
        el, n = gt(pair_bf16, 2000, 100)
        rec(f"pair from bf16 (q8_1 inside the call) m={m}", el / n,
            Wa.nbytes + Wb.nbytes + xq.numel() + 2 * m * K + 4 * m * 1536, m)
    del Was, Wbs

    # grouped (block-diagonal) wo_a MMVQ, the next row: 8 groups of 1024 rows, 2048 values per group
    G, Rg, Kg = 8, 1024, 2048
    Wg = synth.q2k_matrix(0, "grouped.wo_a", G * Rg, Kg)
    R = copies_for(Wg.nbytes, l2)
    Wgs = [torch.from_numpy(Wg).cuda() for _ in range(R)]
    for m in (1, 8):
        x = synth.bf16_normal(0, f"grouped.x{m}", (m, G * Kg))
        xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        xq = q.q8_1_quantize_rows(xd)
        yg = torch.empty((m, G * Rg), dtype=torch.float32, device="cuda")
        el, n = gt(lambda i: check(L.q2k_mmvq_grouped(P(Wgs[i % R]), G, Rg, Kg, P(xq), m, P(yg), cur()),
                                           "grouped"), 2000, 100)
        rec(f"grouped wo_a MMVQ {G}x[{Rg},{Kg}] m={m}", el / n, Wg.nbytes + xq.numel() + 4 * m * G * Rg, m)
    del Wgs

    # Q3_K twins (moe_v41/init.rs names them beside the Q2_K kernels): one matrix, and the
    # experts batches at the MoE shapes (64 experts resident, selection varies per call)
    for N, ms in ((4096, (1, 8)), (16384, (1, 2, 4, 8))):
        K = N
        W3 = synth.q3k_matrix(0, f"sweep.q3.W{N}", N, K)
        R = copies_for(W3.nbytes, l2)
        W30 = torch.from_numpy(W3).cuda()
        W3s = [W30] + [W30.clone() for _ in range(R - 1)]
        for m in ms:
            xq = q.q8_1_quantize_rows(torch.from_numpy(synth.bf16_normal(0, f"sweep.q3.x{m}", (m, K)).view(np.int16))
                                      .cuda().view(torch.bfloat16))
            y = torch.empty((m, N), dtype=torch.float32, device="cuda")
            el, n = gt(lambda i: check(L.q3k_mmvq_q8_1(P(W3s[i % R]), N, K, P(xq), m, P(y), N, cur()),
                                               "q3k"), 2000, 100)
            rec(f"q3k mmvq_q8_1 N={N} K={K} m={m}", el / n, W3.nbytes + xq.numel() + 4 * m * N, m)
        del W3s, W30
        torch.cuda.empty_cache()
    E_pool, topk, dim, inter = 64, 8, 4096, 2048
    q3 = {}
    for e in range(E_pool):
        for kind, shape in (("gate", (inter, dim)), ("up", (inter, dim)), ("down", (dim, inter))):
            q3[(kind, e)] = torch.from_numpy(synth.q3k_matrix(0, f"q3moe.{kind}{e}", *shape)).cuda()
    rng = np.random.default_rng(1)
    gu_t, dn_t = [], []
    for _ in range(32):
        sel = [int(e) for e in rng.choice(E_pool, topk, replace=False)]
        gu_t.append(q.pointer_table([q3[("gate", e)] for e in sel] + [q3[("up", e)] for e in sel]))
        dn_t.append(q.pointer_table([q3[("down", e)] for e in sel]))
    xq = q.q8_1_quantize_rows(torch.from_numpy(synth.bf16_normal(0, "q3moe.x", (1, dim)).view(np.int16))
                              .cuda().view(torch.bfloat16))
    hq = q.q8_1_quantize_rows(torch.from_numpy(synth.bf16_normal(0, "q3moe.h", (topk, inter)).view(np.int16))
                              .cuda().view(torch.bfloat16))
    y_gu = torch.empty((2 * topk, inter), dtype=torch.float32, device="cuda")
    y_dn = torch.empty((topk, dim), dtype=torch.float32, device="cuda")
    ys = torch.empty(dim, dtype=torch.float32, device="cuda")
    wd = torch.from_numpy(synth.expert_route(0, 256, topk)[1]).cuda()
    mb = inter * (dim // 256) * 110
    el, n = gt(lambda i: check(L.q3k_mmvq_experts(P(gu_t[i % 32]), 2 * topk, inter, dim, P(xq), 0, P(y_gu),
                                                          None, None, cur()), "q3k_ex"), 1000, 50)
    rec("q3k experts gate/up batch 16x[2048,4096] m=1", el / n, 2 * topk * mb, 1)
    el, n = gt(lambda i: check(L.q3k_mmvq_experts(P(dn_t[i % 32]), topk, dim, inter, P(hq), 1, P(y_dn),
                                                          P(wd), P(ys), cur()), "q3k_ex"), 1000, 50)
    rec("q3k experts down batch 8x[4096,2048] + weighted sum", el / n, topk * mb, 1, {"launches_per_call": 2})
    del q3, gu_t, dn_t
    torch.cuda.empty_cache()

    # cfg3: routed experts for one token (256 experts resident, selection varies per call)
    E_all, topk, dim, inter = 256, 8, 4096, 2048
    mats = {}
    for e in range(E_all):
        for kind, shape in (("gate", (inter, dim)), ("up", (inter, dim)), ("down", (dim, inter))):
            mats[(kind, e)] = torch.from_numpy(synth.q2k_matrix(0, f"cfg3.{kind}{e}", *shape)).cuda()
    rng = np.random.default_rng(0)
    tables = []
    for _ in range(64):
        sel = rng.choice(E_all, topk, replace=False)
        tables.append(q.pointer_table([mats[("gate", int(e))] for e in sel] + [mats[("up", int(e))] for e in sel] +
                                      [mats[("down", int(e))] for e in sel]))
    x = synth.bf16_normal(0, "cfg3.x", (1, dim))
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    _, w = synth.expert_route(0, E_all, topk)
    wd = torch.from_numpy(w).cuda()
    yo = torch.empty(dim, dtype=torch.float32, device="cuda")
    wsb = q.q2k_moe_m1_workspace_bytes(topk, dim, inter)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    el, n = gt(lambda i: check(L.q2k_moe_m1(P(tables[i % 64]), topk, dim, inter, P(xd), P(wd), P(yo), P(ws),
                                                    wsb, cur()), "moe"), 1000, 50)
    moe_bytes = 3 * topk * inter * (dim // 256) * 84
    rec("moe_m1 (8 of 256 experts, gate/up -> SwiGLU -> down)", el / n, moe_bytes, 1, {"launches_per_call": 3})
    del mats, tables
    torch.cuda.empty_cache()

    # cfg1: engram rows + GEMM m=16
    n_table = 1 << 20
    table = torch.from_numpy(synth.q2k_blocks(0, "cfg1.table", n_table)).cuda()
    ids = torch.from_numpy(synth.row_ids(0, "cfg1.ids", 128, n_table)).cuda()
    wkv = synth.bf16_normal(0, "cfg1.wkv", (20480, 2048), std=0.02)
    R = copies_for(wkv.nbytes, l2)
    wkvs = [torch.from_numpy(wkv.view(np.int16)).cuda() for _ in range(R)]
    rows = torch.empty((128, 256), dtype=torch.int16, device="cuda")
    yk = torch.empty((16, 20480), dtype=torch.float32, device="cuda")

    def engram(i):
        check(L.q2k_dequant_rows(P(table), n_table, 256, P(ids), 128, P(rows), None, cur()), "dequant")
        check(L.dense_gemm_bf16(P(rows), 16, 2048, 2048, P(wkvs[i % R]), 20480, P(yk), 20480, cur()), "gemm")
    el, n = gt(engram, 500, 20)
    rec("engram rows(128) + dense_gemm m=16 [20480x2048]", el / n, wkv.nbytes + 128 * 84 + 2 * 128 * 256 * 2 +
        16 * 20480 * 4, 16)

    # the engram chain on the device: n-gram hash of 16 tokens (3-grams, 2 layers, 4 heads) -> one
    # layer's 128 row ids -> rows -> the m = 16 GEMM (no host round trip)
    rng = np.random.default_rng(0)
    tm = torch.from_numpy(rng.integers(0, 1 << 40, size=1 << 16).astype(np.int64)).cuda()
    hc = torch.zeros(4096, dtype=torch.int64, device="cuda")
    toks = torch.from_numpy(rng.integers(0, 1 << 16, size=16).astype(np.uint32)).cuda()
    mults = torch.from_numpy(rng.integers(-(1 << 62), 1 << 62, size=(2, 3)).astype(np.int64)).cuda()
    primes = torch.full((2, 2, 4), 131071, dtype=torch.int64, device="cuda")
    offs = torch.from_numpy((np.arange(16, dtype=np.int64) % 8 * 65536).reshape(2, 8)).cuda()  # ids < 2^20
    hout = torch.empty((16, 2, 8), dtype=torch.int64, device="cuda")
    lids = torch.empty((16, 8), dtype=torch.int32, device="cuda")

    def engram_chain(i):
        check(L.q2k_engram_hash(P(tm), tm.numel(), P(hc), hc.numel(), P(toks), 16, 0, 3, 2, 4, P(mults), P(primes),
                                P(offs), 0, P(hout), P(lids), 1, None, cur()), "hash")
        check(L.q2k_dequant_rows(P(table), n_table, 256, P(lids), 128, P(rows), None, cur()), "dequant")
        check(L.dense_gemm_bf16(P(rows), 16, 2048, 2048, P(wkvs[i % R]), 20480, P(yk), 20480, cur()), "gemm")
    el, n = gt(engram_chain, 500, 20)
    rec("engram hash(16 tok) + rows(128) + dense_gemm m=16 [20480x2048]", el / n,
        wkv.nbytes + 128 * 84 + 2 * 128 * 256 * 2 + 16 * 20480 * 4, 16)
    del wkvs

    # the page's single-token engram path (engram_v41/apply.rs, `apply`: one
    # token reads `wkv_q2k`): hash of the decode token -> its 8 row ids ->
    # rows -> the Q2_K GEMV against wkv_q2k [20480, 2048]
    wq = synth.q2k_matrix(0, "engram.wkv_q2k", 20480, 2048)
    R = copies_for(wq.nbytes, l2)
    wqs = [torch.from_numpy(wq).cuda() for _ in range(R)]
    rows1 = torch.empty((8, 256), dtype=torch.int16, device="cuda")
    y1 = torch.empty((1, 20480), dtype=torch.float32, device="cuda")
    lids1 = torch.empty((1, 8), dtype=torch.int32, device="cuda")
    hout1 = torch.empty((1, 2, 8), dtype=torch.int64, device="cuda")

    def engram_one(i):
        check(L.q2k_engram_hash(P(tm), tm.numel(), P(hc), hc.numel(), P(toks), 1, 16, 3, 2, 4, P(mults), P(primes),
                                P(offs), 0, P(hout1), P(lids1), 1, None, cur()), "hash")
        check(L.q2k_dequant_rows(P(table), n_table, 256, P(lids1), 8, P(rows1), None, cur()), "dequant")
        check(L.q2k_gemv_bf16(P(wqs[i % R]), 20480, 2048, P(rows1), 1, 2048, P(y1), 20480, cur()), "gemv")
    el, n = gt(engram_one, 2000, 100)
    rec("engram one token: hash + rows(8) + q2k_gemv_bf16 [20480x2048] (wkv_q2k)", el / n,
        wq.nbytes + 8 * 84 + 2 * 8 * 256 * 2 + 20480 * 4, 1, {"launches_per_call": 3})

    # the whole engram step: the same chains, then the gate on the fp32
    # streams [T, hc=4, dim=4096] (engram_v41.rs module doc, step 4)
    qk = torch.from_numpy(np.random.default_rng(2).uniform(0.5, 1.5, (4, 4096)).astype(np.float32)).cuda()
    st1 = torch.from_numpy(np.random.default_rng(3).standard_normal((1, 4, 4096)).astype(np.float32)).cuda()
    st16 = torch.from_numpy(np.random.default_rng(4).standard_normal((16, 4, 4096)).astype(np.float32)).cuda()

    def engram_step_one(i):
        engram_one(i)
        check(L.q2k_engram_gate(P(st1), P(y1), 20480, P(qk), 1, 4, 4096, ctypes.c_float(1e-6), None, cur()), "gate")
    el, n = gt(engram_step_one, 2000, 100)
    rec("engram step one token: hash + rows(8) + q2k_gemv_bf16 (wkv_q2k) + gate [4x4096]", el / n,
        wq.nbytes + 8 * 84 + 2 * 8 * 256 * 2 + 20480 * 4 + 20480 * 4 + 3 * 4 * 4096 * 4, 1, {"launches_per_call": 4})
    del wqs
    wkvs = [torch.from_numpy(wkv.view(np.int16)).cuda() for _ in range(copies_for(wkv.nbytes, l2))]
    R = len(wkvs)

    def engram_step16(i):
        engram_chain(i)
        check(L.q2k_engram_gate(P(st16), P(yk), 20480, P(qk), 16, 4, 4096, ctypes.c_float(1e-6), None, cur()), "gate")
    el, n = gt(engram_step16, 500, 20)
    rec("engram step 16 tokens: hash + rows(128) + dense_gemm m=16 + gate [16x4x4096]", el / n,
        wkv.nbytes + 128 * 84 + 2 * 128 * 256 * 2 + 16 * 20480 * 4 * 2 + 16 * 3 * 4 * 4096 * 4, 16,
        {"launches_per_call": 4})
    del wkvs

    # cfg4: dense GEMM m in {64, 256}
    for Nn in (4096, 8192, 16384):
        Wdn = synth.bf16_normal(0, f"sweep.dense.W{Nn}", (Nn, Nn), std=0.02)
        R = copies_for(Wdn.nbytes, l2)
        Wds = [torch.from_numpy(Wdn.view(np.int16)).cuda() for _ in range(R)]
        for m in (64, 256):
            xx = torch.from_numpy(synth.bf16_normal(0, f"sweep.dense.x{m}.{Nn}", (m, Nn)).view(np.int16)).cuda()
            yy = torch.empty((m, Nn), dtype=torch.float32, device="cuda")
            el, n = gt(lambda i: check(L.dense_gemm_bf16(P(xx), m, Nn, Nn, P(Wds[i % R]), Nn, P(yy), Nn, cur()),
                                               "gemm"), 200, 10)
            flops = 2.0 * m * Nn * Nn
            rec(f"dense_gemm_bf16 m={m} N=K={Nn}", el / n, Wdn.nbytes + 2 * m * Nn + 4 * m * Nn, m,
                {"TFLOPs": flops / (el / n) / 1e12})
        del Wds
        torch.cuda.empty_cache()

    # m > 8: the Q2_K matmul on the tensor cores (weights expanded on-chip)
    for Nn in (4096, 8192, 16384):
        Wq = synth.q2k_matrix(0, f"sweep.W{Nn}x{Nn}", Nn, Nn)
        R = copies_for(Wq.nbytes, l2)
        Wqs = [torch.from_numpy(Wq).cuda() for _ in range(R)]
        for m in (64, 256):
            xx = torch.from_numpy(synth.bf16_normal(0, f"sweep.dense.x{m}.{Nn}", (m, Nn)).view(np.int16)).cuda()
            yy = torch.empty((m, Nn), dtype=torch.float32, device="cuda")
            el, n = gt(lambda i: check(L.q2k_mmq_bf16(P(Wqs[i % R]), Nn, Nn, P(xx), m, Nn, P(yy), Nn, cur()),
                                               "mmq"), 200, 10)
            flops = 2.0 * m * Nn * Nn
            rec(f"q2k_mmq_bf16 m={m} N=K={Nn}", el / n, Wq.nbytes + 2 * m * Nn + 4 * m * Nn, m,
                {"TFLOPs": flops / (el / n) / 1e12})
            xq = q.q8_1_quantize_rows(xx.view(torch.bfloat16))
            ws = torch.empty(q.q2k_mmq_q8_1_workspace_bytes(m, Nn), dtype=torch.uint8, device="cuda")
            el, n = gt(lambda i: check(L.q2k_mmq_q8_1(P(Wqs[i % R]), Nn, Nn, P(xq), m, P(yy), Nn, P(ws),
                                                              ws.numel(), cur()), "mmq8"), 200, 10)
            rec(f"q2k_mmq_q8_1 m={m} N=K={Nn}", el / n, Wq.nbytes + xq.numel() + 4 * m * Nn, m,
                {"TFLOPs": flops / (el / n) / 1e12, "launches_per_call": 2})
        del Wqs
        torch.cuda.empty_cache()

    if rank == 0 and all_out:
        with open(all_out, "w") as f:
            for d in out:
                f.write(json.dumps(d) + "\n")
    return out


# ---- reference arm: the CPU oracle -------------------------------------------------------------

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    W = synth.q2k_matrix(0, "sweep.W16384", N_HEAD, K_HEAD)
    x = synth.bf16_normal(0, "sweep.x1", (1, K_HEAD))
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    nc = host_cores()
    oracle_matvec_threads(W[:8], xf, 1)  # loads the oracle library
    t0 = time.perf_counter()
    oracle_matvec_threads(W[:16 * nc], xf, nc)
    t_row = (time.perf_counter() - t0) / (16 * nc)  # wall time per row on every core
    budget = 150.0  # seconds for warm-up + timed steps together
    rows = int(max(nc, min(N_HEAD, budget / max(1, args.steps + args.warmup) / max(t_row, 1e-9))))
    sample = np.ascontiguousarray(W[:rows])
    for _ in range(args.warmup):
        oracle_matvec_threads(sample, xf, nc)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_matvec_threads(sample, xf, nc)
    dt = time.perf_counter() - t0
    value = args.steps * rows * (K_HEAD // 256) * 84 / dt / 1e9
    desc = f"{rows} of {N_HEAD} rows of the N=K=16384 m=1 workload per step, {nc} threads over rows"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "q2k_gemv_bf16 m=1 N=K=16384 (Q2_K weights, bf16 x) - CPU oracle sample",
                   "parallelism": f"{nc} host threads"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nc, "host_cores": nc, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def _ncu_small_case(q):
    """One call of every other kernel, at the configurations' shapes: the
    engram rows + m=16 GEMM (cfg1), the pair at m=1 (cfg2, q8_1 made
    separately and inside the launch), the MoE step (cfg3, three launches),
    the standalone SwiGLU, the fused-sum expert batch and the weighted sum,
    and a dense GEMM below 16 tokens (the mma.sync kernel)."""
    import torch
    dev = lambda a: torch.from_numpy(a).cuda()
    bf = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    # cfg1: 128 engram rows of a 2^20-row table, then [16, 2048] x wkv^T
    table = dev(synth.q2k_blocks(0, "cfg1.table", 1 << 20))
    ids = dev(synth.row_ids(0, "cfg1.ids", 128, 1 << 20))
    wkv = bf(synth.bf16_normal(0, "cfg1.wkv", (20480, 2048), std=0.02))
    rows = q.q2k_dequant_rows(table, 256, ids=ids)
    q.dense_gemm_bf16(rows.view(16, 2048), wkv)
    q.dense_gemm_bf16(rows.view(16, 2048)[:8], wkv)  # m = 8: the mma.sync kernel
    # cfg2: the pair at m = 1
    Wa = dev(synth.q2k_matrix(0, "cfg2.wq_a", 1024, 4096))
    Wb = dev(synth.q2k_matrix(0, "cfg2.wkv", 512, 4096))
    x = bf(synth.bf16_normal(0, "cfg2.x1", (1, 4096)))
    xq = q.q8_1_quantize_rows(x)
    q.q2k_mmvq_pair(Wa, Wb, xq, 4096)
    q.q2k_mmvq_pair_bf16(Wa, Wb, x, 4096)
    # cfg3: 8 experts; the MoE step, then its pieces
    E, dim, inter = 8, 4096, 2048
    mats = [dev(synth.q2k_matrix(0, f"cfg3.{k}{e}", *shape)) for k, shape in
            (("gate", (inter, dim)), ("up", (inter, dim)), ("down", (dim, inter))) for e in range(E)]
    tbl = q.pointer_table(mats)
    w = torch.full((E,), 0.125, dtype=torch.float32, device="cuda")
    xm = bf(synth.bf16_normal(0, "cfg3.x", (dim,)))
    q.q2k_moe_m1(tbl, E, dim, inter, xm, w)
    gu, _ = q.q2k_mmvq_experts(q.pointer_table(mats[:2 * E]), inter, dim, q.q8_1_quantize_rows(xm.view(1, dim)))
    hq, _ = q.swiglu_q8_1_rows(gu)
    ys = torch.empty(dim, dtype=torch.float32, device="cuda")
    q.q2k_mmvq_experts(q.pointer_table(mats[2 * E:]), dim, inter, hq, x_per_matrix=True, route_w=w, y_sum=ys,
                       want_y=False)
    q.q2k_mmvq_experts(q.pointer_table(mats[2 * E:]), dim, inter, hq, x_per_matrix=True, route_w=w, y_sum=ys)


def run_ncu_case(which: str = "mv", calls: int = 3):
    """A small fixed workload for a profiler (the profiler flushes the caches
    between passes; one weight copy).  mv: `calls` eager calls of
    q2k_gemv_bf16, then of q2k_mmvq_q8_1, at m=1 N=K=16384 (88 MB of
    weights).  mt: the same at m=8.  gemm: dense_gemm_bf16 at m=64, then
    m=256, N=K=16384 (537 MB of bf16 weights), one call each.  q3k:
    `calls` calls of q3k_mmvq_q8_1 at m=1, then at m=2, then at m=8,
    N=K=16384 (115 MB of Q3_K weights).  mmq: q2k_mmq_bf16 at m=64, then m=256, N=K=16384 (88 MB
    of Q2_K weights), one call each.  moe: `calls` calls of q2k_moe_m1 on
    the configuration's 8 selected experts (66 MB)."""
    import torch
    from mmvq_q2_gb300 import build as b
    b.build()
    import mmvq_q2_gb300 as q
    if which == "small":
        _ncu_small_case(q)
        torch.cuda.synchronize()
        print("ncu case done", file=sys.stderr)
        return
    if which == "q3k":
        W = synth.q3k_matrix(0, "sweep.q3.W16384", N_HEAD, K_HEAD)
        Wd = torch.from_numpy(W).cuda()
        for m in (1, 2, 8):
            x = synth.bf16_normal(0, f"sweep.q3.x{m}", (m, K_HEAD))
            xq = q.q8_1_quantize_rows(torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16))
            for _ in range(calls):
                q.q3k_mmvq_q8_1(Wd, xq, K_HEAD)
        torch.cuda.synchronize()
        print("ncu case done", file=sys.stderr)
        return
    if which == "moe":
        dim, inter, E = 4096, 2048, 8
        mats = [torch.from_numpy(synth.q2k_matrix(0, f"ncu.moe.{kind}{e}", *shape)).cuda()
                for kind, shape in (("gate", (inter, dim)), ("up", (inter, dim)), ("down", (dim, inter)))
                for e in range(E)]
        x = torch.from_numpy(synth.bf16_normal(0, "cfg3.x", (dim,)).view(np.int16)).cuda().view(torch.bfloat16)
        w = torch.full((E,), 1.0 / E, dtype=torch.float32, device="cuda")
        tbl = q.pointer_table(mats)
        for _ in range(calls):
            q.q2k_moe_m1(tbl, E, dim, inter, x, w)
        torch.cuda.synchronize()
        print("ncu case done", file=sys.stderr)
        return
    if which == "mmq":
        W = synth.q2k_matrix(0, "sweep.W16384", N_HEAD, K_HEAD)
        Wd = torch.from_numpy(W).cuda()
        for m in (64, 256):
            x = synth.bf16_normal(0, f"sweep.dense.x{m}", (m, K_HEAD))
            q.q2k_mmq_bf16(Wd, torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16))
        torch.cuda.synchronize()
        print("ncu case done", file=sys.stderr)
        return
    if which == "gemm":
        W = synth.bf16_normal(0, "sweep.dense.W", (N_HEAD, K_HEAD), std=0.02)
        Wd = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
        for m in (64, 256):
            x = synth.bf16_normal(0, f"sweep.dense.x{m}", (m, K_HEAD))
            xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
            q.dense_gemm_bf16(xd, Wd)
    else:
        m = 8 if which == "mt" else 1
        W = synth.q2k_matrix(0, "sweep.W16384", N_HEAD, K_HEAD)
        x = synth.bf16_normal(0, f"sweep.x{m}", (m, K_HEAD))
        Wd = torch.from_numpy(W).cuda()
        xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        xq = q.q8_1_quantize_rows(xd)
        for _ in range(calls):
            q.q2k_gemv_bf16(Wd, xd)
        for _ in range(calls):
            q.q2k_mmvq_q8_1(Wd, xq, K_HEAD)
    torch.cuda.synchronize()
    print("ncu case done", file=sys.stderr)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--all", action="store_true")
    ap.add_argument("--all-out", default=None, help="also write the --all records here, one JSON object a line")
    ap.add_argument("--no-configs", action="store_true", help="skip timing the other configurations after the headline")
    ap.add_argument("--ncu-case", nargs="?", const="mv", choices=["mv", "mt", "gemm", "small", "q3k", "mmq", "moe"], default=None)
    args = ap.parse_args(argv)
    if args.ncu_case:
        run_ncu_case(args.ncu_case)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
