"""Benchmark of the block-scaled FP8 GEMM hot path on GB300.

One step = one pass of the hot path over the V3-like linear workload: the six
GEMMs M in {128, 4096} x (N, K) in {(2112, 7168), (24576, 1536), (7168, 16384)}
computed by dg_fp8_gemm_nt from operands and packed MN-major UE8M0 scales
(the pre-packed-scale path; weights B and their 128x128 scales stay resident,
as in serving).  The same step with the activation scales packed from FP32 by
dg_transform_sf inside it is reported as `with_transform`.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is whole-job TFLOP/s (2*M*N*K summed
over the six GEMMs, all ranks) with inputs resident in HBM; `e2e` is the same
metric through the public API with the activations copied from pinned host
memory and D copied back inside the timed region.  --impl reference times the
CPU oracle (fp64, all host cores) on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "block-scaled FP8 GEMM TFLOP/s and % of GB300 dense FP8 peak (1 GPU)"
UNIT = "TFLOP/s"
WORKLOAD = "dense NT V3-like linear shapes M in {128,4096} x (N,K) in {(2112,7168),(24576,1536),(7168,16384)}"
SHAPES = [(m, n, k) for m in (128, 4096) for (n, k) in ((2112, 7168), (24576, 1536), (7168, 16384))]
NOMINAL_FP8_TFLOPS = 4500.0
NOMINAL_BF16_TFLOPS = 2250.0


def flops(m, n, k):
    return 2.0 * m * n * k


def gemm_bytes(m, n, k):
    """Algorithmic bytes of one GEMM: A + B + D + logical 1-byte scales."""
    return m * k + n * k + 2 * m * n + m * (k // 128) + (n // 128) * (k // 128)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]), "hbm_gbs": float(p["hbm_gbs"]),
                "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "source": "fallback"}


def load_traffic():
    """Per-launch DRAM traffic of the GEMM kernel from an ncu capture, valid
    only while the kernel sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "gemm_dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        from block_scaled_fp8_gb300.build import source_digest
        if rec.get("source_digest") != source_digest():
            return None
        return rec
    except Exception:
        return None


def read_ncu_csv(path):
    """Launches of an ncu --csv metrics log: a list of {"kernel": name, metric:
    value in bytes / ns}, in capture order (ncu's own lines before the header
    are skipped)."""
    import csv
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9,
             "ns": 1, "nsecond": 1, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6}
    with open(path) as f:
        lines = f.read().splitlines()
    start = next(i for i, ln in enumerate(lines) if ln.startswith('"ID"'))
    launches = {}
    for row in csv.DictReader(lines[start:]):
        rec = launches.setdefault(row["ID"], {"kernel": row["Kernel Name"]})
        val = float(row["Metric Value"].replace(",", ""))
        rec[row["Metric Name"]] = val * scale.get(row["Metric Unit"], 1)
    return [launches[k] for k in sorted(launches, key=int)]


def record_traffic(capture_dir, out_path, command):
    """Writes the per-launch DRAM traffic record of the benchmark's six GEMMs
    from one ncu capture per GEMM (capture_dir/traffic_M,N,K.csv, the captured
    launch of `bench.py --case M,N,K`), stamped with the digest of the kernel
    sources this tree holds (the tree that was captured)."""
    from block_scaled_fp8_gb300.build import source_digest
    per = {}
    for (m, n, k) in SHAPES:
        launches = read_ncu_csv(os.path.join(capture_dir, f"traffic_{m},{n},{k}.csv"))
        if len(launches) != 1:
            raise RuntimeError(f"{m}x{n}x{k}: expected one captured launch, got {len(launches)}")
        x = launches[0]
        per[f"{m}x{n}x{k}"] = {"kernel": x["kernel"].split("(")[0].replace("void ", ""),
                               "bytes": int(x["dram__bytes_read.sum"] + x["dram__bytes_write.sum"]),
                               "read": int(x["dram__bytes_read.sum"]), "write": int(x["dram__bytes_write.sum"]),
                               "ncu_us": round(x["gpu__time_duration.sum"] / 1e3, 2),
                               "algorithmic_bytes": gemm_bytes(m, n, k)}
    mean = lambda keys: int(round(statistics.mean(per[k]["bytes"] for k in keys)))
    big = [f"{m}x{n}x{k}" for (m, n, k) in SHAPES if m > 128]
    small = [f"{m}x{n}x{k}" for (m, n, k) in SHAPES if m <= 128]
    rec = {"what": "dram__bytes_read.sum + dram__bytes_write.sum per launch, one ncu capture per GEMM "
                   "of the benchmark step",
           "command": command,
           "source_digest": source_digest(),
           "m4096_mean_bytes_per_launch": mean(big),
           "m128_mean_bytes_per_launch": mean(small),
           "per_gemm": per,
           "note": "m4096: the 256-row pair kernel's three launches; m128: the three M=128 GEMMs. "
                   "Writes of D still in L2 when the kernel ends are not counted. The digest is "
                   "computed by this writer from the comment-stripped kernel sources."}
    with open(out_path, "w") as f:
        json.dump(rec, f, indent=2)
        f.write("\n")
    return rec


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 10 ms; stop(t0, t1)
    keeps the samples whose nvidia-smi timestamp lies in the host wall-clock
    window [t0, t1] of the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self, t0: float, t1: float):
        import datetime
        if self.proc is None:
            return None
        time.sleep(0.05)   # let the last samples of the window arrive
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        use = inside if inside else rows
        if not use:
            return None
        reasons = sorted({n for r in use for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use),
                "window": "timed region" if inside else "whole run (no sample fell inside the timed region)"}


# --------------------------------------------------------------------- other workloads

def _time_launches(fn, flush, reps, stream):
    """Median device time (ms) of fn() over reps launches, each behind an L2
    flush, bracketed by CUDA events on the launching stream."""
    import torch
    ts = []
    for r in range(reps):
        flush.fill_(r)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def measure_other_workloads(dev, flush, reps, stream):
    """The other workloads of the method, each timed alone (not part of the
    step): C-accumulate dense GEMM, the two contiguous grouped MoE shapes and
    the masked grouped decode shape.  Inputs are drawn and quantised on the
    GPU (same recipe as the parity tests, another random stream)."""
    import torch

    from block_scaled_fp8_gb300 import binding, inputs

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = []

    def record(name, fn, fl, by, extra):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ms = _time_launches(fn, flush, reps, stream)
        cfg = binding.last_config()
        out.append({"workload": name, "us": round(ms * 1e3, 2),
                    "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                    "gbs": round(by / (ms * 1e-3) / 1e9, 1),
                    "block_m": cfg["block_m"], "block_n": cfg["block_n"], **extra})

    # dense with C accumulate, B block-scale exponents spread over 2^-8..2^4
    m, n, k = 4096, 7168, 2048
    c_ = inputs.dense_case(m, n, k, seed=2, with_c=True, b_scale_exp_range=(-8, 4), device=dev)
    sfa = binding.transform_sf(c_.sfa, 1, m)
    sfb = binding.transform_sf(c_.sfb, 128, n)
    d = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
    record(f"dense NT + C {m}x{n}x{k}",
           lambda: binding.dg_fp8_gemm_nt(c_.a, sfa, c_.b, sfb, d, c=c_.c, status=status),
           flops(m, n, k), gemm_bytes(m, n, k) + 2 * m * n, {})
    # the same GEMM given FP32 scales: the exact two-level promotion kernel
    sfa32, sfb32 = c_.sfa.contiguous(), c_.sfb.contiguous()
    record(f"dense NT + C {m}x{n}x{k}, FP32 scales (promotion)",
           lambda: binding.dg_fp8_gemm_nt(c_.a, sfa32, c_.b, sfb32, d, c=c_.c, status=status),
           flops(m, n, k), gemm_bytes(m, n, k) + 2 * m * n, {"scales": "fp32"})
    # the same GEMM with FP32 C and D
    c32 = c_.c.float()
    d32 = torch.empty(m, n, dtype=torch.float32, device=dev)
    record(f"dense NT + C {m}x{n}x{k}, FP32 C and D",
           lambda: binding.dg_fp8_gemm_nt_f32(c_.a, sfa, c_.b, sfb, d32, c=c32, status=status),
           flops(m, n, k), gemm_bytes(m, n, k) + 2 * m * n + 4 * m * n, {"d": "fp32"})
    # the same with C = D (accumulated in place at L2; D keeps growing, which the timing ignores)
    record(f"dense NT + C {m}x{n}x{k}, FP32 C = D in place",
           lambda: binding.dg_fp8_gemm_nt_f32(c_.a, sfa, c_.b, sfb, c32, c=c32, status=status),
           flops(m, n, k), gemm_bytes(m, n, k) + 2 * m * n + 4 * m * n, {"d": "fp32, in place"})
    # the same GEMM with M- / N-contiguous operands (A stored [K, M], B [K, N])
    a_t = c_.a.view(torch.uint8).t().contiguous().view(torch.float8_e4m3fn)
    b_t = c_.b.view(torch.uint8).t().contiguous().view(torch.float8_e4m3fn)
    for name, fn, a_, b_ in (("NN", binding.dg_fp8_gemm_nn, c_.a, b_t),
                             ("TN", binding.dg_fp8_gemm_tn, a_t, b_t),
                             ("TT", binding.dg_fp8_gemm_tt, a_t, c_.b)):
        record(f"dense {name} + C {m}x{n}x{k}",
               lambda fn=fn, a_=a_, b_=b_: fn(a_, sfa, b_, sfb, d, c=c_.c, status=status),
               flops(m, n, k), gemm_bytes(m, n, k) + 2 * m * n, {"layout": name.lower()})
    del c_, sfa, sfb, sfa32, sfb32, d, c32, d32, a_t, b_t

    # FP8 activations x FP4 (E2M1) weights with one scale per 32 K: the largest V3-like
    # shape and its M=128 decode form (where the weight bytes bound the time)
    for (m, n, k) in ((4096, 7168, 16384), (128, 7168, 16384)):
        fc = inputs.fp4_case(m, n, k, seed=5, device=dev)
        sfa = binding.transform_sf(fc.sfa, 1, m)
        sfb = binding.transform_sf(fc.sfb.contiguous(), 1, n)
        d = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        record(f"dense FP8 x FP4 {m}x{n}x{k}",
               lambda: binding.dg_fp8_fp4_gemm_nt(fc.a, sfa, fc.b, sfb, d, status=status),
               flops(m, n, k), m * k + n * k // 2 + 4 * (m * k // 128 + n * k // 32) // 4 + 2 * m * n,
               {"weights": "e2m1, 1x32 UE8M0 scales"})
        del fc, sfa, sfb, d

    # contiguous grouped: 8 experts, M_e ~ U[128, 4096] padded to 128
    for (n, k) in ((4096, 7168), (7168, 2048)):
        cc = inputs.contiguous_case(8, n, k, seed=3, device=dev)
        mt = cc.a.shape[0]
        sfa = binding.transform_sf(cc.sfa, 1, mt)
        sfb = binding.transform_sf(cc.sfb, 128, n)
        d = torch.empty(mt, n, dtype=torch.bfloat16, device=dev)
        valid = sum(cc.m_per_expert)
        used = sum(1 for v in cc.m_per_expert if v)
        record(f"m-grouped contiguous 8 experts N={n} K={k}",
               lambda: binding.dg_m_grouped_fp8_gemm_nt_contiguous(cc.a, sfa, cc.b, sfb, d,
                                                                   cc.grouped_layout,
                                                                   status=status),
               flops(valid, n, k), valid * k + used * n * k + 2 * valid * n,
               {"valid_rows": valid, "rows": mt})
        if n == 4096:
            # the same problem with the groups given as PSUM offsets (gap rows written 0)
            psum = torch.tensor(cc.m_per_expert, dtype=torch.int32).cumsum(0).to(torch.int32).to(dev)
            record(f"m-grouped contiguous PSUM offsets 8 experts N={n} K={k}",
                   lambda: binding.dg_m_grouped_fp8_gemm_nt_contiguous_psum(cc.a, sfa, cc.b, sfb, d, psum,
                                                                            status=status),
                   flops(valid, n, k), valid * k + used * n * k + 2 * mt * n,
                   {"valid_rows": valid, "rows": mt})
        if n == 4096:
            # the same experts with FP4 (E2M1) weights, one scale per 32 K
            fb = [inputs.fp4_case(1, n, k, seed=40 + e, device=dev) for e in range(8)]
            b4 = torch.stack([f.b for f in fb])
            sfb4 = binding.transform_sf(torch.stack([f.sfb for f in fb]).contiguous(), 1, n)
            del fb
            record(f"m-grouped contiguous FP8 x FP4 8 experts N={n} K={k}",
                   lambda: binding.dg_m_grouped_fp8_fp4_gemm_nt_contiguous(cc.a, sfa, b4, sfb4, d, cc.grouped_layout,
                                                                           status=status),
                   flops(valid, n, k), valid * k + used * n * k // 2 + 2 * valid * n,
                   {"valid_rows": valid, "rows": mt, "weights": "e2m1"})
            del b4, sfb4
        del cc, sfa, sfb, d

    # K-grouped weight gradient of the contiguous MoE layer (8 experts, N=4096 x K=7168
    # weights): D_e[4096, 7168] += dY_e^T X_e over each expert's tokens, in place in FP32
    kc = inputs.k_grouped_case(8, 4096, 7168, seed=3, device=dev)
    sfa = binding.dg_transform_sf_k_grouped(kc.sfa, kc.ks)
    sfb = binding.dg_transform_sf_k_grouped(kc.sfb, kc.ks)
    ks_dev = torch.tensor(kc.ks, dtype=torch.int32, device=dev)
    kt = sum(kc.ks)
    record(f"k-grouped weight gradient 8 groups M=4096 N=7168 K_total={kt}",
           lambda: binding.dg_k_grouped_fp8_gemm_tn_contiguous(kc.a, sfa, kc.b, sfb, kc.c, kc.ks, ks_dev=ks_dev,
                                                               c=kc.c, status=status),
           flops(4096, 7168, kt), kt * (4096 + 7168) + 2 * 4 * 8 * 4096 * 7168,
           {"d": "fp32, in place", "ks": kc.ks})
    del kc, sfa, sfb, ks_dev
    # the same weight gradient with its scales every 32 rows of K (the pages' pre-packed form)
    kc = inputs.k_grouped_case(8, 4096, 7168, seed=3, device=dev, gran_k=32)
    sfa = binding.dg_transform_sf_k_grouped_k32(kc.sfa, kc.ks)
    sfb = binding.dg_transform_sf_k_grouped_k32(kc.sfb, kc.ks)
    ks_dev = torch.tensor(kc.ks, dtype=torch.int32, device=dev)
    kt = sum(kc.ks)
    record(f"k-grouped weight gradient 8 groups M=4096 N=7168 K_total={kt}, 32-row scales",
           lambda: binding.dg_k_grouped_fp8_gemm_tn_contiguous_k32(kc.a, sfa, kc.b, sfb, kc.c, kc.ks, ks_dev=ks_dev,
                                                                   c=kc.c, status=status),
           flops(4096, 7168, kt), kt * (4096 + 7168) + 2 * 4 * 8 * 4096 * 7168,
           {"d": "fp32, in place", "ks": kc.ks, "scales": "every 32 rows of K"})
    del kc, sfa, sfb, ks_dev

    # masked grouped decode: 32 experts, max_m 256
    n, k, e, max_m = 4096, 7168, 32, 256
    mc = inputs.masked_case(e, max_m, n, k, seed=4, device=dev)
    sfa = binding.transform_sf(mc.sfa, 1, max_m)
    sfb = binding.transform_sf(mc.sfb, 128, n)
    d = torch.empty(e, max_m, n, dtype=torch.bfloat16, device=dev)
    valid = int(mc.masked_m.sum())
    used = int((mc.masked_m > 0).sum())
    record(f"m-grouped masked {e} experts max_m={max_m} N={n} K={k}",
           lambda: binding.dg_m_grouped_fp8_gemm_nt_masked(mc.a, sfa, mc.b, sfb, d, mc.masked_m,
                                                           mc.expected_m, status=status),
           flops(valid, n, k), valid * k + used * n * k + 2 * valid * n,
           {"valid_rows": valid, "bound": "hbm"})
    # the same decode with FP4 (E2M1) expert weights: half the weight bytes
    fb = [inputs.fp4_case(1, n, k, seed=80 + i, device=dev) for i in range(e)]
    b4 = torch.stack([f.b for f in fb])
    sfb4 = binding.transform_sf(torch.stack([f.sfb for f in fb]).contiguous(), 1, n)
    del fb
    record(f"m-grouped masked FP8 x FP4 {e} experts max_m={max_m} N={n} K={k}",
           lambda: binding.dg_m_grouped_fp8_fp4_gemm_nt_masked(mc.a, sfa, b4, sfb4, d, mc.masked_m, mc.expected_m,
                                                               status=status),
           flops(valid, n, k), valid * k + used * n * k // 2 + 2 * valid * n,
           {"valid_rows": valid, "bound": "hbm", "weights": "e2m1"})
    del mc, sfa, sfb, d, b4, sfb4
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the other workloads")
    return out


def measure_library_fp8_peak(dev, stream):
    """Context only: a library FP8 matmul (torch._scaled_mm, per-tensor scales)
    at 8192^3, the best of 10 back-to-back runs."""
    import torch
    try:
        n = 8192
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        best = None
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return round(2.0 * n ** 3 / (best * 1e-3) / 1e12, 1)
    except Exception as exc:  # the library may not offer an FP8 GEMM here
        return f"unavailable: {type(exc).__name__}"


# --------------------------------------------------------------------- ranks

def reduce_job_times(local_ms, world, device):
    """Maximum over ranks of each per-rank time in `local_ms` (a list, ms); every
    rank receives the same list."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(local_ms, dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_tflops(flops_per_step, steps, world, total_ms):
    """Whole-job throughput: each of `world` ranks runs `steps` steps of its own
    replica of the workload in at most `total_ms`."""
    return flops_per_step * steps * world / (total_ms * 1e-3) / 1e12


# --------------------------------------------------------------------- ours

def bind_host_to_gpu(dev_index):
    """Pin this process to the host CPUs local to the GPU (its sysfs
    local_cpulist), so that pinned host buffers allocated afterwards are placed
    on the GPU's own memory node.  Returns the CPU list, or None if unknown."""
    import torch
    try:
        pr = torch.cuda.get_device_properties(dev_index)
        addr = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{addr}/local_cpulist") as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return None
        os.sched_setaffinity(0, cpus)
        return spec
    except Exception:
        return None


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from block_scaled_fp8_gb300 import binding, build, inputs

    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    host_cpus = bind_host_to_gpu(local_rank)
    stream = torch.cuda.current_stream()

    # Problems: seeded synthetic data of the workload's shapes (rank-distinct seeds).
    probs = []
    for i, (m, n, k) in enumerate(SHAPES):
        case = inputs.dense_case(m, n, k, seed=1000 * rank + i)
        sfb = binding.transform_sf(case.sfb.to(dev), 128, n)           # weights: packed once
        p = {
            "shape": (m, n, k),
            "a": case.a.to(dev), "sfa_f32": case.sfa.to(dev), "b": case.b.to(dev), "sfb": sfb,
            "sfa": torch.empty((case.sfa.shape[1] + 3) // 4, (m + 3) // 4 * 4, dtype=torch.int32,
                               device=dev),
            "d": torch.empty(m, n, dtype=torch.bfloat16, device=dev),
            # host side for the end-to-end leg
            "a_host": case.a.pin_memory(),
            "d_host": torch.empty(m, n, dtype=torch.bfloat16).pin_memory(),
        }
        probs.append(p)
        del case
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    step_flops = sum(flops(*p["shape"]) for p in probs)
    launches_per_step = len(probs)

    gemm_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in probs]

    def step_with_transform():
        for i, p in enumerate(probs):
            m, n, k = p["shape"]
            binding.dg_transform_sf(p["sfa_f32"], 1, m, p["sfa"], status=status)
            binding.dg_fp8_gemm_nt(p["a"], p["sfa"], p["b"], p["sfb"], p["d"], status=status)

    def step():
        for p in probs:
            binding.dg_fp8_gemm_nt(p["a"], p["sfa"], p["b"], p["sfb"], p["d"], status=status)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush.fill_(1)
        step_with_transform()   # also packs every activation's scales for the step
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")
    bn_used = []
    for p in probs:
        binding.dg_fp8_gemm_nt(p["a"], p["sfa"], p["b"], p["sfb"], p["d"], status=status)
        bn_used.append(binding.last_config())
    torch.cuda.synchronize()

    # ---------------- device-timed steps (inputs resident, L2 flushed between steps)
    # The step is captured once in a CUDA graph and replayed, so host launch
    # latency never shows up as device idle time inside the timed region.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph_t = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_t):
        step_with_transform()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    barrier()
    t_wall0 = time.time()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for s in range(args.steps):
        flush.fill_(s)
        ev[s][0].record(stream)
        graph.replay()
        ev[s][1].record(stream)
    barrier()
    clocks = sampler.stop(t_wall0, time.time())
    step_ms = [a.elapsed_time(b) for a, b in ev]
    local_ms = sum(step_ms)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in timed region")
    # the same steps with the activation-scale transform inside (12 launches per step)
    ev_t = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    barrier()
    for s in range(args.steps):
        flush.fill_(s)
        ev_t[s][0].record(stream)
        graph_t.replay()
        ev_t[s][1].record(stream)
    barrier()
    local_t_ms = sum(a.elapsed_time(b) for a, b in ev_t)
    del graph_t

    # ---------------- per-kernel device time of each GEMM (the dominant kernel)
    # Each launch sits behind an L2-flush kernel, so the host enqueues it while
    # the GPU is busy and the events bracket only the GEMM.
    gemm_ms = [0.0] * len(probs)
    reps = max(3, args.steps // 2)
    for i, p in enumerate(probs):
        for r in range(reps):
            flush.fill_(r)
            gemm_ev[i][0].record(stream)
            binding.dg_fp8_gemm_nt(p["a"], p["sfa"], p["b"], p["sfb"], p["d"], status=status)
            gemm_ev[i][1].record(stream)
            torch.cuda.synchronize()
            gemm_ms[i] += gemm_ev[i][0].elapsed_time(gemm_ev[i][1]) / reps
    del graph

    # ---------------- per-kernel device time of each GEMM inside the step
    # The step's six launches captured with a timing event between launches (event
    # record nodes, so each GEMM starts when the previous one has finished), replayed
    # behind the L2 flush like the timed steps: the time between two events is one
    # GEMM's launch inside the step.  None where torch cannot record timing events in
    # a captured graph.
    step_gemm_ms = measure_step_launches(probs, flush, reps, status, stream)
    # the same with events only where the kernel changes (after the M=128 GEMMs, which
    # come first, and after the M=4096 ones): each kernel's launches keep their overlap
    n_skinny = sum(1 for p in probs if p["shape"][0] <= 128)
    assert all(p["shape"][0] <= 128 for p in probs[:n_skinny]), "the M=128 GEMMs lead the step"
    step_group_ms = measure_step_launches(probs, flush, reps, status, stream, cuts=[n_skinny, len(probs)])

    # ---------------- end to end through the public API with host buffers
    for p in probs:
        p["sfa_packed_host"] = p["sfa"].cpu().pin_memory()
    h2d = sum(p["a_host"].numel() * p["a_host"].element_size() +
              p["sfa_packed_host"].numel() * 4 for p in probs)
    d2h = sum(p["d_host"].numel() * 2 for p in probs)
    e2e_steps = min(20, max(3, args.steps // 2))
    # untimed warm-up of the end-to-end leg (first use of its pinned buffers, streams
    # and second device buffer set), then the timed steps
    e2e_pipelined(probs, max(3, args.warmup), status, stream)
    barrier()
    e2e_ms, e2e_host_ms = e2e_pipelined(probs, e2e_steps, status, stream)
    raw_copy = measure_pinned_copies(dev, stream)

    # ---------------- reductions over ranks (max time)
    total_ms, e2e_total_ms, total_t_ms = reduce_job_times([local_ms, e2e_ms, local_t_ms], world, dev)
    value = job_tflops(step_flops, args.steps, world, total_ms)
    e2e_value = job_tflops(step_flops, e2e_steps, world, e2e_total_ms)

    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * NOMINAL_FP8_TFLOPS / NOMINAL_BF16_TFLOPS
    # The dominant kernel is the CTA-pair kernel of the three M=4096 GEMMs
    # (tensor-bound); the three M=128 GEMMs run the single-CTA kernel (HBM-bound).
    big = [i for i, p in enumerate(probs) if p["shape"][0] > 128]
    skinny = [i for i, p in enumerate(probs) if p["shape"][0] <= 128]
    launch_ms = step_gemm_ms if step_gemm_ms is not None else gemm_ms
    if step_group_ms is not None:
        skinny_ms, big_ms = step_group_ms
    else:
        big_ms = sum(launch_ms[i] for i in big)
        skinny_ms = sum(launch_ms[i] for i in skinny)
    achieved = sum(flops(*probs[i]["shape"]) for i in big) / (big_ms * 1e-3) / 1e12
    skinny_gbs = sum(gemm_bytes(*probs[i]["shape"]) for i in skinny) / (skinny_ms * 1e-3) / 1e9
    other = measure_other_workloads(dev, flush, min(20, max(5, args.steps // 4)), stream) if rank == 0 else []
    lib_fp8 = measure_library_fp8_peak(dev, stream) if rank == 0 else None
    per_gemm = []
    for i, (p, ms, cfg) in enumerate(zip(probs, gemm_ms, bn_used)):
        m, n, k = p["shape"]
        lm = launch_ms[i]
        per_gemm.append({"m": m, "n": n, "k": k, "us": round(lm * 1e3, 2),
                         "tflops": round(flops(m, n, k) / (lm * 1e-3) / 1e12, 1),
                         "gbs": round(gemm_bytes(m, n, k) / (lm * 1e-3) / 1e9, 1),
                         "isolated_us": round(ms * 1e3, 2),
                         "block_n": cfg["block_n"], "grid": cfg["grid"]})
    launch_timing = ("the kernel's three launches inside the step, between CUDA events recorded before "
                     "and after them in the step's graph (replayed behind the L2 flush; the launches "
                     "between the events keep their programmatic overlap); per_gemm.us: each launch "
                     "between events after every launch; per_gemm.isolated_us: one launch alone "
                     "after the flush"
                     if step_group_ms is not None else
                     "each GEMM's launch inside the step (CUDA events between the step's launches, "
                     "replayed behind the L2 flush); per_gemm.isolated_us: one launch alone after the flush"
                     if step_gemm_ms is not None else
                     "one launch alone after the L2 flush (CUDA events around it)")
    traffic = load_traffic()
    big_traffic = skinny_traffic = None
    if traffic is not None:
        big_traffic = traffic.get("m4096_mean_bytes_per_launch")
        skinny_traffic = traffic.get("m128_mean_bytes_per_launch")

    result = None
    if rank == 0:
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8e4m3 (fp32 accumulate, bf16 out)",
            "data": "synthetic (seeded N(0,1) quantised per 1x128 / 128x128, power-of-two scales)",
            "config": {"workload": WORKLOAD, "shapes_mnk": SHAPES,
                       "step": "the six dg_fp8_gemm_nt calls with pre-packed UE8M0 scales, "
                               "replayed as one CUDA graph",
                       "l2": "flushed between steps (256 MB write)",
                       "parallelism": f"replicas x{world}"},
            "pct_of_nominal_fp8_peak": round(100.0 * value / NOMINAL_FP8_TFLOPS, 2),
            "with_transform": {
                "value": round(job_tflops(step_flops, args.steps, world, total_t_ms), 2),
                "ms_per_step": round(total_t_ms / args.steps, 4),
                "step": "dg_transform_sf of each activation's FP32 scales + dg_fp8_gemm_nt "
                        "(12 launches per step, one CUDA graph)"},
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1),
                         "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                         "frac": round(achieved / fp8_peak, 4),
                         "peak_note": f"fp8 = {peaks['source']} bf16 burst x 2 (nominal fp8/bf16 ratio), of {peaks['source']}",
                         "kernel": "dg_bs2_gemm_kernel (CTA pairs): the three M=4096 GEMMs, "
                                   "flops / the three launches' time in the step",
                         "timing": launch_timing,
                         "launches_us": round(big_ms * 1e3, 2),
                         "traffic": big_traffic},
            "roofline_skinny": {"bound": "hbm", "achieved": round(skinny_gbs, 1),
                                "peak": round(peaks["hbm_gbs"], 1), "unit": "GB/s",
                                "frac": round(skinny_gbs / peaks["hbm_gbs"], 4),
                                "kernel": "the three M=128 GEMMs (dg_bs2_gemm_kernel on 128-row CTA pairs "
                                          "where the load model prefers them, else dg_bs_gemm_kernel): "
                                          "algorithmic bytes / the three launches' time in the step, of " + peaks["source"],
                                "timing": launch_timing,
                                "launches_us": round(skinny_ms * 1e3, 2),
                                "traffic": skinny_traffic},
            "per_gemm": per_gemm,
            "other_workloads": other,
            "library_fp8_matmul_8192_tflops": lib_fp8,
            "pct_of_library_fp8_8192": (round(100.0 * value / lib_fp8, 2) if lib_fp8 else None),
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "pipeline": "per GEMM: copy A and packed scales in, dg_fp8_gemm_nt, copy D out; "
                                "D out in two row halves on two streams; two device buffer sets",
                    "host_enqueue_ms_per_step": round(e2e_host_ms / e2e_steps, 3),
                    "host_cpus": host_cpus or "unbound",
                    "raw_pinned_copy_gbs": raw_copy,
                    "copy_bound_value": (round(step_flops / (max(h2d / raw_copy["h2d"], d2h / raw_copy["d2h"]) / 1e9)
                                               / 1e12, 2) if raw_copy else None),
                    "copy_bound_note": "the TFLOP/s the step could reach if its copies were the only cost and "
                                       "the two directions overlapped completely: flops / max(h2d bytes / H2D "
                                       "rate, d2h bytes / D2H rate), each direction's rate measured alone in "
                                       "this run (both at once each ran at h2d_concurrent)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
    return result


# --------------------------------------------------------------------- oracle (CPU)

def oracle_sample(target_s: float, seed: int = 0):
    """Times the oracle (as it stands) on sampled elements of the six GEMMs.
    Returns (TFLOP/s, threads, description)."""
    import numpy as np
    import torch

    import oracle
    from block_scaled_fp8_gb300 import inputs

    oracle.build()
    threads = oracle.max_threads()
    # Small operands suffice for sampling: the oracle reads one A row and one B
    # row per element, so rows beyond the sample are never touched.
    rng = np.random.default_rng(seed)
    prepared = []
    for i, (m, n, k) in enumerate(SHAPES):
        rows_a, rows_b = min(m, 64), min(n, 256)
        case = inputs.dense_case(rows_a, rows_b, k, seed=seed + i)
        a = case.a.view(torch.uint8).numpy()
        b = case.b.view(torch.uint8).numpy()
        sa = case.sfa.double().numpy()
        sb = case.sfb.double().numpy()[np.arange(rows_b) // 128]
        prepared.append((m, n, k, a, b, sa, sb, rows_a, rows_b))
    # calibrate: time a small sample, then size the run to target_s
    def run(samples_per_gemm):
        fl, t0 = 0.0, time.perf_counter()
        for (m, n, k, a, b, sa, sb, ra, rb) in prepared:
            rows = rng.integers(0, ra, samples_per_gemm)
            cols = rng.integers(0, rb, samples_per_gemm)
            oracle.gemm_nt_sampled(a, sa, b, sb, rows, cols)
            fl += 2.0 * k * samples_per_gemm
        return fl, time.perf_counter() - t0
    fl, dt = run(256)
    per_sample = dt / (256 * len(prepared))
    n = max(256, int(target_s / max(per_sample, 1e-9) / len(prepared)))
    fl, dt = run(n)
    desc = (f"{n} sampled output elements of each of the six GEMMs (full-K fp64 dot products, "
            f"{threads} OpenMP threads), {dt:.1f} s")
    return fl / dt / 1e12, threads, desc


def oracle_small_config_s(seed: int = 0):
    """Seconds the oracle takes for the whole of the small workload (M=128, N=256,
    K=512, full D), on one thread and on all of them."""
    import numpy as np
    import torch

    import oracle
    from block_scaled_fp8_gb300 import inputs

    oracle.build()
    m, n, k = 128, 256, 512
    case = inputs.dense_case(m, n, k, seed=seed)
    a, b = case.a.view(torch.uint8).numpy(), case.b.view(torch.uint8).numpy()
    sa, sb = case.sfa.double().numpy(), case.sfb.double().numpy()[np.arange(n) // 128]
    out = {}
    # (an explicit count each time: a count of 0 keeps the previous call's setting)
    for label, thr in (("1_thread", 1), ("all_threads", oracle.max_threads())):
        best = None
        for _ in range(3):
            t0 = time.perf_counter()
            oracle.gemm_nt(a, sa, b, sb, nthreads=thr)
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        out[label] = round(best, 5)
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return None
    target = max(3.0, 20.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(target * 0.3, seed=1)
    vals, thr, desc = [], 0, ""
    t0 = time.perf_counter()
    for s in range(args.steps):
        v, thr, desc = oracle_sample(target, seed=100 + s)
        vals.append(v)
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(wall * 1e3 / max(1, args.steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "shapes_mnk": SHAPES,
                   "step": "oracle on a bounded sample of the workload"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_case_k_grouped(args):
    """One K-grouped weight-gradient GEMM, `warmup` + `steps` launches (for ncu
    captures); prints the median per-launch device time."""
    import torch

    from block_scaled_fp8_gb300 import binding, build, inputs
    build.build()
    e, m, n, k = (int(x) for x in args.case_k_grouped.split(","))
    dev = torch.device("cuda", 0)
    kc = inputs.k_grouped_case(e, m, n, seed=0, ks=[k] * e, device=dev)
    sfa = binding.dg_transform_sf_k_grouped(kc.sfa, kc.ks)
    sfb = binding.dg_transform_sf_k_grouped(kc.sfb, kc.ks)
    ks_dev = torch.tensor(kc.ks, dtype=torch.int32, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        binding.dg_k_grouped_fp8_gemm_tn_contiguous(kc.a, sfa, kc.b, sfb, kc.c, kc.ks, ks_dev=ks_dev, c=kc.c,
                                                    status=status)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    times = []
    for i in range(args.steps):
        flush.fill_(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    assert int(status.item()) == 0, int(status.item())
    us = statistics.median(times) * 1e3
    kt = e * k
    by = kt * (m + n) + 2 * 4 * e * m * n
    print(json.dumps({"case_k_grouped": [e, m, n, k], "median_us": round(us, 2),
                      "tflops": round(flops(m, n, kt) / (us * 1e-6) / 1e12, 1),
                      "gbs": round(by / (us * 1e-6) / 1e9, 1), "config": binding.last_config()}))


def run_case_grouped(args):
    """One M-grouped GEMM of the MoE workloads, `warmup` + `steps` launches (for ncu
    captures): `contiguous` (8 experts, M_e ~ U[128, 4096] padded to 128, N=4096,
    K=7168) or `masked` (32 experts, max_m 256, N=4096, K=7168); prints the median
    per-launch device time."""
    import torch

    from block_scaled_fp8_gb300 import binding, build, inputs
    build.build()
    dev = torch.device("cuda", 0)
    n, k = 4096, 7168
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if args.case_grouped == "contiguous":
        cc = inputs.contiguous_case(8, n, k, seed=3, device=dev)
        mt = cc.a.shape[0]
        sfa = binding.transform_sf(cc.sfa, 1, mt)
        sfb = binding.transform_sf(cc.sfb, 128, n)
        d = torch.empty(mt, n, dtype=torch.bfloat16, device=dev)
        valid = sum(cc.m_per_expert)
        used = sum(1 for v in cc.m_per_expert if v)

        def call():
            binding.dg_m_grouped_fp8_gemm_nt_contiguous(cc.a, sfa, cc.b, sfb, d, cc.grouped_layout, status=status)
    else:
        mc = inputs.masked_case(32, 256, n, k, seed=4, device=dev)
        sfa = binding.transform_sf(mc.sfa, 1, 256)
        sfb = binding.transform_sf(mc.sfb, 128, n)
        d = torch.empty(32, 256, n, dtype=torch.bfloat16, device=dev)
        valid = int(mc.masked_m.sum())
        used = int((mc.masked_m > 0).sum())

        def call():
            binding.dg_m_grouped_fp8_gemm_nt_masked(mc.a, sfa, mc.b, sfb, d, mc.masked_m, mc.expected_m,
                                                    status=status)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    times = []
    for i in range(args.steps):
        flush.fill_(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    assert int(status.item()) == 0, int(status.item())
    us = statistics.median(times) * 1e3
    by = valid * k + used * n * k + 2 * valid * n
    print(json.dumps({"case_grouped": args.case_grouped, "valid_rows": valid, "median_us": round(us, 2),
                      "tflops": round(flops(valid, n, k) / (us * 1e-6) / 1e12, 1),
                      "gbs": round(by / (us * 1e-6) / 1e9, 1), "config": binding.last_config()}))


def run_case(args):
    """One dense GEMM shape, `warmup` + `steps` launches (for ncu captures and
    per-shape timing); prints per-launch device time."""
    import torch

    from block_scaled_fp8_gb300 import binding, build, inputs
    build.build()
    m, n, k = (int(x) for x in args.case.split(","))
    dev = torch.device("cuda", 0)
    if args.fp4:
        case = inputs.fp4_case(m, n, k, seed=0, with_c=args.with_c, device=dev)
        sfb = binding.transform_sf(case.sfb.contiguous(), 1, n)
        gemm = binding.dg_fp8_fp4_gemm_nt
    else:
        case = inputs.dense_case(m, n, k, seed=0, with_c=args.with_c, device=dev)
        sfb = binding.transform_sf(case.sfb, 128, n)
        gemm = binding.dg_fp8_gemm_nt
    a, b = case.a.to(dev), case.b.to(dev)
    sfa = binding.transform_sf(case.sfa.to(dev), 1, m)
    c = case.c.to(dev) if args.with_c else None
    d = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        gemm(a, sfa, b, sfb, d, c=c, status=status)
    torch.cuda.synchronize()
    times = []
    for i in range(args.steps):
        flush.fill_(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        gemm(a, sfa, b, sfb, d, c=c, status=status)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    assert int(status.item()) == 0, int(status.item())
    us = statistics.median(times) * 1e3
    cfg = binding.last_config()
    print(json.dumps({"case": [m, n, k], "with_c": args.with_c, "fp4": args.fp4, "median_us": round(us, 2),
                      "tflops": round(flops(m, n, k) / (us * 1e-6) / 1e12, 1),
                      "gbs": round((m * k + n * k // 2 + 2 * m * n if args.fp4 else gemm_bytes(m, n, k))
                                   / (us * 1e-6) / 1e9, 1), "config": cfg}))


def measure_step_launches(probs, flush, reps, status, stream, cuts=None):
    """Device time (ms, mean over `reps` replays) of runs of the step's GEMM
    launches: the six launches captured in a CUDA graph with a timing event before
    the first and after each launch count in `cuts` (default: after every launch),
    each replay behind the L2 flush.  An event between two launches makes the second
    wait for the first to finish, where the plain step lets it start early
    (programmatic dependent launch); launches between two events keep that overlap.
    Returns one time per run; None if torch cannot record timing events inside a
    captured graph."""
    import torch

    from block_scaled_fp8_gb300 import binding
    cuts = list(range(1, len(probs) + 1)) if cuts is None else list(cuts)
    try:
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(cuts) + 1)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            evs[0].record()
            j = 0
            for i, p in enumerate(probs):
                binding.dg_fp8_gemm_nt(p["a"], p["sfa"], p["b"], p["sfb"], p["d"], status=status)
                if j < len(cuts) and i + 1 == cuts[j]:
                    j += 1
                    evs[j].record()
        torch.cuda.synchronize()
        out = [0.0] * len(cuts)
        for r in range(reps + 1):
            flush.fill_(r)
            g.replay()
            torch.cuda.synchronize()
            if r == 0:
                continue   # the graph's first replay uploads it
            for i in range(len(cuts)):
                out[i] += evs[i].elapsed_time(evs[i + 1]) / reps
        del g
        return out
    except (TypeError, RuntimeError):
        torch.cuda.synchronize()
        return None


def measure_pinned_copies(dev, stream, nbytes=256 * 1024 * 1024, reps=5):
    """Raw copy rates (GB/s, best of `reps`) between pinned host memory and the
    device in this process: host to device alone, device to host alone (two
    halves on two streams, as the e2e pipeline copies D out), and both
    directions at once (all three streams)."""
    import torch
    try:
        h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        d_out = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        s_in, s_o = torch.cuda.Stream(), [torch.cuda.Stream(), torch.cuda.Stream()]
        h = nbytes // 2

        def timed(do_in, do_out):
            best = None
            for _ in range(reps):
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for s_ in [s_in] + s_o:
                    s_.wait_event(e0)
                if do_in:
                    with torch.cuda.stream(s_in):
                        d_in.copy_(h_in, non_blocking=True)
                if do_out:
                    for j, s_ in enumerate(s_o):
                        with torch.cuda.stream(s_):
                            h_out[j * h:(j + 1) * h].copy_(d_out[j * h:(j + 1) * h], non_blocking=True)
                for s_ in [s_in] + s_o:
                    stream.wait_stream(s_)
                e1.record(stream)
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1)
                best = ms if best is None else min(best, ms)
            return nbytes / (best * 1e-3) / 1e9
        h2d = timed(True, False)
        d2h = timed(False, True)
        both = timed(True, True)   # each direction moved nbytes in that time
        return {"h2d": round(h2d, 1), "d2h": round(d2h, 1), "h2d_concurrent": round(both, 1),
                "d2h_concurrent": round(both, 1), "bytes": nbytes}
    except Exception:
        return None


def e2e_pipelined(probs, steps, status, stream):
    """End-to-end steps through the public API: every GEMM of every step copies
    its activations and their packed scales in from pinned host memory, runs,
    and copies D back to pinned host memory.  Copies in, GEMMs and copies out
    run on their own streams, so the input copy of one GEMM and the output copy
    of the previous one overlap a GEMM; D goes out in two row halves on two
    streams (two copy engines); device buffers alternate between two sets from
    step to step.  Returns the elapsed ms of all steps (CUDA events)."""
    import torch
    from block_scaled_fp8_gb300 import binding

    s_in = torch.cuda.Stream()
    s_outs = [torch.cuda.Stream(), torch.cuda.Stream()]
    sets = [[(p["a"], p["sfa"], p["d"]) for p in probs],
            [(torch.empty_like(p["a"]), torch.empty_like(p["sfa"]), torch.empty_like(p["d"]))
             for p in probs]]
    n = len(probs)
    ev_in = [[torch.cuda.Event() for _ in range(n)] for _ in range(2)]     # inputs on the device
    ev_done = [[torch.cuda.Event() for _ in range(n)] for _ in range(2)]   # GEMM finished
    # D on the host, per output stream
    ev_out = [[[torch.cuda.Event() for _ in s_outs] for _ in range(n)] for _ in range(2)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for so in s_outs:
        so.wait_event(e0)
    t_host = time.perf_counter()
    for step_i in range(steps):
        b = step_i % 2
        for i, p in enumerate(probs):
            a, sfa, d = sets[b][i]
            if step_i >= 2:
                s_in.wait_event(ev_done[b][i])     # the GEMM two steps back has read this set
                for ev in ev_out[b][i]:            # and its D has been copied out
                    stream.wait_event(ev)
            with torch.cuda.stream(s_in):
                a.copy_(p["a_host"], non_blocking=True)
                sfa.copy_(p["sfa_packed_host"], non_blocking=True)
                ev_in[b][i].record(s_in)
            stream.wait_event(ev_in[b][i])
            binding.dg_fp8_gemm_nt(a, sfa, p["b"], p["sfb"], d, status=status, stream=stream)
            ev_done[b][i].record(stream)
            h = d.shape[0] // 2
            for j, (so, rows) in enumerate(zip(s_outs, (slice(0, h), slice(h, d.shape[0])))):
                so.wait_event(ev_done[b][i])
                with torch.cuda.stream(so):
                    p["d_host"][rows].copy_(d[rows], non_blocking=True)
                    ev_out[b][i][j].record(so)
    stream.wait_stream(s_in)
    for so in s_outs:
        stream.wait_stream(so)
    e1.record(stream)
    host_ms = (time.perf_counter() - t_host) * 1e3
    torch.cuda.synchronize()
    del sets[1]
    return e0.elapsed_time(e1), host_ms


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", default=None, help="M,N,K: time one dense GEMM shape only")
    ap.add_argument("--with-c", action="store_true")
    ap.add_argument("--fp4", action="store_true", help="with --case: FP4 (E2M1) weights, dg_fp8_fp4_gemm_nt")
    ap.add_argument("--case-k-grouped", default=None,
                    help="E,M,N,K: time one K-grouped GEMM (E groups of K rows each, C = D in place)")
    ap.add_argument("--case-grouped", choices=["contiguous", "masked"], default=None,
                    help="time one M-grouped MoE GEMM: contiguous (8 experts) or masked (32 experts)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--record-traffic", default=None, metavar="DIR",
                    help="write the DRAM traffic record from DIR/traffic_M,N,K.csv (one ncu capture per "
                         "GEMM of the step) to --traffic-out, stamped with this tree's source digest")
    ap.add_argument("--traffic-out", default=os.path.join(ROOT, "profiles", "gemm_dram_traffic.json"))
    ap.add_argument("--traffic-command", default="", help="the capture command, stored in the record")
    args = ap.parse_args()
    if args.record_traffic:
        rec = record_traffic(args.record_traffic, args.traffic_out, args.traffic_command)
        print(json.dumps({"traffic_record": args.traffic_out, "source_digest": rec["source_digest"]}))
        return
    if args.warmup < 3 and not (args.case or args.case_k_grouped or args.case_grouped):
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        world = max(world, 1)

    if args.case:
        run_case(args)
        return
    if args.case_k_grouped:
        run_case_k_grouped(args)
        return
    if args.case_grouped:
        run_case_grouped(args)
        return
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            v, thr, desc = oracle_sample(10.0)
            res["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": thr, "kind": "oracle",
                                   "sample": desc,
                                   "small_workload_128x256x512_full_s": oracle_small_config_s()}
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
