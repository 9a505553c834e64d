"""Benchmark: bit-exact emulated block-FMAs/s on GB300 (and emulated-GEMM GFLOP/s).

A step is one pass of the block-FMA stream over the randomized-validation workload:
10^7 vector sets for each of FP16 K=4, BF16 K=4, XF32 K=2, FP8 E4M3 K=8, FP8 E5M2
K=8 (OCP) under three models (truncate, round-to-nearest-even, exact-then-round) and
INT8 K=16 (int32 accumulate); inputs by independent bit sampling with 1% each of
zeros, subnormals, Inf and NaN.  16 launches, 1.6e8 block FMAs per step and GPU.
The dense BF16 (2048^3), 2:4 sparse E4M3 (4096^3) and multi-word FP64 (4096^3)
GEMMs are timed in the same run and reported under "gemm".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  Under torchrun each rank processes its own vector
sets (weak scaling, no collective on the data path).
"""
import argparse
import hashlib
import re
import json
import os
import subprocess
import sys
import time
from fractions import Fraction

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_exact_emulation_gb300 import workloads as W  # noqa: E402

N_VEC = 10_000_000
FORMATS = [("fp16", 4), ("bf16", 4), ("xf32", 2), ("e4m3", 8), ("e5m2", 8), ("int8", 16)]
MODELS = ("ga_trunc", "ga_rne", "ieee_exact")
METRIC = "bit-exact emulated block-FMAs/sec (10^7 vector sets x 6 formats x 3 models)"
VEC_BYTES = {f: k * (1 if f in ("e4m3", "e5m2", "int8") else (2 if f in ("fp16", "bf16") else 4))
             for f, k in FORMATS}


def workload_config(n_vec):
    """The workload both arms report (the reference arm times a bounded sample of it)."""
    return {"workload": f"randomized block-FMA vector sets: {n_vec:.0e} each of FP16 K=4, BF16 K=4, XF32 K=2, "
                        "E4M3 K=8, E5M2 K=8 (OCP) x {truncate, RNE, exact} + INT8 K=16",
            "vector_sets_per_step_per_gpu": n_vec * 16, "launches_per_step": 16,
            "l2": "inputs larger than L2 (200-400 MB read per launch)"}


def rank_seed(k, rank):
    """Seed of one rank's vector sets: every rank streams its own sets (weak scaling)."""
    return 2 + k + 1000 * rank


def max_over_ranks(x, dist, device):
    """The largest value of x over all ranks (the job takes as long as its slowest rank)."""
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step, world, ms_per_step):
    """Units all ranks processed per second, over the slowest rank's step time."""
    return units_per_rank_step * world / (ms_per_step / 1e3)


def workload_models(fmt, k):
    """(name, model description) of the stream models for one format (library presets)."""
    from bit_exact_emulation_gb300 import binding as L
    if fmt == "int8":
        return [("int", L.preset_desc("ieee_exact", "int8", k))]
    return [(name, L.preset_desc(name, fmt, k)) for name in MODELS]


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sms, mx, reasons = [], None, set()
        for line in out.strip().splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sms.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), p[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sms)) if sms else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


# ---------------------------------------------------------------------------
# the CPU baseline (the oracle, as it stands) -- also the bench's parity sample
# ---------------------------------------------------------------------------
def cpu_baseline(data, outputs, per_combo, threads):
    import oracle
    from oracle.presets import block_models
    total, t_total, mismatches = 0, 0.0, 0
    for fmt, k in FORMATS:
        a, b, c = data[fmt]
        idx = np.random.default_rng(99).choice(a.shape[0], per_combo, replace=False)
        idx.sort()
        for name, spec in block_models(fmt, k).items():
            t0 = time.perf_counter()
            want = oracle.block_fma_parallel(spec, a[idx], b[idx], c[idx], threads)
            t_total += time.perf_counter() - t0
            total += per_combo
            got = outputs.get((fmt, name))
            if got is not None:
                mismatches += int((got[idx] != want).sum())
    return total, t_total, mismatches


def run_reference(args, rank):
    """The reference arm: the oracle on the host cores, a bounded sample per step."""
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    per_combo = 30000
    data = {fmt: W.gen_block_fma_set(fmt, 2 * per_combo, k, seed=2 + k) for fmt, k in FORMATS}
    for _ in range(args.warmup):
        cpu_baseline(data, {}, per_combo // 10, threads)
    n = 0
    t = 0.0
    for _ in range(args.steps):
        cnt, dt, _ = cpu_baseline(data, {}, per_combo, threads)
        n += cnt
        t += dt
    value = n / t
    sample = f"{per_combo} vector sets per (format, model) pair per step, 16 pairs, CPU oracle"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "block-FMA/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int (exact big-integer)",
            "data": "synthetic", "config": workload_config(N_VEC),
            "cpu_baseline": {"value": value, "unit": "block-FMA/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "block-FMA/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
STREAM_SOURCES = ("core.cuh", "model.h", "stream.cu", "stream_fp8.cu", "stream_pair.cuh")


def _code_only(text):
    """C/C++ source without its comments and with whitespace runs collapsed: what the
    compiler sees, so that a comment edit leaves the hash unchanged."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash():
    """Hash of the code (comments stripped) the block-FMA stream kernels are compiled from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_exact_emulation_gb300", "csrc")
    paths = [os.path.join(csrc, name) for name in STREAM_SOURCES] + [os.path.join(ROOT, "include", "mcemu.h")]
    for path in paths:
        with open(path, encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def read_profile_row(kernel_key):
    """The committed ncu figures of a stream kernel (profiles/traffic.md): DRAM bytes per
    launch at 10^7 sets, thread instructions per set, ALU-pipe and issue utilisation --
    when they were taken on the current kernel sources, else None."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash()
    for line in open(path):
        p = [x.strip() for x in line.strip().strip("|").split("|")]
        if len(p) >= 6 and p[0] == kernel_key and p[-1] == cur:
            try:
                return {"traffic": float(p[1]), "inst_per_set": float(p[2]), "alu_pct": float(p[3]),
                        "issue_pct": float(p[4])}
            except ValueError:
                return None
    return None


def c1_launch(L, torch, dev, reps=200):
    """The 65,536-set FP16 K=4 cancellation workload under global alignment with 3
    extra bits and truncation: 1.5 MiB of inputs stay in L2, so one launch is short and
    latency-bound; reported per launch, parity checked in the tests."""
    a, b, c = W.gen_fp16_cancellation(65536, 4, seed=1)
    da, db, dc = dev(a), dev(b), dev(c)
    m = L.Model(L.preset_desc("ga_trunc", "fp16", 4))
    d = torch.empty(65536, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    for _ in range(3):
        L.block_fma(m, da, db, dc, d)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a device-side wait ahead of the start event lets the host queue the launches, so the
    # events measure the GPU's time per launch rather than the host's call rate
    torch.cuda._sleep(20_000_000)
    e0.record(s)
    t0 = time.perf_counter()
    for _ in range(reps):
        L.block_fma(m, da, db, dc, d)
    host_us = (time.perf_counter() - t0) / reps * 1e6
    e1.record(s)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    return {"sets": 65536, "us_per_launch": us, "block_fma_per_s": 65536 / (us * 1e-6),
            "host_us_per_call": host_us,
            "note": "L2-resident inputs, back-to-back launches queued ahead of the GPU; host_us_per_call is the "
                    "Python call through the C ABI"}


def int_pipe_peaks(torch):
    """Measured lane-operation rates of the integer pipes (csrc/peak.cu): lop3 and shf on
    the ALU pipe, mad.lo on the FMA pipe; the best of three launches each."""
    import ctypes
    from bit_exact_emulation_gb300 import build
    P = ctypes.CDLL(build.build_peak())
    P.mcpeak_int_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_double)]
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = {}
    for kind, name in ((0, "alu_lop3"), (1, "alu_shf"), (2, "fma_imad")):
        best = 0.0
        for _ in range(3):
            r = ctypes.c_double(0.0)
            if P.mcpeak_int_rate(kind, 4096, ctypes.c_void_p(sink.data_ptr()), ctypes.byref(r)) == 0:
                best = max(best, r.value)
        out[name] = best
    out["unit"] = "lane-ops/s"
    return out


# minimum integer work per multiply-accumulate of an emulated GEMM: one significand
# product, one exponent add, one maximum, one alignment shift, one add (per-block
# normalisation and rounding on top); the ALU pipe's measured rate is the roof
OPS_PER_MAC = 5


def gemm_roofline(macs_per_s, peaks):
    if not peaks or not peaks.get("alu_lop3"):
        return None
    achieved = macs_per_s * OPS_PER_MAC
    return {"bound": "alu", "ops_per_mac": OPS_PER_MAC, "achieved": achieved, "peak": peaks["alu_lop3"],
            "peak_source": "measured (lop3 chains, csrc/peak.cu)", "unit": "lane-ops/s",
            "frac": achieved / peaks["alu_lop3"]}


def gemm_section(L, torch, dev, steps, parts=("dense", "sparse", "multiword"), peaks=None):
    """Time the emulated-GEMM workloads named in `parts`; returns their summary dict."""
    out = {}
    s = torch.cuda.current_stream()

    def timed(fn, reps):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(reps):
            fn()
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps / 1000.0

    # dense BF16 2048^3, 32x32x8 bf16 tile semantics
    if "dense" in parts:
        out["dense_bf16_2048"] = gemm_dense(L, torch, dev, timed, steps, peaks)
    if "sparse" in parts:
        out["sparse24_e4m3_4096"] = gemm_sparse(L, torch, dev, timed, steps, peaks)
    if "multiword" in parts:
        out["multiword_fp64_4096"] = gemm_multiword(L, torch, timed, steps, peaks)
    return out


def gemm_dense(L, torch, dev, timed, steps, peaks=None):
    M = N = K = 2048
    A, Bt, C = W.gen_dense_bf16(M, N, K, seed=3)
    dA, dB, dC = dev(A), dev(Bt), dev(C)
    t = L.tile(0, 32, 32, 8, 4)
    dense = {}
    for name, desc in (("cdna3_bf16", L.preset_desc("cdna3_bf16")), ("ga_trunc_k4", L.preset_desc("ga_trunc", "bf16", 4)),
                       ("ga_rne_k4", L.preset_desc("ga_rne", "bf16", 4)), ("ieee_exact_k4", L.preset_desc("ieee_exact", "bf16", 4))):
        m = L.Model(desc)
        D = torch.empty((M, N), dtype=torch.int32, device="cuda")
        sec = timed(lambda: L.tile_gemm(m, t, dA, dB, dC, D), steps)
        dense[name] = {"ms": sec * 1e3, "gflops": 2.0 * M * N * K / sec / 1e9,
                       "roofline": gemm_roofline(M * N * K / sec, peaks)}
    return dense


def gemm_sparse(L, torch, dev, timed, steps, peaks=None):
    """2:4 sparse E4M3 4096^3, 16x16x32 tile semantics."""
    M = N = K = 4096
    A, Bt, C = W.gen_sparse_e4m3(M, N, K, seed=4)
    dA, dB, dC = dev(A), dev(Bt), dev(C)
    Ac, meta, viol = L.sparse24_compress("e4m3", dA)
    tcomp = timed(lambda: L.sparse24_compress("e4m3", dA), steps)
    ts = L.tile(1, 16, 16, 32, 8)
    sparse = {"compress_ms": tcomp * 1e3, "compress_gbs": (M * K * 1.5 + M * K / 2 + M * K / 4) / tcomp / 1e9,
              "violations": int(viol.item())}
    for name in ("ga_trunc", "ga_rne"):
        m = L.Model(L.preset_desc(name, "e4m3", 8))
        D = torch.empty((M, N), dtype=torch.int32, device="cuda")
        sec = timed(lambda: L.sparse24_gemm(m, ts, Ac, meta, dB, dC, D), steps)
        sparse[name] = {"ms": sec * 1e3, "gflops_effective": 2.0 * M * N * (K // 2) / sec / 1e9,
                        "gflops_dense_equivalent": 2.0 * M * N * K / sec / 1e9,
                        "roofline": gemm_roofline(M * N * (K // 2) / sec, peaks)}
    return sparse


def gemm_multiword(L, torch, timed, steps, peaks=None):
    """Multi-word FP64 4096^3: 3 BF16 words, 9 and 6 word products, CDNA3 BF16 word model."""
    M = N = K = 4096
    t = L.tile(0, 32, 32, 8, 4)
    A, Bt = W.gen_multiword_fp64(M, N, K, seed=5)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda()
    m = L.Model(L.preset_desc("cdna3_bf16"))
    ws = torch.empty(L.multiword_workspace(3, M, N, K), dtype=torch.uint8, device="cuda")
    D = torch.empty((M, N), dtype=torch.float64, device="cuda")
    R = dA @ dB.T
    # exact values of 256 sampled entries: every binary64 product is an integer times a
    # power of two, so the dot product is summed exactly in Python integers
    rng = np.random.default_rng(21)
    si, sj = rng.integers(0, M, 256), rng.integers(0, N, 256)
    exact = [exact_dot(A[i], Bt[j]) for i, j in zip(si, sj)]
    mw = {}
    for label, trunc, npairs in (("9_products", False, 9), ("6_products", True, 6)):
        sec = timed(lambda: L.multiword_gemm(m, t, 3, trunc, dA, dB, D, ws), max(1, steps // 2))
        e2, r2 = L.fro_error(D, R).cpu().numpy()
        Dh = D.cpu().numpy()
        rel = [abs(Fraction(float(Dh[i, j])) - x) / abs(x) for (i, j), x in zip(zip(si, sj), exact) if x != 0]
        mw[label] = {"ms": sec * 1e3, "gflops_emulated": npairs * 2.0 * M * N * K / sec / 1e9,
                     "roofline": gemm_roofline(npairs * M * N * K / sec, peaks),
                     "rel_fro_error": float(np.sqrt(e2 / r2)),
                     "rel_err_exact_sampled": {"max": float(max(rel)), "median": float(np.median([float(r) for r in rel])),
                                               "entries": len(rel)}}
    return mw


def oracle_gemm_sample(fn, M, N, entries, gpu_ms):
    """The oracle on `entries` sampled outputs of a GEMM, single host thread: its time per
    output, and the whole GEMM extrapolated from it (labelled as such)."""
    rng = np.random.default_rng(17)
    ii = rng.integers(0, M, entries).astype(np.int32)
    jj = rng.integers(0, N, entries).astype(np.int32)
    t0 = time.perf_counter()
    fn(ii, jj)
    dt = time.perf_counter() - t0
    per = dt / entries
    return {"entries": entries, "threads": 1, "s_per_output": per,
            "whole_gemm_s_extrapolated": per * M * N, "gpu_speedup_extrapolated": per * M * N / (gpu_ms / 1e3)}


def cpu_gemm_baseline(gemm):
    """CPU-baseline leg for the GEMM workloads: the oracle on sampled outputs of each
    (the inputs regenerated from their seeds), one host thread."""
    import oracle
    from oracle.presets import PRESETS, block_models
    out = {}
    if "dense_bf16_2048" in gemm:
        M = N = K = 2048
        A, Bt, C = W.gen_dense_bf16(M, N, K, seed=3)
        out["dense_bf16_2048 cdna3_bf16"] = oracle_gemm_sample(
            lambda ii, jj: oracle.gemm_entries(PRESETS["cdna3_bf16"], K, 8, A, Bt, C, ii, jj), M, N, 64,
            gemm["dense_bf16_2048"]["cdna3_bf16"]["ms"])
    if "sparse24_e4m3_4096" in gemm:
        M = N = K = 4096
        A, Bt, C = W.gen_sparse_e4m3(M, N, K, seed=4)
        Ac, meta, _ = oracle.sparse24_compress("e4m3", A)
        spec = block_models("e4m3", 8)["ga_trunc"]
        out["sparse24_e4m3_4096 ga_trunc"] = oracle_gemm_sample(
            lambda ii, jj: oracle.sparse24_entries(spec, K, 32, Ac, meta, Bt, C, ii, jj), M, N, 32,
            gemm["sparse24_e4m3_4096"]["ga_trunc"]["ms"])
    if "multiword_fp64_4096" in gemm:
        M = N = K = 4096
        A, Bt = W.gen_multiword_fp64(M, N, K, seed=5)
        out["multiword_fp64_4096 9_products"] = oracle_gemm_sample(
            lambda ii, jj: oracle.multiword_entries(PRESETS["cdna3_bf16"], 8, 3, False, A, Bt, ii, jj), M, N, 4,
            gemm["multiword_fp64_4096"]["9_products"]["ms"])
    return out


def exact_dot(x, y):
    """Exact sum of x[k] * y[k] for binary64 vectors, as a Fraction."""
    terms = []
    for u, v in zip(x.tolist(), y.tolist()):
        pu, qu = u.as_integer_ratio()
        pv, qv = v.as_integer_ratio()
        terms.append((pu * pv, qu * qv))
    den = max(q for _, q in terms)                  # denominators are powers of two
    num = sum(p * (den // q) for p, q in terms)
    return Fraction(num, den)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-gemm", action="store_true", help="skip the GEMM section (stream numbers only)")
    ap.add_argument("--gemm-parts", default="dense,sparse,multiword",
                    help="comma list of the GEMM workloads to time (dense, sparse, multiword)")
    ap.add_argument("--vectors", type=int, default=N_VEC,
                    help="vector sets per (format, model) launch; smaller values are for profiling runs only")
    ap.add_argument("--only", default="",
                    help="profiling runs only: comma list of format:model stream launches to keep (e.g. "
                         "bf16:ieee_exact); the end-to-end, GEMM and CPU legs are skipped")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    from bit_exact_emulation_gb300 import build
    build.build()
    from bit_exact_emulation_gb300 import binding as L

    def dev(x):
        x = np.ascontiguousarray(x)
        if x.dtype == np.uint16:
            x = x.view(np.int16)
        elif x.dtype == np.uint32:
            x = x.view(np.int32)
        return torch.from_numpy(x).cuda()

    n_vec = args.vectors
    only = {tuple(x.split(":")) for x in args.only.split(",") if x}
    # inputs: this rank's own vector sets (weak scaling)
    data, gpu, launches = {}, {}, []
    for fmt, k in FORMATS:
        if only and not any(f == fmt for f, _ in only):
            continue
        a, b, c = W.gen_block_fma_set(fmt, n_vec, k, seed=rank_seed(k, rank))
        data[fmt] = (a, b, c)
        gpu[fmt] = (dev(a), dev(b), dev(c))
        for name, desc in workload_models(fmt, k):
            if only and (fmt, name) not in only:
                continue
            m = L.Model(desc)
            d = torch.empty(n_vec, dtype=torch.int32, device="cuda")
            launches.append((fmt, name, m, d))
    stream = torch.cuda.current_stream()
    # one pair of events per launch and step: they are read after the timed loop, so the
    # host never waits inside it and launches stay queued ahead of the GPU
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in launches]
           for _ in range(args.steps)]

    def step(ev=None):
        for li, (fmt, name, m, d) in enumerate(launches):
            a, b, c = gpu[fmt]
            if ev is not None:
                ev[li][0].record(stream)
            L.block_fma(m, a, b, c, d)
            if ev is not None:
                ev[li][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    per_launch = np.zeros(len(launches))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    # a short device-side wait ahead of the start event lets the host queue the first
    # launches before the timed region begins, so no launch in it waits on the host
    torch.cuda._sleep(4_000_000)
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize()
    elapsed_ms = t0.elapsed_time(t1)
    for k in range(args.steps):
        for li in range(len(launches)):
            per_launch[li] += evs[k][li][0].elapsed_time(evs[k][li][1])
    clk = clocks.stop()
    if world > 1:
        elapsed_ms = max_over_ranks(elapsed_ms, dist, "cuda")
        dist.barrier()
    ms_per_step = elapsed_ms / args.steps
    fmas_per_step = n_vec * len(launches)
    value = whole_job_rate(fmas_per_step, world, ms_per_step)

    # outputs of the last step for the parity sample
    outputs = {(fmt, name): d.cpu().numpy().view(np.uint32) for fmt, name, m, d in launches}

    # roofline of the dominant kernel: algorithmic bytes = n * (2 * vector bytes + 8) per launch
    per_launch /= args.steps
    dom = int(np.argmax(per_launch))
    dfmt, dname = launches[dom][0], launches[dom][1]
    algo_bytes = n_vec * (2 * VEC_BYTES[dfmt] + 8)
    achieved = algo_bytes / (per_launch[dom] / 1e3) / 1e9
    peak, peak_kind = hbm_peak()
    prof = read_profile_row(f"block_fma {dfmt} {dname}")
    roofline = {"bound": "hbm", "kernel": f"block_fma {dfmt} {dname}", "achieved": achieved, "peak": peak,
                "peak_source": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                "traffic": prof["traffic"] if prof else None,
                # the stream kernels are instruction-issue bound: ncu's figures for this kernel (6e6-set capture)
                "pipes_ncu": ({"inst_per_set": prof["inst_per_set"], "alu_pipe_pct": prof["alu_pct"],
                               "issue_active_pct": prof["issue_pct"]} if prof else None),
                "algorithmic_bytes_per_launch": algo_bytes,
                "per_kernel_gbs": {f"{f} {n}": n_vec * (2 * VEC_BYTES[f] + 8) / (t / 1e3) / 1e9
                                   for (f, n, _, _), t in zip(launches, per_launch)}}

    if only:
        if rank == 0:
            print(json.dumps({"profiling_only": sorted(f"{f}:{n}" for f, n in only), "vectors": n_vec,
                              "ms_per_step": ms_per_step, "roofline": roofline}), flush=True)
        return

    # end to end through the host-buffer entry point (pinned host memory, copies timed)
    e2e = None
    if rank == 0:
        pinned = {}
        for fmt, k in FORMATS:
            a, b, c = data[fmt]
            pinned[fmt] = tuple(torch.from_numpy(np.ascontiguousarray(x).view(
                {np.uint16: np.int16, np.uint32: np.int32}.get(x.dtype.type, x.dtype))).pin_memory() for x in (a, b, c))
        outs = [torch.empty(n_vec, dtype=torch.int32).pin_memory() for _ in launches]
        ws = torch.empty(max(L.block_fma_host_workspace(m) for _, _, m, _ in launches), dtype=torch.uint8,
                         device="cuda")

        def e2e_step():
            for li, (fmt, name, m, d) in enumerate(launches):
                a, b, c = pinned[fmt]
                L.block_fma_host(m, a, b, c, outs[li], ws)

        e2e_step()
        torch.cuda.synchronize()
        step_ms = []
        for _ in range(max(1, min(args.steps, 5))):
            t0 = time.perf_counter()
            e2e_step()                       # each host call returns after its last copy back
            torch.cuda.synchronize()
            step_ms.append((time.perf_counter() - t0) * 1e3)
        # the median step: one slow step of the host (paging, another process) does not
        # stand for the link; every step's time is listed beside it
        te = float(np.median(step_ms)) / 1e3
        h2d = sum(n_vec * (2 * VEC_BYTES[f] + 4) for f, _, _, _ in launches)
        e2e = {"value": fmas_per_step / te, "unit": "block-FMA/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": n_vec * 4 * len(launches), "ms_per_step": te * 1e3,
               "step_ms": [round(x, 2) for x in step_ms], "stat": "median step",
               "api": "mcemu_block_fma_host"}
        for li, (fmt, name, m, d) in enumerate(launches):
            if not np.array_equal(outs[li].numpy().view(np.uint32), outputs[(fmt, name)]):
                e2e["mismatch"] = f"{fmt} {name}"

    peaks = int_pipe_peaks(torch) if rank == 0 else None
    c1 = c1_launch(L, torch, dev) if rank == 0 else None
    gemm = None
    if rank == 0 and not args.no_gemm:
        gemm = gemm_section(L, torch, dev, max(1, min(args.steps, 3)), tuple(args.gemm_parts.split(",")), peaks)

    if world > 1:
        dist.barrier()
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    per_combo = min(100_000, n_vec // 2)
    n_cpu, t_cpu, mism = cpu_baseline(data, outputs, per_combo, threads)
    n_1, t_1, _ = cpu_baseline(data, {}, min(10_000, per_combo), 1)
    cpu = {"value": n_cpu / t_cpu, "unit": "block-FMA/s", "cores": threads, "kind": "oracle",
           "sample": f"{per_combo} seeded vector sets of each (format, model) pair of the step, "
                     f"{n_cpu} block FMAs; the same sample checks the GPU outputs",
           "single_thread": {"value": n_1 / t_1, "unit": "block-FMA/s", "cores": 1,
                             "sample": f"{min(10_000, per_combo)} sets of each pair"}}
    if gemm:
        cpu["gemm_sampled_outputs"] = cpu_gemm_baseline(gemm)
    line = {"metric": METRIC, "value": value, "unit": "block-FMA/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bit-exact: integer significands and error-free fp32 sums", "data": "synthetic",
            "config": dict(workload_config(n_vec), parity_sample_mismatches=mism, parity_sample=n_cpu),
            "gpu_launches": len(launches) * args.steps, "clocks": clk, "roofline": roofline,
            "cpu_baseline": cpu, "e2e": e2e, "int_pipe_peaks": peaks, "c1_fp16_cancellation": c1, "gemm": gemm}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
