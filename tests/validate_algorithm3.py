"""Randomized validation of the GPU emulator at the scale of "Accurate Models of AMD
Matrix Cores" (Sec. 5, Table 2) -- TEST INFRASTRUCTURE: it runs the CPU oracle.

The paper validates its CDNA 3 model against MI300A/X hardware with exponent-mantissa
sampling (Sec. 5.1, Algorithm 3, an MT19937 stream seeded with 0) and reports, for
each input format, the ensemble size N_ens, the mismatches m and the Bayesian upper
bound p_eps on the mismatch probability (Sec. 5.4, eps = 10^-6).  Its final refinement
iteration (Table 2, iteration 4) ran 10^7 vector sets for fp16, bf16 and tf32 and
2 x 10^7 for binary8 (fp8 and bf8).  Here the GPU library plays the part of the
device under test and the oracle the part of the model:

  - every ensemble uses the instruction inner size k of Sec. 5.1 (fp16 and bf16 16,
    tf19 8, binary8 16), evaluated as the chain of ceil(k / N_FMA) block FMAs that one
    MFMA instruction performs, with the fp32 result of each block the addend of the
    next;
  - each format's ensemble is split evenly over the two exponent ranges of Sec. 5.1
    (normal and subnormal limits); binary8 is 10^7 E4M3 plus 10^7 E5M2 sets, FNUZ;
  - a further ensemble mixes E4M3 and E5M2 operands ("any combination", Sec. 4.3.4);
  - the GPU runs through the C ABI (the stream entry point), the oracle on all host
    cores; the outputs are compared bit for bit.

    python tests/validate_algorithm3.py [--scale 1.0] [--out record.json]

`--scale` multiplies every ensemble size (1.0 reproduces Table 2's final sizes).
The record lists, per ensemble and per Table 2 row, N_ens, m and p_eps.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time
from math import expm1, log

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle.presets import PRESETS  # noqa: E402
from bit_exact_emulation_gb300 import workloads as W  # noqa: E402

EPS = 1e-6
# Table 2 row, preset, format of a, format of b, k, exponent range of a and b, of c,
# share of the row's N_ens, seed of the MT19937 stream (Sec. 5.1 limits)
ENSEMBLES = [
    ("fp16", "cdna3_fp16", "fp16", "fp16", 16, (-14, 15), (-126, 127), 0.5, 0),
    ("fp16", "cdna3_fp16", "fp16", "fp16", 16, (-24, -14), (-149, -126), 0.5, 0),
    ("bf16", "cdna3_bf16", "bf16", "bf16", 16, (-126, 63), (-126, 127), 0.5, 0),
    ("bf16", "cdna3_bf16", "bf16", "bf16", 16, (-133, -126), (-149, -126), 0.5, 0),
    ("tf32", "cdna3_xf32", "xf32", "xf32", 8, (-126, 63), (-126, 127), 0.5, 0),
    ("tf32", "cdna3_xf32", "xf32", "xf32", 8, (-136, -126), (-149, -126), 0.5, 0),
    ("binary8", "cdna3_fp8", "e4m3", "e4m3", 16, (-7, 7), (-126, 127), 0.25, 0),
    ("binary8", "cdna3_fp8", "e4m3", "e4m3", 16, (-10, -7), (-149, -126), 0.25, 0),
    ("binary8", "cdna3_bf8", "e5m2", "e5m2", 16, (-15, 15), (-126, 127), 0.25, 0),
    ("binary8", "cdna3_bf8", "e5m2", "e5m2", 16, (-17, -15), (-149, -126), 0.25, 0),
]
TABLE2_N = {"binary8": 20_000_000, "fp16": 10_000_000, "bf16": 10_000_000, "tf32": 10_000_000}
MIXED = ("binary8 mixed", "cdna3_fp8", "e4m3", "e5m2", 16, (-7, 7), (-15, 15), (-126, 127), 2_000_000)


def p_eps(n: int, m: int, eps: float = EPS) -> float:
    """Upper bound p_eps on the mismatch probability after m mismatches in n trials with a
    uniform prior: the (1 - eps) quantile of the Beta(m + 1, n - m + 1) posterior
    (Sec. 5.4); for m = 0 it is 1 - eps^(1 / (n + 1))."""
    if m == 0:
        return -expm1(log(eps) / (n + 1))
    from scipy.special import betaincinv
    return float(betaincinv(m + 1, n - m + 1, 1.0 - eps))


def _draw(fmt_a, fmt_b, n, k, eab, eb, ec, rng_a, rng_b, enc):
    """One chunk of an ensemble: Algorithm 3 draws of a (and b, from its own stream when
    the formats differ), c drawn with a."""
    a, b, c = W.gen_exp_mantissa(fmt_a, n, k, eab, ec, enc=enc, rng=rng_a)
    if rng_b is not None:
        b, _, _ = W.gen_exp_mantissa(fmt_b, n, k, eb, ec, enc=enc, rng=rng_b)
    return a, b, c


def _chain(block, spec, k, a, b, c):
    """The ceil(k / N_FMA) block FMAs of one instruction: the result of block j is the
    addend of block j + 1 (fp32 between blocks)."""
    nf = spec["n_fma"]
    d = c
    for j in range(0, k, nf):
        d = block(spec, np.ascontiguousarray(a[:, j:j + nf]), np.ascontiguousarray(b[:, j:j + nf]), d)
    return d


def run(scale: float = 1.0, chunk: int = 1_000_000, threads: int | None = None, log_fn=print) -> dict:
    import torch
    from bit_exact_emulation_gb300 import build
    build.build()
    from bit_exact_emulation_gb300 import binding as L

    threads = threads or os.cpu_count() or 1
    models = {}

    def dev(x):
        x = np.ascontiguousarray(x)
        return torch.from_numpy(x.view({np.uint16: np.int16, np.uint32: np.int32}.get(x.dtype.type, x.dtype))).cuda()

    def gpu_block(spec, a, b, c):
        key = json.dumps(spec, sort_keys=True)
        if key not in models:
            models[key] = L.Model(spec)
        cd = c if isinstance(c, torch.Tensor) else dev(c)
        return L.block_fma(models[key], dev(a), dev(b), cd)

    def cpu_block(spec, a, b, c):
        return oracle.block_fma_parallel(spec, a, b, c, threads)

    jobs = [dict(row=r, preset=p, fmt_a=fa, fmt_b=fb, k=k, eab=eab, eb=eab, ec=ec,
                 n=int(round(TABLE2_N[r] * share * scale)), seed=seed)
            for r, p, fa, fb, k, eab, ec, share, seed in ENSEMBLES]
    r, p, fa, fb, k, eab, eb, ec, n = MIXED
    jobs.append(dict(row=r, preset=p, fmt_a=fa, fmt_b=fb, k=k, eab=eab, eb=eb, ec=ec, n=int(round(n * scale)),
                     seed=0))
    t_gpu = t_cpu = 0.0
    out = []
    for job in jobs:
        spec = dict(PRESETS[job["preset"]], fmt_b=job["fmt_b"])
        enc = spec.get("fp8_enc", "ocp")
        rng_a = W.algorithm3_rng(job["seed"])
        rng_b = W.algorithm3_rng(job["seed"] + 1) if job["fmt_b"] != job["fmt_a"] else None
        mism, done, first = 0, 0, []
        while done < job["n"]:
            n = min(chunk, job["n"] - done)
            a, b, c = _draw(job["fmt_a"], job["fmt_b"], n, job["k"], job["eab"], job["eb"], job["ec"],
                            rng_a, rng_b, enc)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            got = _chain(gpu_block, spec, job["k"], a, b, c)
            got = got.cpu().numpy().view(np.uint32)
            t_gpu += time.perf_counter() - t0
            t0 = time.perf_counter()
            want = _chain(cpu_block, spec, job["k"], a, b, c)
            t_cpu += time.perf_counter() - t0
            bad = np.nonzero(got != want)[0]
            mism += len(bad)
            for v in bad[:4 - len(first)]:
                first.append({"set": int(done + v), "gpu": f"{int(got[v]):#010x}", "oracle": f"{int(want[v]):#010x}"})
            done += n
        entry = dict(job, eab=list(job["eab"]), eb=list(job["eb"]), ec=list(job["ec"]),
                     n_fma=spec["n_fma"], blocks=-(-job["k"] // spec["n_fma"]), mismatches=mism,
                     p_eps=p_eps(job["n"], mism), first_mismatches=first)
        out.append(entry)
        log_fn(f"{job['row']:14s} {job['preset']:11s} {job['fmt_a']}x{job['fmt_b']} k={job['k']} "
               f"e_ab={job['eab']} e_c={job['ec']} N={job['n']} m={mism}")
    rows = []
    for row in ("binary8", "fp16", "bf16", "tf32", "binary8 mixed"):
        ents = [e for e in out if e["row"] == row]
        n = sum(e["n"] for e in ents)
        m = sum(e["mismatches"] for e in ents)
        rows.append({"row": row, "n_ens": n, "mismatches": m, "p_eps": p_eps(n, m),
                     "table2_n_ens": TABLE2_N.get(row)})
    return {"what": "Algorithm 3 exponent-mantissa sampling, CDNA 3 presets, GPU library vs CPU oracle",
            "eps": EPS, "scale": scale, "host_threads": threads,
            "gpu": torch.cuda.get_device_name(0), "gpu_seconds": t_gpu, "oracle_seconds": t_cpu,
            "table2": rows, "ensembles": out}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--scale", type=float, default=1.0)
    ap.add_argument("--chunk", type=int, default=1_000_000)
    ap.add_argument("--out", default="")
    args = ap.parse_args()
    rec = run(args.scale, args.chunk)
    text = json.dumps(rec, indent=1)
    if args.out:
        with open(args.out, "w") as f:
            f.write(text + "\n")
    for r in rec["table2"]:
        print(f"{r['row']:14s} N_ens={r['n_ens']:>10d} m={r['mismatches']} p_eps={r['p_eps']:.3g}")
    sys.exit(0 if all(r["mismatches"] == 0 for r in rec["table2"]) else 1)


if __name__ == "__main__":
    main()
