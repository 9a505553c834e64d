"""Randomized validation at the paper's scale ("Accurate Models of AMD Matrix Cores",
Sec. 5): Algorithm 3 exponent-mantissa sampling for every CDNA 3 preset at the exponent
bounds of Sec. 5.1, 10^6 vector sets per range, every GPU output compared with the
oracle.  With no mismatch in n trials, the Bayesian bound of Sec. 5.3 (m = 0, confidence
1 - 10^-6) limits the mismatch probability to 1 - 10^(-6/(n+1)), 1.38e-5 at n = 10^6."""
from math import expm1, log

import numpy as np
import pytest

import oracle
from oracle.presets import PRESETS
from bit_exact_emulation_gb300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

N = 1_000_000
RANGES = [  # preset, format, exponent range of a and b, exponent range of c (Sec. 5.1)
    ("cdna3_fp16", "fp16", (-14, 15), (-126, 127)), ("cdna3_fp16", "fp16", (-24, -14), (-149, -126)),
    ("cdna3_bf16", "bf16", (-126, 63), (-126, 127)), ("cdna3_bf16", "bf16", (-133, -126), (-149, -126)),
    ("cdna3_xf32", "xf32", (-126, 63), (-126, 127)), ("cdna3_xf32", "xf32", (-136, -126), (-149, -126)),
    ("cdna3_fp8", "e4m3", (-7, 7), (-126, 127)), ("cdna3_fp8", "e4m3", (-10, -7), (-149, -126)),
    ("cdna3_bf8", "e5m2", (-15, 15), (-126, 127)), ("cdna3_bf8", "e5m2", (-17, -15), (-149, -126)),
]


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_exact_emulation_gb300 import build
    build.build()
    from bit_exact_emulation_gb300 import binding
    return binding


def dev(x):
    x = np.ascontiguousarray(x)
    return torch.from_numpy(x.view({np.uint16: np.int16, np.uint32: np.int32}.get(x.dtype.type, x.dtype))).cuda()


@pytest.mark.parametrize("preset,fmt,eab,ec", RANGES)
def test_algorithm3_validation(L, preset, fmt, eab, ec):
    spec = PRESETS[preset]
    a, b, c = W.gen_exp_mantissa(fmt, N, spec["n_fma"], eab, ec, seed=0, enc=spec.get("fp8_enc", "ocp"))
    m = L.Model(spec)
    got = L.block_fma(m, dev(a), dev(b), dev(c)).cpu().numpy().view(np.uint32)
    want = oracle.block_fma_parallel(spec, a, b, c, threads=16)
    mismatches = int((got != want).sum())
    assert mismatches == 0, f"{preset} {eab} {ec}: {mismatches} of {N} differ"
    bound = -expm1(log(1e-6) / (N + 1))
    assert bound < 1.39e-5
