"""The multi-word GEMM entry point that allocates nothing (its word scratch is a
fixed array of the library's device memory), through the C ABI, against the
entry point that takes caller workspace.

Both entry points run the same kernels, so the tolerance is zero: the binary64
outputs must agree bit for bit, on every call of a run of calls."""
import numpy as np
import pytest

from oracle.presets import PRESETS, block_models
from bit_exact_emulation_gb300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_exact_emulation_gb300 import build
    build.build()
    from bit_exact_emulation_gb300 import binding
    return binding


def bits(t):
    return t.cpu().numpy().view(np.uint64)


CASES = [  # word model, words, truncated product set, M, N, K
    ("cdna3_bf16", 3, False, 64, 48, 256),
    ("ga_trunc", 3, True, 37, 29, 100),
    ("cdna3_bf16", 2, False, 5, 130, 72),
    # a word model the per-pair fast GEMM does not take (exact-then-round): the words
    # go through the fused general kernel, which also reads the fixed scratch
    ("ieee_exact", 3, False, 33, 41, 96),
    ("ieee_exact", 2, True, 16, 16, 40),
]


def spec_of(name):
    if name == "cdna3_bf16":
        return PRESETS["cdna3_bf16"]
    return block_models("bf16", 8)[name]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_static_scratch_matches_workspace_entry(L, case):
    name, nw, trunc, M, N, K = CASES[case]
    A, Bt = W.gen_multiword_fp64(M, N, K, seed=40 + case)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda()
    m = L.Model(spec_of(name))
    t = L.tile(0, 32, 32, 8, 4)
    want = bits(L.multiword_gemm(m, t, nw, trunc, dA, dB))
    for call in range(2):                      # two calls in a row reuse the same scratch
        got = bits(L.multiword_gemm_static(m, t, nw, trunc, dA, dB))
        assert np.array_equal(got, want), f"call {call}: {int((got != want).sum())} outputs differ"


def test_static_scratch_after_a_larger_call(L):
    """A smaller problem right after a larger one: stale words left in the scratch
    must not reach the result."""
    m = L.Model(PRESETS["cdna3_bf16"])
    t = L.tile(0, 32, 32, 8, 4)
    for (M, N, K) in ((96, 80, 512), (7, 9, 24)):
        A, Bt = W.gen_multiword_fp64(M, N, K, seed=M)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda()
        want = bits(L.multiword_gemm(m, t, 3, False, dA, dB))
        got = bits(L.multiword_gemm_static(m, t, 3, False, dA, dB))
        assert np.array_equal(got, want)


def test_static_scratch_rejects_sizes_beyond_the_array(L):
    M = N = K = 1024                           # 3 words: 12 MiB of words > 8 MiB
    assert L.multiword_workspace(3, M, N, K) > L.MULTIWORD_STATIC_BYTES
    dA = torch.zeros((M, K), dtype=torch.float64, device="cuda")
    m = L.Model(PRESETS["cdna3_bf16"])
    with pytest.raises(L.McemuError) as e:
        L.multiword_gemm_static(m, L.tile(0, 32, 32, 8, 4), 3, False, dA, dA)
    assert e.value.status == 7                 # MCEMU_ERR_WORKSPACE
