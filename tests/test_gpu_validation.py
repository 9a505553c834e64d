"""Randomized validation at the paper's scale ("Accurate Models of AMD Matrix Cores",
Sec. 5): Algorithm 3 exponent-mantissa sampling for every CDNA 3 preset at the exponent
limits of Sec. 5.1, with the instruction inner sizes k of Sec. 5.1 (chains of block
FMAs), every GPU output compared with the oracle by the harness in
validate_algorithm3.py.  Here at 5 % of Table 2's final ensemble sizes; the harness
run at full size writes the record in tests/records/."""
import numpy as np
import pytest

import validate_algorithm3 as V

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_algorithm3_campaign():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rec = V.run(scale=0.05, chunk=500_000, log_fn=lambda s: None)
    bad = [e for e in rec["ensembles"] if e["mismatches"]]
    assert not bad, bad[:3]
    rows = {r["row"]: r for r in rec["table2"]}
    assert rows["fp16"]["n_ens"] == 500_000 and rows["binary8"]["n_ens"] == 1_000_000
    for r in rec["table2"]:
        assert r["mismatches"] == 0
        assert np.isclose(r["p_eps"], -np.expm1(np.log(1e-6) / (r["n_ens"] + 1)))
