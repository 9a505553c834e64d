"""Loader of the paper-vector fixtures in tests/golden/*.txt."""
import os

from bit_exact_emulation_gb300.workloads import encode_exact, parse_value

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_vectors(name):
    """Rows of a fixture: dict(id, preset, fmt, kt, c, prods=[(a, b)], expect, cite)."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            cols = [c.strip() for c in line.split("|", 7)]
            id_, preset, fmt, kt, c, prods, expect, cite = cols
            pairs = []
            for p in prods.split(","):
                a, b = p.split("@")
                pairs.append((a.strip(), b.strip()))
            rows.append(dict(id=id_, preset=preset, fmt=fmt, kt=int(kt), c=c, prods=pairs,
                             expect=expect, cite=cite))
    return rows


def fp32_expect_bits(expect: str, nan_bits: int) -> int:
    v = parse_value(expect)
    if v in ("nan", "-nan"):
        return nan_bits
    if v == "0":
        return 0
    return encode_exact(v, "fp32")


def encode_row(row, enc="ocp"):
    """(a bits list, b bits list, c bits) of a fixture row in its input format."""
    fmt = row["fmt"]
    a = [encode_exact(parse_value(x), fmt, enc) for x, _ in row["prods"]]
    b = [encode_exact(parse_value(y), fmt, enc) for _, y in row["prods"]]
    c = encode_exact(parse_value(row["c"]), "fp32")
    return a, b, c
