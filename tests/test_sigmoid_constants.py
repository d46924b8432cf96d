"""The constants of the library's fp32 sigmoid (csrc/sigmoid.cuh) against
decimal arithmetic: the 2^(j/32) table pairs, the three-part ln2/32 split and
32/ln2.  Reads the header as text; no GPU."""

import os
import re
from decimal import Decimal, getcontext

import numpy as np

from conftest import ROOT

getcontext().prec = 80
HDR = os.path.join(ROOT, "confidence_scheduled_speculative_gb300", "csrc", "sigmoid.cuh")


def _hexf(s: str) -> Decimal:
    return Decimal(float.fromhex(s.rstrip("f")))


def _text():
    with open(HDR) as f:
        return f.read()


def test_exp2_table_pairs():
    body = _text().split("kExp2Tab[32] = {")[1].split("};")[0]
    pairs = re.findall(r"\{(-?0x[0-9a-fp.+-]+f), (-?0x[0-9a-fp.+-]+f)\}", body)
    assert len(pairs) == 32
    for j, (hi, lo) in enumerate(pairs):
        v = Decimal(2) ** (Decimal(j) / 32)
        h, l = _hexf(hi), _hexf(lo)
        assert h == Decimal(float(np.float32(float(v)))), j      # hi: the fp32 rounding
        assert abs(h + l - v) / v < Decimal(2) ** -49, j          # pair within 2^-49
        assert Decimal(float(np.float32(float(l)))) == l          # lo is an fp32 value


def test_ln2_split_and_inverse():
    t = _text()
    get = lambda name: _hexf(re.search(rf"{name} = (-?0x[0-9a-fp.+-]+f);", t).group(1))
    L1, L2, L3, inv = get("kL1"), get("kL2"), get("kL3"), get("kInvL")
    L = Decimal(2).ln() / 32
    # L1 has at most 12 significant bits, so k*L1 is exact for |k| < 4096
    m = L1 * Decimal(2) ** 17
    assert m == m.to_integral_value() and m < 4096
    assert abs(L1 + L2 + L3 - L) < Decimal(2) ** -68
    assert inv == Decimal(float(np.float32(float(Decimal(32) / Decimal(2).ln()))))
    # |t| <= 60 keeps k*32 in range of 12 bits and 2^m normal
    assert 60 * float(inv) < 4096
