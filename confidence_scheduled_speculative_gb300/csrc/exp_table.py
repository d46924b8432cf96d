"""Print the constants of sigmoid.cuh from decimal arithmetic.

2^(j/32) for j = 0..31 as an fp32 pair (hi = the fp32 rounding, lo = the fp32
rounding of the remainder), ln2/32 as kL1 (12 significant bits) + kL2 (24) +
kL3, and 32/ln2 rounded to fp32.  Run: python exp_table.py
"""

from decimal import Decimal, getcontext

import numpy as np

getcontext().prec = 80


def f32_hex(d) -> str:
    mant, exp = float(np.float32(float(d))).hex().split("p")
    mant = mant.rstrip("0")
    return (mant + "0" if mant.endswith(".") else mant) + "p" + exp


def round_bits(d: Decimal, bits: int) -> Decimal:
    e, a = 0, abs(d)
    while a >= 1:
        a /= 2
        e += 1
    while a < Decimal("0.5"):
        a *= 2
        e -= 1
    scale = Decimal(2) ** (bits - e)
    return (d * scale).to_integral_value() / scale


def main() -> None:
    ln2 = Decimal(2).ln()
    L = ln2 / 32
    L1 = round_bits(L, 12)
    L2 = round_bits(L - L1, 24)
    L3 = L - L1 - L2
    print(f"kL1 = {f32_hex(L1)}f  kL2 = {f32_hex(L2)}f  kL3 = {f32_hex(L3)}f  "
          f"kInvL = {f32_hex(Decimal(32) / ln2)}f")
    for j in range(32):
        v = Decimal(2) ** (Decimal(j) / 32)
        hi = np.float32(float(v))
        lo = np.float32(float(v - Decimal(float(hi))))
        print(f"{{{f32_hex(Decimal(float(hi)))}f, {f32_hex(Decimal(float(lo)))}f}},")


if __name__ == "__main__":
    main()
