"""Writes int8_block0_mnn_fill.txt: the Int8-Block0 codes the benchmark page's weight fill
must produce, derived by exact rational arithmetic from the page's formula alone.

Source: "MNN GemmSpeed 基准测试实战", section «为什么用 Conv1x1 来测 GEMM»: weight shape
{ic, oc} = {K, N}, fill ((i % 127) - 63) / 1000, Int8-Block0 = nbit 8 with one block over all
of K. With K = 4096 = 32 (mod 127) and gcd(32, 127) = 1, every channel n sees every residue
r = (32 k + n) mod 127, so each channel's min is -63/1000 and max 63/1000; the asymmetric
8-bit code of residue r is then round(r * 255 / 126). Where that quotient is exactly half way
(r = 21, 63, 105) float32 rounding may land on either neighbour, so both are listed.
This script uses only integer/rational arithmetic (no oracle, no GPU).
"""
import os
from fractions import Fraction

HERE = os.path.dirname(os.path.abspath(__file__))


def main():
    lines = [
        "# Int8-Block0 codes of the benchmark page's fill ((i % 127) - 63) / 1000, K = N = 4096",
        "# source: 'MNN GemmSpeed 基准测试实战', «为什么用 Conv1x1 来测 GEMM»; written by make_int8_fill_golden.py",
        "# every channel: offset = -63/1000 (as float32), max = 63/1000, 255 levels",
        "# columns: residue r (value (r - 63)/1000) and the allowed codes",
    ]
    for r in range(127):
        x = Fraction(r * 255, 126)
        lo = x.numerator // x.denominator
        frac = x - lo
        if frac == Fraction(1, 2):
            codes = [lo, lo + 1]
        elif frac < Fraction(1, 2):
            codes = [lo]
        else:
            codes = [lo + 1]
        lines.append(f"{r} " + "|".join(str(c) for c in codes))
    with open(os.path.join(HERE, "int8_block0_mnn_fill.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
