"""Writes e4m3_positive_values.txt: the value of every non-negative finite FP8 E4M3 code,
from the format's definition alone (exact rational arithmetic; nothing from oracle/ or the
library). Definition (OCP 8-bit Floating Point Specification, E4M3): 1 sign, 4 exponent and
3 mantissa bits, exponent bias 7; exponent field 0 holds the subnormals m/8 * 2^-6; there are
no infinities, and only S.1111.111 is NaN, so the largest finite value is 1.75 * 2^8 = 448."""

import os
from fractions import Fraction


def value(code):
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0:
        return Fraction(m, 8) * Fraction(1, 2 ** 6)
    return (1 + Fraction(m, 8)) * (Fraction(2) ** (e - 7))


def main():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "e4m3_positive_values.txt")
    with open(path, "w") as f:
        f.write("# FP8 E4M3 (OCP 8-bit floating point specification): bias 7, subnormals m/8*2^-6,\n")
        f.write("# no infinities, 0x7F = NaN. Written by make_e4m3_table.py from the definition.\n")
        f.write("# code value(exact fraction)\n")
        for code in range(0x7F):
            v = value(code)
            f.write(f"0x{code:02X} {v.numerator}/{v.denominator}\n")


if __name__ == "__main__":
    main()
