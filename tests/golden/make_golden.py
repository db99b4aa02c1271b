"""Writes the stored expected values under tests/golden/ from the oracle alone.

Run from the repository root: python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import nf4_oracle as o  # noqa: E402


def main():
    lv = o.nf4_levels()
    with open(os.path.join(HERE, "nf4_levels.txt"), "w") as f:
        f.write("# NF4 levels, fp32, index / hex bits / value.\n")
        f.write("# Definition: standard-normal quantiles at evenly spaced probabilities,\n")
        f.write("# 7 negative, exact 0, 8 positive, normalised to [-1, 1]\n")
        f.write("# (\"bitsandbytes\", NF4 paragraph; \"Zenbit\", zenbit.nf4 bullet).\n")
        f.write("# Written by tests/golden/make_golden.py from the oracle.\n")
        for i, v in enumerate(lv):
            f.write(f"{i} {int(v.view('uint32')):08x} {float(v)!r}\n")


if __name__ == "__main__":
    main()
