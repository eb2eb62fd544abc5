"""Writes the oracle-derived regression fixtures in this folder.

Calls only ``oracle``; run from the repository root:
    python tests/golden/make_golden.py
"""

import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as orc  # noqa: E402


def main():
    om = orc.build_omega(0, 8, 4, orthogonal=True)
    np.savetxt(os.path.join(HERE, "omega_seed0_m8_d4.txt"), om, fmt="%.17e",
               header="Omega (ORF, seed 0, m 8, d 4) from oracle.build_omega; regression pin")


if __name__ == "__main__":
    main()
