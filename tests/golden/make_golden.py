"""Writes tests/golden/h_k3_seed1.txt from the CPU oracle (and only the oracle).

The stored example: the proving-key-shaped synthetic problem of a 2^3 domain drawn with
seed 1, and the oracle's h in both encodings. Run from the repository root:
    python tests/golden/make_golden.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle import fr_int as F  # noqa: E402
from bn254_scalar_field_gb300 import synth  # noqa: E402


def main():
    A, B, w = synth.problem(3, seed=1)
    hm, hs = oracle.compute_h(3, A, B, w)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "h_k3_seed1.txt")
    with open(path, "w") as f:
        f.write("# h for synth.problem(3, seed=1), written by tests/golden/make_golden.py\n")
        f.write("# from the CPU oracle: '<encoding> <index> <value as hex>'.\n")
        for name, arr in (("h_mont", hm), ("h_std", hs)):
            for i, v in enumerate(F.array_to_ints(arr)):
                f.write("%s %d 0x%064x\n" % (name, i, v))


if __name__ == "__main__":
    main()
