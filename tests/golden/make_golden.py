"""Writes the stored expected values under tests/golden/ using only ``oracle``.

    python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def write_local_lens():
    path = os.path.join(HERE, "dcp_local_lens.txt")
    with open(path, "w") as f:
        f.write("# Rank-local lengths under the round-robin owner rule (token t -> rank t mod P).\n")
        f.write("# P and L are the grid of the decode-layout test in sglang pull 33926\n")
        f.write("# (test snippet TestDcpDecodeLayout: SIZES = 1,2,3,4,8; LENS = 0..40).\n")
        f.write("# columns: P L len(rank 0) ... len(rank P-1)\n")
        for p in [1, 2, 3, 4, 8]:
            for L in range(0, 41):
                lens = [oracle.local_len(L, p, r) for r in range(p)]
                f.write(f"{p} {L} " + " ".join(map(str, lens)) + "\n")


if __name__ == "__main__":
    write_local_lens()
