"""Writes the stored expected values under tests/golden/.

Calls only the oracle (``oracle/``); nothing here touches the CUDA library.
Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def mulberry32_draws():
    path = os.path.join(HERE, "mulberry32_draws.txt")
    with open(path, "w") as f:
        f.write("# mulberry32 raw uint32 draws (\"PlayTrain\", Appendix F.2 listing\n")
        f.write("# \"seeded RNG\"; the listing divides these by 2^32).\n")
        f.write("# Written by tests/golden/make_golden.py from the oracle.\n")
        f.write("# columns: seed draw_index value\n")
        for seed in (0, 1, 12345, 0xFFFFFFFF):
            d = oracle.mulberry32_stream(seed, 8)
            for k in range(8):
                f.write(f"{seed} {k} {int(d[k])}\n")


if __name__ == "__main__":
    mulberry32_draws()
