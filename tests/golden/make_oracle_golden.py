"""Write oracle_rows_causal_L2048.txt: fp64 oracle rows for the causal L=2048 workload.

Calls only ``oracle/`` (and the seeded input generator). The stored values guard the
oracle against unintended changes; they are not an independent pin.
Run from the repository root:  python tests/golden/make_oracle_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from seeded_inputs import CAUSAL_B1_H4_L2048_D64 as W, bits16, make_qkv  # noqa: E402

ROWS = [0, 1, 2, 127, 128, 1000, 2047, 2048 + 5, 3 * 2048 + 2047]


def main():
    q, k, v = make_qkv(W)
    o, lse = oracle.default().attn_rows(bits16(q), bits16(k), bits16(v), W.dtype, W.causal,
                                        W.window_left, W.scale, np.array(ROWS))
    with open(os.path.join(HERE, "oracle_rows_causal_L2048.txt"), "w") as f:
        f.write(f"# workload {W.name} seed {W.seed}; row = (b*Hq + h)*L + i; "
                "written by tests/golden/make_oracle_golden.py (oracle only)\n")
        for r, orow, l in zip(ROWS, o, lse):
            f.write(f"{r} {float(l)!r} " + " ".join(repr(float(x)) for x in orow) + "\n")


if __name__ == "__main__":
    main()
