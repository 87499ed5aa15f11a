"""Writes tiny_oracle_rows.txt: oracle outputs for a few rows of the tiny
configuration (1 sequence, 256 + 5 tokens, 4 q / 1 kv heads, D = 64, bf16
KV).  It calls only the oracle and the seeded input generator; the stored
values are a regression pin for the oracle, not an independent check."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from speculative_decoding_verify_causal_gb300 import workloads as wl  # noqa: E402

ROWS = [(0, 0, 0), (0, 2, 1), (0, 4, 3), (0, 3, 2)]


def main():
    w = wl.config_workload("tiny")
    o, l = oracle.verify_attn_rows(w, ROWS)
    with open(os.path.join(HERE, "tiny_oracle_rows.txt"), "w") as f:
        f.write("# b t h lse out[0..63]; tiny config, seed 20260; written by make_golden.py\n")
        for (b, t, h), lse, out in zip(ROWS, l, o):
            f.write(f"{b} {t} {h} {float(lse)!r} " + " ".join(repr(float(x)) for x in out) + "\n")


if __name__ == "__main__":
    main()
