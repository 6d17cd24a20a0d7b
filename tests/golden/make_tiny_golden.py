"""Write tests/golden/tiny_step.txt: the oracle's result for the tiny workload.

Calls only the oracle (and the seeded input generator).  The file is a
regression pin: it changes only when the oracle's arithmetic changes, and such
a change must name the passage that justifies it.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from paged_gqa_decode_step_gb300 import workloads as wl  # noqa: E402


def compute():
    w = wl.TINY
    a = {k: wl.to_numpy(v) for k, v in wl.generate(w, "cpu").items()}
    shape = oracle.make_shape(w.rows, w.heads, w.kv_heads, w.head_dim, w.pages_per_row,
                              a["k_pool"].shape[0], oracle.BF16, window=w.window, rope_theta=w.rope_theta)
    q_rot, out, _, rc = oracle.step(shape, a["q"], a["k_new"], a["v_new"], a["positions"], a["table"],
                                    a["k_pool"], a["v_pool"])
    assert rc == 0
    return q_rot, out


def main():
    q_rot, out = compute()
    path = os.path.join(HERE, "tiny_step.txt")
    with open(path, "w") as f:
        f.write("# tiny workload (Rows 2, Heads 8, KvHeads 8, D 64, positions 37 and 100, theta 1e4,\n")
        f.write("# seed 1000): bf16 bit patterns (hex) of the oracle's rotated q and attention output.\n")
        f.write("# Written by tests/golden/make_tiny_golden.py from the oracle alone.\n")
        for name, arr in (("q_rot", q_rot), ("out", out)):
            flat = arr.reshape(-1)
            f.write(f"{name} {arr.shape[0]} {arr.shape[1]} {arr.shape[2]}\n")
            for i in range(0, flat.size, 16):
                f.write(" ".join(f"{int(v):04x}" for v in flat[i:i + 16]) + "\n")
    print(path)


if __name__ == "__main__":
    main()
