"""Write the regression fixture ``c0_oracle.txt`` from the oracle alone.

The pages print no worked example (no attention values, no LSE, no
acceptance counts), so nothing here is a page value.  This fixture records
the oracle's own c0 results so that any later change of the oracle's
arithmetic shows up as a diff; it is not an independent pin (those live in
tests/pins.py).  Run:  python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from oracle import ref_verify_step  # noqa: E402
from workloads import make_inputs  # noqa: E402


def main():
    inp = make_inputs("c0", seed=0)
    ref = ref_verify_step(inp)
    lines = ["# c0 (seed 0) oracle results: lse[t][h] (natural log), out checksums, greedy outputs",
             "# written by tests/golden/make_golden.py from oracle/ only"]
    for t in range(inp["T"]):
        lines.append("lse %d " % t + " ".join("%.15e" % v for v in ref["lse"][t]))
    for t in range(inp["T"]):
        lines.append("outsum %d " % t + " ".join("%.15e" % v for v in ref["out"][t].sum(axis=1)))
    for key in ("argmax", "accepted", "next_tokens", "kv_lens_out"):
        lines.append(key + " " + " ".join(str(int(v)) for v in ref[key]))
    with open(os.path.join(HERE, "c0_oracle.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
