"""Writes the stored container fixtures from the CPU oracle (and nothing else).

Run from the repository root:  python tests/golden/make_golden.py
The fixtures freeze container version 1 for a small seeded tensor (5 x 200,
Student-t(4) at std 0.02 with 5% N(0, 100^2) outliers, so both schemes carry escapes and the
element count is not a multiple of the 32-element group).
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from decode_gemv_sign_gb300 import synth  # noqa: E402
from oracle import wcomp_oracle as O  # noqa: E402

SPEC = synth.WeightSpec("golden", 5, 200, "t4", 0.02, 0.05, "normal", 100.0, seed=77)


def build():
    w = synth.gen_weights_np(SPEC)
    out = {"_source": "written by tests/golden/make_golden.py from the CPU oracle",
           "N": SPEC.N, "K": SPEC.K, "weights_hex": w.astype("<u2").tobytes().hex()}
    for scheme, name in ((O.BYTESPLIT, "bytesplit"), (O.K15, "k15")):
        c = O.encode(w, scheme)
        out[name] = {"E": c.E, "table": [int(t) for t in c.table],
                     "container_hex": O.serialize(c).hex()}
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "containers_5x200.json"), "w") as f:
        json.dump(build(), f, indent=1)
        f.write("\n")
