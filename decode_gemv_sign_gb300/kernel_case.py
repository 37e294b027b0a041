"""Run one library operation on one seeded workload tensor set, for profiler captures.

    python -m decode_gemv_sign_gb300.kernel_case --op decode --scheme k15 --reps 3
    python -m decode_gemv_sign_gb300.kernel_case --op gemv --scheme bytesplit --batch 1

The inputs are the first `--tensors` tensors of the dense-layer workload (all
seven by default: 4 x 4096x4096 and 3 x 4096x11008, 386 MB of BF16, larger
than L2), drawn on the device; the operation runs `--reps` times after the
containers are built, as one batched launch per repetition.  Exits non-zero if
a decode is not bit-exact.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch

    from decode_gemv_sign_gb300 import build, synth
    from decode_gemv_sign_gb300 import wcomp as W

    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["encode", "decode", "gemv", "gemv_bf16"], required=True)
    ap.add_argument("--scheme", choices=["bytesplit", "k15", "both"], default="bytesplit",
                    help="both: every tensor in both schemes, one batch (the benchmark's decode launch)")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--tensors", type=int, default=7)
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args()
    build.build()
    dev = torch.device("cuda")
    specs = synth.workload_dense_layers()[: a.tensors]
    ws = [synth.gen_weights_torch(s, dev) for s in specs]
    if a.scheme == "both":
        specs = [s for s in specs for _ in (0, 1)]
        ws = [w for w in ws for _ in (0, 1)]
        schemes = [0, 1] * (len(ws) // 2)
    else:
        schemes = [W.SCHEMES[a.scheme]] * len(ws)
    if a.op == "encode":
        for _ in range(a.reps):
            for c in W.encode_batched(ws, schemes):
                c.free()
        torch.cuda.synchronize()
        return
    cs = W.encode_batched(ws, schemes)
    xs = [synth.gen_x_torch(a.batch, s.K, 5 + i, dev) for i, s in enumerate(specs)]
    outs = [torch.empty_like(w) for w in ws]
    for _ in range(a.reps):
        if a.op == "decode":
            W.decode_batched(cs, outs)
        elif a.op == "gemv":
            W.gemv_batched(cs, xs)
        else:
            W.gemv_bf16_batched(ws, xs)
    torch.cuda.synchronize()
    if a.op == "decode":
        for w, o in zip(ws, outs):
            if not torch.equal(w, o):
                sys.exit("decode mismatch")


if __name__ == "__main__":
    main()
