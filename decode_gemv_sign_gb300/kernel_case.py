"""Run one library operation on a seeded slice of the benchmark's workload, for profiler captures.

    python -m decode_gemv_sign_gb300.kernel_case --op decode --scheme both --reps 2
    python -m decode_gemv_sign_gb300.kernel_case --op gemv --scheme k15 --batch 1 --rows 4096

Inputs, drawn on the device:
  * encode / decode: one layer of the checkpoint-shaped set (the 17 tensors
    that follow the two embeddings in its first 16 GiB batch: 4 x 6144x6144,
    2 x 16384x6144, 6144x16384, 8 x 2048x6144, 2 norms; 1.1 GB of BF16, far
    larger than L2), or the first `--tensors` of them;
  * gemv / gemv_bf16: the first `--rows` rows of the 16384x53248 GEMV weight
    (all of them by default; 4096 rows are 436 MB of BF16), or with
    `--dense12` the escape-free weight of the same shape.
The operation runs `--reps` times after the containers are built, one
batched launch per repetition.  Exits non-zero if a decode is not bit-exact
or a GEMV kernel reports an error.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def layer_specs(count: int):
    from decode_gemv_sign_gb300 import synth

    return synth.checkpoint_batch(0)[2:2 + count]


def main():
    import torch

    from decode_gemv_sign_gb300 import accounting, build, synth
    from decode_gemv_sign_gb300 import wcomp as W

    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["encode", "decode", "gemv", "gemv_bf16"], required=True)
    ap.add_argument("--scheme", choices=["bytesplit", "k15", "both"], default="bytesplit",
                    help="both: every tensor in both schemes, one batch (the benchmark's encode and decode)")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--tensors", type=int, default=17)
    ap.add_argument("--rows", type=int, default=16384)
    ap.add_argument("--dense12", action="store_true")
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args()
    build.build()
    dev = torch.device("cuda")
    if a.op in ("gemv", "gemv_bf16"):
        base = synth.dense12_spec() if a.dense12 else synth.checkpoint_gemv_spec()
        specs = [dataclasses.replace(base, N=min(a.rows, base.N))]
    else:
        specs = layer_specs(a.tensors)
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
    xs = [synth.gen_x_torch(a.batch, s.K, 5 + i, dev) for i, s in enumerate(specs)]
    if a.op == "gemv_bf16":
        for _ in range(a.reps):
            W.gemv_bf16_batched(ws, xs)
        torch.cuda.synchronize()
        print(json.dumps({"op": a.op, "algorithmic_bytes_per_rep": sum(
            accounting.plain_bytes(s.N, s.K, a.batch) for s in specs)}))
        return
    cs = W.encode_batched(ws, schemes)
    outs = [torch.empty_like(w) for w in ws]
    for _ in range(a.reps):
        if a.op == "decode":
            W.decode_batched(cs, outs)
        else:
            W.gemv_batched(cs, xs)
    torch.cuda.synchronize()
    if a.op == "decode":
        for w, o in zip(ws, outs):
            if not torch.equal(w, o):
                sys.exit("decode mismatch")
    if W.lib().wcomp_device_check(None) != W.OK:
        sys.exit("device error word set")
    infos = [c.info() for c in cs]
    per = [accounting.decode_bytes(i) if a.op == "decode" else accounting.gemv_bytes(i, a.batch) for i in infos]
    print(json.dumps({"op": a.op, "algorithmic_bytes_per_rep": sum(per),
                      "elements": sum(i["n"] for i in infos), "escapes": sum(i["n_escapes"] for i in infos)}))


if __name__ == "__main__":
    main()
