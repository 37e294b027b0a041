"""Streamed whole-checkpoint validation on the GPU.

The counterpart of the pages' reproduction protocol ("Compresión de pesos LLM
sin pérdida vs 8-bit GGUF", section "¿Qué demostró realmente el
experimento con GLM-5.2?"; "Prueba de GLM-5.2 reduce la memoria BF16 en casi
un 25%", closing paragraph): stream a checkpoint tensor by tensor, check the
byte-split reconstruction bit for bit, compute the K15 accounting, and keep
going without holding the whole checkpoint.  Here the checkpoint is the
seeded checkpoint-shaped synthetic set (the real one is not available), the
tensors are drawn on the device in batches of at most ``batch_bytes`` of
BF16, and each batch is encoded with one batched call per scheme, decoded
with one batched call, and compared with the source on the device.

Every (tensor, scheme) result is appended to a JSON-lines log; a rerun with
the same log skips what is already there (resume after an interruption).

    python -m decode_gemv_sign_gb300.validate --workload checkpoint --log run.jsonl
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time
from typing import Dict, List, Optional, Sequence

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

SCHEME_NAMES = {0: "bytesplit", 1: "k15"}


def _batches(specs, batch_bytes: int):
    cur, size = [], 0
    for s in specs:
        b = 2 * s.n
        if cur and size + b > batch_bytes:
            yield cur
            cur, size = [], 0
        cur.append(s)
        size += b
    if cur:
        yield cur


def _read_log(path: Optional[str]) -> Dict[tuple, dict]:
    """Finished (tensor, scheme) records of a JSON-lines log.

    Only newline-terminated lines count: text after the last newline is a
    record an interruption cut short, and its tensor is validated again.  A
    malformed line before that is an error (the log was damaged otherwise).
    """
    done = {}
    if path and os.path.exists(path):
        with open(path) as f:
            complete = f.read().split("\n")[:-1]
        for line in complete:
            line = line.strip()
            if not line:
                continue
            r = json.loads(line)
            done[(r["name"], r["scheme"])] = r
    return done


def _open_log(path: str):
    """Open the log for appending, after dropping an unterminated last line
    (see _read_log) so the next record starts on a line of its own."""
    if os.path.exists(path):
        with open(path, "r+b") as f:
            data = f.read()
            keep = data.rfind(b"\n") + 1
            if keep != len(data):
                f.truncate(keep)
    return open(path, "a")


def validate(specs: Sequence, schemes: Sequence[int] = (0, 1), batch_bytes: int = 16 << 30,
             log_path: Optional[str] = None, device: str = "cuda") -> dict:
    """Encode, decode and compare every tensor of ``specs`` in every scheme.

    Returns totals per scheme: tensors, elements, escapes, serialized bytes,
    entropy-accounting bits, both bits/weight figures, the reduction against
    BF16, and the list of tensors whose round trip was not bit-exact (empty
    when everything matched).
    """
    import torch

    from decode_gemv_sign_gb300 import synth
    from decode_gemv_sign_gb300 import wcomp as W

    dev = torch.device(device)
    done = _read_log(log_path)
    log = _open_log(log_path) if log_path else None
    t0 = time.perf_counter()
    try:
        for batch in _batches(specs, batch_bytes):
            todo = [(s, sc) for s in batch for sc in schemes if (s.name, sc) not in done]
            if not todo:
                continue
            need = {s.name: s for s, _ in todo}
            ws = {name: synth.gen_weights_torch(s, dev) for name, s in need.items()}
            for sc in schemes:
                items = [s for s, c in todo if c == sc]
                if not items:
                    continue
                cs = W.encode_batched([ws[s.name] for s in items], sc)
                outs = W.decode_batched(cs)
                for s, c, o in zip(items, cs, outs):
                    inf = c.info()
                    exact = bool(torch.equal(ws[s.name].view(-1), o.view(-1)))
                    rec = {"name": s.name, "scheme": sc, "N": s.N, "K": s.K, "n": inf["n"],
                           "escapes": inf["n_escapes"], "serialized_bytes": inf["serialized_bytes"],
                           "serialized_compact_bytes": inf["serialized_compact_bytes"],
                           "entropy_bpw": inf["entropy_bpw"], "exact": exact}
                    done[(s.name, sc)] = rec
                    if log:
                        log.write(json.dumps(rec) + "\n")
                for c in cs:
                    c.free()
                del outs
            if log:
                log.flush()
            del ws
            torch.cuda.synchronize()
    finally:
        if log:
            log.close()
    elapsed = time.perf_counter() - t0
    names = [s.name for s in specs]
    out = {"tensors": len(specs), "seconds": round(elapsed, 2), "schemes": {}}
    for sc in schemes:
        recs = [done[(nm, sc)] for nm in names if (nm, sc) in done]
        n = sum(r["n"] for r in recs)
        ser = sum(r["serialized_bytes"] for r in recs)
        ser_c = sum(r.get("serialized_compact_bytes", r["serialized_bytes"]) for r in recs)
        ebits = sum(r["entropy_bpw"] * r["n"] for r in recs)
        bpw_e = ebits / n if n else 0.0
        out["schemes"][SCHEME_NAMES[sc]] = {
            "tensors": len(recs), "elements": n, "escapes": sum(r["escapes"] for r in recs),
            "serialized_bytes": ser, "source_bytes": 2 * n,
            "entropy_bpw": round(bpw_e, 5), "physical_bpw": round(8.0 * ser / n, 5) if n else 0.0,
            "entropy_reduction_pct": round(100.0 * (1 - bpw_e / 16.0), 3) if n else 0.0,
            "physical_reduction_pct": round(100.0 * (1 - ser / (2.0 * n)), 3) if n else 0.0,
            "serialized_compact_bytes": ser_c,
            "physical_compact_bpw": round(8.0 * ser_c / n, 5) if n else 0.0,
            "physical_compact_reduction_pct": round(100.0 * (1 - ser_c / (2.0 * n)), 3) if n else 0.0,
            "not_exact": [r["name"] for r in recs if not r["exact"]],
        }
    return out


def main(argv: Optional[List[str]] = None):
    from decode_gemv_sign_gb300 import build, synth

    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="checkpoint", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--layers", type=int, default=None, help="checkpoint workload: number of layers (default 113)")
    ap.add_argument("--batch-gib", type=float, default=16.0)
    ap.add_argument("--log", default=None, help="JSON-lines result log; finished tensors are skipped on rerun")
    ap.add_argument("--schemes", default="bytesplit,k15")
    a = ap.parse_args(argv)
    build.build()
    if a.workload == "checkpoint" and a.layers is not None:
        specs = synth.workload_checkpoint(a.layers)
    else:
        specs = synth.WORKLOADS[a.workload]()
    schemes = [{"bytesplit": 0, "k15": 1}[x] for x in a.schemes.split(",")]
    res = validate(specs, schemes, int(a.batch_gib * (1 << 30)), a.log)
    print(json.dumps(res))
    bad = any(v["not_exact"] for v in res["schemes"].values())
    sys.exit(1 if bad else 0)


if __name__ == "__main__":
    main()
