"""Streamed whole-checkpoint validation on the GPU.

The counterpart of the pages' reproduction protocol and production pilot
("Compresión de pesos LLM sin pérdida vs 8-bit GGUF", sections "¿Qué demostró
realmente el experimento con GLM-5.2?" and "Un piloto de producción de 14
días": decode every tensor, compare byte by byte, validate hashes, inject
corruption; "Prueba de GLM-5.2 reduce la memoria BF16 en casi un 25%",
closing paragraph: the checkpoint is checked tensor by tensor without holding
it whole).  Here the checkpoint is the seeded checkpoint-shaped synthetic set
(the real one is not available).

Tensors are taken in batches of at most ``batch_bytes`` of BF16.  A batch is
encoded with one batched call per scheme, decoded with one batched call and
compared with its source on the device.  With ``source="host"`` the batches
live in pinned host memory, as a checkpoint read from storage would: each one
is copied to the device on a copy stream while the previous batch is encoded
and decoded (two host and two device buffers alternate); the host buffers are
filled by drawing the synthetic tensors on the device and copying them back,
in place of reading shards.  With ``source="device"`` each batch is drawn
straight on the device (no transfer), for runs over the whole set.  Both
modes draw the same bytes.

Optional checks per tensor:
  * ``hashes``: BLAKE2b-128 of the source bytes (taken on the host from the
    bytes the pipeline was given) and of every decoded copy (read back); the
    two must agree.  The hashes run in a pool of host threads while the GPU
    goes on, and a batch's records are logged once its hashes are in;
  * ``corrupt_every`` (k > 0): every k-th tensor (and scheme) is serialized in
    both forms, one seeded byte of each is flipped on the host, and
    wcomp_deserialize must refuse both as corrupt (the CRC-32 over header and
    payload detects every error burst up to 32 bits long).

Every (tensor, scheme) result is appended to a JSON-lines log; a rerun with
the same log skips what is already there (resume after an interruption).

    python -m decode_gemv_sign_gb300.validate --workload checkpoint --log run.jsonl
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
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
    from decode_gemv_sign_gb300 import synth

    return synth.batches(specs, batch_bytes)


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


def tensor_hash(t) -> str:
    """BLAKE2b-128 of a tensor's bytes (a host tensor is hashed in place)."""
    import numpy as np

    a = t.cpu() if t.is_cuda else t
    return hashlib.blake2b(np.ascontiguousarray(a.numpy()).view(np.uint8), digest_size=16).hexdigest()


def corruption_check(W, c, seed: int) -> dict:
    """Serialize c in both forms, flip one seeded byte of each (header or
    payload) and check that wcomp_deserialize refuses it."""
    import numpy as np

    rng = np.random.default_rng(seed)
    out = {}
    for form, compact in (("v1", False), ("compact", True)):
        buf = bytearray(W.serialize(c, compact=compact))
        off = int(rng.integers(0, len(buf)))
        buf[off] ^= int(rng.integers(1, 256))
        try:
            W.deserialize(bytes(buf)).free()
            out[form] = {"offset": off, "detected": False}
        except W.CorruptContainer:
            out[form] = {"offset": off, "detected": True}
    return out


class _HostStream:
    """Batches staged in pinned host memory and copied to the device on a copy
    stream, two buffers deep: batch k+1 is filled and copied while batch k is
    processed."""

    def __init__(self, torch, batches, batch_bytes: int, device, fill):
        self.torch = torch
        self.batches = batches
        elems = max(sum((s.n + 7) // 8 * 8 for s in b) for b in batches) if batches else 0
        from decode_gemv_sign_gb300.hostmem import PinnedBuffer

        self._bufs = [PinnedBuffer(torch, elems, torch.int16) for _ in range(2)]
        self.host = [b.tensor for b in self._bufs]
        self.dev = [torch.empty(elems, dtype=torch.int16, device=device) for _ in range(2)]
        self.copy = torch.cuda.Stream(device=device)
        self.ready = [torch.cuda.Event(), torch.cuda.Event()]
        self.free = [torch.cuda.Event(), torch.cuda.Event()]
        self.fill = fill
        self.pending = {}

    @staticmethod
    def views(flat, specs):
        out, o = [], 0
        for s in specs:
            out.append(flat[o:o + s.n].view(s.N, s.K))
            o += (s.n + 7) // 8 * 8
        return out

    def start(self, k: int):
        """Fill host buffer k % 2 with batch k and queue its copy to the device."""
        if k >= len(self.batches) or k in self.pending:
            return
        i = k % 2
        self.free[i].synchronize()  # the device buffer's previous batch is done with it
        hv = self.views(self.host[i], self.batches[k])
        self.fill(self.batches[k], hv)
        used = sum((s.n + 7) // 8 * 8 for s in self.batches[k])
        self.copy.wait_event(self.free[i])
        with self.torch.cuda.stream(self.copy):
            self.dev[i][:used].copy_(self.host[i][:used], non_blocking=True)
        self.ready[i].record(self.copy)
        self.pending[k] = (hv, self.views(self.dev[i], self.batches[k]))

    def take(self, k: int, stream):
        """Host and device views of batch k, ordered after its copy on `stream`."""
        self.start(k)
        stream.wait_event(self.ready[k % 2])
        return self.pending.pop(k)

    def release(self, k: int, stream):
        self.free[k % 2].record(stream)


def _fill_host(specs, views):
    """Fill the batch's pinned host views, standing in for reading the shards
    from storage.  Each tensor is drawn on the device (the same draw as
    ``source="device"``, so both modes validate the same bytes) on a stream of
    its own and copied into its host view; torch's CPU generator took tens of
    seconds per GB, which would have made the synthetic draw, not the
    pipeline, the bound of a host-streamed run."""
    import torch

    from decode_gemv_sign_gb300 import synth

    fill_stream = torch.cuda.Stream()
    with torch.cuda.stream(fill_stream):
        for s, v in zip(specs, views):
            v.copy_(synth.gen_weights_torch(s, "cuda"), non_blocking=True)
    fill_stream.synchronize()


def validate(specs: Sequence, schemes: Sequence[int] = (0, 1), batch_bytes: int = 16 << 30,
             log_path: Optional[str] = None, device: str = "cuda", source: str = "device",
             hashes: bool = False, corrupt_every: int = 0, fill=None) -> dict:
    """Encode, decode and compare every tensor of ``specs`` in every scheme.

    Returns totals per scheme: tensors, elements, escapes, serialized bytes,
    entropy-accounting bits, both bits/weight figures, the reduction against
    BF16, the list of tensors whose round trip was not bit-exact, those whose
    hashes differ (when hashed) and the corruption checks run and missed.
    """
    import torch

    from decode_gemv_sign_gb300 import synth
    from decode_gemv_sign_gb300 import wcomp as W

    if source not in ("device", "host"):
        raise ValueError("source must be 'device' or 'host'")
    dev = torch.device(device)
    done = _read_log(log_path)
    log = _open_log(log_path) if log_path else None
    batches = [b for b in _batches(specs, batch_bytes) if any((s.name, sc) not in done for s in b for sc in schemes)]
    stream = torch.cuda.current_stream(dev)
    feeder = _HostStream(torch, batches, batch_bytes, dev, fill or _fill_host) if source == "host" else None
    hasher = cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) if hashes else None
    index = {s.name: i for i, s in enumerate(specs)}
    t0 = time.perf_counter()
    try:
        for k, batch in enumerate(batches):
            todo = [(s, sc) for s in batch for sc in schemes if (s.name, sc) not in done]
            if feeder:
                hv, dv = feeder.take(k, stream)
                src = {s.name: v for s, v in zip(batch, dv)}
                host_src = {s.name: v for s, v in zip(batch, hv)}
            else:
                src = {s.name: synth.gen_weights_torch(s, dev) for s in batch}
                host_src = None
            # source hashes from the bytes the pipeline was given, computed on
            # the host while the GPU works
            src_hash = {}
            if hasher:
                todo_names = {s.name for s, _ in todo}
                for s in batch:
                    if s.name in todo_names:
                        src_hash[s.name] = hasher.submit(tensor_hash, host_src[s.name] if host_src else src[s.name].cpu())
            # records of this batch, completed once their hashes are in
            pending = []
            for sc in schemes:
                items = [s for s, c in todo if c == sc]
                if not items:
                    continue
                cs = W.encode_batched([src[s.name] for s in items], sc, stream=stream)
                outs = W.decode_batched(cs, stream=stream)
                if feeder and k + 1 < len(batches) and sc == schemes[-1]:
                    feeder.start(k + 1)  # the next batch's copy overlaps this one's work
                for s, c, o in zip(items, cs, outs):
                    inf = c.info()
                    exact = bool(torch.equal(src[s.name].view(-1), o.view(-1)))
                    rec = {"name": s.name, "scheme": sc, "N": s.N, "K": s.K, "n": inf["n"],
                           "escapes": inf["n_escapes"], "serialized_bytes": inf["serialized_bytes"],
                           "serialized_compact_bytes": inf["serialized_compact_bytes"],
                           "entropy_bpw": inf["entropy_bpw"], "exact": exact}
                    # the decoded bytes are read back here (in stream order) and
                    # hashed by the pool while the GPU goes on
                    dec_hash = hasher.submit(tensor_hash, o.cpu()) if hasher else None
                    if corrupt_every > 0 and index[s.name] % corrupt_every == 0:
                        rec["corruption"] = corruption_check(W, c, 7919 * index[s.name] + sc)
                    pending.append((s.name, sc, rec, dec_hash))
                for c in cs:
                    c.free(stream)
                del outs
            for name, sc, rec, dec_hash in pending:
                if hasher:
                    rec["source_hash"] = src_hash[name].result()
                    rec["decoded_hash"] = dec_hash.result()
                done[(name, sc)] = rec
                if log:
                    log.write(json.dumps(rec) + "\n")
            if log:
                log.flush()
            if feeder:
                feeder.release(k, stream)
            del src
            torch.cuda.synchronize()
    finally:
        if log:
            log.close()
        if hasher:
            hasher.shutdown()
    elapsed = time.perf_counter() - t0
    names = [s.name for s in specs]
    out = {"tensors": len(specs), "seconds": round(elapsed, 2), "source": source, "schemes": {}}
    for sc in schemes:
        recs = [done[(nm, sc)] for nm in names if (nm, sc) in done]
        n = sum(r["n"] for r in recs)
        ser = sum(r["serialized_bytes"] for r in recs)
        ser_c = sum(r.get("serialized_compact_bytes", r["serialized_bytes"]) for r in recs)
        ebits = sum(r["entropy_bpw"] * r["n"] for r in recs)
        bpw_e = ebits / n if n else 0.0
        corr = [r["corruption"] for r in recs if "corruption" in r]
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
            "hashed": sum(1 for r in recs if "source_hash" in r),
            "hash_mismatch": [r["name"] for r in recs if "source_hash" in r and r["source_hash"] != r["decoded_hash"]],
            "corruption_checks": sum(len(c) for c in corr),
            "corruption_missed": sum(1 for c in corr for v in c.values() if not v["detected"]),
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
    ap.add_argument("--source", default="device", choices=["device", "host"])
    ap.add_argument("--hashes", action="store_true", help="BLAKE2b of every source and decoded tensor")
    ap.add_argument("--corrupt-every", type=int, default=0, help="flip a byte of every k-th serialized tensor")
    a = ap.parse_args(argv)
    build.build()
    if a.workload == "checkpoint" and a.layers is not None:
        specs = synth.workload_checkpoint(a.layers)
    else:
        specs = synth.WORKLOADS[a.workload]()
    schemes = [{"bytesplit": 0, "k15": 1}[x] for x in a.schemes.split(",")]
    res = validate(specs, schemes, int(a.batch_gib * (1 << 30)), a.log, source=a.source, hashes=a.hashes,
                   corrupt_every=a.corrupt_every)
    print(json.dumps(res))
    bad = any(v["not_exact"] or v["hash_mismatch"] or v["corruption_missed"] for v in res["schemes"].values())
    sys.exit(1 if bad else 0)


if __name__ == "__main__":
    main()
