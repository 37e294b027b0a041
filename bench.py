"""Benchmark of the lossless BF16 weight-coding hot path on one GB300 (or N replicas).

Workload: the checkpoint-shaped set (1,923 BF16 tensors, 120 GiB; hidden 6144,
vocabulary 151552) and its 16384x53248 GEMV.  One step is one pass of the
whole hot path over one HBM-sized batch of that set:

  1. encode the batch's 208 tensors (16 GiB of BF16, both embeddings and the
     first layers) in both schemes: histogram, top-15 table, pack, tile scan,
     escape compaction, row index
  2. decode all 416 containers to exact BF16 (batched launches)
  3. fused decode-GEMV on the 16384x53248 weight (byte-split and K15
     containers, encoded once before timing) at batch 1, 4, 8 and 16
  4. plain BF16 GEMV on the same weight at the same batches

`value` is the step's algorithmic HBM bytes (the minimum each launch must
move, see `*_bytes` below) divided by the device time of the step, in GB/s.
Each row is also reported as decoded GB/s (2n / t, BF16 produced or
consumed) and compressed-read GB/s (container bytes read / t), with the
fused / plain GEMV time ratio per batch.  Inputs (17 GB of BF16 plus ~24 GB of
containers) are far larger than the 129 MB L2 and are swept in order, so no
launch finds its inputs in L2.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs the same workload on its own GPU (replicas,
weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused decode-GEMV & decode HBM GB/s (% of GB300 peak); GEMV time vs plain BF16"
BATCHES = (1, 4, 8, 16)
BATCH_BYTES = 16 << 30
SCHEME_NAMES = {0: "bytesplit", 1: "k15"}
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0

# Algorithmic bytes per launch (the minimum traffic each operation implies).
from decode_gemv_sign_gb300.accounting import (container_read_bytes, decode_bytes, encode_bytes,  # noqa: E402,F401
                                               gemv_bytes, plain_bytes)


# ---------------------------------------------------------------------------
# Clocks sampled during the timed region.
# ---------------------------------------------------------------------------
REASON_FIELDS = ["clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                 "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampled every 20 ms in the background; only samples taken
    between mark_start() and mark_end() count."""

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.rows = []
        self.t0 = self.t1 = None

    def start(self):
        import threading

        q = "clocks.sm,clocks.max.sm,power.draw," + ",".join(REASON_FIELDS)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.rows.append((time.time(), line))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        # let the sampler come up before the timed region starts
        deadline = time.time() + 3.0
        while not self.rows and time.time() < deadline:
            time.sleep(0.01)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        inside = [r for r in self.rows if self.t0 is not None and self.t0 <= r[0] <= (self.t1 or 1e30)]
        use = inside if inside else self.rows[-3:]
        for _, line in use:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 3 + len(REASON_FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(REASON_FIELDS, parts[3:]):
                if v.lower() == "active":
                    reasons.add(name.split(".")[-1])
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "samples_in_timed_region": len(inside)}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample of the workload.
# ---------------------------------------------------------------------------
CPU_SAMPLE = ("per process: one 2048x6144 tensor of the batch (each process its own): encode, decode, fused "
              "GEMV B=1,4,8,16 and plain GEMV B=1,4,8,16, both schemes")


def _sample_spec(i: int):
    from decode_gemv_sign_gb300 import synth

    # the batch's 2048x6144 tensors, taken in turn
    sq = [s for s in synth.checkpoint_batch(0, BATCH_BYTES) if (s.N, s.K) == (2048, 6144)]
    return sq[i % len(sq)]


def oracle_sample(i: int) -> dict:
    """One bounded sample of the workload through the oracle (runs in a worker
    process with BLAS limited to one thread)."""
    import numpy as np

    from decode_gemv_sign_gb300 import synth
    from oracle import wcomp_oracle as O

    spec = _sample_spec(i)
    w = synth.gen_weights_np(spec)
    xs = {B: synth.gen_x_np(B, spec.K, 77 + B) for B in BATCHES}
    total = 0
    t0 = time.perf_counter()
    for scheme in (0, 1):
        c = O.encode(w, scheme)
        buf = O.serialize(c)
        info = {"n": c.n, "N": c.N, "K": c.K, "n_tiles": c.n_tiles, "n_escapes": c.E, "scheme": scheme,
                "serialized_bytes": len(buf)}
        sizes = dict(O.section_sizes(scheme, c.N, c.K, c.E))
        info["bytes_codes"] = O._pad(sizes["codes"])
        info["bytes_raw"] = sum(O._pad(sizes[k]) for k in ("raw", "plane_a", "plane_b", "plane_c") if k in sizes)
        total += encode_bytes(info)
        d = O.decode(O.deserialize(buf))
        assert np.array_equal(d, w)
        total += decode_bytes(info)
        for B in BATCHES:
            O.gemv_container(c, xs[B])
            total += gemv_bytes(info, B)
    for B in BATCHES:
        O.gemv(w, xs[B])
        total += plain_bytes(spec.N, spec.K, B)
    return {"bytes": total, "seconds": time.perf_counter() - t0}


def _pool_init():
    os.environ["CUDA_VISIBLE_DEVICES"] = ""


class OraclePool:
    """Worker processes (spawned, one BLAS thread each) that run oracle samples."""

    def __init__(self, procs: int):
        import multiprocessing as mp

        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
        self.procs = procs
        self.pool = mp.get_context("spawn").Pool(procs, initializer=_pool_init)

    def run(self, first: int, rounds: int = 1) -> dict:
        """`rounds` samples per process, all processes at once; bytes over wall time."""
        t0 = time.perf_counter()
        res = self.pool.map(oracle_sample, range(first, first + self.procs * rounds), chunksize=1)
        wall = time.perf_counter() - t0
        return {"bytes": sum(r["bytes"] for r in res), "seconds": wall,
                "busy_seconds": sum(r["seconds"] for r in res)}

    def close(self):
        self.pool.close()
        self.pool.join()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


CPU_ROUNDS = 4  # samples per process: about 10 s of oracle work per core


def cpu_baseline() -> dict:
    """The oracle on one core and on every host core (one process per core)."""
    one = OraclePool(1)
    r1 = one.run(0, CPU_ROUNDS)
    one.close()
    cores = host_cores()
    allp = OraclePool(cores)
    ra = allp.run(0, CPU_ROUNDS)
    allp.close()
    sample = f"{CPU_ROUNDS} samples per process, " + CPU_SAMPLE
    return {"value": round(ra["bytes"] / ra["seconds"] / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{cores} processes at once, " + sample, "seconds": round(ra["seconds"], 2),
            "cpu_seconds": round(ra["busy_seconds"], 1),
            "single_core": {"value": round(r1["bytes"] / r1["seconds"] / 1e9, 4), "unit": "GB/s", "cores": 1,
                            "sample": "1 process, " + sample, "seconds": round(r1["seconds"], 2)}}


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas; barrier and max-over-ranks timing).
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world):
    """NCCL on GPUs (one rank per GPU); gloo when the ranks have no GPU (host-side tests)."""
    if world <= 1:
        return None
    import torch
    import torch.distributed as dist

    dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def _all_reduce(dist, v: float, op) -> float:
    import torch

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def allmax(dist, v: float) -> float:
    return v if dist is None else _all_reduce(dist, v, dist.ReduceOp.MAX)


def allsum(dist, v: float) -> float:
    return v if dist is None else _all_reduce(dist, v, dist.ReduceOp.SUM)


def aggregate_rate(dist, local_bytes: float, local_ms: float) -> tuple:
    """Whole-job rate of replicas: the bytes all ranks moved over the slowest rank's time."""
    t_max = allmax(dist, local_ms)
    return allsum(dist, local_bytes) / (t_max / 1e3) / 1e9, t_max


# ---------------------------------------------------------------------------
# The GPU arm.
# ---------------------------------------------------------------------------
def workload_config(batch_specs, gemv_spec, world: int) -> dict:
    """The `config` of both arms' lines: the workload a step covers."""
    return {"workload": (f"checkpoint-shaped set (1,923 BF16 tensors, 120 GiB), one HBM-sized batch of "
                         f"{len(batch_specs)} tensors (the first 16 GiB: both 151552x6144 embeddings and the first "
                         f"layers), both schemes: encode + batched decode; GEMV {gemv_spec.N}x{gemv_spec.K} "
                         f"fused (byte-split, K15) and plain BF16 at B=1,4,8,16"),
            "tensors": len(batch_specs), "elements": int(sum(s.n for s in batch_specs)),
            "gemv": [gemv_spec.N, gemv_spec.K], "batches": list(BATCHES),
            "l2": "inputs far larger than L2 (17 GB BF16 batch, ~24 GB containers, 1.7 GB GEMV weight), swept in order",
            "parallelism": f"replicas x{world}"}


def alloc_batch(specs, dev):
    """One flat device buffer holding the batch's tensors back to back (16-byte aligned views)."""
    import torch

    offs, total = [], 0
    for s in specs:
        offs.append(total)
        total += (s.n + 7) // 8 * 8
    flat = torch.empty(total, dtype=torch.int16, device=dev)
    views = [flat[o:o + s.n].view(s.N, s.K) for o, s in zip(offs, specs)]
    return flat, views


class HotPath:
    """The step's device state: batch sources, decode outputs, GEMV inputs and outputs."""

    def __init__(self, W, torch, src_views, specs, gemv_w, gemv_cs, xs, stream):
        self.W = W
        self.torch = torch
        self.src = src_views
        self.specs = specs
        self.gemv_w = gemv_w
        self.gemv_cs = gemv_cs
        self.xs = xs
        self.stream = stream
        dev = gemv_w.device
        self.out_flat, self.outs0 = alloc_batch(specs, dev)
        self.out_flat1, self.outs1 = alloc_batch(specs, dev)
        self.outs = [o for pair in zip(self.outs0, self.outs1) for o in pair]
        N = gemv_w.shape[0]
        self.yf = {(s, B): torch.empty((B, N), dtype=torch.float32, device=dev) for s in (0, 1) for B in BATCHES}
        self.yp = {B: torch.empty((B, N), dtype=torch.float32, device=dev) for B in BATCHES}
        self.containers = []
        self.infos = None

    def step(self, marks=None):
        """One pass of the hot path; `marks` (list) receives (name, start event, end event)."""
        W, torch = self.W, self.torch

        def mark():
            e = torch.cuda.Event(enable_timing=True)
            e.record(self.stream)
            return e

        for c in self.containers:
            c.free(self.stream)
        prev = mark() if marks is not None else None
        cs = W.encode_batched([w for w in self.src for _ in (0, 1)], [0, 1] * len(self.src), stream=self.stream)
        self.containers = cs
        if marks is not None:
            e = mark()
            marks.append(("encode", prev, e))
            prev = e
        W.decode_batched(cs, self.outs, stream=self.stream)
        if marks is not None:
            e = mark()
            marks.append(("decode", prev, e))
            prev = e
        for B in BATCHES:
            for s in (0, 1):
                W.gemv(self.gemv_cs[s], self.xs[B], self.yf[(s, B)], stream=self.stream)
                if marks is not None:
                    e = mark()
                    marks.append((f"gemv_fused_{SCHEME_NAMES[s]}_b{B}", prev, e))
                    prev = e
            W.gemv_bf16(self.gemv_w, self.xs[B], self.yp[B], stream=self.stream)
            if marks is not None:
                e = mark()
                marks.append((f"gemv_plain_b{B}", prev, e))
                prev = e
        if self.infos is None:
            self.infos = [c.info() for c in cs]

    def row_bytes(self) -> dict:
        """Algorithmic bytes of every row of the step, with the bytes of
        BF16 produced / consumed and the container bytes read."""
        out = {"encode": {"bytes": sum(encode_bytes(i) for i in self.infos), "bf16": sum(2 * i["n"] for i in self.infos),
                          "compressed": sum(i["serialized_bytes"] - 96 for i in self.infos)},
               "decode": {"bytes": sum(decode_bytes(i) for i in self.infos), "bf16": sum(2 * i["n"] for i in self.infos),
                          "compressed": sum(container_read_bytes(i, "decode") for i in self.infos)}}
        gi = {s: self.gemv_cs[s].info() for s in (0, 1)}
        N, K = self.gemv_w.shape
        for B in BATCHES:
            for s in (0, 1):
                out[f"gemv_fused_{SCHEME_NAMES[s]}_b{B}"] = {"bytes": gemv_bytes(gi[s], B), "bf16": 2 * N * K,
                                                             "compressed": container_read_bytes(gi[s], "gemv")}
            out[f"gemv_plain_b{B}"] = {"bytes": plain_bytes(N, K, B), "bf16": 2 * N * K, "compressed": 2 * N * K}
        return out


def time_launches(fn, stream, reps: int = 10) -> float:
    """Average device time (ms) of one call of fn, over reps back-to-back calls.

    One untimed call first keeps the GPU busy while the timed calls are
    enqueued, so host launch latency does not enter the measurement."""
    import torch

    fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / reps


def layer_rows(W, torch, hp, stream, peak) -> dict:
    """GEMV over the first layer of the batch (its 15 matrices, two norms left
    out) in one batched call per scheme, against one batched plain GEMV: the
    serving-shaped use of the same containers the step encodes."""
    from decode_gemv_sign_gb300 import synth

    idx = [i for i in range(2, 19) if hp.specs[i].N > 1]
    dev = hp.gemv_w.device
    n = sum(hp.specs[i].n for i in idx)
    infos = hp.infos
    out = {"tensors": len(idx), "weights": n,
           "shapes": sorted({f"{hp.specs[i].N}x{hp.specs[i].K}" for i in idx})}
    for B in BATCHES:
        xs = [synth.gen_x_torch(B, hp.specs[i].K, 7000 + 31 * B + i, dev) for i in idx]
        ys = [torch.empty((B, hp.specs[i].N), dtype=torch.float32, device=dev) for i in idx]
        tp = time_launches(lambda: W.gemv_bf16_batched([hp.src[i] for i in idx], xs, ys, stream=stream), stream)
        row = {"plain_ms": round(tp, 4),
               "plain_GB/s": round(plain_bytes_total(hp, idx, B) / (tp / 1e3) / 1e9, 1)}
        for s in (0, 1):
            cs = [hp.containers[2 * i + s] for i in idx]
            tf = time_launches(lambda: W.gemv_batched(cs, xs, ys, stream=stream), stream)
            nbytes = sum(gemv_bytes(infos[2 * i + s], B) for i in idx)
            row[f"{SCHEME_NAMES[s]}_ms"] = round(tf, 4)
            row[f"{SCHEME_NAMES[s]}_over_plain"] = round(tf / tp, 4)
            row[f"{SCHEME_NAMES[s]}_frac_of_peak"] = round(nbytes / (tf / 1e3) / 1e9 / peak, 4)
        out[f"b{B}"] = row
    return out


def plain_bytes_total(hp, idx, B) -> int:
    return sum(plain_bytes(hp.specs[i].N, hp.specs[i].K, B) for i in idx)


def make_gemv(W, torch, dev):
    """The 16384x53248 GEMV weight, its containers and x per batch size."""
    from decode_gemv_sign_gb300 import synth

    spec = synth.checkpoint_gemv_spec()
    w = synth.gen_weights_torch(spec, dev)
    cs = {s: W.encode(w, s) for s in (0, 1)}
    xs = {B: synth.gen_x_torch(B, spec.K, 9000 + B, dev) for B in BATCHES}
    return spec, w, cs, xs


def run_ours(args):
    import torch

    from decode_gemv_sign_gb300 import build, synth
    from decode_gemv_sign_gb300 import wcomp as W

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world)
    build.build()
    W.lib()
    dev = torch.device("cuda", local)
    specs = synth.checkpoint_batch(0, BATCH_BYTES)
    src_flat, src = alloc_batch(specs, dev)
    for s, v in zip(specs, src):
        v.copy_(synth.gen_weights_torch(s, dev))
    gspec, gw, gcs, xs = make_gemv(W, torch, dev)
    stream = torch.cuda.current_stream()
    hp = HotPath(W, torch, src, specs, gw, gcs, xs, stream)
    for _ in range(args.warmup):
        hp.step()
    torch.cuda.synchronize()
    # every decode of the warm-up steps was bit-exact
    exact = all(bool(torch.equal(a, w) and torch.equal(b, w)) for a, b, w in zip(hp.outs0, hp.outs1, src))

    # ---- timed region: K steps, device time, clocks sampled meanwhile
    clocks = ClockSampler(local)
    clocks.start()
    marks = []
    barrier(dist)
    torch.cuda.synchronize()
    clocks.mark_start()
    n0 = W.launch_count()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        hp.step(marks)
    end.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    barrier(dist)
    launches = W.launch_count() - n0
    clk = clocks.stop()
    t_ms = start.elapsed_time(end)
    dev_check = W.lib().wcomp_device_check(None)

    phase_ms = {}
    for name, a, b in marks:
        phase_ms[name] = phase_ms.get(name, 0.0) + a.elapsed_time(b)
    phase_ms = {k: v / args.steps for k, v in phase_ms.items()}
    rb = hp.row_bytes()
    step_bytes = sum(r["bytes"] for r in rb.values())
    value, t_ms_max = aggregate_rate(dist, step_bytes * args.steps, t_ms)

    peaks = measured_peaks()
    peak = peaks["hbm_gbs"]

    def rates(name, ms):
        r = rb[name]
        gbs = r["bytes"] / (ms / 1e3) / 1e9
        return {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                "frac_of_8TBps": round(gbs / NOMINAL_HBM_GBS, 4), "bytes": r["bytes"],
                "decoded_GB/s": round(r["bf16"] / (ms / 1e3) / 1e9, 1),
                "compressed_read_GB/s": round(r["compressed"] / (ms / 1e3) / 1e9, 1)}

    rows = {k: rates(k, ms) for k, ms in phase_ms.items()}
    # per-launch times (back-to-back calls of each operation, device clock)
    kt = {"decode_batch": time_launches(lambda: W.decode_batched(hp.containers, hp.outs, stream=stream), stream, 5)}
    for B in BATCHES:
        for s in (0, 1):
            kt[f"gemv_fused_{SCHEME_NAMES[s]}_b{B}"] = time_launches(
                lambda: W.gemv(gcs[s], xs[B], hp.yf[(s, B)], stream=stream), stream)
        kt[f"gemv_plain_b{B}"] = time_launches(lambda: W.gemv_bf16(gw, xs[B], hp.yp[B], stream=stream), stream)
    rb["decode_batch"] = rb["decode"]
    kernels = {k: rates(k, ms) for k, ms in kt.items()}
    ratio = {f"b{B}": {SCHEME_NAMES[s]: round(kt[f"gemv_fused_{SCHEME_NAMES[s]}_b{B}"] / kt[f"gemv_plain_b{B}"], 4)
                       for s in (0, 1)} for B in BATCHES}
    # the dense 12-bit ablation: the same GEMV on an escape-free weight (byte-split E = 0)
    ablation = dense12_rows(W, torch, dev, stream, peak)
    # one layer's matrices in one batched call (serving-shaped GEMVs)
    layer = layer_rows(W, torch, hp, stream, peak)

    # Dominant kernel: decode_kernel, the step's largest share of library GPU
    # time (launch list in profiles/); its launches in the batched decode
    # call carry the batch's 416 containers.
    dom_ms = kt["decode_batch"]
    dom_gbs = rb["decode"]["bytes"] / (dom_ms / 1e3) / 1e9
    roofline = {"kernel": "decode_kernel (batched decode of the batch's 416 containers)", "bound": "hbm",
                "achieved": round(dom_gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(dom_gbs / peak, 4),
                "frac_of_8TBps": round(dom_gbs / NOMINAL_HBM_GBS, 4),
                "peak_source": peaks["source"] + " (hbm_gbs: read+write copy)",
                "algorithmic_bytes_per_call": rb["decode"]["bytes"], "call_ms": round(dom_ms, 4),
                "traffic": load_traffic("decode_kernel_checkpoint_batch", rb["decode"]["bytes"])}

    infos = hp.infos
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u16 codec / fp32 GEMV accumulate",
        "data": "synthetic (seeded checkpoint-shaped BF16 tensors: Normal / Student-t(4), sigma ~ U(0.005, 0.05), "
                "0.1% outliers; x ~ N(0,1) BF16)",
        "config": workload_config(specs, gspec, world),
        "rows": rows,
        "kernels": kernels,
        "fused_over_plain_time": ratio,
        "dense12_ablation": ablation,
        "layer_gemv": layer,
        "decode_exact": exact,
        "device_check": dev_check,
        "escape_rate": {SCHEME_NAMES[s]: round(sum(i["n_escapes"] for i in infos if i["scheme"] == s) /
                                               sum(i["n"] for i in infos if i["scheme"] == s), 6) for s in (0, 1)},
        "gemv_escape_rate": {SCHEME_NAMES[s]: round(gcs[s].info()["n_escapes"] / gcs[s].info()["n"], 6)
                             for s in (0, 1)},
        "bpw": {SCHEME_NAMES[s]: {"entropy": round(sum(i["entropy_bpw"] * i["n"] for i in infos if i["scheme"] == s) /
                                                   sum(i["n"] for i in infos if i["scheme"] == s), 4),
                                  "physical": round(sum(8 * i["serialized_bytes"] for i in infos if i["scheme"] == s) /
                                                    sum(i["n"] for i in infos if i["scheme"] == s), 4),
                                  "physical_compact": round(
                                      sum(8 * i["serialized_compact_bytes"] for i in infos if i["scheme"] == s) /
                                      sum(i["n"] for i in infos if i["scheme"] == s), 4)}
                for s in (0, 1)},
        "roofline": roofline,
        "clocks": clk,
        "gpu_launches": int(launches),
    }
    # ---- end to end through the public API with host buffers
    result["e2e"] = run_e2e(args, W, torch, hp, specs, src_flat, dist)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def dense12_rows(W, torch, dev, stream, peak) -> dict:
    """Fused byte-split GEMV on an escape-free 16384x53248 weight (every high
    byte in the table, so the kernel reads exactly 12 bits per weight and
    corrects nothing) beside the plain GEMV, at B = 1 and 4."""
    from decode_gemv_sign_gb300 import synth

    spec = synth.dense12_spec()
    w = synth.gen_weights_torch(spec, dev)
    c = W.encode(w, 0)
    inf = c.info()
    out = {"weight": [spec.N, spec.K], "escapes": inf["n_escapes"]}
    for B in (1, 4):
        x = synth.gen_x_torch(B, spec.K, 9100 + B, dev)
        y = torch.empty((B, spec.N), dtype=torch.float32, device=dev)
        tf = time_launches(lambda: W.gemv(c, x, y, stream=stream), stream)
        tp = time_launches(lambda: W.gemv_bf16(w, x, y, stream=stream), stream)
        gbs = gemv_bytes(inf, B) / (tf / 1e3) / 1e9
        out[f"b{B}"] = {"fused_ms": round(tf, 4), "plain_ms": round(tp, 4), "fused_over_plain": round(tf / tp, 4),
                        "fused_GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)}
    c.free(stream)
    del w
    return out


def run_e2e(args, W, torch, hp, specs, src_flat, dist):
    """The same step through the public API, its inputs copied from pinned host
    memory every step (the batch's 16 GiB of BF16 and every x) and every GEMV
    result read back.  Two device copies of the batch alternate, so step k+1's
    inputs are copied on a second stream while step k computes (the copy of
    the first timed step lies inside the timed region too)."""
    from decode_gemv_sign_gb300.hostmem import PinnedBuffer

    host_buf = PinnedBuffer(torch, src_flat.numel(), src_flat.dtype)
    host_src = host_buf.tensor
    host_src.copy_(src_flat)
    host_x = {B: hp.xs[B].cpu().pin_memory() for B in BATCHES}
    host_y = {k: torch.empty(y.shape, dtype=y.dtype).pin_memory() for k, y in hp.yf.items()}
    host_yp = {B: torch.empty(y.shape, dtype=y.dtype).pin_memory() for B, y in hp.yp.items()}
    h2d = host_src.numel() * 2 + sum(x.numel() * 2 for x in host_x.values())
    d2h = sum(y.numel() * 4 for y in host_y.values()) + sum(y.numel() * 4 for y in host_yp.values())
    sets = [(src_flat, hp.src, hp.xs)]
    flat2, views2 = alloc_batch(specs, src_flat.device)
    sets.append((flat2, views2, {B: torch.empty_like(hp.xs[B]) for B in BATCHES}))
    copy_stream = torch.cuda.Stream()
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(i):
        flat, _, xs = sets[i]
        copy_stream.wait_event(done[i])  # the set's previous step has finished with it
        with torch.cuda.stream(copy_stream):
            flat.copy_(host_src, non_blocking=True)
            for B in BATCHES:
                xs[B].copy_(host_x[B], non_blocking=True)
        ready[i].record(copy_stream)

    def run(steps):
        done[0].record(hp.stream)
        done[1].record(hp.stream)
        copy_in(0)
        for k in range(steps):
            i = k % 2
            if k + 1 < steps:
                copy_in(1 - i)
            hp.stream.wait_event(ready[i])
            hp.src, hp.xs = sets[i][1], sets[i][2]
            hp.step()
            for key, h in host_y.items():
                h.copy_(hp.yf[key], non_blocking=True)
            for B, h in host_yp.items():
                h.copy_(hp.yp[B], non_blocking=True)
            done[i].record(hp.stream)

    run(max(2, args.warmup))
    torch.cuda.synchronize()
    barrier(dist)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(hp.stream)
    copy_stream.wait_event(a)
    run(args.steps)
    b.record(hp.stream)
    torch.cuda.synchronize()
    barrier(dist)
    hp.src, hp.xs = sets[0][1], sets[0][2]
    ms = allmax(dist, a.elapsed_time(b))
    step_bytes = sum(r["bytes"] for r in hp.row_bytes().values())
    v = allsum(dist, step_bytes * args.steps) / (ms / 1e3) / 1e9
    del flat2, views2, host_src
    host_buf.release()
    return {"value": round(v, 1), "unit": "GB/s", "ms_per_step": round(ms / args.steps, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "overlap": "step k+1's inputs are copied on a second stream while step k computes"}


def _source_digest(files) -> str:
    import hashlib

    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "decode_gemv_sign_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(key: str, algorithmic_bytes: int):
    """DRAM bytes (read + write) per call from the committed ncu summary, or None
    when the summary has no such line or the kernel's sources changed since the
    capture.  The summary stores DRAM bytes per algorithmic byte of a smaller
    capture of the same kernel; the call's traffic is that ratio times its
    algorithmic bytes."""
    p = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if len(parts) == 4 and parts[0] == "bench-traffic" and parts[1] == key:
            files, digest = parts[3].split("=")
            if _source_digest(files.split("+")) != digest:
                return None
            return int(round(float(parts[2]) * algorithmic_bytes))
    return None


# ---------------------------------------------------------------------------
# The reference arm: the CPU oracle, timed on the host cores.
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from decode_gemv_sign_gb300 import synth

    cores = host_cores()
    pool = OraclePool(cores)
    try:
        for i in range(args.warmup):
            pool.run(cores * i)
        t_total, b_total = 0.0, 0.0
        for i in range(args.steps):
            r = pool.run(cores * (args.warmup + i))
            t_total += r["seconds"]
            b_total += r["bytes"]
    except Exception as e:  # a failing oracle run is reported, not hidden
        print(json.dumps({"impl": "reference", "unavailable": f"oracle run failed: {e}"}))
        return
    finally:
        pool.close()
    v = b_total / t_total / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_total / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16 codec / f64 GEMV",
        "data": "synthetic (seeded numpy draw of the same workload recipe)",
        # the same workload as our arm's line; each step times a bounded sample of it
        "config": workload_config(synth.checkpoint_batch(0, BATCH_BYTES), synth.checkpoint_gemv_spec(), world),
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {cores} processes at once, " + CPU_SAMPLE},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 20 for ours, about half a second of device time; 3 for the "
                         "reference arm, whose steps take seconds each)")
    ap.add_argument("--warmup", type=int, default=None, help="untimed steps first (default 3; ours takes at least 3)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 20 if args.impl == "ours" else 3
    if args.warmup is None:
        args.warmup = 3 if args.impl == "ours" else 1
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
