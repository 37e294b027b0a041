"""Benchmark of the lossless BF16 weight-coding hot path on one GB300 (or N replicas).

One step = one pass of the whole hot path over the dense-layer workload
(4 x 4096x4096 and 3 x 4096x11008 BF16 weights, N(0, 0.02) with 0.1%
N(0, 0.5) outliers), in both schemes (byte-split and K15):

  1. encode every tensor (histogram, top-15 table, pack, tile scan, escape
     compaction, row index)
  2. decode all 14 containers to exact BF16 in one batched launch
  3. fused decode-GEMV over all 14 containers at batch 1 and batch 4
  4. plain BF16 GEMV over the 7 raw tensors at batch 1 and batch 4 (one
     batched launch each, the same launch structure as the fused GEMV)

`value` is the step's algorithmic HBM bytes (the minimum each launch must
move, see `bytes_*` below) divided by the device time of the step, in GB/s.
Per-row rates, the fused / plain GEMV time ratio and the roofline of the
dominant kernel are reported beside it.  Inputs (386 MB of BF16 weights plus
~580 MB of containers) are larger than the 129 MB L2 and are swept in order,
so successive launches do not find their inputs in L2.

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
WORKLOAD = "dense_layers"
BATCHES = (1, 4)
SCHEME_NAMES = {0: "bytesplit", 1: "k15"}
FALLBACK_HBM_GBS = 6800.0

# ---------------------------------------------------------------------------
# Algorithmic bytes per launch (the minimum traffic each operation implies).
# ---------------------------------------------------------------------------


def container_read_bytes(info: dict, part: str) -> int:
    """Bytes a decode ("decode") or fused GEMV ("gemv") must read from a container."""
    n_tiles_b = 4 * (info["n_tiles"] + 1)
    rows_b = 4 * (info["N"] + 1)
    E = info["n_escapes"]
    val = E if info["scheme"] == 0 else 2 * E
    streams = info["bytes_codes"] + info["bytes_raw"]
    if part == "decode":
        return streams + n_tiles_b + 4 * E + val
    return streams + rows_b + 4 * E + val


def encode_bytes(info: dict) -> int:
    # read the source once, write the container once
    return 2 * info["n"] + info["serialized_bytes"] - 96


def decode_bytes(info: dict) -> int:
    return container_read_bytes(info, "decode") + 2 * info["n"]


def gemv_bytes(info: dict, B: int) -> int:
    return container_read_bytes(info, "gemv") + 2 * B * info["K"] + 4 * B * info["N"]


def plain_bytes(N: int, K: int, B: int) -> int:
    return 2 * N * K + 2 * B * K + 4 * B * N


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
CPU_SAMPLE = "one 4096x4096 tensor of the dense-layer workload: encode, decode, GEMV B=1,4, plain GEMV B=1,4, both schemes"


def oracle_sample_run() -> dict:
    """Runs in a child process with BLAS limited to one thread."""
    import numpy as np

    from decode_gemv_sign_gb300 import synth
    from oracle import wcomp_oracle as O

    spec = synth.workload_dense_layers()[0]
    w = synth.gen_weights_np(spec)
    xs = {B: synth.gen_x_np(B, spec.K, 77 + B) for B in BATCHES}
    total_bytes = 0
    t0 = time.perf_counter()
    for scheme in (0, 1):
        c = O.encode(w, scheme)
        buf = O.serialize(c)
        info = {"n": c.n, "N": c.N, "K": c.K, "n_tiles": c.n_tiles, "n_escapes": c.E, "scheme": scheme,
                "serialized_bytes": len(buf)}
        sizes = dict(O.section_sizes(scheme, c.N, c.K, c.E))
        info["bytes_codes"] = O._pad(sizes["codes"])
        info["bytes_raw"] = sum(O._pad(sizes[k]) for k in ("raw", "plane_a", "plane_b", "plane_c") if k in sizes)
        total_bytes += encode_bytes(info)
        d = O.decode(O.deserialize(buf))
        assert np.array_equal(d, w)
        total_bytes += decode_bytes(info)
        for B in BATCHES:
            O.gemv_container(c, xs[B])
            total_bytes += gemv_bytes(info, B)
    for B in BATCHES:
        O.gemv(w, xs[B])
        total_bytes += plain_bytes(spec.N, spec.K, B)
    dt = time.perf_counter() - t0
    return {"bytes": total_bytes, "seconds": dt}


def cpu_baseline(repeats: int = 1) -> dict:
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    tot_b, tot_s = 0.0, 0.0
    for _ in range(repeats):
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample"], env=env,
                           capture_output=True, text=True, timeout=900)
        if r.returncode != 0:
            return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": CPU_SAMPLE,
                    "error": r.stderr.strip().splitlines()[-1:] or ["failed"]}
        d = json.loads(r.stdout.strip().splitlines()[-1])
        tot_b += d["bytes"]
        tot_s += d["seconds"]
    return {"value": tot_b / tot_s / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{repeats} x " + CPU_SAMPLE, "seconds": round(tot_s, 2)}


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
class HotPath:
    def __init__(self, W, weights, specs, xs, stream):
        import torch

        self.W = W
        self.torch = torch
        self.weights = weights
        self.specs = specs
        self.xs = xs  # {B: [x per tensor]}
        self.stream = stream
        self.outs = [torch.empty((s.N, s.K), dtype=torch.int16, device="cuda") for s in specs for _ in (0, 1)]
        self.ys = {B: [torch.empty((B, s.N), dtype=torch.float32, device="cuda") for s in specs for _ in (0, 1)]
                   for B in BATCHES}
        self.yp = {B: [torch.empty((B, s.N), dtype=torch.float32, device="cuda") for s in specs] for B in BATCHES}
        self.containers = []
        self.infos = None

    def step(self, ev=None):
        """One pass of the hot path; `ev` (list) receives (name, start, end) events."""
        W, torch = self.W, self.torch

        def mark():
            e = torch.cuda.Event(enable_timing=True)
            e.record(self.stream)
            return e

        for c in self.containers:
            c.free(self.stream)
        t0 = mark() if ev is not None else None
        cs = W.encode_batched([w for w in self.weights for _ in (0, 1)], [0, 1] * len(self.weights),
                              stream=self.stream)
        self.containers = cs
        t1 = mark() if ev is not None else None
        W.decode_batched(cs, self.outs, stream=self.stream)
        t2 = mark() if ev is not None else None
        marks = [("encode", t0, t1), ("decode", t1, t2)]
        prev = t2
        for B in BATCHES:
            xs2 = [x for x in self.xs[B] for _ in (0, 1)]
            W.gemv_batched(cs, xs2, self.ys[B], stream=self.stream)
            e = mark() if ev is not None else None
            marks.append((f"gemv_fused_b{B}", prev, e))
            prev = e
        for B in BATCHES:
            W.gemv_bf16_batched(self.weights, self.xs[B], self.yp[B], stream=self.stream)
            e = mark() if ev is not None else None
            marks.append((f"gemv_plain_b{B}", prev, e))
            prev = e
        if ev is not None:
            ev.append(marks)
        if self.infos is None:
            self.infos = [c.info() for c in cs]

    def algorithmic_bytes(self) -> dict:
        out = {"encode": 0, "decode": 0}
        for B in BATCHES:
            out[f"gemv_fused_b{B}"] = 0
            out[f"gemv_plain_b{B}"] = 0
        for inf in self.infos:
            out["encode"] += encode_bytes(inf)
            out["decode"] += decode_bytes(inf)
            for B in BATCHES:
                out[f"gemv_fused_b{B}"] += gemv_bytes(inf, B)
        for s in self.specs:
            for B in BATCHES:
                out[f"gemv_plain_b{B}"] += plain_bytes(s.N, s.K, B)
        return out

    def per_scheme_bytes(self, B: int) -> dict:
        d = {0: 0, 1: 0}
        for inf in self.infos:
            d[inf["scheme"]] += gemv_bytes(inf, B)
        return d


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


def time_kernels(hp, W, torch) -> dict:
    """Per-launch device time of each kernel kind of the step (ms)."""
    res = {}
    # the step's decode launch: all containers of both schemes in one batch
    res["decode_all"] = time_launches(lambda: W.decode_batched(hp.containers, hp.outs, stream=hp.stream), hp.stream)
    by = {s: [c for c in hp.containers if c.scheme == s] for s in (0, 1)}
    outs = {s: [o for o, c in zip(hp.outs, hp.containers) if c.scheme == s] for s in (0, 1)}
    for s in (0, 1):
        nm = SCHEME_NAMES[s]
        res[f"decode_{nm}"] = time_launches(lambda: W.decode_batched(by[s], outs[s], stream=hp.stream), hp.stream)
        for B in BATCHES:
            ys = [torch.empty((B, c.N), dtype=torch.float32, device="cuda") for c in by[s]]
            res[f"gemv_fused_{nm}_b{B}"] = time_launches(
                lambda: W.gemv_batched(by[s], hp.xs[B], ys, stream=hp.stream), hp.stream)
    for B in BATCHES:
        res[f"gemv_plain_b{B}"] = time_launches(
            lambda: W.gemv_bf16_batched(hp.weights, hp.xs[B], hp.yp[B], stream=hp.stream), hp.stream)
    return res


def run_ours(args):
    import numpy as np
    import torch

    from decode_gemv_sign_gb300 import build, synth
    from decode_gemv_sign_gb300 import wcomp as W

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world)
    build.build()
    W.lib()
    specs = synth.WORKLOADS[WORKLOAD]()
    dev = torch.device("cuda", local)
    weights = [synth.gen_weights_torch(s, dev) for s in specs]
    xs = {B: [synth.gen_x_torch(B, s.K, 9000 + 10 * B + i, dev) for i, s in enumerate(specs)] for B in BATCHES}
    stream = torch.cuda.current_stream()
    hp = HotPath(W, weights, specs, xs, stream)
    for _ in range(args.warmup):
        hp.step()
    torch.cuda.synchronize()

    # ---- timed region: K steps, device time, clocks sampled meanwhile
    clocks = ClockSampler(local)
    clocks.start()
    ev = []
    barrier(dist)
    torch.cuda.synchronize()
    clocks.mark_start()
    n0 = W.launch_count()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        hp.step(ev)
    end.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    barrier(dist)
    launches = W.launch_count() - n0
    clk = clocks.stop()
    t_ms = start.elapsed_time(end)

    phase_ms = {}
    for marks in ev:
        for name, a, b in marks:
            phase_ms[name] = phase_ms.get(name, 0.0) + a.elapsed_time(b)
    phase_ms = {k: v / args.steps for k, v in phase_ms.items()}
    bytes_ = hp.algorithmic_bytes()
    step_bytes = sum(bytes_.values())
    value, t_ms_max = aggregate_rate(dist, step_bytes * args.steps, t_ms)

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(args, W, torch, hp, specs, dist)

    peaks = measured_peaks()
    peak = peaks["hbm_gbs"]
    rows = {}
    for k, ms in phase_ms.items():
        gbs = bytes_[k] / (ms / 1e3) / 1e9
        rows[k] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                   "frac_of_8TBps": round(gbs / 8000.0, 4), "bytes": bytes_[k]}
    # per-launch kernel times (back-to-back launches, device clock)
    kt = time_kernels(hp, W, torch)
    kbytes = {"decode_all": sum(decode_bytes(i) for i in hp.infos)}
    for s_ in (0, 1):
        nm = SCHEME_NAMES[s_]
        infos = [i for i in hp.infos if i["scheme"] == s_]
        kbytes[f"decode_{nm}"] = sum(decode_bytes(i) for i in infos)
        for B in BATCHES:
            kbytes[f"gemv_fused_{nm}_b{B}"] = sum(gemv_bytes(i, B) for i in infos)
    for B in BATCHES:
        kbytes[f"gemv_plain_b{B}"] = sum(plain_bytes(sp.N, sp.K, B) for sp in specs)
    kernels = {k: {"ms": round(v, 4), "GB/s": round(kbytes[k] / (v / 1e3) / 1e9, 1),
                   "frac_of_peak": round(kbytes[k] / (v / 1e3) / 1e9 / peak, 4), "bytes": kbytes[k]}
               for k, v in kt.items()}
    ratio = {}
    for B in BATCHES:
        ratio[f"b{B}"] = {SCHEME_NAMES[s_]: round(kt[f"gemv_fused_{SCHEME_NAMES[s_]}_b{B}"] / kt[f"gemv_plain_b{B}"], 4)
                          for s_ in (0, 1)}
    # Dominant kernel: the single launch with the largest device time in the step
    # (the batched decode of all 14 containers; the launch list in profiles/
    # confirms it has the largest share of the library's GPU time).
    dom = "decode_all"
    dom_gbs = kbytes[dom] / (kt[dom] / 1e3) / 1e9
    traffic = load_traffic("decode_kernel_both")
    roofline = {"kernel": "decode_kernel (batched, 7 tensors x 2 schemes)", "bound": "hbm", "achieved": round(dom_gbs, 1),
                "peak": peak, "unit": "GB/s", "frac": round(dom_gbs / peak, 4),
                "peak_source": peaks["source"] + " (hbm_gbs: read+write copy)",
                "algorithmic_bytes_per_launch": kbytes[dom], "launch_ms": round(kt[dom], 4),
                "traffic": traffic}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u16 codec / fp32 GEMV accumulate",
        "data": "synthetic (seeded N(0,0.02) BF16 weights with 0.1% N(0,0.5) outliers, x ~ N(0,1) BF16)",
        "config": workload_config(specs, world),
        "rows": rows,
        "kernels": kernels,
        "fused_over_plain_time": ratio,
        "escape_rate": {SCHEME_NAMES[s]: round(sum(i["n_escapes"] for i in hp.infos if i["scheme"] == s) /
                                               sum(i["n"] for i in hp.infos if i["scheme"] == s), 6) for s in (0, 1)},
        "bpw": {SCHEME_NAMES[s]: {"entropy": round(sum(i["entropy_bpw"] * i["n"] for i in hp.infos if i["scheme"] == s) /
                                                   sum(i["n"] for i in hp.infos if i["scheme"] == s), 4),
                                  "physical": round(sum(8 * i["serialized_bytes"] for i in hp.infos if i["scheme"] == s) /
                                                    sum(i["n"] for i in hp.infos if i["scheme"] == s), 4),
                                  "physical_compact": round(
                                      sum(8 * i["serialized_compact_bytes"] for i in hp.infos if i["scheme"] == s) /
                                      sum(i["n"] for i in hp.infos if i["scheme"] == s), 4)}
                for s in (0, 1)},
        "roofline": roofline,
        "clocks": clk,
        "gpu_launches": int(launches),
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(repeats=2)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(args, W, torch, hp, specs, dist):
    """Same hot path through the public API, inputs copied from pinned host memory each step
    and every GEMV result read back to the host.  Two device input sets alternate: step k+1's
    weights and x are copied on a second stream while step k computes (the copy of step 0
    and every later one lies inside the timed region)."""
    host_w = [w.cpu().pin_memory() for w in hp.weights]
    host_x = {B: [x.cpu().pin_memory() for x in hp.xs[B]] for B in BATCHES}
    host_y = {B: [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in hp.ys[B]] for B in BATCHES}
    host_yp = {B: [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in hp.yp[B]] for B in BATCHES}
    h2d = sum(w.numel() * 2 for w in host_w) + sum(x.numel() * 2 for B in BATCHES for x in host_x[B])
    d2h = sum(y.numel() * 4 for B in BATCHES for y in host_y[B]) + sum(
        y.numel() * 4 for B in BATCHES for y in host_yp[B])
    sets = []
    for _ in range(2):
        dev_w = [torch.empty_like(w) for w in hp.weights]
        dev_x = {B: [torch.empty_like(x) for x in hp.xs[B]] for B in BATCHES}
        sets.append((dev_w, dev_x, HotPath(W, dev_w, specs, dev_x, hp.stream)))
    copy_stream = torch.cuda.Stream()
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(i):
        dev_w, dev_x, _ = sets[i]
        copy_stream.wait_event(done[i])  # the set's previous step has finished with it
        with torch.cuda.stream(copy_stream):
            for d, h in zip(dev_w, host_w):
                d.copy_(h, non_blocking=True)
            for B in BATCHES:
                for d, h in zip(dev_x[B], host_x[B]):
                    d.copy_(h, non_blocking=True)
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
            e2e_hp = sets[i][2]
            e2e_hp.step()
            for B in BATCHES:
                for h, d in zip(host_y[B], e2e_hp.ys[B]):
                    h.copy_(d, non_blocking=True)
                for h, d in zip(host_yp[B], e2e_hp.yp[B]):
                    h.copy_(d, non_blocking=True)
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
    ms = allmax(dist, a.elapsed_time(b))
    for _, _, e2e_hp in sets:
        for c in e2e_hp.containers:
            c.free(hp.stream)
    step_bytes = sum(hp.algorithmic_bytes().values())
    v = allsum(dist, step_bytes * args.steps) / (ms / 1e3) / 1e9
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


def load_traffic(key: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary, or None when
    the summary has no such line or the kernel's sources changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic_dense_layers.md")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if len(parts) == 4 and parts[0] == "bench-traffic" and parts[1] == key:
            files, digest = parts[3].split("=")
            if _source_digest(files.split("+")) != digest:
                return None
            return int(parts[2])
    return None


def workload_config(specs, world: int) -> dict:
    """The `config` of both arms' lines: the workload a step covers."""
    return {"workload": "dense layer set: 4 x 4096x4096 + 3 x 4096x11008 BF16, both schemes, "
                        "encode + batched decode + fused GEMV B=1,4 + plain GEMV B=1,4",
            "tensors": len(specs), "elements": int(sum(s.n for s in specs)), "batches": list(BATCHES),
            "l2": "inputs larger than L2 (386 MB BF16, ~580 MB containers), swept in order",
            "parallelism": f"replicas x{world}"}


# ---------------------------------------------------------------------------
# The reference arm: the CPU oracle, timed on the host cores.
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from decode_gemv_sign_gb300 import synth
    vals = []
    for _ in range(args.warmup):
        cpu_baseline()
    t_total, b_total = 0.0, 0.0
    last = None
    for _ in range(args.steps):
        last = cpu_baseline()
        if last["value"] is None:
            print(json.dumps({"impl": "reference", "unavailable": "oracle run failed: " + str(last.get("error"))}))
            return
        t_total += last["seconds"]
        b_total += last["value"] * last["seconds"] * 1e9
        vals.append(last["value"])
    v = b_total / t_total / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_total / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16 codec / f64 GEMV",
        "data": "synthetic (seeded numpy draw of the same workload recipe)",
        # the same workload as our arm's line; each step times a bounded sample of it (cpu_baseline)
        "config": workload_config(synth.workload_dense_layers(), world),
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": CPU_SAMPLE},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 200 for ours, so the timed region spans several clock "
                         "samples; 10 for the reference arm, whose steps take seconds each)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_sample:
        print(json.dumps(oracle_sample_run()))
        return
    if args.steps is None:
        args.steps = 200 if args.impl == "ours" else 10
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
