"""Seeded synthetic BF16 weights and activations.

This module only produces inputs.  It holds none of the codec's arithmetic
(no symbols, tables, codes or streams): it draws floats, rounds them to BF16
bit patterns and hands out ``uint16`` arrays.  Both the CPU oracle and the
CUDA path consume what it returns, so neither side regenerates inputs.

Two generators are provided:

* ``numpy`` (PCG64): platform-independent, used for every case the oracle
  checks element by element and for the stored golden values.
* ``torch`` on a CUDA device: used for workloads too large to draw on the
  host in seconds (hundreds of millions of weights).  The bits it produces
  are copied to the host whenever the oracle has to look at them.

Distributions follow the five workloads defined below (weights
drawn N(0, sigma) or Student-t(4) scaled to sigma, with a fixed fraction of
outlier positions taken from a seeded permutation).  Heavy Student-t tails
are the shape the quantization-survey page on weight distributions reports
for trained weights.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

BF16_NAN = 0x7FC0


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (round to nearest, ties to even); return uint16 bits.

    NaN inputs become a quiet NaN that keeps the sign.  This matches
    ``torch.Tensor.to(torch.bfloat16)``.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    rounded = ((u + 0x7FFF + lsb) >> 16).astype(np.uint32)
    nan = np.isnan(a)
    if nan.any():
        sign = ((u >> 16) & 0x8000).astype(np.uint32)
        rounded = np.where(nan, sign | BF16_NAN, rounded)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class WeightSpec:
    """One synthetic weight tensor W[N, K] (row-major, y = x @ W.T)."""

    name: str
    N: int
    K: int
    dist: str  # "normal" | "t4"
    sigma: float
    outlier_frac: float = 0.0
    outlier_kind: str = "none"  # "normal" (N(0, outlier_scale)) | "pm" (+-outlier_scale)
    outlier_scale: float = 0.0
    seed: int = 0
    offset: float = 0.0  # added after drawing (norm weights sit around 1.0)

    @property
    def n(self) -> int:
        return self.N * self.K


def _outlier_count(n: int, frac: float) -> int:
    return int(round(frac * n))


def gen_weights_np(spec: WeightSpec) -> np.ndarray:
    """Draw ``spec`` with numpy's PCG64; return uint16 BF16 bits of shape [N, K]."""
    rng = np.random.Generator(np.random.PCG64(spec.seed))
    n = spec.n
    if spec.dist in ("normal", "normal_clamped"):
        v = rng.standard_normal(n, dtype=np.float32) * np.float32(spec.sigma)
        if spec.dist == "normal_clamped":
            v = np.sign(v + np.float32(1e-30)) * np.clip(np.abs(v), np.float32(2.0**-14), np.float32(2.0**-2 * 0.99))
            v = v.astype(np.float32)
    elif spec.dist == "t4":
        # Student-t with 4 degrees of freedom has variance 2: scale to std sigma.
        v = rng.standard_t(4, size=n).astype(np.float32) * np.float32(spec.sigma / math.sqrt(2.0))
    else:
        raise ValueError(f"unknown distribution {spec.dist!r}")
    if spec.offset:
        v = v + np.float32(spec.offset)
    m = _outlier_count(n, spec.outlier_frac)
    if m:
        pos = rng.permutation(n)[:m]
        if spec.outlier_kind == "normal":
            v[pos] = rng.standard_normal(m, dtype=np.float32) * np.float32(spec.outlier_scale)
        elif spec.outlier_kind == "pm":
            sgn = np.where(rng.integers(0, 2, size=m) == 1, 1.0, -1.0).astype(np.float32)
            v[pos] = sgn * np.float32(spec.outlier_scale)
        else:
            raise ValueError(f"unknown outlier kind {spec.outlier_kind!r}")
    return f32_to_bf16_bits(v).reshape(spec.N, spec.K)


def gen_weights_torch(spec: WeightSpec, device):
    """Draw ``spec`` on a torch device; return an int16 tensor [N, K] holding BF16 bits.

    The values follow the same recipe as :func:`gen_weights_np` but come from
    torch's device generator, so the bits differ from the numpy draw.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(spec.seed)
    n = spec.n
    if spec.dist in ("normal", "normal_clamped"):
        v = torch.randn(n, generator=g, device=device, dtype=torch.float32) * spec.sigma
        if spec.dist == "normal_clamped":
            sgn = torch.where(v < 0, -1.0, 1.0)
            v = sgn * v.abs().clamp_(2.0**-14, 2.0**-2 * 0.99)
            del sgn
    elif spec.dist == "t4":
        # t4 = Z / sqrt(chi2_4 / 4); chi2_4 = -2 log(U1 U2).
        z = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        u = torch.rand(2, n, generator=g, device=device, dtype=torch.float32).clamp_min_(1e-30)
        chi2 = -2.0 * torch.log(u[0] * u[1])
        v = z / torch.sqrt(chi2 / 4.0) * (spec.sigma / math.sqrt(2.0))
        del z, u, chi2
    else:
        raise ValueError(f"unknown distribution {spec.dist!r}")
    if spec.offset:
        v += spec.offset
    m = _outlier_count(n, spec.outlier_frac)
    if m:
        pos = torch.randperm(n, generator=g, device=device)[:m]
        if spec.outlier_kind == "normal":
            v[pos] = torch.randn(m, generator=g, device=device, dtype=torch.float32) * spec.outlier_scale
        else:
            sgn = torch.randint(0, 2, (m,), generator=g, device=device).to(torch.float32) * 2 - 1
            v[pos] = sgn * spec.outlier_scale
        del pos
    return v.to(torch.bfloat16).view(torch.int16).reshape(spec.N, spec.K)


def gen_x_np(B: int, K: int, seed: int) -> np.ndarray:
    """Activations x[B, K] ~ N(0, 1) as BF16 bits (numpy draw)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return f32_to_bf16_bits(rng.standard_normal(B * K, dtype=np.float32)).reshape(B, K)


def gen_x_torch(B: int, K: int, seed: int, device):
    """Activations x[B, K] ~ N(0, 1) as an int16 tensor of BF16 bits (device draw)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    v = torch.randn(B * K, generator=g, device=device, dtype=torch.float32)
    return v.to(torch.bfloat16).view(torch.int16).reshape(B, K)


# --------------------------------------------------------------------------
# The five workloads.  "N x K" is read as W[N, K] of y = x @ W.T.
# Tensor i of workload c uses seed 1000 * c + i (workload 1 uses seed 0).
# --------------------------------------------------------------------------

def workload_small() -> List[WeightSpec]:
    """One 1024x1024 matrix, N(0, 0.02) with 0.05% N(0, 1) outliers, seed 0."""
    return [WeightSpec("w1024", 1024, 1024, "normal", 0.02, 0.0005, "normal", 1.0, seed=0)]


def workload_dense_layers() -> List[WeightSpec]:
    """4 x 4096x4096 and 3 x 4096x11008, N(0, 0.02) with 0.1% N(0, 0.5) outliers."""
    out = []
    for i in range(4):
        out.append(WeightSpec(f"attn{i}", 4096, 4096, "normal", 0.02, 0.001, "normal", 0.5, seed=2000 + i))
    for i in range(3):
        out.append(WeightSpec(f"mlp{i}", 4096, 11008, "normal", 0.02, 0.001, "normal", 0.5, seed=2004 + i))
    return out


def workload_block6144() -> List[WeightSpec]:
    """q/k/v/o 6144x6144 and 3 x 6144x16384, Student-t(4) scaled to std 0.02."""
    out = []
    for i, nm in enumerate("qkvo"):
        out.append(WeightSpec(nm, 6144, 6144, "t4", 0.02, seed=3000 + i))
    for i in range(3):
        out.append(WeightSpec(f"mlp{i}", 6144, 16384, "t4", 0.02, seed=3004 + i))
    return out


def workload_moe(n_experts: int = 128) -> List[WeightSpec]:
    """Per expert: 2048x6144 and 6144x2048, N(0, s) with s ~ U(0.005, 0.05), 0.2% outliers at +-50 s."""
    rng = np.random.Generator(np.random.PCG64(4000))
    sig = rng.uniform(0.005, 0.05, size=n_experts)
    out = []
    for e in range(n_experts):
        s = float(sig[e])
        out.append(WeightSpec(f"e{e}.up", 2048, 6144, "normal", s, 0.002, "pm", 50 * s, seed=4000 + 2 * e + 1))
        out.append(WeightSpec(f"e{e}.down", 6144, 2048, "normal", s, 0.002, "pm", 50 * s, seed=4000 + 2 * e + 2))
    return out


def moe_selected_experts(k: int = 8, n_experts: int = 128, seed: int = 4999) -> List[int]:
    """The seeded choice of experts the batch-1 MoE GEMV runs on."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return sorted(int(e) for e in rng.choice(n_experts, size=k, replace=False))


def workload_checkpoint(layers: int = 113) -> List[WeightSpec]:
    """Checkpoint-shaped set: 2 embeddings 151552x6144 and, per layer, 4 x 6144^2,
    2 x 16384x6144, 1 x 6144x16384, 8 x 2048x6144 and 2 norms [6144].

    Even-indexed matrices are Normal, odd ones Student-t(4); sigma ~ U(0.005, 0.05);
    0.1% N(0, 25 sigma^2) outliers; norms are 1 + N(0, 0.02).
    """
    rng = np.random.Generator(np.random.PCG64(5000))
    shapes = [(151552, 6144), (151552, 6144)]
    kinds = ["mat", "mat"]
    for _ in range(layers):
        shapes += [(6144, 6144)] * 4 + [(16384, 6144)] * 2 + [(6144, 16384)] + [(2048, 6144)] * 8
        kinds += ["mat"] * 15
        shapes += [(1, 6144)] * 2
        kinds += ["norm"] * 2
    out = []
    m = 0
    for i, ((N, K), kind) in enumerate(zip(shapes, kinds)):
        if kind == "norm":
            out.append(WeightSpec(f"t{i}", N, K, "normal", 0.02, seed=5001 + i, offset=1.0))
            continue
        s = float(rng.uniform(0.005, 0.05))
        dist = "normal" if m % 2 == 0 else "t4"
        m += 1
        out.append(WeightSpec(f"t{i}", N, K, dist, s, 0.001, "normal", 5 * s, seed=5001 + i))
    return out


def batches(specs: Sequence[WeightSpec], batch_bytes: int) -> List[List[WeightSpec]]:
    """Consecutive groups of specs holding at most ``batch_bytes`` of BF16 each
    (a tensor larger than the limit forms a group of its own)."""
    out, cur, size = [], [], 0
    for s in specs:
        b = 2 * s.n
        if cur and size + b > batch_bytes:
            out.append(cur)
            cur, size = [], 0
        cur.append(s)
        size += b
    if cur:
        out.append(cur)
    return out


def checkpoint_batch(index: int = 0, batch_bytes: int = 16 << 30) -> List[WeightSpec]:
    """Batch ``index`` of the checkpoint-shaped set in HBM-sized groups."""
    return batches(workload_checkpoint(), batch_bytes)[index]


def checkpoint_gemv_spec() -> WeightSpec:
    """The single large GEMV weight of the checkpoint workload: 16384x53248."""
    return WeightSpec("gemv16384x53248", 16384, 53248, "t4", 0.02, 0.001, "normal", 0.1, seed=5999)


def dense12_spec(N: int = 16384, K: int = 53248, seed: int = 6000) -> WeightSpec:
    """Escape-free weights: N(0, 0.02) with every magnitude clamped into
    [2^-14, 2^-2), so only 14 high bytes occur (sign x exponent bits 7..1 of
    113..124) and byte-split needs no escape at all: exactly 4 code bits plus 8
    raw bits per weight, the dense 12-bit form of the pages' GPU prototype."""
    return WeightSpec("dense12", N, K, "normal_clamped", 0.02, seed=seed)


WORKLOADS = {
    "small": workload_small,
    "dense_layers": workload_dense_layers,
    "block6144": workload_block6144,
    "moe": workload_moe,
    "checkpoint": workload_checkpoint,
}


def total_elements(specs: Sequence[WeightSpec]) -> int:
    return sum(s.n for s in specs)


def pick(specs: Sequence[WeightSpec], names: Optional[Sequence[str]] = None) -> List[WeightSpec]:
    if names is None:
        return list(specs)
    d = {s.name: s for s in specs}
    return [d[n] for n in names]
