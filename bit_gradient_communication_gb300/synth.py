"""Seeded synthetic gradient generators and the workload recipes.

This module holds none of the codec's arithmetic: it only draws inputs.  The
tests hand the same bytes to the CUDA path and to the CPU oracle, and the
benchmark times the CUDA path on them.  Distributions stand in for the
gradients of the workloads (no dataset is involved):
  normal          N(0, sigma^2)
  student_t3      Student-t with 3 degrees of freedom times a scale (heavy tails)
  laplace         Laplace(0, b) as b * (E1 - E2), E1, E2 ~ Exp(1)
  normal_outliers N(0, sigma^2) with a fraction p of positions times a factor
Device draws use one torch.Generator per call, advanced chunk by chunk, so a
(kind, n, seed) triple gives the same bytes on a given device and torch build.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 27


def _fill_chunk(torch, kind, m, g, device, params):
    if kind == "normal":
        return torch.randn(m, generator=g, device=device) * params.get("sigma", 1.0)
    if kind == "student_t3":
        z = torch.randn(m, generator=g, device=device)
        c = torch.zeros(m, device=device)
        for _ in range(3):
            c += torch.randn(m, generator=g, device=device) ** 2
        return z / torch.sqrt(c / 3.0) * params.get("scale", 1e-3)
    if kind == "laplace":
        e1 = torch.empty(m, device=device).exponential_(1.0, generator=g)
        e2 = torch.empty(m, device=device).exponential_(1.0, generator=g)
        return (e1 - e2) * params.get("b", 1e-3)
    if kind == "normal_outliers":
        x = torch.randn(m, generator=g, device=device) * params.get("sigma", 1e-4)
        hit = torch.rand(m, generator=g, device=device) < params.get("p", 1e-3)
        return torch.where(hit, x * params.get("factor", 100.0), x)
    raise ValueError(kind)


def gradients(kind: str, n: int, seed: int, dtype=None, device="cuda", out=None, **params):
    """n gradients of the given kind as a torch tensor (fp32 or bf16)."""
    import torch
    dtype = dtype or torch.float32
    if out is None:
        out = torch.empty(n, dtype=dtype, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    for lo in range(0, n, CHUNK):
        m = min(CHUNK, n - lo)
        out[lo:lo + m].copy_(_fill_chunk(torch, kind, m, g, device, params))
    return out


def np_gradients(kind: str, n: int, seed: int, **params) -> np.ndarray:
    """Host (numpy) draws of the same families, fp32, for CPU-only tests."""
    rng = np.random.default_rng(seed)
    if kind == "normal":
        x = rng.standard_normal(n) * params.get("sigma", 1.0)
    elif kind == "student_t3":
        x = rng.standard_t(3, n) * params.get("scale", 1e-3)
    elif kind == "laplace":
        x = rng.laplace(0.0, params.get("b", 1e-3), n)
    elif kind == "normal_outliers":
        x = rng.standard_normal(n) * params.get("sigma", 1e-4)
        hit = rng.random(n) < params.get("p", 1e-3)
        x = np.where(hit, x * params.get("factor", 100.0), x)
    else:
        raise ValueError(kind)
    return x.astype(np.float32)


@dataclass
class Workload:
    """One workload: its inputs and the codec parameters it runs with."""
    name: str
    n: int                      # elements per rank
    dtype: str                  # "f32" or "bf16"
    kind: str
    params: dict = field(default_factory=dict)
    bits: int = 4
    block: int = 128
    rounding: int = 0           # 0 RTN, 1 SR
    ef: bool = False
    ranks: int = 1
    ef2: bool = False
    bucket_bytes: int = 0
    seed: int = 0
    sr_seed: int = 0
    hadamard: int = 0           # Walsh-Hadamard transform block H, 0 = none


MiB = 1024 * 1024

# Workload recipes.  Sizes, distributions and codec parameters are those of
# the five benchmark configurations; seeds the configurations leave open are
# fixed here.
WORKLOADS = {
    "roundtrip_1m": Workload("roundtrip_1m", 1_048_576, "f32", "normal", {"sigma": 1.0},
                             bits=4, block=128, seed=0),
    "bucket25mb_f32": Workload("bucket25mb_f32", 6_553_600, "f32", "student_t3", {"scale": 1e-3},
                               bits=4, block=256, rounding=1, ef=True, seed=0, sr_seed=42,
                               bucket_bytes=25 * MiB),
    "allreduce_w8_gpt1p3b": Workload("allreduce_w8_gpt1p3b", 1_300_000_000, "bf16", "normal",
                                     {"sigma": 1e-3}, bits=4, block=128, ef=True, ranks=8, ef2=True,
                                     seed=1000),
    "gpt6p7b_2bit_buckets": Workload("gpt6p7b_2bit_buckets", 6_700_000_000, "bf16", "normal_outliers",
                                     {"sigma": 1e-4, "p": 1e-3, "factor": 100.0}, bits=2, block=64,
                                     rounding=1, ef=True, seed=4, sr_seed=4242, bucket_bytes=25 * MiB),
    "tlq_hs_w8_gpt1p3b": Workload("tlq_hs_w8_gpt1p3b", 1_300_000_000, "bf16", "normal", {"sigma": 1e-3},
                                  bits=8, block=512, ef=True, ranks=8, ef2=True, seed=1000),
    "qwd_gpt6p7b_w8": Workload("qwd_gpt6p7b_w8", 6_700_000_000, "bf16", "normal", {"sigma": 2e-2},
                               bits=4, block=2048, ranks=8, seed=7),
    "allgather_decode_gpt1p3b": Workload("allgather_decode_gpt1p3b", 1_300_000_000, "bf16", "normal",
                                         {"sigma": 1e-3}, bits=4, block=128, ranks=8, seed=1000),
    # the same decode of the two-level Hadamard-smoothed all-reduce's stage-2
    # codes (4-bit blocks of 128, rotated by H = 128): the inverse rotation runs
    # in the decode
    "allgather_decode_hs_gpt1p3b": Workload("allgather_decode_hs_gpt1p3b", 1_300_000_000, "bf16", "normal",
                                            {"sigma": 1e-3}, bits=4, block=128, ranks=8, seed=1000,
                                            hadamard=128),
    "sweep_laplace_256m": Workload("sweep_laplace_256m", 268_435_456, "f32", "laplace", {"b": 1e-3},
                                   bits=4, block=128, seed=5, sr_seed=55),
    # pipeline-A without local quantisation: the node leader's rank-ordered fp32
    # sum of its 8 local ranks' GPT-1.3B-shaped gradients
    "local_sum_w8_gpt1p3b": Workload("local_sum_w8_gpt1p3b", 1_300_000_000, "bf16", "normal", {"sigma": 1e-3},
                                     ranks=8, seed=1000),
    # pipeline-A with local quantisation: the node leader's decode of its 8 local
    # ranks' 4-bit codes into their rank-ordered fp32 sum (no requantisation)
    "local_decode_w8_gpt1p3b": Workload("local_decode_w8_gpt1p3b", 1_300_000_000, "bf16", "normal",
                                        {"sigma": 1e-3}, bits=4, block=128, ranks=8, seed=1000),
}
