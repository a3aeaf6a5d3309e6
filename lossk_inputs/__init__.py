"""Seeded synthetic inputs for the fused LM-head loss.

This module only draws random numbers; it holds none of the loss arithmetic,
so both the oracle side and the CUDA side may use it.  Every array is drawn
with ``numpy.random.default_rng([seed, stream])`` (streams: hidden 1,
weight 2, targets 3, mask 4, teacher 5), so each tensor is independent of the
others' shapes.  Normals are drawn in float32 and, for the bf16 workloads,
rounded to bf16 (round-to-nearest-even, via torch); the oracle and the GPU
then see the same bits.

Workloads (named by what they are):

=====================  =====  =====  ======  ======  =========================================
name                   n_tok  d      vocab   chunk   distributions
=====================  =====  =====  ======  ======  =========================================
tiny_fp32_ce           64     64     1000    16      H~N(0,1), W~N(0,0.02), y~U[0,V); fp32
ce_512x1024x32000      512    1024   32000   128     H~N(0,1), W~N(0,0.02), y~U
qwen3_0p6b_head        2048   1024   151936  256     H~N(0,1), W~N(0,0.02), y~Zipf(1.1)
ce_z_8192x4096x128256  8192   4096   128256  1024    W~N(0,0.015), y~U, z weight 1e-4, 5% masked
distill_z_4096x2048    4096   2048   151936  512     W~N(0,0.02), teacher~N(0,3) bf16, T=2,
                                                     10% masked, z weight 1e-4
=====================  =====  =====  ======  ======  =========================================

"N(0, s)" is read as standard deviation s.  Zipf(s) over vocabulary ids is
P(v) proportional to (v+1)^-s on [0, V), sampled by inverse CDF in float64.
Masks mark exactly round(f*n) tokens as excluded, chosen without replacement.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

STREAM_HIDDEN, STREAM_WEIGHT, STREAM_TARGETS, STREAM_MASK, STREAM_TEACHER = 1, 2, 3, 4, 5


@dataclass(frozen=True)
class Workload:
    name: str
    n_tok: int
    d_model: int
    vocab: int
    chunk: int
    dtype: str = "bf16"            # "bf16" or "fp32"
    hidden_std: float = 1.0
    weight_std: float = 0.02
    targets: str = "uniform"       # "uniform" or "zipf1.1"
    mask_frac: float = 0.0
    z_weight: float = 0.0
    teacher_std: float = 0.0       # > 0: distillation workload
    temperature: float = 1.0
    directions: tuple = field(default=())


WORKLOADS = {
    "tiny_fp32_ce": Workload("tiny_fp32_ce", 64, 64, 1000, 16, dtype="fp32"),
    "ce_512x1024x32000": Workload("ce_512x1024x32000", 512, 1024, 32000, 128),
    "qwen3_0p6b_head": Workload("qwen3_0p6b_head", 2048, 1024, 151936, 256, targets="zipf1.1"),
    "ce_z_8192x4096x128256": Workload("ce_z_8192x4096x128256", 8192, 4096, 128256, 1024,
                                      weight_std=0.015, mask_frac=0.05, z_weight=1e-4),
    "distill_z_4096x2048": Workload("distill_z_4096x2048", 4096, 2048, 151936, 512,
                                    teacher_std=3.0, temperature=2.0, mask_frac=0.10,
                                    z_weight=1e-4, directions=("fkl", "rkl", "ce")),
}


def rng(seed: int, stream: int, batch: int = 0) -> np.random.Generator:
    """Batch 0 is the workload's own batch; batch b > 0 is another batch drawn
    with the same recipe (a data-parallel rank's share), same weight."""
    return np.random.default_rng([seed, stream] if batch == 0 else [seed, stream, batch])


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (RNE) and return them widened to float32."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).to(torch.float32).numpy()


def to_f16_values(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE half (RNE) and return them widened to float32."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """The values a tensor of `dtype` ("bf16", "f16" or "fp32") holds."""
    if dtype == "bf16":
        return to_bf16_values(x)
    if dtype == "f16":
        return to_f16_values(x)
    return x


def _normal(seed, stream, shape, std, dtype, batch=0):
    x = rng(seed, stream, batch).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return round_to(x, dtype)


def hidden(seed, n, d, std=1.0, dtype="bf16", batch=0):
    return _normal(seed, STREAM_HIDDEN, (n, d), std, dtype, batch)


def weight(seed, V, d, std=0.02, dtype="bf16"):
    return _normal(seed, STREAM_WEIGHT, (V, d), std, dtype)


def teacher(seed, n, V, std=3.0, batch=0, dtype="bf16"):
    return _normal(seed, STREAM_TEACHER, (n, V), std, dtype, batch)


def targets(seed, n, V, kind="uniform", batch=0):
    g = rng(seed, STREAM_TARGETS, batch)
    if kind == "uniform":
        return g.integers(0, V, size=n, dtype=np.int64)
    if kind.startswith("zipf"):
        s = float(kind[4:])
        p = np.arange(1, V + 1, dtype=np.float64) ** (-s)
        cdf = np.cumsum(p)
        cdf /= cdf[-1]
        u = g.random(n)
        return np.minimum(np.searchsorted(cdf, u, side="right"), V - 1).astype(np.int64)
    raise ValueError(kind)


def mask(seed, n, frac, batch=0):
    """uint8 mask, 1 = token counts; exactly round(frac*n) tokens are 0."""
    m = np.ones(n, dtype=np.uint8)
    k = int(round(frac * n))
    if k:
        m[rng(seed, STREAM_MASK, batch).choice(n, k, replace=False)] = 0
    return m


def make(w: Workload | str, seed: int = 0, n_tok=None, d_model=None, vocab=None, batch=0):
    """Draw a workload's inputs (optionally at overridden sizes, same recipe).

    Returns a dict of float32/int64/uint8 numpy arrays: hidden [n][d],
    weight [V][d], targets [n], mask [n] or None, teacher [n][V] or None.
    `batch` selects another batch (hidden, targets, mask, teacher) for the
    same weight.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    n = n_tok or w.n_tok
    d = d_model or w.d_model
    V = vocab or w.vocab
    out = {
        "hidden": hidden(seed, n, d, w.hidden_std, w.dtype, batch),
        "weight": weight(seed, V, d, w.weight_std, w.dtype),
        "targets": targets(seed, n, V, w.targets, batch),
        "mask": mask(seed, n, w.mask_frac, batch) if w.mask_frac > 0 else None,
        "teacher": teacher(seed, n, V, w.teacher_std, batch) if w.teacher_std > 0 else None,
    }
    return out
