"""Seeded synthetic inputs for the TSP layer forward.

This module is shared by the oracle side (tests, CPU baseline) and the CUDA side
(tests, bench). It holds no arithmetic of the method itself: it only draws
numbers, rounds them to bfloat16 bit patterns and names the workloads.

Workloads follow the evaluation setup of "Folding Tensor and Sequence
Parallelism for Memory-Efficient Transformer Training & Inference" (section 4,
Results): a 7B-parameter dense transformer at 16K-128K tokens, plus two small
shapes that the oracle finishes in seconds. All are batch 1 (a micro-batch of
several sequences is drawn on request) with
x ~ N(0, 1) and every weight ~ N(0, 0.02), drawn from a Philox counter-based
generator (NumPy) and rounded to bfloat16 with round-to-nearest-even.

Weights use the ``nn.Linear`` layout ``[out_features, in_features]``:
Wq, Wk, Wv, Wo are ``[H, H]``; W1 (gate) and W3 (up) are ``[F, H]``; W2 (down)
is ``[H, F]``.
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "LayerConfig",
    "CONFIGS",
    "config_by_name",
    "bf16_bits_from_f32",
    "normal_bf16_bits",
    "layer_inputs",
    "sample_rows",
]


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """One TSP layer workload: D logical ranks, S tokens, hidden H, heads, ffn F."""

    name: str
    D: int
    S: int
    hidden: int
    heads: int
    ffn: int
    seed: int

    @property
    def head_dim(self) -> int:
        return self.hidden // self.heads

    @property
    def tokens_per_rank(self) -> int:
        return self.S // self.D

    @property
    def chunk(self) -> int:
        """Zigzag chunk length: the sequence is cut into 2D equal chunks."""
        return self.S // (2 * self.D)

    def describe(self) -> str:
        return (f"{self.name}: D={self.D} S={self.S} hidden={self.hidden} "
                f"heads={self.heads}x{self.head_dim} ffn={self.ffn}")


# The five workloads. The seed of each is 1234 + its index.
CONFIGS = (
    LayerConfig("tiny", D=2, S=256, hidden=256, heads=4, ffn=688, seed=1234),
    LayerConfig("small", D=4, S=4096, hidden=1024, heads=16, ffn=2816, seed=1235),
    LayerConfig("7b-16k", D=8, S=16384, hidden=4096, heads=32, ffn=11008, seed=1236),
    LayerConfig("7b-64k", D=8, S=65536, hidden=4096, heads=32, ffn=11008, seed=1237),
    LayerConfig("7b-128k", D=8, S=131072, hidden=4096, heads=32, ffn=11008, seed=1238),
)


def config_by_name(name: str) -> LayerConfig:
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(f"unknown workload {name!r}; known: {[c.name for c in CONFIGS]}")


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even); return uint16 bits.

    Inputs are finite (normal draws), so no NaN handling is needed.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def normal_bf16_bits(shape, std: float, seed: int, stream: int) -> np.ndarray:
    """Draw N(0, std^2) float32 values from Philox(key=(seed, stream)); return bf16 bits."""
    rng = np.random.Generator(np.random.Philox(key=[seed, stream]))
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    step = 1 << 24  # draw in slices to bound the float32 temporary
    for lo in range(0, flat.size, step):
        n = min(step, flat.size - lo)
        v = rng.standard_normal(n, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        flat[lo:lo + n] = bf16_bits_from_f32(v)
    return out


_STREAMS = {"x": 0, "Wq": 1, "Wk": 2, "Wv": 3, "Wo": 4, "W1": 5, "W3": 6, "W2": 7}


def layer_inputs(cfg: LayerConfig, seed: int | None = None, names=None, batch: int = 1) -> dict:
    """Return the seeded bf16 bit patterns (uint16 arrays) of one workload.

    Keys: x [S, H] (or [batch, S, H] for a micro-batch of `batch` sequences);
    Wq, Wk, Wv, Wo [H, H]; W1, W3 [F, H]; W2 [H, F]. ``names`` restricts the draw
    to a subset of keys. The sequences of a micro-batch are consecutive draws of
    the same stream, so sequence 0 equals the batch-1 x of the same seed.
    """
    seed = cfg.seed if seed is None else seed
    H, F, S = cfg.hidden, cfg.ffn, cfg.S
    xshape = (S, H) if batch == 1 else (batch, S, H)
    shapes = {"x": xshape, "Wq": (H, H), "Wk": (H, H), "Wv": (H, H), "Wo": (H, H),
              "W1": (F, H), "W3": (F, H), "W2": (H, F)}
    out = {}
    for k in (names or shapes):
        std = 1.0 if k == "x" else 0.02
        out[k] = normal_bf16_bits(shapes[k], std, seed, _STREAMS[k])
    return out


def sample_rows(S: int, n: int, seed: int) -> np.ndarray:
    """n distinct sorted token positions in [0, S), always holding 0 and S-1."""
    n = min(n, S)
    rng = np.random.Generator(np.random.Philox(key=[seed, 99]))
    inner = rng.choice(np.arange(1, S - 1), size=max(n - 2, 0), replace=False) if S > 2 else []
    rows = np.unique(np.concatenate([[0, S - 1], np.asarray(inner, dtype=np.int64)]))
    return rows.astype(np.int64)
