"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws numbers: ternary weight matrices with a given zero
fraction, fp32 activations, per-layer zero fractions, and positions to corrupt.
It contains none of the method's arithmetic (no packing, quantisation or
products); each side -- the CUDA library and the CPU oracle -- consumes the
same int8 / fp32 arrays through its own code.

Workloads follow BitNet b1.58 2B4T's shapes ("Tritium: One Weight Format for
Ternary Inference ..." -- The model: 30 layers, hidden 2560, FFN 6912, 20
query heads with 5 key/value heads) and its measured zero statistics ("BITCOS:
Intel's Ternary LLM Weight Format Goes Below 1.58 Bits" -- The zeros nobody was
counting: 42.19% zeros model-wide, 38.5%-50.8% across tensors).  No checkpoint
is used: every weight is drawn i.i.d. from a seeded generator.

Every array is a pure function of (seed, layer, projection, stream), so any
single projection can be regenerated without drawing the rest.
"""
from __future__ import annotations

import numpy as np

# (name, N rows = output features, K cols = input features) of the seven
# ternary projections of one decoder layer.
PROJECTIONS = (
    ("q", 2560, 2560),
    ("k", 640, 2560),
    ("v", 640, 2560),
    ("o", 2560, 2560),
    ("gate", 6912, 2560),
    ("up", 6912, 2560),
    ("down", 2560, 6912),
)
FFN = ("gate", "up", "down")
LAYERS = 30
P_ZERO = 0.4219            # model-wide zero fraction of the 2B4T checkpoint
Z_RANGE = (0.385, 0.508)   # per-tensor zero fractions measured on that checkpoint
BATCH_SWEEP = (1, 2, 4, 8, 16, 32, 64)
PREFILL_M = (512, 2048)
CORRUPT_RATE = 0.001

# streams within one (seed, layer, projection) key
_W, _X, _Z, _C = 0, 1, 2, 3


def rng_for(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def ternary(rng: np.random.Generator, N: int, K: int, p0: float) -> np.ndarray:
    """int8 [N, K] with P(0) = p0 and P(+1) = P(-1) = (1 - p0) / 2, drawn by
    thresholding uniform 16-bit integers."""
    t0 = int(round(p0 * 65536))
    t1 = t0 + (65536 - t0) // 2
    lut = np.zeros(65536, dtype=np.int8)
    lut[t0:t1] = 1
    lut[t1:] = -1
    u = rng.integers(0, 65536, N * K, dtype=np.uint16)
    return lut[u].reshape(N, K)


def activations(rng: np.random.Generator, M: int, K: int, kind: str = "normal") -> np.ndarray:
    """fp32 [M, K]: 'normal' is N(0, 1); 'relu2' is relu(z)^2 with z ~ N(0, 1)
    (the squared-ReLU input of the down projection)."""
    z = rng.standard_normal((M, K), dtype=np.float32)
    if kind == "normal":
        return z
    if kind == "relu2":
        r = np.maximum(z, np.float32(0))
        return r * r
    raise ValueError(kind)


def w_scale(w: np.ndarray) -> np.float32:
    """The per-tensor fp32 scale 1 / mean|W| of a drawn ternary matrix."""
    nnz = int(np.count_nonzero(w))
    return np.float32(w.size / nnz) if nnz else np.float32(1.0)


def act_kind(name: str) -> str:
    return "relu2" if name == "down" else "normal"


def layer_zero_fraction(seed: int, layer: int) -> float:
    """Per-layer zero fraction, uniform in Z_RANGE, shared by the layer's seven projections."""
    return float(rng_for(seed, layer, 0, _Z).uniform(*Z_RANGE))


def projection_weights(seed: int, layer: int, idx: int, p0: float | None = None) -> np.ndarray:
    name, N, K = PROJECTIONS[idx]
    if p0 is None:
        p0 = P_ZERO
    return ternary(rng_for(seed, layer, idx, _W), N, K, p0)


def projection_acts(seed: int, layer: int, idx: int, M: int) -> np.ndarray:
    name, N, K = PROJECTIONS[idx]
    return activations(rng_for(seed, layer, idx, _X), M, K, act_kind(name))


def corrupt_positions(seed: int, layer: int, idx: int, n_beats: int, rate: float = CORRUPT_RATE):
    """Choose round(rate * n_beats) distinct beat indices and one bit position
    (0..63) for each.  Returns (beats int64 [n], bits int64 [n]), sorted by beat."""
    rng = rng_for(seed, layer, idx, _C)
    n = max(1, int(round(rate * n_beats)))
    beats = np.sort(rng.choice(n_beats, size=n, replace=False)).astype(np.int64)
    bits = rng.integers(0, 64, n).astype(np.int64)
    return beats, bits


# ---- the five workloads ----------------------------------------------------

def config0(seed: int = 0):
    """Single 2560 x 2560 GEMV at batch 1, P(0) = 0.4219, x ~ N(0, 1)."""
    rng = rng_for(seed, 0, 0, _W)
    w = ternary(rng, 2560, 2560, P_ZERO)
    x = activations(rng_for(seed, 0, 0, _X), 1, 2560, "normal")
    return w, x


def config1(seed: int = 1):
    """One layer: the seven projections at batch 1, P(0) = 0.4219; list of
    (name, W, x) with x relu(z)^2 for down and N(0, 1) otherwise."""
    out = []
    for idx, (name, N, K) in enumerate(PROJECTIONS):
        out.append((name, projection_weights(seed, 0, idx), projection_acts(seed, 0, idx, 1)))
    return out


def stack_items(layers: int = LAYERS):
    """(layer, idx, name, N, K) of the 30-layer stack in layer order."""
    for layer in range(layers):
        for idx, (name, N, K) in enumerate(PROJECTIONS):
            yield layer, idx, name, N, K


def stack_weights(seed: int, layer: int, idx: int) -> np.ndarray:
    """Weights of one projection of the 30-layer stack (per-layer zero fraction)."""
    return projection_weights(seed, layer, idx, layer_zero_fraction(seed, layer))


def prefill_items(layers: int = LAYERS):
    """(layer, idx, name, N, K) of the gate/up/down GEMMs of the prefill workload."""
    for layer in range(layers):
        for idx, (name, N, K) in enumerate(PROJECTIONS):
            if name in FFN:
                yield layer, idx, name, N, K
