"""Seeded synthetic workload for the 4-bit weight-only decode GEMVs.

This module only draws random numbers and names shapes.  It holds none of the
method's arithmetic (no quantisation, packing, scaling or dot products), so both
the CUDA path and the CPU oracle may take their inputs from it.

Workload (the decode step the pages measure):
  * "Do Quantization and Sparsity make LLM Inference Faster ?", section
    "What we did": eight matrix shapes of one Qwen2.5-1.5B decode step, 197
    matrix multiplications per generated token, tested at batches 1, 8, 32, 128.
  * "LLM Quantization on RTX 4060: Where 4-bit Decode Falls Behind FP16",
    section "Why k/v Projections": q/o 1536 -> 1536, k/v 1536 -> 256.
  * "My Triton Kernel Ties bitsandbytes -- and Both Lose to Math", section
    "The roofline first": 3.087 GB of bf16 weights, 0.772 GB at int4, so the
    step holds 1,543,569,408 weights.

No trained weights are used: W ~ N(0, 0.02) and x ~ N(0, 1) stand in for the
model's weights and hidden states, with the model's shapes.
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 20261202

# (name, N = out features, K = in features, count per decode step)
DECODE_SHAPES = (
    ("q", 1536, 1536, 28),
    ("k", 256, 1536, 28),
    ("v", 256, 1536, 28),
    ("o", 1536, 1536, 28),
    ("gate", 8960, 1536, 28),
    ("up", 8960, 1536, 28),
    ("down", 1536, 8960, 28),
    ("lm_head", 151936, 1536, 1),
)
N_LAYERS = 28
PROJ_INDEX = {"q": 0, "k": 1, "v": 2, "o": 3, "gate": 4, "up": 5, "down": 6, "lm_head": 0}

# Activation slots of one layer: which projections read the same input vector
# (q, k and v read the attention input; gate and up read the MLP input).
X_SLOT = {"q": 0, "k": 0, "v": 0, "o": 1, "gate": 2, "up": 2, "down": 3, "lm_head": 0}


def shape_of(name: str) -> tuple[int, int]:
    for nm, n, k, _ in DECODE_SHAPES:
        if nm == name:
            return n, k
    raise KeyError(name)


def weight_seed(layer: int, proj: str) -> int:
    """Seed of one weight matrix; the lm_head sits at layer 28."""
    return BASE_SEED + 1000 * layer + PROJ_INDEX[proj]


def x_seed(layer: int, slot: int, batch: int) -> int:
    return BASE_SEED + 1000 * layer + 500 + 10 * slot + 100000 * batch


def decode_step_gemvs():
    """The 197 GEMVs of one decode step in execution order.

    Yields (layer, proj, N, K).  Execution order follows one decoder layer:
    q, k, v, o, gate, up, down; the lm_head closes the step.
    """
    order = ("q", "k", "v", "o", "gate", "up", "down")
    for layer in range(N_LAYERS):
        for proj in order:
            n, k = shape_of(proj)
            yield layer, proj, n, k
    n, k = shape_of("lm_head")
    yield N_LAYERS, "lm_head", n, k


def weights(seed: int, n: int, k: int, sigma: float = 0.02,
            outlier_frac: float = 0.0, outlier_sigmas: float = 10.0) -> np.ndarray:
    """FP32 weight matrix [n, k] with entries N(0, sigma).

    With outlier_frac > 0, exactly round(outlier_frac * n * k) distinct positions,
    drawn without replacement, are replaced by +-outlier_sigmas * sigma with a
    random sign (the 0.1 % outliers at 10 sigma of the outlier sweep).
    """
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((n, k), dtype=np.float32)
    w *= np.float32(sigma)
    if outlier_frac > 0.0:
        count = int(round(outlier_frac * n * k))
        pos = rng.choice(n * k, size=count, replace=False)
        sign = np.where(rng.random(count) < 0.5, -1.0, 1.0)
        w.reshape(-1)[pos] = (sign * outlier_sigmas * sigma).astype(np.float32)
    return w


def activations(seed: int, m: int, k: int) -> np.ndarray:
    """FP16 activations [m, k]: N(0, 1) draws rounded to FP16 (round to nearest even)."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((m, k)).astype(np.float16)


def step_weight_count() -> int:
    return sum(n * k * c for _, n, k, c in DECODE_SHAPES)


def step_gemv_count() -> int:
    return sum(c for *_, c in DECODE_SHAPES)
