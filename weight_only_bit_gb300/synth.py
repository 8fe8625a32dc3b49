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

import os
from concurrent.futures import ThreadPoolExecutor

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


ROW_BLOCK = 1024   # rows per independently seeded generator block


def _fill_block(seed: int, b: int, k: int, rows: int, sigma: float) -> np.ndarray:
    out = np.empty((rows, k), dtype=np.float32)
    np.random.Generator(np.random.PCG64([seed, b])).standard_normal(out=out, dtype=np.float32)
    out *= np.float32(sigma)
    return out


def _outliers(seed: int, n: int, k: int, frac: float, sigmas: float, sigma: float):
    count = int(round(frac * n * k))
    rng = np.random.Generator(np.random.PCG64([seed, 1 << 40]))
    pos = rng.choice(n * k, size=count, replace=False)
    sign = np.where(rng.random(count) < 0.5, -1.0, 1.0)
    return pos, (sign * sigmas * sigma).astype(np.float32)


def weights(seed: int, n: int, k: int, sigma: float = 0.02,
            outlier_frac: float = 0.0, outlier_sigmas: float = 10.0) -> np.ndarray:
    """FP32 weight matrix [n, k] with entries N(0, sigma).

    Rows come in blocks of ROW_BLOCK, block b drawn by PCG64 seeded with (seed, b), so the matrix
    is the same whatever the number of threads, and any rows can be regenerated alone.
    With outlier_frac > 0, exactly round(outlier_frac * n * k) distinct positions, drawn without
    replacement, are replaced by +-outlier_sigmas * sigma with a random sign (the 0.1 % outliers
    at 10 sigma of the outlier sweep).
    """
    nb = (n + ROW_BLOCK - 1) // ROW_BLOCK
    w = np.empty((n, k), dtype=np.float32)

    def fill(b):
        r0 = b * ROW_BLOCK
        r1 = min(n, r0 + ROW_BLOCK)
        w[r0:r1] = _fill_block(seed, b, k, r1 - r0, sigma)

    if nb > 1:
        with ThreadPoolExecutor(max_workers=min(nb, os.cpu_count() or 4)) as ex:
            list(ex.map(fill, range(nb)))
    else:
        fill(0)
    if outlier_frac > 0.0:
        pos, val = _outliers(seed, n, k, outlier_frac, outlier_sigmas, sigma)
        w.reshape(-1)[pos] = val
    return w


def weights_rows(seed: int, n: int, k: int, rows, sigma: float = 0.02,
                 outlier_frac: float = 0.0, outlier_sigmas: float = 10.0) -> np.ndarray:
    """Rows `rows` of weights(seed, n, k, ...), generating only the blocks that hold them."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((len(rows), k), dtype=np.float32)
    blocks = {}
    for i, r in enumerate(rows):
        b = int(r) // ROW_BLOCK
        if b not in blocks:
            r0 = b * ROW_BLOCK
            blocks[b] = _fill_block(seed, b, k, min(n, r0 + ROW_BLOCK) - r0, sigma)
        out[i] = blocks[b][int(r) - b * ROW_BLOCK]
    if outlier_frac > 0.0:
        pos, val = _outliers(seed, n, k, outlier_frac, outlier_sigmas, sigma)
        pr, pc = pos // k, pos % k
        for i, r in enumerate(rows):
            sel = pr == r
            out[i, pc[sel]] = val[sel]
    return out


def activations(seed: int, m: int, k: int) -> np.ndarray:
    """FP16 activations [m, k]: N(0, 1) draws rounded to FP16 (round to nearest even)."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((m, k)).astype(np.float16)


def step_weight_count() -> int:
    return sum(n * k * c for _, n, k, c in DECODE_SHAPES)


def step_gemv_count() -> int:
    return sum(c for *_, c in DECODE_SHAPES)
