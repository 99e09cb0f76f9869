"""Seeded synthetic inputs for the AWQ W4A16 linear layer.

This module is shared by the CPU oracle, the tests and the benchmark. It
holds no arithmetic of the quantization method: it only draws random numbers
and rounds them to fp16, so that both sides of every parity check start from
the same bytes.

Recipe (the same for every layer shape):

* ``W`` ~ N(0, 0.02^2), drawn in fp32 and rounded to fp16 (RNE), shape
  ``[N, K]`` (row = output channel, column = input channel).
* ``X`` ~ N(0, 1), drawn in fp32; ``max(1, round(0.01 * K))`` input
  channels, picked by a seeded permutation, are multiplied by 20 before the
  fp16 cast.  These are the "salient" channels with large activations that the
  method protects ("AWQ量化实战" §2.1: a small fraction, 0.1%-1%, of channels
  carries most of the activation magnitude).  The same outlier channels are
  used for the calibration tokens and for the timed tokens of a layer.
* Seeds: ``1000 + layer_id`` for W, ``2000 + layer_id`` for calibration
  tokens, ``3000 + layer_id`` for timed tokens, ``4000 + layer_id`` for the
  outlier permutation.

The generator is numpy's PCG64; draws are made in fixed-size row chunks so
that the bytes do not depend on available memory.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "LAYERS", "MODELS", "layer", "outlier_channels", "weight", "activations",
    "calib_tokens", "timed_tokens",
]

# Llama-2 linear-layer shapes, K (input dim) -> N (output dim).  qkv and
# gate_up are the fused projections; 70B qkv is the grouped-query shape.
MODELS = {
    "toy": {"linear": (512, 512)},
    "llama2-7b": {"qkv": (4096, 12288), "o": (4096, 4096),
                  "gate_up": (4096, 22016), "down": (11008, 4096)},
    "llama2-13b": {"qkv": (5120, 15360), "o": (5120, 5120),
                   "gate_up": (5120, 27648), "down": (13824, 5120)},
    "llama2-70b": {"qkv": (8192, 10240), "o": (8192, 8192),
                   "gate_up": (8192, 57344), "down": (28672, 8192)},
}

# Stable per-layer ids for the seeds.
_MODEL_BASE = {"toy": 0, "llama2-7b": 10, "llama2-13b": 20, "llama2-70b": 30}
_LAYER_OFF = {"linear": 0, "qkv": 1, "o": 2, "gate_up": 3, "down": 4}

LAYERS = [(m, l) for m in MODELS for l in MODELS[m]]

_CHUNK = 1 << 22  # elements per draw


def layer(model: str, name: str):
    """Return ``(K, N, layer_id)`` for a named layer."""
    K, N = MODELS[model][name]
    return K, N, _MODEL_BASE[model] + _LAYER_OFF[name]


def _normal(rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.float32)
    flat = out.reshape(-1)
    for s in range(0, flat.size, _CHUNK):
        e = min(flat.size, s + _CHUNK)
        flat[s:e] = rng.standard_normal(e - s, dtype=np.float32)
    return out


def outlier_channels(K: int, layer_id: int) -> np.ndarray:
    """Sorted indices of the ``max(1, round(0.01*K))`` outlier input channels."""
    n_out = max(1, int(round(0.01 * K)))
    perm = np.random.Generator(np.random.PCG64(4000 + layer_id)).permutation(K)
    return np.sort(perm[:n_out])


def weight(N: int, K: int, layer_id: int, std: float = 0.02) -> np.ndarray:
    """fp16 ``[N, K]`` weight ~ N(0, std^2)."""
    rng = np.random.Generator(np.random.PCG64(1000 + layer_id))
    w = _normal(rng, N, K)
    w *= np.float32(std)
    return w.astype(np.float16)


def activations(T: int, K: int, layer_id: int, seed_base: int,
                outlier_gain: float = 20.0) -> np.ndarray:
    """fp16 ``[T, K]`` tokens ~ N(0,1) with the layer's outlier channels scaled."""
    rng = np.random.Generator(np.random.PCG64(seed_base + layer_id))
    idx = outlier_channels(K, layer_id)
    out = np.empty((T, K), dtype=np.float16)
    rows = max(1, _CHUNK // K)
    for r in range(0, T, rows):
        e = min(T, r + rows)
        x = _normal(rng, e - r, K)
        x[:, idx] *= np.float32(outlier_gain)
        out[r:e] = x.astype(np.float16)
    return out


def calib_tokens(T: int, K: int, layer_id: int) -> np.ndarray:
    """Calibration tokens for the scale search (seed 2000 + layer_id)."""
    return activations(T, K, layer_id, 2000)


def timed_tokens(M: int, K: int, layer_id: int) -> np.ndarray:
    """Tokens fed to the timed matmul (seed 3000 + layer_id)."""
    return activations(M, K, layer_id, 3000)
