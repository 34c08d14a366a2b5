"""Seeded synthetic inputs for the Gated DeltaNet prefill scan (host side).

Inputs only: counter-based random numbers (the streams of ``synth.gen``),
the unit-norm queries and keys a Gated DeltaNet layer hands its scan, and
rounding to the storage types.  No scan arithmetic lives here.

Recipe (one layer, one prompt or several):

* q, k [T, Hk, dk]: N(0, 1) vectors divided by their fp32 L2 norm, then
  rounded to bf16 (so their norms are 1 up to bf16 rounding);
* v [T, Hv, dv]: N(0, 1), bf16;
* g [T, Hv]: log(alpha) with alpha uniform in [0.9, 1.0), fp32 (a memory of
  ten tokens to the whole prompt);
* beta [T, Hv]: sigmoid of N(0, 1), fp32;
* initial state [N, Hv, dv, dk]: zero, or N(0, state_std) fp32.

Shape of the Qwen3.6-35B-A3B-style linear-attention layer: Hk = 16 query/key
heads, Hv = 32 value heads, dk = dv = 128.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import gen

TAG_GDN_Q = 21
TAG_GDN_K = 22
TAG_GDN_V = 23
TAG_GDN_GATE = 24
TAG_GDN_BETA = 25
TAG_GDN_STATE = 26


@dataclass
class GdnShape:
    Hk: int = 16
    Hv: int = 32
    dk: int = 128
    dv: int = 128


@dataclass
class GdnInputs:
    q: np.ndarray       # uint16 bf16 bits [T, Hk, dk]
    k: np.ndarray       # uint16 bf16 bits [T, Hk, dk]
    v: np.ndarray       # uint16 bf16 bits [T, Hv, dv]
    g: np.ndarray       # fp32 [T, Hv]
    beta: np.ndarray    # fp32 [T, Hv]
    state0: np.ndarray | None  # fp32 [N, Hv, dv, dk]
    offsets: np.ndarray  # int32 [N + 1]


def _uniform01(key: int, count: int) -> np.ndarray:
    """count values uniform in [0, 1): the top 24 bits of each draw."""
    d = gen.draws(key, np.arange(count, dtype=np.uint64))
    return (d >> np.uint64(40)).astype(np.float64) / float(1 << 24)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float32)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))


def make_inputs(seed: int, lengths, shape: GdnShape = GdnShape(), state_std: float = 0.0,
                layer: int = 0) -> GdnInputs:
    """Inputs for sequences of the given lengths, packed one after another."""
    lengths = [int(n) for n in lengths]
    T = sum(lengths)
    offsets = np.zeros(len(lengths) + 1, np.int32)
    offsets[1:] = np.cumsum(lengths)
    Hk, Hv, dk, dv = shape.Hk, shape.Hv, shape.dk, shape.dv

    def normal(tag, count, std=1.0):
        return gen.normal_fp32(gen.stream_key(seed, tag, layer, 0), 0, count, std)

    q = _unit_rows(normal(TAG_GDN_Q, T * Hk * dk).reshape(T, Hk, dk))
    k = _unit_rows(normal(TAG_GDN_K, T * Hk * dk).reshape(T, Hk, dk))
    v = normal(TAG_GDN_V, T * Hv * dv).reshape(T, Hv, dv)
    alpha = 0.9 + 0.1 * _uniform01(gen.stream_key(seed, TAG_GDN_GATE, layer, 0), T * Hv)
    g = np.log(alpha).astype(np.float32).reshape(T, Hv)
    z = normal(TAG_GDN_BETA, T * Hv).astype(np.float64)
    beta = (1.0 / (1.0 + np.exp(-z))).astype(np.float32).reshape(T, Hv)
    state0 = None
    if state_std > 0:
        state0 = normal(TAG_GDN_STATE, len(lengths) * Hv * dv * dk, state_std).reshape(
            len(lengths), Hv, dv, dk)
    return GdnInputs(q=gen.round_to_bf16_bits(q), k=gen.round_to_bf16_bits(k),
                     v=gen.round_to_bf16_bits(v), g=g, beta=beta, state0=state0,
                     offsets=offsets)
