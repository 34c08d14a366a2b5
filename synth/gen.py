"""Seeded synthetic inputs for the sparse 4-bit MoE block (host side).

This module only makes INPUTS: counter-based random numbers, rounding to the
storage types (bf16, fp16) and the group-affine 4-bit quantiser that turns
fp32 weights into the checkpoint format the block consumes.  It holds none of
the block's own arithmetic (no routing, no matmul, no activation), so both the
CUDA path and the oracle can be fed from it without sharing method code.

Random numbers
--------------
Every value is a pure function of (seed, tag, layer, expert, element index):

* ``mix64`` is the SplitMix64 output function (Steele, Lea & Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014).
* a stream key is ``mix64`` chained over (seed, tag, layer, expert);
* draw ``i`` of a stream is ``mix64(key + (i + 1) * GAMMA)`` mod 2**64;
* a value ``n`` uses draws ``2n`` and ``2n + 1``: their eight 16-bit fields are
  summed as integers (Irwin-Hall with eight uniform terms), centred, and
  multiplied once, in fp32, by ``std / sigma_S``.  This is bell-shaped with the
  requested standard deviation and uses only integer operations plus one IEEE
  fp32 multiply, so the device generator (``synth/csrc/synth_gen.cu``)
  reproduces it bit for bit.

Quantiser (per group of ``group`` consecutive values along K)
-----------------------------------------------------------
``s = r((max - min) / 15)``, ``beta = r(min)`` with r the rounding to the
scale type, fp16 or bf16 (fp32 arithmetic, one rounding per step,
round-to-nearest-even), and
``q = clamp(rint((w - beta) / s), 0, 15)`` computed with the ROUNDED s and beta;
``q = 0`` where ``s == 0``.  Two codes share a byte, the even K index in the
low nibble.  Weights are [out, in] row-major with the groups contiguous along
``in``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX_A = 0xBF58476D1CE4E5B9
MIX_B = 0x94D049BB133111EB

# Tags of the independent streams of one layer.
TAG_ROUTER = 1
TAG_SHARED_GATE = 2
TAG_GATE_UP = 3
TAG_DOWN = 4
TAG_SH_GATE_UP = 5
TAG_SH_DOWN = 6
TAG_X = 7
TAG_RANKING = 8

# standard deviation of the sum of eight uniform 16-bit integers
SIGMA_S = math.sqrt(8.0 * (65536.0 * 65536.0 - 1.0) / 12.0)
CENTRE_S = 8 * 65535 // 2  # 262140, the mean of the sum


def _u64(v) -> np.ndarray:
    return np.asarray(v, dtype=np.uint64)


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on uint64 arrays (wrapping arithmetic)."""
    z = _u64(z)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX_A)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX_B)
        z = z ^ (z >> np.uint64(31))
    return z


def mix64_int(z: int) -> int:
    """Scalar SplitMix64 output function on Python ints."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX_A) & MASK64
    z = ((z ^ (z >> 27)) * MIX_B) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tag: int, layer: int = 0, expert: int = 0) -> int:
    """Key of one random stream: mix64 chained over its identifiers."""
    k = mix64_int((seed + GAMMA) & MASK64)
    for v in (tag, layer, expert):
        k = mix64_int(k ^ ((v + GAMMA) & MASK64))
    return k


def draws(key: int, idx: np.ndarray) -> np.ndarray:
    """Draw number ``idx`` (uint64 array) of the stream with ``key``."""
    idx = _u64(idx)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (idx + np.uint64(1)) * np.uint64(GAMMA)
    return mix64(z)


def fp32_scale(std: float) -> np.float32:
    """The single fp32 multiplier that maps the centred sum to ``std``."""
    return np.float32(std / SIGMA_S)


def normal_fp32(key: int, start: int, count: int, std: float) -> np.ndarray:
    """Values start..start+count-1 of a stream, fp32, mean 0, given std."""
    n = np.arange(start, start + count, dtype=np.uint64)
    a = draws(key, n * np.uint64(2))
    b = draws(key, n * np.uint64(2) + np.uint64(1))
    m16 = np.uint64(0xFFFF)
    s = np.zeros(count, dtype=np.int64)
    for w in (a, b):
        for sh in (0, 16, 32, 48):
            s += ((w >> np.uint64(sh)) & m16).astype(np.int64)
    z = (s - CENTRE_S).astype(np.float32)  # |z| < 2**19: exact
    return z * fp32_scale(std)  # one IEEE fp32 multiply


def round_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (finite)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def bf16_bits_to_fp32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def quantize_rows(w: np.ndarray, group: int = 64, scale_dtype: str = "f16"):
    """Group-affine 4-bit quantiser.  ``w``: fp32 [rows, K].

    Returns (packed uint8 [rows, K/2], scale [rows, K/group],
    bias [rows, K/group]); scale and bias are fp16 (np.float16) or, with
    ``scale_dtype="bf16"``, bf16 bit patterns (np.uint16).
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, K = w.shape
    assert K % group == 0 and K % 2 == 0
    g = w.reshape(rows, K // group, group)
    mn = g.min(axis=2)
    mx = g.max(axis=2)
    if scale_dtype == "bf16":
        s16 = round_to_bf16_bits((mx - mn) / np.float32(15.0))
        b16 = round_to_bf16_bits(mn)
        s = bf16_bits_to_fp32(s16)[:, :, None]
        b = bf16_bits_to_fp32(b16)[:, :, None]
    else:
        assert scale_dtype == "f16"
        s16 = ((mx - mn) / np.float32(15.0)).astype(np.float16)
        b16 = mn.astype(np.float16)
        s = s16.astype(np.float32)[:, :, None]
        b = b16.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (g - b) / s
    q = np.where(s == 0, np.float32(0), np.rint(t))
    q = np.clip(q, 0, 15).astype(np.uint8).reshape(rows, K)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return packed, s16, b16


def quantized_matrix(seed, tag, layer, expert, rows, K, std=0.02, group=64, scale_dtype="f16"):
    """Quantised [rows, K] weight matrix of one stream (fp32 draws -> 4-bit)."""
    key = stream_key(seed, tag, layer, expert)
    w = normal_fp32(key, 0, rows * K, std).reshape(rows, K)
    return quantize_rows(w, group, scale_dtype)


def bf16_matrix(seed, tag, layer, expert, rows, K, std, row0=0):
    """bf16 bit patterns of rows row0..row0+rows-1 of a [*, K] stream."""
    key = stream_key(seed, tag, layer, expert)
    v = normal_fp32(key, row0 * K, rows * K, std)
    return round_to_bf16_bits(v).reshape(rows, K)


@dataclass
class MoEShape:
    d: int
    E: int
    k: int
    I: int
    group: int = 64
    scale_dtype: str = "f16"  # "f16" (np.float16) or "bf16" (bit patterns, np.uint16)


@dataclass
class LayerWeights:
    """One layer in the canonical (caller) layout; bf16 as uint16 bits."""
    shape: MoEShape
    w_router: np.ndarray      # uint16 [E, d]
    w_shared_gate: np.ndarray  # uint16 [d]
    gu_codes: np.ndarray      # uint8 [E, 2I, d/2]  rows 0..I-1 gate, I..2I-1 up
    gu_scale: np.ndarray      # fp16 or bf16 bits [E, 2I, d/g]
    gu_bias: np.ndarray       # fp16 or bf16 bits [E, 2I, d/g]
    dn_codes: np.ndarray      # uint8 [E, d, I/2]
    dn_scale: np.ndarray      # fp16 or bf16 bits [E, d, I/g]
    dn_bias: np.ndarray       # fp16 or bf16 bits [E, d, I/g]
    sh_gu_codes: np.ndarray   # uint8 [2I, d/2]
    sh_gu_scale: np.ndarray
    sh_gu_bias: np.ndarray
    sh_dn_codes: np.ndarray   # uint8 [d, I/2]
    sh_dn_scale: np.ndarray
    sh_dn_bias: np.ndarray


def expert_weights(seed, layer, expert, shape: MoEShape, std=0.02):
    """(gu_codes, gu_scale, gu_bias, dn_codes, dn_scale, dn_bias) of one
    routed expert (``expert`` < E) or of the shared expert (``expert`` == E)."""
    d, I, g, sd = shape.d, shape.I, shape.group, shape.scale_dtype
    if expert == shape.E:
        gu = quantized_matrix(seed, TAG_SH_GATE_UP, layer, 0, 2 * I, d, std, g, sd)
        dn = quantized_matrix(seed, TAG_SH_DOWN, layer, 0, d, I, std, g, sd)
    else:
        gu = quantized_matrix(seed, TAG_GATE_UP, layer, expert, 2 * I, d, std, g, sd)
        dn = quantized_matrix(seed, TAG_DOWN, layer, expert, d, I, std, g, sd)
    return gu + dn


def make_layer(seed: int, layer: int, shape: MoEShape, std=0.02) -> LayerWeights:
    """All weights of one layer on the host (use for small shapes)."""
    E, d, I, g = shape.E, shape.d, shape.I, shape.group
    sdt = np.uint16 if shape.scale_dtype == "bf16" else np.float16
    gu_c = np.empty((E, 2 * I, d // 2), np.uint8)
    gu_s = np.empty((E, 2 * I, d // g), sdt)
    gu_b = np.empty_like(gu_s)
    dn_c = np.empty((E, d, I // 2), np.uint8)
    dn_s = np.empty((E, d, I // g), sdt)
    dn_b = np.empty_like(dn_s)
    for e in range(E):
        gu_c[e], gu_s[e], gu_b[e], dn_c[e], dn_s[e], dn_b[e] = expert_weights(
            seed, layer, e, shape, std)
    sh = expert_weights(seed, layer, E, shape, std)
    return LayerWeights(
        shape=shape,
        w_router=bf16_matrix(seed, TAG_ROUTER, layer, 0, E, d, std),
        w_shared_gate=bf16_matrix(seed, TAG_SHARED_GATE, layer, 0, 1, d, std)[0],
        gu_codes=gu_c, gu_scale=gu_s, gu_bias=gu_b,
        dn_codes=dn_c, dn_scale=dn_s, dn_bias=dn_b,
        sh_gu_codes=sh[0], sh_gu_scale=sh[1], sh_gu_bias=sh[2],
        sh_dn_codes=sh[3], sh_dn_scale=sh[4], sh_dn_bias=sh[5],
    )


def make_x(seed: int, T: int, d: int, row0: int = 0, layer: int = 0) -> np.ndarray:
    """Activations, bf16 bits [T, d], N(0, 1)-shaped; rows row0..row0+T-1."""
    return bf16_matrix(seed, TAG_X, layer, 0, T, d, 1.0, row0=row0)


def expert_ranking(seed: int, E: int) -> np.ndarray:
    """rank_e in 1..E from a seeded random permutation of the experts."""
    key = stream_key(seed, TAG_RANKING, 0, 0)
    r = draws(key, np.arange(E, dtype=np.uint64))
    order = np.argsort(r, kind="stable")
    rank = np.empty(E, dtype=np.int64)
    rank[order] = np.arange(1, E + 1)
    return rank


def zipf_bias(seed: int, E: int, alpha: float = 1.5) -> np.ndarray:
    """Per-expert logit bias b_e = alpha * ln(1 / rank_e), fp32 [E]."""
    rank = expert_ranking(seed, E)
    return (alpha * np.log(1.0 / rank.astype(np.float64))).astype(np.float32)
