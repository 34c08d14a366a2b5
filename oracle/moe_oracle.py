"""Plain fp64 CPU oracle of the sparse 4-bit Mixture-of-Experts block.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` call it.  It shares no code with the CUDA path.

Source: Perplexity, "Optimizing on-device inference for Apple Silicon"
(2026-09-01), cited below by section:

* §"Qwen creates three different workload shapes": a router scores 256
  experts per token and selects eight; one shared expert processes every token.
* §"Dequantize weights during matrix multiplication": every weight is a 4-bit
  integer code; each group of 64 weights shares a scale and a bias that
  reconstruct its values; accumulation is fp32, the result bf16.
* §"Keep expert routing on the GPU": a histogram counts the assignments per
  expert, a prefix scan turns the counts into start offsets, a scatter places
  the rows into their expert groups, a block map lists the blocks to process.
* §"Reduce intermediate and state traffic": the expert output projection is
  combined with its routing score and with the shared expert's result.

Where the pages leave a step open this module takes the plain reading:
softmax over the router logits, keep the top k
ordered by (logit descending, expert index ascending) and renormalise over
those k; SwiGLU experts ``down(silu(gate x) * (up x))``; the shared expert
weighted by ``sigmoid(w_sg . x)``; dequantised value ``s * q + beta``.

Everything is fp64 with no intermediate rounding.  The method skips the
unselected experts, which is exact (their weight is zero), so the plain dense
definition written out here is what the fast path must reproduce.
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit

F64 = np.float64


# --------------------------------------------------------------------------
# Weight format (§"Dequantize weights during matrix multiplication")
# --------------------------------------------------------------------------

def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] -> integer codes uint8 [..., K].

    Two codes per byte; the even K index is in the low nibble."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = packed & 0x0F
    out[..., 1::2] = packed >> 4
    return out


def scale_values(a) -> np.ndarray:
    """Exact fp64 values of a scale or bias array: np.uint16 arrays are bf16
    bit patterns (the checkpoint format on the pages, §"Dequantize weights
    during matrix multiplication"), anything else holds values (fp16)."""
    a = np.asarray(a)
    return bf16_values(a) if a.dtype == np.uint16 else a.astype(F64)


def dequantize(packed, scale, bias, group: int = 64) -> np.ndarray:
    """Reconstruct a [rows, K] matrix: w[n, c] = s[n, c // g] * q[n, c] + beta[n, c // g].

    ``scale`` and ``bias`` are [rows, K/g]: fp16 values, or bf16 bit patterns
    (np.uint16); ``g`` is the quantisation group along K."""
    q = unpack_codes(packed).astype(F64)
    s = np.repeat(scale_values(scale), group, axis=-1)
    b = np.repeat(scale_values(bias), group, axis=-1)
    assert s.shape == q.shape, (s.shape, q.shape)
    return s * q + b


# --------------------------------------------------------------------------
# Router (§"Qwen creates three different workload shapes")
# --------------------------------------------------------------------------

def router_logits(x, w_router, logit_bias=None) -> np.ndarray:
    """l[t, e] = sum_c x[t, c] * W_r[e, c] (+ b_e), fp64.  x, W_r given as the
    exact values of their bf16 storage."""
    lg = np.asarray(x, F64) @ np.asarray(w_router, F64).T
    if logit_bias is not None:
        lg = lg + np.asarray(logit_bias, F64)[None, :]
    return lg


def select_top_k(logits, k: int):
    """Top-k experts per token, ordered by (logit descending, index ascending),
    and their softmax weights renormalised over the k kept experts:
    w_j = exp(l_j - l_max) / sum_{i in top-k} exp(l_i - l_max).

    Returns (idx int32 [T, k], w fp64 [T, k])."""
    lg = np.asarray(logits, F64)
    T, E = lg.shape
    ids = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((ids, -lg), axis=-1)  # primary: -logit, then index
    idx = order[:, :k].astype(np.int32)
    top = np.take_along_axis(lg, idx.astype(np.int64), axis=1)
    m = top[:, :1]
    with np.errstate(invalid="ignore"):
        ex = np.exp(top - m)
    w = ex / ex.sum(axis=1, keepdims=True)
    # Infinite logits (the pages are silent; the limit of the softmax): if the
    # largest kept logit is +inf, the +inf experts share the weight equally;
    # if every kept logit is -inf, the k experts share it equally.
    pos = m[:, 0] == np.inf
    if pos.any():
        hit = (top[pos] == np.inf).astype(F64)
        w[pos] = hit / hit.sum(axis=1, keepdims=True)
    neg = m[:, 0] == -np.inf
    if neg.any():
        w[neg] = 1.0 / k
    return idx, w


# --------------------------------------------------------------------------
# Grouping (§"Keep expert routing on the GPU")
# --------------------------------------------------------------------------

def group_by_expert(idx, E: int):
    """Histogram, prefix scan and scatter of the T*k assignments.

    counts[e]  = number of (t, j) with idx[t, j] == e
    offsets[e] = sum of counts of experts below e; offsets[E] = T*k
    perm[r]    = token of row r, rows grouped by expert, ascending token
                 within an expert (a stable counting sort by (expert, token))
    slot[t, j] = row that holds assignment (t, j)."""
    idx = np.asarray(idx)
    T, k = idx.shape
    flat = idx.reshape(-1).astype(np.int64)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(flat, kind="stable")  # flat index = t*k + j
    perm = (order // k).astype(np.int32)
    slot = np.empty(T * k, dtype=np.int32)
    slot[order] = np.arange(T * k, dtype=np.int32)
    return counts, offsets, perm, slot.reshape(T, k)


# --------------------------------------------------------------------------
# Experts (SwiGLU FFN with dequantised weights)
# --------------------------------------------------------------------------

def silu(z):
    z = np.asarray(z, F64)
    return z * expit(z)


def swiglu_expert(xrows, w_gate, w_up, w_down) -> np.ndarray:
    """y = W_down (silu(W_gate x) * (W_up x)) for each row x, fp64."""
    xr = np.asarray(xrows, F64)
    g = xr @ w_gate.T
    u = xr @ w_up.T
    return (silu(g) * u) @ w_down.T


def expert_matrices(gu_codes, gu_scale, gu_bias, dn_codes, dn_scale, dn_bias, group=64):
    """Dequantised (W_gate, W_up, W_down) of one expert; gate/up rows stacked
    as rows 0..I-1 gate and I..2I-1 up."""
    wgu = dequantize(gu_codes, gu_scale, gu_bias, group)
    I = wgu.shape[0] // 2
    return wgu[:I], wgu[I:], dequantize(dn_codes, dn_scale, dn_bias, group)


def shared_gate(x, w_shared_gate) -> np.ndarray:
    """sigma_t = sigmoid(sum_c w_sg[c] * x[t, c])."""
    return expit(np.asarray(x, F64) @ np.asarray(w_shared_gate, F64))


# --------------------------------------------------------------------------
# The whole block
# --------------------------------------------------------------------------

def moe_layer(x, lw, logit_bias=None, logits=None, expert_source=None):
    """Output of one MoE block for the token rows ``x`` (values of bf16 [T, d]).

    ``lw``: synth.gen.LayerWeights-like object (bf16 fields as uint16 bits are
    NOT accepted: pass values; see ``layer_values``).
    ``logits``: optional fp32 router logits to route from (parity mode: the
    fast path's own logits, so that both sides take the same decision).
    ``expert_source(e)``: optional callable returning the six quantised arrays
    of expert e (e == E is the shared expert); default reads them from ``lw``.

    out[t] = sum_j w[t, j] * FFN_{idx[t, j]}(x_t) + sigma_t * FFN_shared(x_t),
    summed in slot order j = 0..k-1, then the shared term."""
    x = np.asarray(x, F64)
    T = x.shape[0]
    E, k, group = lw["E"], lw["k"], lw["group"]
    if logits is None:
        logits = router_logits(x, lw["w_router"], logit_bias)
    else:
        logits = np.asarray(logits, F64)
    idx, w = select_top_k(logits, k)
    counts, offsets, perm, slot = group_by_expert(idx, E)

    if expert_source is None:
        def expert_source(e):
            if e == E:
                return lw["shared"]
            return tuple(a[e] for a in lw["experts"])

    y = np.zeros((T, k, x.shape[1]), F64)
    for e in np.unique(idx):
        rows = np.nonzero(idx == e)  # (token indices, slot indices)
        wg, wu, wd = expert_matrices(*expert_source(int(e)), group=group)
        y[rows[0], rows[1]] = swiglu_expert(x[rows[0]], wg, wu, wd)
    out = np.zeros((T, x.shape[1]), F64)
    for j in range(k):
        out += w[:, j:j + 1] * y[:, j]
    sigma = None
    if lw.get("has_shared", True):
        sigma = shared_gate(x, lw["w_shared_gate"])
        wg, wu, wd = expert_matrices(*expert_source(E), group=group)
        out += sigma[:, None] * swiglu_expert(x, wg, wu, wd)
    return dict(out=out, logits=logits, idx=idx, w=w, counts=counts,
                offsets=offsets, perm=perm, slot=slot, sigma=sigma)


def rms_norm(v, eps: float = 1e-6) -> np.ndarray:
    """v / sqrt(mean(v^2) + eps) along the last axis (no learned weight)."""
    v = np.asarray(v, F64)
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps)


def bf16_values(bits) -> np.ndarray:
    """Exact fp64 values of bf16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(F64)


def layer_values(lw_bits, has_shared=True) -> dict:
    """Adapt a synth.gen.LayerWeights (bf16 as bits) into the dict moe_layer takes."""
    s = lw_bits.shape
    return dict(
        E=s.E, k=s.k, group=s.group, has_shared=has_shared,
        w_router=bf16_values(lw_bits.w_router),
        w_shared_gate=bf16_values(lw_bits.w_shared_gate),
        experts=(lw_bits.gu_codes, lw_bits.gu_scale, lw_bits.gu_bias,
                 lw_bits.dn_codes, lw_bits.dn_scale, lw_bits.dn_bias),
        shared=(lw_bits.sh_gu_codes, lw_bits.sh_gu_scale, lw_bits.sh_gu_bias,
                lw_bits.sh_dn_codes, lw_bits.sh_dn_scale, lw_bits.sh_dn_bias),
    )
