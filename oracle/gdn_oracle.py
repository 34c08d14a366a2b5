"""Plain fp64 CPU oracle of the Gated DeltaNet prefill scan.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` call it.  It shares no code with the CUDA path.

Source: Perplexity, "Optimizing on-device inference for Apple Silicon"
(2026-09-01), cited below by section:

* §"Qwen creates three different workload shapes": a Gated DeltaNet layer
  folds everything before the current token into a recurrent state of fixed
  size; a learned gate decides how much of that state is kept and a delta
  update writes the current token into it; every token depends on the state
  left by the token before it.
* §"Keep recurrent state on chip": the state is a matrix; the prefill scan
  carries it through the whole prompt in order and writes it back once at
  the end; the state and its gate are fp32, queries and keys bf16.

The pages do not print the update itself.  The plain reading taken here is
the gated delta rule of the Gated DeltaNet paper (Yang, Kautz & Hatamizadeh,
"Gated Delta Networks: Improving Mamba2 with Delta Rule", ICLR 2025), for
each value head and each token t in order:

    S_t = S_{t-1} (alpha_t (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T
    o_t = scale * S_t q_t

with S in R^{dv x dk} (it maps keys to values), alpha_t = exp(g_t) in (0, 1]
the gate, beta_t in [0, 1] the write strength.  Grouped heads: value head h
reads query/key head h // (Hv / Hk).  Several sequences are scanned
independently, each from its own initial state.

Everything is fp64 with no intermediate rounding: the inputs are taken at
their exact values (bf16 q, k, v; fp32 g, beta, initial state).
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def bf16_values(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> their exact fp64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(F64)


def as_values(a) -> np.ndarray:
    """uint16 arrays are bf16 bit patterns; anything else holds values."""
    a = np.asarray(a)
    return bf16_values(a) if a.dtype == np.uint16 else a.astype(F64)


def gated_delta_step_dense(S, q, k, v, g, beta, scale):
    """One token of one head, written exactly as the gated delta rule:
    the transition matrix alpha (I - beta k k^T) is formed explicitly
    (dk x dk).  Slow; used on small heads to check ``gated_delta_step``."""
    S, q, k, v = (np.asarray(a, F64) for a in (S, q, k, v))
    dk = k.shape[0]
    alpha = np.exp(F64(g))
    transition = alpha * (np.eye(dk) - F64(beta) * np.outer(k, k))
    S_new = S @ transition + F64(beta) * np.outer(v, k)
    return S_new, F64(scale) * (S_new @ q)


def gated_delta_step(S, q, k, v, g, beta, scale):
    """The same token, batched over heads, with the transition applied as a
    rank-one correction: S (I - beta k k^T) = S - beta (S k) k^T.

    S [H, dv, dk]; q, k [H, dk]; v [H, dv]; g, beta [H]."""
    alpha = np.exp(g)[:, None, None]
    Sk = np.einsum("hij,hj->hi", S, k)                      # S_{t-1} k_t
    S_new = alpha * (S - beta[:, None, None] * Sk[:, :, None] * k[:, None, :]) \
        + beta[:, None, None] * v[:, :, None] * k[:, None, :]
    o = scale * np.einsum("hij,hj->hi", S_new, q)           # readout after the write
    return S_new, o


def gdn_scan(q, k, v, g, beta, scale=None, state0=None, offsets=None):
    """The prefill scan over one or more sequences.

    q, k  [T, Hk, dk]  (bf16 bit patterns as uint16, or values)
    v     [T, Hv, dv]  (same)
    g     [T, Hv]      log of the gate alpha (fp32 values)
    beta  [T, Hv]      write strength (fp32 values)
    scale              readout scale; default 1/sqrt(dk)
    state0 [N, Hv, dv, dk] or None (zero state)
    offsets [N+1]      token boundaries of the N sequences; None = one sequence

    Returns (o [T, Hv, dv], state [N, Hv, dv, dk]), fp64."""
    q, k, v = as_values(q), as_values(k), as_values(v)
    g, beta = np.asarray(g, F64), np.asarray(beta, F64)
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    assert k.shape == q.shape and v.shape[0] == T and Hv % Hk == 0
    assert g.shape == (T, Hv) and beta.shape == (T, Hv)
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    if offsets is None:
        offsets = [0, T]
    offsets = [int(x) for x in offsets]
    N = len(offsets) - 1
    head_of = np.arange(Hv) // (Hv // Hk)                    # value head -> q/k head
    states = np.zeros((N, Hv, dv, dk), F64)
    if state0 is not None:
        states[:] = np.asarray(state0, F64)
    o = np.zeros((T, Hv, dv), F64)
    for n in range(N):
        S = states[n].copy()
        for t in range(offsets[n], offsets[n + 1]):
            S, o[t] = gated_delta_step(S, q[t, head_of], k[t, head_of], v[t], g[t], beta[t],
                                       F64(scale))
        states[n] = S
    return o, states
