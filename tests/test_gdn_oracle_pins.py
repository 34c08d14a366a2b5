"""Pins of the Gated DeltaNet scan oracle to facts fixed by the pages and by
mathematics: a hand-worked example (tests/golden/gdn_hand.txt), closed forms
of special cases (no write, pure overwrite, no decay), the delta rule as one
gradient step of an online regression loss (checked with autograd), an
independent chunked evaluation (a triangular solve per chunk of tokens), and
the structure of the scan (state carried across chunks, sequences
independent, grouped heads, readout scale).  A dropped term, a wrong sign, a swapped
operand or a wrong head index in oracle/gdn_oracle.py fails at least one.
"""
import importlib.util
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_oracle():
    """The oracle under test; GDN_ORACLE_FILE points at a planted-mistake copy
    when tests/test_oracle_mutations.py runs these pins against one."""
    path = os.environ.get("GDN_ORACLE_FILE")
    if not path:
        from oracle import gdn_oracle
        return gdn_oracle
    spec = importlib.util.spec_from_file_location("gdn_oracle_under_test", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


G = _load_oracle()


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *vals = line.split()
                out[key] = np.array([float(v) for v in vals])
    return out


def _random(rng, T, Hk, Hv, dk, dv, unit=True):
    q = rng.standard_normal((T, Hk, dk))
    k = rng.standard_normal((T, Hk, dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, Hv, dv))
    g = np.log(rng.uniform(0.8, 1.0, (T, Hv)))
    beta = rng.uniform(0.0, 1.0, (T, Hv))
    return q, k, v, g, beta


# ------------------------------------------------------------ worked example

def _hand():
    h = _golden("gdn_hand.txt")
    T = 3
    q = h["q"].reshape(T, 1, 2)
    k = h["k"].reshape(T, 1, 2)
    v = h["v"].reshape(T, 1, 3)
    g = np.log(h["alpha"]).reshape(T, 1)
    beta = h["beta"].reshape(T, 1)
    return q, k, v, g, beta, float(h["scale"][0]), h["o"].reshape(T, 3), h["state"].reshape(3, 2)


def test_hand_example_scan():
    q, k, v, g, beta, scale, o_ref, s_ref = _hand()
    o, S = G.gdn_scan(q, k, v, g, beta, scale=scale)
    np.testing.assert_allclose(o[:, 0], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S[0, 0], s_ref, rtol=0, atol=1e-12)


def test_hand_example_dense_rule():
    q, k, v, g, beta, scale, o_ref, s_ref = _hand()
    S = np.zeros((3, 2))
    for t in range(3):
        S, o = G.gated_delta_step_dense(S, q[t, 0], k[t, 0], v[t, 0], g[t, 0], beta[t, 0], scale)
        np.testing.assert_allclose(o, o_ref[t], rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, s_ref, rtol=0, atol=1e-12)


def test_rank_one_form_matches_dense_rule():
    rng = np.random.default_rng(1)
    q, k, v, g, beta = _random(rng, 6, 1, 1, 5, 3, unit=False)
    S = rng.standard_normal((3, 5))
    Sb = S[None].copy()
    for t in range(6):
        S, o = G.gated_delta_step_dense(S, q[t, 0], k[t, 0], v[t, 0], g[t, 0], beta[t, 0], 0.7)
        Sb, ob = G.gated_delta_step(Sb, q[t, :1], k[t, :1], v[t, :1], g[t, :1], beta[t, :1], 0.7)
        np.testing.assert_allclose(ob[0], o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Sb[0], S, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ closed forms

def test_no_write_is_pure_decay():
    """beta = 0: nothing is written, S_t = (prod alpha) S_0 and
    o_t = scale (prod_{s<=t} alpha_s) S_0 q_t."""
    rng = np.random.default_rng(2)
    T, dk, dv = 9, 4, 3
    q, k, v, g, _ = _random(rng, T, 1, 2, dk, dv)
    S0 = rng.standard_normal((1, 2, dv, dk))
    o, S = G.gdn_scan(q, k, v, g, np.zeros((T, 2)), scale=0.5, state0=S0)
    decay = np.exp(np.cumsum(g, axis=0))                        # [T, Hv]
    for h in range(2):
        expect = 0.5 * decay[:, h, None] * np.einsum("ij,tj->ti", S0[0, h], q[:, 0])
        np.testing.assert_allclose(o[:, h], expect, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(S[0, h], decay[-1, h] * S0[0, h], rtol=1e-12, atol=1e-14)


def test_full_write_overwrites_the_key():
    """alpha = 1, beta = 1, keys from an orthonormal basis: writing (k, v)
    replaces the value stored under k and leaves the other keys alone, so a
    query equal to a written key reads back the last value written there."""
    rng = np.random.default_rng(3)
    dk, dv = 6, 4
    basis = np.linalg.qr(rng.standard_normal((dk, dk)))[0]    # orthonormal columns
    order = [0, 3, 1, 3, 5, 0, 3]
    T = len(order)
    k = basis[:, order].T.reshape(T, 1, dk)
    q = k.copy()
    v = rng.standard_normal((T, 1, dv))
    S0 = rng.standard_normal((1, 1, dv, dk))
    o, S = G.gdn_scan(q, k, v, np.zeros((T, 1)), np.ones((T, 1)), scale=1.0, state0=S0)
    np.testing.assert_allclose(o[:, 0], v[:, 0], rtol=0, atol=1e-12)
    stored = {j: S0[0, 0] @ basis[:, j] for j in range(dk)}
    for t, j in enumerate(order):
        stored[j] = v[t, 0]
    for j in range(dk):
        np.testing.assert_allclose(S[0, 0] @ basis[:, j], stored[j], rtol=0, atol=1e-12)


def test_write_shrinks_the_residual_by_one_minus_beta():
    """No decay, unit key: S_t k - v = (1 - beta)(S_{t-1} k - v)."""
    rng = np.random.default_rng(4)
    dk, dv = 5, 7
    S = rng.standard_normal((1, dv, dk))
    k = rng.standard_normal((1, dk))
    k /= np.linalg.norm(k)
    v = rng.standard_normal((1, dv))
    for beta in (0.0, 0.25, 0.9, 1.0):
        S_new, _ = G.gated_delta_step(S, k, k, v, np.zeros(1), np.array([beta]), 1.0)
        before = S[0] @ k[0] - v[0]
        after = S_new[0] @ k[0] - v[0]
        np.testing.assert_allclose(after, (1.0 - beta) * before, rtol=1e-12, atol=1e-12)


def test_update_is_one_gradient_step_after_the_decay():
    """The gated delta rule decays the state by alpha and then takes one step
    of size beta down the gradient of 1/2 ||S k - v||^2 (Gated DeltaNet
    paper, the online-regression view); the gradient is taken by autograd."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    dk, dv = 4, 6
    S = rng.standard_normal((1, dv, dk))
    q = rng.standard_normal((1, dk))
    k = rng.standard_normal((1, dk))
    v = rng.standard_normal((1, dv))
    g, beta = np.array([math.log(0.7)]), np.array([0.35])
    Sd = torch.tensor(0.7 * S[0], dtype=torch.float64, requires_grad=True)
    loss = 0.5 * torch.sum((Sd @ torch.tensor(k[0]) - torch.tensor(v[0])) ** 2)
    loss.backward()
    expect = (Sd - 0.35 * Sd.grad).detach().numpy()
    S_new, o = G.gated_delta_step(S, q, k, v, g, beta, 1.0)
    np.testing.assert_allclose(S_new[0], expect, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o[0], expect @ q[0], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ structure

def test_default_scale_is_inverse_sqrt_dk():
    rng = np.random.default_rng(6)
    q, k, v, g, beta = _random(rng, 5, 1, 1, 16, 4)
    o1, S1 = G.gdn_scan(q, k, v, g, beta)
    o2, S2 = G.gdn_scan(q, k, v, g, beta, scale=0.25)
    np.testing.assert_allclose(o1, o2, rtol=1e-14, atol=0)
    np.testing.assert_array_equal(S1, S2)


def test_scale_touches_only_the_readout():
    rng = np.random.default_rng(7)
    q, k, v, g, beta = _random(rng, 7, 1, 1, 4, 4)
    o1, S1 = G.gdn_scan(q, k, v, g, beta, scale=1.0)
    o3, S3 = G.gdn_scan(q, k, v, g, beta, scale=3.0)
    np.testing.assert_allclose(o3, 3.0 * o1, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(S1, S3)


def test_linear_in_values_and_initial_state():
    rng = np.random.default_rng(8)
    q, k, v1, g, beta = _random(rng, 8, 1, 2, 4, 3)
    v2 = rng.standard_normal(v1.shape)
    A, B = rng.standard_normal((2, 1, 2, 3, 4))
    oa, Sa = G.gdn_scan(q, k, v1, g, beta, state0=A[None])
    ob, Sb = G.gdn_scan(q, k, v2, g, beta, state0=B[None])
    oc, Sc = G.gdn_scan(q, k, 2 * v1 - v2, g, beta, state0=(2 * A - B)[None])
    np.testing.assert_allclose(oc, 2 * oa - ob, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(Sc, 2 * Sa - Sb, rtol=1e-11, atol=1e-12)


def test_state_carries_across_chunks():
    """Scanning [0, T1) and then [T1, T) from the carried state equals one
    scan of [0, T): the prompt may be cut into chunks."""
    rng = np.random.default_rng(9)
    q, k, v, g, beta = _random(rng, 13, 2, 4, 4, 3)
    S0 = rng.standard_normal((1, 4, 3, 4))
    o, S = G.gdn_scan(q, k, v, g, beta, state0=S0)
    oa, Sa = G.gdn_scan(q[:5], k[:5], v[:5], g[:5], beta[:5], state0=S0)
    ob, Sb = G.gdn_scan(q[5:], k[5:], v[5:], g[5:], beta[5:], state0=Sa)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Sb, S, rtol=1e-12, atol=1e-12)


def test_sequences_are_independent():
    rng = np.random.default_rng(10)
    lens = [4, 0, 7, 1]
    T = sum(lens)
    q, k, v, g, beta = _random(rng, T, 1, 2, 4, 3)
    S0 = rng.standard_normal((4, 2, 3, 4))
    off = np.concatenate([[0], np.cumsum(lens)])
    o, S = G.gdn_scan(q, k, v, g, beta, state0=S0, offsets=off)
    for n in range(4):
        a, b = off[n], off[n + 1]
        on, Sn = G.gdn_scan(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], state0=S0[n:n + 1])
        np.testing.assert_allclose(o[a:b], on, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(S[n], Sn[0], rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(S[1], S0[1])                 # empty sequence


@pytest.mark.parametrize("Hk,Hv", [(2, 4), (4, 8), (2, 6)])
def test_value_heads_share_their_query_key_head(Hk, Hv):
    """Hv value heads over Hk query/key heads: value head h reads q/k head
    h // (Hv / Hk) (e.g. Hv = 4 over Hk = 2: heads 0, 1 read 0 and 2, 3 read 1)."""
    rng = np.random.default_rng(11)
    q, k, v, g, beta = _random(rng, 6, Hk, Hv, 4, 3)
    o, S = G.gdn_scan(q, k, v, g, beta)
    for h in range(Hv):
        hk = h // (Hv // Hk)
        oh, Sh = G.gdn_scan(q[:, hk:hk + 1], k[:, hk:hk + 1], v[:, h:h + 1], g[:, h:h + 1],
                            beta[:, h:h + 1])
        np.testing.assert_allclose(o[:, h], oh[:, 0], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(S[0, h], Sh[0, 0], rtol=1e-13, atol=1e-14)


def test_bf16_bit_inputs_read_exactly():
    bits = np.array([[[0x3F80, 0xC000, 0x3E80, 0x0000]]], dtype=np.uint16)   # 1, -2, 0.25, 0
    np.testing.assert_array_equal(G.as_values(bits), [[[1.0, -2.0, 0.25, 0.0]]])


def _chunked_scan(q, k, v, g, beta, scale, S0, C):
    """The same rule evaluated a chunk of C tokens at a time, derived
    independently of the oracle's token loop.  Unrolling the rule inside a
    chunk that starts from state S_0, with gamma_i the product of the gates up
    to token i and c_i = beta_i (v_i - alpha_i S_{i-1} k_i):
        S_i = gamma_i S_0 + sum_{j<=i} (gamma_i / gamma_j) c_j k_j^T,
    so the c_i solve the unit lower-triangular system
        c_i + beta_i sum_{j<i} (gamma_i/gamma_j)(k_i.k_j) c_j
            = beta_i (v_i - gamma_i S_0 k_i),
    and o_i = scale (gamma_i S_0 q_i + sum_{j<=i} (gamma_i/gamma_j)(q_i.k_j) c_j).
    One head: q, k [T, dk], v [T, dv], g, beta [T], S0 [dv, dk]."""
    from scipy.linalg import solve_triangular
    T = q.shape[0]
    S = S0.copy()
    o = np.zeros((T, v.shape[1]))
    for a in range(0, T, C):
        b = min(T, a + C)
        Q, K, V = q[a:b], k[a:b], v[a:b]
        gam = np.exp(np.cumsum(g[a:b]))
        ratio = gam[:, None] / gam[None, :]
        L = np.tril(beta[a:b, None] * ratio * (K @ K.T), -1)
        rhs = beta[a:b, None] * (V - gam[:, None] * (K @ S.T))
        Cm = solve_triangular(np.eye(b - a) + L, rhs, lower=True, unit_diagonal=True)
        M = np.tril(ratio * (Q @ K.T))
        o[a:b] = scale * (gam[:, None] * (Q @ S.T) + M @ Cm)
        S = gam[-1] * S + Cm.T @ ((gam[-1] / gam)[:, None] * K)
    return o, S


@pytest.mark.parametrize("C", [1, 4, 16])
def test_chunked_form_matches_the_token_loop(C):
    """An independent evaluation (chunks, a triangular solve, matrix
    products: the blockwise way the pages mention) gives the same outputs and
    state as the oracle's token-by-token scan."""
    rng = np.random.default_rng(12)
    T, dk, dv = 37, 8, 5
    q, k, v, g, beta = _random(rng, T, 1, 1, dk, dv)
    S0 = rng.standard_normal((1, 1, dv, dk))
    o, S = G.gdn_scan(q, k, v, g, beta, scale=0.6, state0=S0)
    oc, Sc = _chunked_scan(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], 0.6, S0[0, 0], C)
    np.testing.assert_allclose(o[:, 0], oc, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(S[0, 0], Sc, rtol=1e-10, atol=1e-11)


def _wy_scan(q, k, v, g, beta, scale, S0, C):
    """The chunked form with everything that depends on the inputs alone
    folded into four per-chunk matrices, so that the sequential pass over the
    chunks touches the state only through products with them:
        A = (I + L)^{-1} diag(beta)          (L as in _chunked_scan)
        U = A V,   W = A diag(gamma) K,   P = diag(gamma) Q~ - M W,   R = M U
        c-vectors  C = U - W S_0^T
        outputs    O = P S_0^T + R
        end state  S = gamma_C S_0 + C^T diag(gamma_C / gamma) K."""
    from scipy.linalg import solve_triangular
    T = q.shape[0]
    S = S0.copy()
    o = np.zeros((T, v.shape[1]))
    for a in range(0, T, C):
        b = min(T, a + C)
        Q, K, V = scale * q[a:b], k[a:b], v[a:b]
        gam = np.exp(np.cumsum(g[a:b]))
        ratio = gam[:, None] / gam[None, :]
        L = np.tril(beta[a:b, None] * ratio * (K @ K.T), -1)
        A = solve_triangular(np.eye(b - a) + L, np.diag(beta[a:b]), lower=True,
                             unit_diagonal=True)
        M = np.tril(ratio * (Q @ K.T))
        U, W = A @ V, A @ (gam[:, None] * K)
        P, R = gam[:, None] * Q - M @ W, M @ U
        Cm = U - W @ S.T
        o[a:b] = P @ S.T + R
        S = gam[-1] * S + Cm.T @ ((gam[-1] / gam)[:, None] * K)
    return o, S


@pytest.mark.parametrize("C", [3, 16, 64])
def test_input_only_chunk_matrices_reproduce_the_scan(C):
    rng = np.random.default_rng(13)
    T, dk, dv = 70, 8, 6
    q, k, v, g, beta = _random(rng, T, 1, 1, dk, dv)
    S0 = rng.standard_normal((1, 1, dv, dk))
    o, S = G.gdn_scan(q, k, v, g, beta, scale=0.4, state0=S0)
    ow, Sw = _wy_scan(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], 0.4, S0[0, 0], C)
    np.testing.assert_allclose(o[:, 0], ow, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(S[0, 0], Sw, rtol=1e-10, atol=1e-11)
