"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

Each test fixes the oracle against something other than itself: a hand-worked
example (tests/golden/), a closed form, an invariant, a brute-force enumeration
on tiny inputs, or a special case that reduces to a textbook routine.  Together
they are chosen so that a dropped term, a wrong sign or index, or a transposed
operand anywhere in oracle/moe_oracle.py fails at least one of them.
"""
import importlib.util
import itertools
import math
import os

import numpy as np
import pytest
from scipy.special import expit, softmax


def _load_oracle():
    """The oracle under test; MOE_ORACLE_FILE points at a planted-mistake copy
    when tests/test_oracle_mutations.py runs these pins against one."""
    path = os.environ.get("MOE_ORACLE_FILE")
    if not path:
        from oracle import moe_oracle
        return moe_oracle
    spec = importlib.util.spec_from_file_location("moe_oracle_under_test", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


O = _load_oracle()

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


# ---------------------------------------------------------------- format ---

def test_dequant_hand_example():
    g = _golden("dequant_hand.txt")
    packed = np.array([[int(b, 16) for b in g["bytes0"]],
                       [int(b, 16) for b in g["bytes1"]]], dtype=np.uint8)
    scale = np.array([[float(v)] for v in g["scale"]], dtype=np.float16)
    bias = np.array([[float(v)] for v in g["bias"]], dtype=np.float16)
    w = O.dequantize(packed, scale, bias, 64)
    assert np.array_equal(w[0], np.array([float(v) for v in g["expect0"]]))
    assert np.array_equal(w[1], np.array([float(v) for v in g["expect1"]]))


def test_dequant_bf16_group128_hand_example():
    # bf16 scale/bias given as bit patterns, one pair per 128 weights
    g = _golden("dequant_bf16_g128.txt")
    packed = np.array([[int(b, 16) for b in g["bytes0"]],
                       [int(b, 16) for b in g["bytes1"]]], dtype=np.uint8)
    scale = np.array([[int(v, 16)] for v in g["scale_bits"]], dtype=np.uint16)
    bias = np.array([[int(v, 16)] for v in g["bias_bits"]], dtype=np.uint16)
    w = O.dequantize(packed, scale, bias, 128)
    assert np.array_equal(w[0], np.array([float(v) for v in g["expect0"]]))
    assert np.array_equal(w[1], np.array([float(v) for v in g["expect1"]]))


def test_bf16_scale_bits_decode_as_bf16():
    # the same 16 bits mean different numbers in bf16 and fp16
    assert O.scale_values(np.array([0x3C00], np.uint16))[0] == 2.0 ** -7
    assert O.scale_values(np.array([0x3C00], np.uint16).view(np.float16))[0] == 1.0
    assert O.scale_values(np.array([0xC0A0], np.uint16))[0] == -5.0


def test_dequant_group128_boundaries():
    # with 128-wide groups, elements 0..127 use pair 0 and 128..255 pair 1
    q = np.zeros((1, 256), np.uint8)
    q[0, 127] = 3
    q[0, 128] = 5
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    s = np.array([[0.5, 2.0]], np.float16)
    b = np.array([[1.0, -4.0]], np.float16)
    w = O.dequantize(packed, s, b, 128)
    assert w[0, 0] == 1.0 and w[0, 64] == 1.0 and w[0, 127] == 1.0 + 0.5 * 3
    assert w[0, 128] == -4.0 + 2.0 * 5 and w[0, 255] == -4.0


def test_nibble_order_low_is_even():
    q = O.unpack_codes(np.array([[0x21, 0xF0]], np.uint8))
    assert q.tolist() == [[1, 2, 0, 15]]


def test_dequant_group_boundaries():
    # two groups in one row with different (s, beta): every element must use
    # the parameters of ITS group (c // 64), not a neighbour's.
    q = np.zeros((1, 128), np.uint8)
    q[0, 63] = 3
    q[0, 64] = 5
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    s = np.array([[0.5, 2.0]], np.float16)
    b = np.array([[1.0, -4.0]], np.float16)
    w = O.dequantize(packed, s, b, 64)
    assert w[0, 0] == 1.0 and w[0, 63] == 1.0 + 0.5 * 3
    assert w[0, 64] == -4.0 + 2.0 * 5 and w[0, 127] == -4.0


# --------------------------------------------------------------- routing ---

def test_page_assignment_count():
    g = _golden("page_figures.txt")
    T, E, k = int(g["tokens"][0]), int(g["experts"][0]), int(g["top_k"][0])
    rng = np.random.default_rng(0)
    idx, w = O.select_top_k(rng.standard_normal((T, E)), k)
    counts, offsets, perm, slot = O.group_by_expert(idx, E)
    assert counts.sum() == int(g["assignments"][0])
    assert counts.sum() / E == int(g["mean_rows_per_expert"][0])
    assert offsets[-1] == int(g["assignments"][0])


def _brute_rank(lg):
    """rank of expert e = number of experts that beat it (higher logit, or the
    same logit and a lower index): O(E^2) enumeration, no sorting."""
    E = lg.shape[0]
    r = np.zeros(E, np.int64)
    for e in range(E):
        for f in range(E):
            if lg[f] > lg[e] or (lg[f] == lg[e] and f < e):
                r[e] += 1
    return r


@pytest.mark.parametrize("k", [1, 2, 5])
def test_topk_matches_bruteforce_rank_with_ties(k):
    rng = np.random.default_rng(1)
    # coarse values: many exact ties between experts
    lg = np.round(rng.standard_normal((64, 16)) * 2) / 2
    idx, w = O.select_top_k(lg, k)
    for t in range(lg.shape[0]):
        r = _brute_rank(lg[t])
        expect = [int(np.nonzero(r == j)[0][0]) for j in range(k)]
        assert idx[t].tolist() == expect


def test_topk_all_pairs_e16_k2():
    # E=16, k=2: among all C(16,2) pairs, the kept pair is the one whose
    # members beat every expert outside it (ties to the lower index).
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((32, 16))
    lg[:, 5] = lg[:, 9]  # a tie in every token
    idx, _ = O.select_top_k(lg, 2)
    beats = lambda f, e, row: row[f] > row[e] or (row[f] == row[e] and f < e)
    for t in range(32):
        row = lg[t]
        winners = [p for p in itertools.combinations(range(16), 2)
                   if all(beats(a, o, row) for a in p for o in range(16) if o not in p)]
        assert len(winners) == 1
        assert sorted(idx[t].tolist()) == list(winners[0])


def test_topk_weights_closed_form_k2():
    lg = np.array([[0.3, 1.7, -0.2, 1.1]])
    idx, w = O.select_top_k(lg, 2)
    assert idx.tolist() == [[1, 3]]
    assert w[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(1.1 - 1.7)), abs=1e-15)
    assert w[0, 1] == pytest.approx(1.0 / (1.0 + math.exp(1.7 - 1.1)), abs=1e-15)


def test_topk_weights_are_renormalised_full_softmax():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((50, 32)) * 3
    idx, w = O.select_top_k(lg, 8)
    p = softmax(lg, axis=1)  # library softmax over ALL experts
    pk = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(w, pk / pk.sum(axis=1, keepdims=True), rtol=0, atol=1e-14)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)  # slots in descending logit order


def test_topk_weights_infinite_logits_are_the_softmax_limit():
    lg = np.array([[1.0, np.inf, 0.0, np.inf, -3.0],
                   [-np.inf] * 5,
                   [np.inf, 2.0, 1.0, 0.0, -1.0]])
    idx, w = O.select_top_k(lg, 3)
    assert idx.tolist() == [[1, 3, 0], [0, 1, 2], [0, 1, 2]]
    assert w.tolist() == [[0.5, 0.5, 0.0], [1 / 3, 1 / 3, 1 / 3], [1.0, 0.0, 0.0]]
    # the finite limit: logits c, c, a with c -> large give the same weights
    idx2, w2 = O.select_top_k(np.array([[1.0, 800.0, 0.0, 800.0, -3.0]]), 3)
    np.testing.assert_allclose(w2[0], [0.5, 0.5, 0.0], atol=1e-300)


def test_router_logits_bias_and_orientation():
    # d != E so a transposed router matrix cannot go unnoticed
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 7))
    W = rng.standard_normal((5, 7))
    b = np.array([0.5, -1.0, 0.0, 2.0, 3.0])
    lg = O.router_logits(x, W, b)
    assert lg.shape == (3, 5)
    # x = 0  ->  logits are exactly the bias
    assert np.array_equal(O.router_logits(np.zeros((1, 7)), W, b)[0], b)
    # unit vector picks one column of W
    e2 = np.zeros((1, 7)); e2[0, 2] = 1.0
    assert np.array_equal(O.router_logits(e2, W)[0], W[:, 2])


# -------------------------------------------------------------- grouping ---

def test_grouping_hand_example():
    g = _golden("grouping_hand.txt")
    idx = np.array([int(v) for v in g["idx"]]).reshape(5, 2)
    counts, offsets, perm, slot = O.group_by_expert(idx, 4)
    assert counts.tolist() == [int(v) for v in g["counts"]]
    assert offsets.tolist() == [int(v) for v in g["offsets"]]
    assert perm.tolist() == [int(v) for v in g["perm"]]
    assert slot.reshape(-1).tolist() == [int(v) for v in g["slot"]]


def test_grouping_invariants():
    rng = np.random.default_rng(5)
    T, E, k = 300, 24, 4
    idx, _ = O.select_top_k(rng.standard_normal((T, E)), k)
    counts, offsets, perm, slot = O.group_by_expert(idx, E)
    assert counts.sum() == T * k
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(np.bincount(perm, minlength=T), np.full(T, k))  # k times each
    for t in range(T):
        assert len(set(idx[t].tolist())) == k  # k distinct experts
        for j in range(k):
            r = slot[t, j]
            assert perm[r] == t
            assert offsets[idx[t, j]] <= r < offsets[idx[t, j] + 1]
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)  # ascending token within an expert


# --------------------------------------------------------------- experts ---

def _const_expert(a, b, c, d, I, dtype=np.float16):
    """Expert whose dequantised gate, up and down matrices are the constants
    a, b, c (all codes 0, scale 0, bias = the constant)."""
    gu_codes = np.zeros((2 * I, d // 2), np.uint8)
    gu_s = np.zeros((2 * I, d // 64), dtype)
    gu_b = np.concatenate([np.full((I, d // 64), a), np.full((I, d // 64), b)]).astype(dtype)
    dn_codes = np.zeros((d, I // 2), np.uint8)
    dn_s = np.zeros((d, I // 64), dtype)
    dn_b = np.full((d, I // 64), c).astype(dtype)
    return gu_codes, gu_s, gu_b, dn_codes, dn_s, dn_b


def _ffn_const(a, b, c, I, S):
    """Closed form of a constant expert on a token with sum(x) = S:
    gate = a*S, up = b*S, h = silu(a*S)*b*S on each of I features,
    y_f = c * I * h (every output feature)."""
    g = a * S
    return c * I * (g / (1.0 + math.exp(-g))) * (b * S)


def _layer(experts, shared, d, k, w_router=None, w_sg=None):
    E = len(experts)
    stack = tuple(np.stack([ex[i] for ex in experts]) for i in range(6))
    return dict(E=E, k=k, group=64, has_shared=shared is not None,
                w_router=w_router if w_router is not None else np.zeros((E, d)),
                w_shared_gate=w_sg if w_sg is not None else np.zeros(d),
                experts=stack, shared=shared)


def test_swiglu_closed_form_and_gate_up_order():
    d, I = 128, 64  # d != I
    x = np.full((1, d), 0.125)  # S = 16
    S = 16.0
    a, b, c = 0.0625, -0.25, 0.5
    lw = _layer([_const_expert(a, b, c, d, I)], None, d, 1)
    out = O.moe_layer(x, lw, logits=np.zeros((1, 1)))["out"]
    assert out.shape == (1, d)
    np.testing.assert_allclose(out[0], _ffn_const(a, b, c, I, S), rtol=1e-13)
    # swapping the roles of gate and up changes the value: the order is pinned
    assert not np.isclose(_ffn_const(b, a, c, I, S), _ffn_const(a, b, c, I, S))


def test_two_experts_weighted_by_routing_closed_form():
    d, I = 128, 64
    x = np.full((1, d), 1.0 / 64)  # S = 2
    S = 2.0
    ex = [_const_expert(0.5, 0.25, 1.0, d, I), _const_expert(-0.125, 2.0, -0.5, d, I)]
    lg = np.array([[0.2, 1.0]])
    lw = _layer(ex, None, d, 2)
    r = O.moe_layer(x, lw, logits=lg)
    w1 = 1.0 / (1.0 + math.exp(0.2 - 1.0))  # expert 1 is slot 0
    y0, y1 = _ffn_const(0.5, 0.25, 1.0, I, S), _ffn_const(-0.125, 2.0, -0.5, I, S)
    assert r["idx"].tolist() == [[1, 0]]
    np.testing.assert_allclose(r["out"][0], w1 * y1 + (1 - w1) * y0, rtol=1e-13)


def test_shared_expert_sigmoid_gate_closed_form():
    d, I = 128, 64
    x = np.full((1, d), 1.0 / 32)  # S = 4
    S = 4.0
    ex = [_const_expert(0.5, 0.25, 1.0, d, I)]
    sh = _const_expert(0.25, -0.5, 0.125, d, I)
    v = 0.1875
    lw = _layer(ex, sh, d, 1, w_sg=np.full(d, v))
    r = O.moe_layer(x, lw, logits=np.zeros((1, 1)))
    sig = 1.0 / (1.0 + math.exp(-v * S))
    assert r["sigma"][0] == pytest.approx(sig, rel=1e-15)
    expect = _ffn_const(0.5, 0.25, 1.0, I, S) + sig * _ffn_const(0.25, -0.5, 0.125, I, S)
    np.testing.assert_allclose(r["out"][0], expect, rtol=1e-13)
    # w_sg = 0  ->  sigma = 1/2 exactly
    lw0 = _layer(ex, sh, d, 1, w_sg=np.zeros(d))
    assert O.moe_layer(x, lw0, logits=np.zeros((1, 1)))["sigma"][0] == 0.5


def _random_layer(rng, E, d, I, k, shared=True):
    def mats():
        gu = rng.integers(0, 256, (2 * I, d // 2), dtype=np.uint8)
        dn = rng.integers(0, 256, (d, I // 2), dtype=np.uint8)
        f = lambda r, c, sc: (rng.standard_normal((r, c)) * sc).astype(np.float16)
        return (gu, f(2 * I, d // 64, 0.01), f(2 * I, d // 64, 0.05),
                dn, f(d, I // 64, 0.01), f(d, I // 64, 0.05))
    experts = [mats() for _ in range(E)]
    return _layer(experts, mats() if shared else None, d, k,
                  w_router=rng.standard_normal((E, d)) * 0.05,
                  w_sg=rng.standard_normal(d) * 0.05)


def test_k_equals_E_is_dense_softmax_mixture():
    rng = np.random.default_rng(6)
    E, d, I = 4, 128, 64
    lw = _random_layer(rng, E, d, I, k=E, shared=False)
    x = rng.standard_normal((5, d))
    r = O.moe_layer(x, lw)
    p = softmax(O.router_logits(x, lw["w_router"]), axis=1)
    dense = np.zeros((5, d))
    for e in range(E):
        wg, wu, wd = O.expert_matrices(*(a[e] for a in lw["experts"]))
        dense += p[:, e:e + 1] * O.swiglu_expert(x, wg, wu, wd)
    np.testing.assert_allclose(r["out"], dense, rtol=1e-12, atol=1e-14)


def test_identical_experts_output_independent_of_routing():
    rng = np.random.default_rng(7)
    E, d, I, k = 6, 128, 64, 3
    base = _random_layer(rng, 1, d, I, 1)
    one = tuple(a[0] for a in base["experts"])
    lw = _layer([one] * E, one, d, k,
                w_router=rng.standard_normal((E, d)), w_sg=rng.standard_normal(d) * 0.1)
    x = rng.standard_normal((4, d))
    o1 = O.moe_layer(x, lw)["out"]
    o2 = O.moe_layer(x, lw, logit_bias=np.arange(E)[::-1] * 10.0)["out"]  # other experts
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)


def test_unselected_experts_never_touched():
    rng = np.random.default_rng(8)
    E, d, I, k = 8, 128, 64, 2
    lw = _random_layer(rng, E, d, I, k)
    x = rng.standard_normal((6, d))
    bias = np.full(E, -1e4); bias[[1, 4, 6]] = 0.0  # only 1, 4, 6 can win
    ref = O.moe_layer(x, lw, logit_bias=bias)
    used = set(np.unique(ref["idx"]).tolist())
    poisoned = dict(lw)
    poisoned["experts"] = tuple(a.copy() for a in lw["experts"])
    for e in range(E):
        if e not in used:
            for a in poisoned["experts"][1:3] + poisoned["experts"][4:6]:
                a[e] = np.nan
    out = O.moe_layer(x, poisoned, logit_bias=bias)["out"]
    assert np.all(np.isfinite(out))
    assert np.array_equal(out, ref["out"])


def test_token_permutation_equivariance():
    rng = np.random.default_rng(9)
    lw = _random_layer(rng, 8, 128, 64, 2)
    x = rng.standard_normal((10, 128))
    p = rng.permutation(10)
    a = O.moe_layer(x, lw)["out"]
    b = O.moe_layer(x[p], lw)["out"]
    np.testing.assert_allclose(b, a[p], rtol=1e-13, atol=1e-15)


def test_doubling_down_projection_doubles_output_exactly():
    rng = np.random.default_rng(10)
    lw = _random_layer(rng, 5, 128, 64, 2)
    x = rng.standard_normal((7, 128))
    a = O.moe_layer(x, lw)["out"]
    dbl = dict(lw)
    ex = list(lw["experts"]); ex[4] = ex[4] * 2; ex[5] = ex[5] * 2
    sh = list(lw["shared"]); sh[4] = sh[4] * 2; sh[5] = sh[5] * 2
    dbl["experts"], dbl["shared"] = tuple(ex), tuple(sh)
    b = O.moe_layer(x, dbl)["out"]
    assert np.array_equal(b, 2 * a)


def test_rms_norm_closed_form():
    v = np.array([[3.0, 4.0, 3.0, 4.0]])
    np.testing.assert_allclose(O.rms_norm(v, 0.0), v / math.sqrt(12.5), rtol=1e-15)
    np.testing.assert_allclose(O.rms_norm(v, 1e-6), v / math.sqrt(12.5 + 1e-6), rtol=1e-15)


def test_silu_textbook():
    z = np.array([-3.0, 0.0, 0.5, 7.0])
    np.testing.assert_allclose(O.silu(z), z / (1 + np.exp(-z)), rtol=1e-15)
    assert O.silu(np.array([0.0]))[0] == 0.0
