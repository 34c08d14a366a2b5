"""Property-based checks of both oracles on many small random cases
(hypothesis): the grouping invariants of the block's routing, the top-k
order, and the scan's chunked evaluation against its token loop, over random
shapes, lengths and chunk sizes.  CPU only."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import gdn_oracle as G  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402
from tests.test_gdn_oracle_pins import _chunked_scan, _wy_scan  # noqa: E402


@settings(max_examples=60, deadline=None)
@given(T=st.integers(1, 40), E=st.integers(2, 24), data=st.data())
def test_grouping_invariants(T, E, data):
    k = data.draw(st.integers(1, min(E, 6)))
    seed = data.draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    # logits with many exact ties (small integers) to exercise the tie-break
    logits = rng.integers(-3, 4, size=(T, E)).astype(np.float64)
    idx, w = O.select_top_k(logits, k)
    counts, offsets, perm, slot = O.group_by_expert(idx, E)
    for t in range(T):
        row = idx[t]
        assert len(set(row.tolist())) == k                       # k distinct experts
        key = [(-logits[t, e], e) for e in row]
        assert key == sorted(key)                                # (logit desc, index asc)
        worst = key[-1]
        others = [(-logits[t, e], e) for e in range(E) if e not in row]
        assert all(o > worst for o in others)                    # nothing better left out
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert counts.sum() == T * k and offsets[0] == 0 and offsets[-1] == T * k
    assert np.array_equal(np.diff(offsets), counts)
    for e in range(E):
        rows = perm[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(rows) > 0)                         # ascending tokens
        assert all(e in idx[t] for t in rows)
    for t in range(T):
        for j in range(k):
            r = slot[t, j]
            assert perm[r] == t and offsets[idx[t, j]] <= r < offsets[idx[t, j] + 1]


@settings(max_examples=40, deadline=None)
@given(T=st.integers(1, 50), dk=st.integers(1, 9), dv=st.integers(1, 7),
       C=st.integers(1, 20), seed=st.integers(0, 2**31 - 1))
def test_scan_chunked_forms_match_the_token_loop(T, dk, dv, C, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, 1, dk))
    k = rng.standard_normal((T, 1, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, 1, dv))
    g = np.log(rng.uniform(0.7, 1.0, (T, 1)))
    beta = rng.uniform(0.0, 1.0, (T, 1))
    S0 = rng.standard_normal((1, 1, dv, dk))
    o, S = G.gdn_scan(q, k, v, g, beta, scale=0.5, state0=S0)
    for form in (_chunked_scan, _wy_scan):
        oc, Sc = form(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], 0.5, S0[0, 0], C)
        np.testing.assert_allclose(oc, o[:, 0], rtol=1e-9, atol=1e-10)
        np.testing.assert_allclose(Sc, S[0, 0], rtol=1e-9, atol=1e-10)
