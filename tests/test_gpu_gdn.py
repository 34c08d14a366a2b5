"""Parity of the Gated DeltaNet prefill scan (include/gdn.h, gdn_scan.cu)
with the fp64 oracle (oracle/gdn_oracle.py), called through the C ABI.

Tolerances, from the arithmetic: q, k, v enter exactly (bf16 -> fp32); the
state is fp32 and every per-token step is non-expansive for unit keys and
beta in [0, 1], so its rounding stays near fp32 epsilon (an fp32 emulation
of the kernel's operation order on these inputs: rel-L2 1.3e-7, max 2.7e-7
of max|S|); the output is rounded to bf16, a relative error up to 2^-8.
Bars: o within 2^-8 |o_ref| + 2e-3 max|o_ref| per element and rel-L2 3e-3;
final state within 1e-5 of max|S_ref| per element and rel-L2 1e-5.
"""
import numpy as np
import pytest
import torch

import sparse_moe_bit_gb300 as M
from oracle import gdn_oracle as G
from synth import gdn
from tests.moe_cases import bits_to_dev, dev_to_bits

pytestmark = pytest.mark.gpu

QWEN = gdn.GdnShape(Hk=16, Hv=32, dk=128, dv=128)


def _to_dev(inp):
    d = dict(q=bits_to_dev(inp.q), k=bits_to_dev(inp.k), v=bits_to_dev(inp.v),
             g=torch.from_numpy(inp.g).cuda(), beta=torch.from_numpy(inp.beta).cuda(),
             offsets=torch.from_numpy(inp.offsets).cuda())
    d["state"] = None if inp.state0 is None else torch.from_numpy(inp.state0).cuda()
    return d


def _bf16_values(t):
    return G.bf16_values(dev_to_bits(t))


def _check_o(o, o_ref, rows=None):
    o_ref = o_ref if rows is None else o_ref[rows]
    o = o if rows is None else o[rows]
    bar = 2.0 ** -8 * np.abs(o_ref) + 2e-3 * np.abs(o_ref).max()
    worst = np.max(np.abs(o - o_ref) / bar)
    assert worst <= 1.0, f"o off by {worst:.3f} of the bar"
    rel = np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref)
    assert rel <= 3e-3, f"o rel-L2 {rel:.2e}"


def _check_state(S, S_ref):
    m = np.abs(S_ref).max()
    assert np.abs(S - S_ref).max() <= 1e-5 * m
    assert np.linalg.norm(S - S_ref) <= 1e-5 * np.linalg.norm(S_ref)


def _run(inp, shape, **kw):
    d = _to_dev(inp)
    o, S = M.gdn_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], offsets=d["offsets"],
                      state=d["state"], **kw)
    torch.cuda.synchronize()
    return o, S


@pytest.mark.parametrize("lens,shape,state_std", [
    ([100], gdn.GdnShape(2, 4, 128, 64), 0.0),            # several token blocks + a ragged tail
    ([37, 0, 200, 5], gdn.GdnShape(2, 4, 128, 32), 0.05),  # ragged sequences, one empty
    ([1], gdn.GdnShape(1, 1, 128, 32), 0.1),               # one token, one head
    ([64, 31, 33], gdn.GdnShape(4, 4, 128, 96), 0.0),      # block-size edges, Hv == Hk
], ids=["T100", "ragged4", "T1", "edges"])
def test_scan_parity(lens, shape, state_std):
    inp = gdn.make_inputs(3, lens, shape, state_std=state_std)
    o_ref, s_ref = G.gdn_scan(inp.q, inp.k, inp.v, inp.g, inp.beta, state0=inp.state0,
                              offsets=inp.offsets)
    o, S = _run(inp, shape)
    _check_o(_bf16_values(o), o_ref)
    _check_state(S.cpu().numpy().astype(np.float64), s_ref)


def test_scan_parity_qwen_prompt_2k():
    """The bench's workload: one 2K-token prompt through a Qwen-shaped layer
    (16 query/key heads, 32 value heads, 128 x 128 state per head)."""
    inp = gdn.make_inputs(0, [2048], QWEN)
    o_ref, s_ref = G.gdn_scan(inp.q, inp.k, inp.v, inp.g, inp.beta, offsets=inp.offsets)
    o, S = _run(inp, QWEN)
    _check_o(_bf16_values(o), o_ref)
    _check_state(S.cpu().numpy().astype(np.float64), s_ref)


def test_prompt_split_over_two_calls():
    """Scanning a prompt in two calls, the state carried in place between
    them, matches one call within the parity bars (the tensor-core scan
    evaluates chunks of 32 tokens from the start of each call, so the two
    ways round differently; the token-by-token kernel gave the same bits)."""
    shape = gdn.GdnShape(2, 4, 128, 64)
    inp = gdn.make_inputs(5, [300], shape, state_std=0.05)
    d = _to_dev(inp)
    o1, S1 = M.gdn_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], state=d["state"])
    st = d["state"].clone()
    o2 = torch.empty_like(o1)
    for a, b in ((0, 77), (77, 300)):
        M.gdn_scan(d["q"][a:b], d["k"][a:b], d["v"][a:b], d["g"][a:b], d["beta"][a:b],
                   state=st, state_out=st, o=o2[a:b])
    torch.cuda.synchronize()
    o_ref, s_ref = G.gdn_scan(inp.q, inp.k, inp.v, inp.g, inp.beta, state0=inp.state0)
    _check_o(_bf16_values(o2), o_ref)
    _check_state(st.cpu().numpy().astype(np.float64), s_ref)
    _check_o(_bf16_values(o2), _bf16_values(o1))
    _check_state(st.cpu().numpy().astype(np.float64), S1.cpu().numpy().astype(np.float64))


def test_grouped_heads_match_repeated_heads():
    """Hv = 4 over Hk = 2 gives the same bits as Hk = 4 with each q/k head
    repeated for its two value heads."""
    shape = gdn.GdnShape(2, 4, 128, 32)
    inp = gdn.make_inputs(6, [90], shape)
    d = _to_dev(inp)
    o1, S1 = M.gdn_scan(d["q"], d["k"], d["v"], d["g"], d["beta"])
    rep = lambda x: x.repeat_interleave(2, dim=1).contiguous()
    o2, S2 = M.gdn_scan(rep(d["q"]), rep(d["k"]), d["v"], d["g"], d["beta"])
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(S1, S2)


def test_deterministic_and_untouched_outside_sequences():
    shape = gdn.GdnShape(2, 4, 128, 32)
    inp = gdn.make_inputs(7, [60], shape)
    d = _to_dev(inp)
    off = torch.tensor([5, 50], dtype=torch.int32, device="cuda")
    sentinel = torch.full((60, 4, 32), 7.0, dtype=torch.bfloat16, device="cuda")
    oa, Sa = M.gdn_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], offsets=off,
                        o=sentinel.clone())
    ob, Sb = M.gdn_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], offsets=off,
                        o=sentinel.clone())
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16)) and torch.equal(Sa, Sb)
    assert torch.all(oa[:5] == 7.0) and torch.all(oa[50:] == 7.0)
    o_ref, s_ref = G.gdn_scan(inp.q[5:50], inp.k[5:50], inp.v[5:50], inp.g[5:50],
                              inp.beta[5:50])
    _check_o(_bf16_values(oa[5:50]), o_ref)
    _check_state(Sa.cpu().numpy().astype(np.float64), s_ref)


def test_empty_scan_copies_the_state():
    shape = gdn.GdnShape(1, 2, 128, 64)
    inp = gdn.make_inputs(8, [4, 0], shape, state_std=0.3)
    d = _to_dev(inp)
    o, S = M.gdn_scan(d["q"][:0], d["k"][:0], d["v"][:0], d["g"][:0], d["beta"][:0],
                      state=d["state"][:1])
    o2, S2 = M.gdn_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], offsets=d["offsets"],
                        state=d["state"])
    torch.cuda.synchronize()
    assert o.numel() == 0 and torch.equal(S, d["state"][:1])
    assert torch.equal(S2[1], d["state"][1])                  # the empty second sequence
