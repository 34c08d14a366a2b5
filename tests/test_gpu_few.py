"""The few-token path (2 <= T <= 8 tokens of one layer in one launch on the
DECODE layout: every token routed on the device, the union of the tokens'
experts streamed once).

Per token its arithmetic is the decode kernel's, so the T rows of one call
must equal T single-token calls (the decode kernel, itself checked against the
oracle layer by layer) bit for bit.  The outputs are also checked against the
fp64 oracle routing from its own fp64 logits (independent mode; tokens whose
k-th and (k+1)-th logits are within 1e-4 are excluded and counted)."""
import numpy as np
import pytest
import torch

import sparse_moe_bit_gb300 as M
from oracle import moe_oracle as O
from synth import device as sd
from synth import gen
from tests.moe_cases import (MID, QWEN, TINY, DeviceLayer, HostCase, bits_to_dev,
                             check_output, near_tie_tokens)

pytestmark = pytest.mark.gpu


def _rows_match_single_calls(moe, x):
    y = moe.forward(x)
    rows = torch.stack([moe.forward(x[t:t + 1])[0] for t in range(x.shape[0])])
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), rows.view(torch.int16)), "rows differ from T=1 calls"
    return y


def _independent(case_oracle, bits, y, k, what):
    ref = case_oracle(O.bf16_values(bits))
    ok = ~near_tie_tokens(ref["logits"], k)
    assert ok.any(), f"{what}: every token is a near tie"
    check_output(y.float().cpu().numpy()[ok], ref["out"][ok], what)


@pytest.fixture(scope="module")
def tiny():
    return HostCase(TINY, seed=2, max_tokens=64)


@pytest.fixture(scope="module")
def mid():
    return HostCase(MID, seed=3, max_tokens=64)


@pytest.mark.parametrize("T", [2, 3, 5, 8])
def test_few_tokens_tiny_and_mid(tiny, mid, T):
    for case, name in ((tiny, "tiny"), (mid, "mid")):
        bits = gen.make_x(40 + T, T, case.shape.d)
        y = _rows_match_single_calls(case.moe, bits_to_dev(bits))
        _independent(lambda xv: O.moe_layer(xv, case.vals), bits, y, case.shape.k,
                     f"{name} T={T}")
        assert case.moe.device_error() == 0


def test_few_tokens_sharing_experts(mid):
    # identical tokens pick identical experts: every union entry serves all T
    bits = np.repeat(gen.make_x(7, 1, MID.d), 6, axis=0)
    bits[3] = gen.make_x(8, 1, MID.d)[0]  # one different token among them
    y = _rows_match_single_calls(mid.moe, bits_to_dev(bits))
    yv = y.view(torch.int16)
    assert torch.equal(yv[0], yv[1]) and torch.equal(yv[0], yv[5])
    _independent(lambda xv: O.moe_layer(xv, mid.vals), bits, y, MID.k, "shared experts")


def test_few_tokens_bias_and_no_shared_expert():
    case = HostCase(MID, seed=4, has_shared=False, max_tokens=16)
    bits = gen.make_x(9, 7, MID.d)
    x = bits_to_dev(bits)
    bias = torch.linspace(-0.3, 0.3, MID.E, device="cuda", dtype=torch.float32)
    y = case.moe.forward(x, bias)
    rows = torch.stack([case.moe.forward(x[t:t + 1], bias)[0] for t in range(7)])
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), rows.view(torch.int16))
    _independent(lambda xv: O.moe_layer(xv, case.vals, logit_bias=bias.cpu().numpy()), bits, y,
                 MID.k, "bias, no shared expert")


@pytest.mark.parametrize("E,k", [(64, 16), (512, 8)])
def test_few_tokens_shape_edges(E, k):
    # k = 16 with 8 tokens: 128 chosen experts of 64, a union of every expert;
    # E = 512: 16 logits per lane in the selection
    shape = gen.MoEShape(d=256, E=E, k=k, I=128)
    case = HostCase(shape, seed=5, max_tokens=16)
    bits = gen.make_x(11, 8, shape.d)
    y = _rows_match_single_calls(case.moe, bits_to_dev(bits))
    _independent(lambda xv: O.moe_layer(xv, case.vals), bits, y, k, f"E={E} k={k}")


@pytest.mark.parametrize("T", [2, 4, 8])
def test_few_tokens_qwen_shape(T):
    layer = DeviceLayer(QWEN, seed=0, layer=0, max_tokens=16, layouts=M.MOE_LAYOUT_DECODE)
    x = sd.make_x(3, T, QWEN.d)
    y = _rows_match_single_calls(layer.moe, x)
    bits = gen.make_x(3, T, QWEN.d)
    xv = O.bf16_values(bits)
    lg = O.router_logits(xv, layer.w_router)
    ok = ~near_tie_tokens(lg, QWEN.k)
    ref = layer.oracle(xv, logits=lg)
    check_output(y.float().cpu().numpy()[ok], ref["out"][ok], f"qwen T={T}")
    assert layer.moe.device_error() == 0
