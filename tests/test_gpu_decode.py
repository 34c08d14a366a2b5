"""Batch-1 decode chain through the C ABI (moe_decode), teacher-forced per
layer against the fp64 oracle: layer l of the oracle takes the GPU's own
input to layer l, x_l = out_{l-1} / sqrt(mean(out_{l-1}^2) + eps), so errors
do not compound; routing is compared given the GPU's fp32 logits."""
import numpy as np
import pytest
import torch

import sparse_moe_bit_gb300 as M
from oracle import moe_oracle as O
from synth import device as sd
from synth import gen
from tests.moe_cases import (QWEN, TINY, DeviceLayer, HostCase, bits_to_dev, check_output,
                             dev_to_bits)

pytestmark = pytest.mark.gpu
EPS = 1e-6


def _check_layer(l, x_l, tr, oracle, k, w_router, bias=None):
    lg = tr["logits"][l]
    # logits vs fp64 from the same input (fp32 accumulation tolerance)
    ref_lg = O.router_logits(x_l[None], w_router, bias)[0]
    absdot = np.abs(x_l) @ np.abs(w_router).T
    assert np.all(np.abs(lg - ref_lg) <= x_l.shape[0] * 2.0 ** -24 * absdot + 1e-6), l
    idx, w = O.select_top_k(lg[None].astype(np.float64), k)
    assert np.array_equal(tr["idx"][l], idx[0]), l
    w32 = w[0].astype(np.float32)
    assert np.all(np.abs(tr["w"][l] - w32) <= np.spacing(np.abs(w32))), l
    ref = oracle(x_l[None], lg[None])
    check_output(O.bf16_values(tr["out_bits"][l])[None], ref["out"], f"layer {l}")
    assert abs(tr["sigma"][l] - ref["sigma"][0]) <= 1e-5


def _trace_np(t):
    return dict(logits=t["logits"].cpu().numpy(), idx=t["idx"].cpu().numpy(),
                w=t["w"].cpu().numpy(), sigma=t["sigma"].cpu().numpy(),
                out_bits=dev_to_bits(t["out"]))


def _inputs(x0_bits, out_bits, L):
    xs = [O.bf16_values(x0_bits)]
    for l in range(1, L):
        xs.append(O.rms_norm(O.bf16_values(out_bits[l - 1]), EPS))
    return xs


def test_decode_chain_tiny_teacher_forced():
    L = 6
    cases = [HostCase(TINY, seed=0, layer=l, max_tokens=4) for l in range(L)]
    x0 = gen.make_x(0, 1, TINY.d)[0]
    y, t = M.decode([c.moe for c in cases], bits_to_dev(x0), eps=EPS, trace=True)
    torch.cuda.synchronize()
    assert cases[0].moe.device_error() == 0
    tr = _trace_np(t)
    assert np.array_equal(dev_to_bits(y), tr["out_bits"][L - 1])
    xs = _inputs(x0, tr["out_bits"], L)
    for l in range(L):
        c = cases[l]
        _check_layer(l, xs[l], tr, lambda xv, lg: O.moe_layer(xv, c.vals, logits=lg),
                     TINY.k, c.vals["w_router"])


def test_decode_single_step_matches_prefill_path():
    case = HostCase(TINY, seed=3, max_tokens=4)
    pre = HostCase(TINY, seed=3, max_tokens=4, layouts=M.MOE_LAYOUT_PREFILL)
    x0 = gen.make_x(5, 1, TINY.d)
    x = bits_to_dev(x0)
    y_dec = case.moe.forward(x)  # T == 1 takes the decode kernel
    y_pre = pre.moe.forward(x)
    r = pre.moe.route(x)
    torch.cuda.synchronize()
    ref = pre.oracle(x0, logits=r["logits"].cpu().numpy())
    check_output(y_dec.float().cpu().numpy(), ref["out"], "decode T=1")
    check_output(y_pre.float().cpu().numpy(), ref["out"], "prefill T=1")


def test_decode_with_bias_and_chained_launch():
    # 70 layers exceed one launch (64): the second launch continues the chain
    L = 70
    cases = [HostCase(TINY, seed=1, layer=l % 3, max_tokens=2) for l in range(3)]
    layers = [cases[l % 3].moe for l in range(L)]
    bias = torch.zeros(L, TINY.E, device="cuda")
    bias[:, 2] = 0.5
    x0 = gen.make_x(2, 1, TINY.d)[0]
    y, t = M.decode(layers, bits_to_dev(x0), bias=bias, eps=EPS, trace=True)
    torch.cuda.synchronize()
    tr = _trace_np(t)
    xs = _inputs(x0, tr["out_bits"], L)
    b = bias.cpu().numpy()
    for l in (0, 1, 63, 64, 69):
        c = cases[l % 3]
        _check_layer(l, xs[l], tr,
                     lambda xv, lg, c=c: O.moe_layer(xv, c.vals, logits=lg),
                     TINY.k, c.vals["w_router"], bias=b[l])


def test_decode_qwen_40_layers():
    L = 40
    layers = [DeviceLayer(QWEN, seed=0, layer=l, max_tokens=1, layouts=M.MOE_LAYOUT_DECODE)
              for l in range(L)]
    x0 = gen.make_x(0, 1, QWEN.d)[0]
    y, t = M.decode([dl.moe for dl in layers], bits_to_dev(x0), eps=EPS, trace=True)
    torch.cuda.synchronize()
    assert layers[0].moe.device_error() == 0
    tr = _trace_np(t)
    xs = _inputs(x0, tr["out_bits"], L)
    for l in range(L):  # routing of every layer, given its logits
        idx, _ = O.select_top_k(tr["logits"][l][None].astype(np.float64), QWEN.k)
        assert np.array_equal(tr["idx"][l], idx[0]), l
    for l in range(L):  # outputs of every layer, teacher-forced
        dl = layers[l]
        _check_layer(l, xs[l], tr, lambda xv, lg, dl=dl: dl.oracle(xv, logits=lg), QWEN.k,
                     dl.w_router)
