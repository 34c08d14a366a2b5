"""Parity of the CUDA path with the fp64 oracle for the other checkpoint
formats: bf16 scale and bias (the format of the pages' checkpoint,
§"Dequantize weights during matrix multiplication") and quantisation groups
of 128.  moe_create converts bf16 scale/bias to fp16 exactly and repeats a
group's pair over its 64-wide K blocks, so these run the same kernels as the
fp16 group-64 cases; the tests check the conversion, the indexing and the
refusal of values fp16 cannot hold exactly."""
import numpy as np
import pytest
import torch

import sparse_moe_bit_gb300 as M
from sparse_moe_bit_gb300 import moe as MM
from synth import device as sd
from synth import gen
from tests.moe_cases import HostCase, bits_to_dev, check_output, near_tie_tokens

pytestmark = pytest.mark.gpu

TINY_BF16 = gen.MoEShape(d=256, E=16, k=2, I=128, scale_dtype="bf16")
MID_BF16_G128 = gen.MoEShape(d=512, E=32, k=4, I=256, group=128, scale_dtype="bf16")
MID_F16_G128 = gen.MoEShape(d=512, E=32, k=4, I=256, group=128)
# the Qwen layer's dimensions with fewer experts (host generation stays fast)
QWENISH_BF16 = gen.MoEShape(d=2048, E=16, k=8, I=512, scale_dtype="bf16")


@pytest.fixture(scope="module", params=["tiny_bf16", "mid_bf16_g128", "mid_f16_g128"])
def case(request):
    shape = {"tiny_bf16": TINY_BF16, "mid_bf16_g128": MID_BF16_G128,
             "mid_f16_g128": MID_F16_G128}[request.param]
    return HostCase(shape, seed=2)


def _x(case, T, seed):
    bits = gen.make_x(seed, T, case.shape.d)
    return bits, bits_to_dev(bits)


@pytest.mark.parametrize("T", [2, 17, 200, 257])
def test_forward_parity_formats(case, T):
    bits, x = _x(case, T, seed=T + 1)
    y = case.moe.forward(x)
    r = case.moe.route(x)
    torch.cuda.synchronize()
    ref = case.oracle(bits, logits=r["logits"].cpu().numpy())
    check_output(y.float().cpu().numpy(), ref["out"], f"{case.shape} T={T}")
    assert case.moe.device_error() == 0


def test_decode_step_parity_formats(case):
    # T = 1 through the decode kernel (the handle has both layouts)
    bits, x = _x(case, 1, seed=9)
    y, t = M.decode([case.moe], x, trace=True)
    torch.cuda.synchronize()
    ref = case.oracle(bits, logits=t["logits"].cpu().numpy())
    check_output(y.float().cpu().numpy()[None], ref["out"], f"{case.shape} decode")


def test_qwen_dims_bf16_parity():
    case = HostCase(QWENISH_BF16, seed=3, max_tokens=1024)
    bits, x = _x(case, 600, seed=4)
    y = case.moe.forward(x).float().cpu().numpy()
    r = case.moe.route(x)
    torch.cuda.synchronize()
    ref = case.oracle(bits, logits=r["logits"].cpu().numpy())
    check_output(y, ref["out"], "qwen dims, bf16 scales")
    # and routed independently by the oracle (near-tie tokens excluded)
    ref2 = case.oracle(bits)
    ok = ~near_tie_tokens(ref2["logits"], QWENISH_BF16.k)
    check_output(y[ok], ref2["out"][ok], "qwen dims, bf16 scales, independent routing")


@pytest.mark.parametrize("bad_bits", [0x0001, 0x4880])  # 9.2e-41 (fp16 rounds it to 0); 2^18
def test_bf16_scale_without_exact_fp16_is_refused(bad_bits):
    lw = gen.make_layer(5, 0, TINY_BF16)
    lw.dn_scale[3, 7, 1] = bad_bits
    w = sd.host_layer_to_device(lw)
    cfg = M.MoEConfig(d=256, E=16, k=2, I=128, scale_dtype=MM.MOE_SCALE_BF16, max_tokens=64)
    with pytest.raises(M.MoEError) as ei:
        M.MoE(cfg, w)
    assert ei.value.status == 2  # MOE_ERR_UNSUPPORTED
    # the boundary values themselves are accepted: 2^-17 and 65280 (bf16 0x7F7F is larger)
    lw.dn_scale[3, 7, 1] = 0x3700  # 2^-17
    lw.dn_bias[3, 7, 1] = 0x477F   # 65280
    M.MoE(cfg, sd.host_layer_to_device(lw)).close()
