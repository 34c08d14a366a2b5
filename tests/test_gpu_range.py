"""Activations over bf16's range, through the prefill path (fp16 tensor-core
operands: each token's row is divided by a power of two that the epilogues
undo) and through the decode path (16-bit integers with a power-of-two scale
per group of 64), against the fp64 oracle given the GPU's own logits.

Token classes (one seeded N(0,1) row each, times a class factor):
  large   2^16 (magnitudes up to ~3e5, above fp16's 65504),
  small   2^-60 (about 1e-18),
  mixed   half of the features times 2^16, the other half times 2^-20,
  tiny    2^-133 (bf16 subnormals only; the output underflows to zero),
  plain   1.
Each class is checked on its own with the usual bars (rel-L2 <= 5e-3,
max-abs <= 3e-2 max|oracle|): a mix of magnitudes in one check would hide
the small classes behind the large one."""
import numpy as np
import pytest
import torch

import sparse_moe_bit_gb300 as M
from oracle import moe_oracle as O
from synth import device as sd
from synth import gen
from tests.moe_cases import MID, HostCase, bits_to_dev, check_output, dev_to_bits

pytestmark = pytest.mark.gpu

CLASSES = {"large": (0, 12), "small": (12, 24), "mixed": (24, 32), "tiny": (32, 40),
           "plain": (40, 48)}


def _range_tokens(d, seed=21):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((48, d))
    v[0:12] *= 2.0 ** 16
    v[12:24] *= 2.0 ** -60
    v[24:32, : d // 2] *= 2.0 ** 16
    v[24:32, d // 2:] *= 2.0 ** -20
    v[32:40] *= 2.0 ** -133
    bits = gen.round_to_bf16_bits(v.astype(np.float32))
    xv = O.bf16_values(bits)
    assert np.abs(xv[0:12]).max() > 65504.0  # beyond fp16
    assert np.abs(xv[32:40]).max() < 2.0 ** -126 and np.abs(xv[32:40]).max() > 0  # subnormal
    return bits, xv


def _check_classes(out, ref, what):
    for name, (a, b) in CLASSES.items():
        if name == "tiny":
            # the exact outputs are below bf16's smallest subnormal (2^-133)
            assert np.all(np.isfinite(out[a:b])), what
            assert np.abs(ref[a:b]).max() < 2.0 ** -134
            assert np.abs(out[a:b]).max() <= 2.0 ** -133, f"{what} {name}"
        else:
            check_output(out[a:b], ref[a:b], f"{what} {name}")


def test_prefill_path_over_bf16_range():
    case = HostCase(MID, seed=4, layouts=M.MOE_LAYOUT_PREFILL)
    bits, xv = _range_tokens(MID.d)
    x = bits_to_dev(bits)
    y = case.moe.forward(x)
    r = case.moe.route(x)
    torch.cuda.synchronize()
    assert case.moe.device_error() == 0
    ref = O.moe_layer(xv, case.vals, logits=r["logits"].cpu().numpy())["out"]
    _check_classes(y.float().cpu().numpy(), ref, "prefill")


def test_decode_path_over_bf16_range():
    case = HostCase(MID, seed=4, layouts=M.MOE_LAYOUT_DECODE)
    bits, xv = _range_tokens(MID.d)
    out = np.zeros_like(xv)
    lgs = np.zeros((xv.shape[0], MID.E))
    for t in range(xv.shape[0]):
        y, tr = M.decode([case.moe], bits_to_dev(bits[t]), trace=True)
        torch.cuda.synchronize()
        out[t] = O.bf16_values(dev_to_bits(y))
        lgs[t] = tr["logits"][0].cpu().numpy()
    assert case.moe.device_error() == 0
    ref = O.moe_layer(xv, case.vals, logits=lgs)["out"]
    _check_classes(out, ref, "decode")


def test_prefill_flags_activations_beyond_its_scaling():
    """A token above 2^61 times fp16's range is reported, not silently wrong."""
    case = HostCase(MID, seed=4, layouts=M.MOE_LAYOUT_PREFILL)
    bits, _ = _range_tokens(MID.d)
    big = gen.round_to_bf16_bits((np.random.default_rng(3).standard_normal((1, MID.d)) *
                                  2.0 ** 90).astype(np.float32))
    x = bits_to_dev(np.concatenate([bits, big]))
    case.moe.forward(x)
    torch.cuda.synchronize()
    assert case.moe.device_error() & M.MOE_DEVERR_FP16_RANGE


def test_large_intermediates_flagged_on_prefill_exact_on_decode():
    """Gate/up weights 1000 times N(0, 0.02)-scale make silu(gate)*up reach
    ~1e5 and more: beyond fp16, which holds the prefill path's H, so the
    prefill path reports MOE_DEVERR_FP16_RANGE (a non-finite output); the
    decode path, which keeps H in fp32 and 16-bit integers with a
    power-of-two scale per block, matches the oracle."""
    from dataclasses import replace
    lw = gen.make_layer(4, 0, MID)
    big = dict(gu_scale=(lw.gu_scale.astype(np.float32) * 1000).astype(np.float16),
               gu_bias=(lw.gu_bias.astype(np.float32) * 1000).astype(np.float16),
               sh_gu_scale=(lw.sh_gu_scale.astype(np.float32) * 1000).astype(np.float16),
               sh_gu_bias=(lw.sh_gu_bias.astype(np.float32) * 1000).astype(np.float16))
    lw = replace(lw, **big)
    vals = O.layer_values(lw)
    w = sd.host_layer_to_device(lw)
    bits = gen.make_x(12, 8, MID.d)
    x = bits_to_dev(bits)
    pf = M.MoE(M.MoEConfig(d=MID.d, E=MID.E, k=MID.k, I=MID.I, max_tokens=16,
                           layouts=M.MOE_LAYOUT_PREFILL), w)
    pf.forward(x)
    torch.cuda.synchronize()
    assert pf.device_error() & M.MOE_DEVERR_FP16_RANGE
    dec = M.MoE(M.MoEConfig(d=MID.d, E=MID.E, k=MID.k, I=MID.I, max_tokens=16,
                            layouts=M.MOE_LAYOUT_DECODE), w)
    outs, lgs = [], []
    for t in range(8):
        y, tr = M.decode([dec], x[t], trace=True)
        torch.cuda.synchronize()
        outs.append(O.bf16_values(dev_to_bits(y)))
        lgs.append(tr["logits"][0].cpu().numpy())
    assert dec.device_error() == 0
    ref = O.moe_layer(O.bf16_values(bits), vals, logits=np.stack(lgs))["out"]
    check_output(np.stack(outs), ref, "decode, large intermediates")
