"""Seeded synthetic inputs generated directly in GPU memory.

Same definition as synth/gen.py, evaluated by synth/libsynth.so (large
layers: 16 G weights for a 40-layer stack are impractical on the host).
``tests/test_gpu_synth.py`` checks host and device agree bit for bit.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import gen

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None


def _load():
    global _lib
    if _lib is None:
        path = os.path.join(_HERE, "libsynth.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built: call synth.build.build()")
        lib = ctypes.CDLL(path)
        lib.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_quantized.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p]
        _lib = lib
    return _lib


def _stream():
    return torch.cuda.current_stream().cuda_stream


def bf16_tensor(seed, tag, layer, expert, count, std, start=0, device="cuda") -> torch.Tensor:
    """bf16 values start..start+count-1 of a stream, as a torch.bfloat16 tensor."""
    out = torch.empty(count, dtype=torch.bfloat16, device=device)
    key = gen.stream_key(seed, tag, layer, expert)
    rc = _load().synth_normal_bf16(key, start, count, float(gen.fp32_scale(std)),
                                   out.data_ptr(), _stream())
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16 failed: {rc}")
    return out


def quantized_into(seed, tag, layer, expert, rows, K, codes, scale, bias, std=0.02):
    key = gen.stream_key(seed, tag, layer, expert)
    rc = _load().synth_quantized(key, rows, K, float(gen.fp32_scale(std)), codes.data_ptr(),
                                 scale.data_ptr(), bias.data_ptr(), _stream())
    if rc != 0:
        raise RuntimeError(f"synth_quantized failed: {rc}")


def make_layer(seed: int, layer: int, shape: gen.MoEShape, has_shared=True, std=0.02,
               device="cuda") -> dict:
    """All weights of one layer, canonical layout, on the GPU."""
    E, d, I, g = shape.E, shape.d, shape.I, shape.group
    u8 = dict(dtype=torch.uint8, device=device)
    f16 = dict(dtype=torch.float16, device=device)
    w = dict(
        gu_codes=torch.empty(E, 2 * I, d // 2, **u8), gu_scale=torch.empty(E, 2 * I, d // g, **f16),
        gu_bias=torch.empty(E, 2 * I, d // g, **f16),
        dn_codes=torch.empty(E, d, I // 2, **u8), dn_scale=torch.empty(E, d, I // g, **f16),
        dn_bias=torch.empty(E, d, I // g, **f16))
    for e in range(E):
        quantized_into(seed, gen.TAG_GATE_UP, layer, e, 2 * I, d, w["gu_codes"][e],
                       w["gu_scale"][e], w["gu_bias"][e], std)
        quantized_into(seed, gen.TAG_DOWN, layer, e, d, I, w["dn_codes"][e], w["dn_scale"][e],
                       w["dn_bias"][e], std)
    if has_shared:
        w.update(sh_gu_codes=torch.empty(2 * I, d // 2, **u8),
                 sh_gu_scale=torch.empty(2 * I, d // g, **f16),
                 sh_gu_bias=torch.empty(2 * I, d // g, **f16),
                 sh_dn_codes=torch.empty(d, I // 2, **u8), sh_dn_scale=torch.empty(d, I // g, **f16),
                 sh_dn_bias=torch.empty(d, I // g, **f16))
        quantized_into(seed, gen.TAG_SH_GATE_UP, layer, 0, 2 * I, d, w["sh_gu_codes"],
                       w["sh_gu_scale"], w["sh_gu_bias"], std)
        quantized_into(seed, gen.TAG_SH_DOWN, layer, 0, d, I, w["sh_dn_codes"], w["sh_dn_scale"],
                       w["sh_dn_bias"], std)
        w["w_shared_gate"] = bf16_tensor(seed, gen.TAG_SHARED_GATE, layer, 0, d, std, device=device)
    w["w_router"] = bf16_tensor(seed, gen.TAG_ROUTER, layer, 0, E * d, std,
                                device=device).view(E, d)
    return w


def make_x(seed: int, T: int, d: int, row0: int = 0, layer: int = 0, device="cuda") -> torch.Tensor:
    """Activations bf16 [T, d], rows row0..row0+T-1 of the x stream."""
    return bf16_tensor(seed, gen.TAG_X, layer, 0, T * d, 1.0, start=row0 * d,
                       device=device).view(T, d)


def host_layer_to_device(lw: gen.LayerWeights, has_shared=True, device="cuda") -> dict:
    """Upload a host-generated synth.gen.LayerWeights in the canonical layout."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    bf = lambda bits: t(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    sc = lambda a: bf(a) if a.dtype == np.uint16 else t(a)  # bf16 bits or fp16 scales
    w = dict(gu_codes=t(lw.gu_codes), gu_scale=sc(lw.gu_scale), gu_bias=sc(lw.gu_bias),
             dn_codes=t(lw.dn_codes), dn_scale=sc(lw.dn_scale), dn_bias=sc(lw.dn_bias),
             w_router=bf(lw.w_router))
    if has_shared:
        w.update(sh_gu_codes=t(lw.sh_gu_codes), sh_gu_scale=sc(lw.sh_gu_scale),
                 sh_gu_bias=sc(lw.sh_gu_bias), sh_dn_codes=t(lw.sh_dn_codes),
                 sh_dn_scale=sc(lw.sh_dn_scale), sh_dn_bias=sc(lw.sh_dn_bias),
                 w_shared_gate=bf(lw.w_shared_gate))
    return w
