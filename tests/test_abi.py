"""The C-ABI library loads, exports every function include/moe.h and
include/gdn.h declare,
and rejects bad arguments before touching the GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401  (makes the CUDA runtime the library links against resolvable)
    from sparse_moe_bit_gb300 import build, moe
    if not os.path.exists(moe.LIB_PATH):
        build.build()
    return moe.load_library()


def _declared():
    names = set()
    for header in ("moe.h", "gdn.h"):
        src = open(os.path.join(ROOT, "include", header)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b((?:moe|gdn)_[a-z_]+)\s*\(", src))
    return sorted(names)


def test_header_and_binding_agree():
    from sparse_moe_bit_gb300 import moe
    assert _declared() == sorted(moe.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert lib.moe_version() == 1
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(1) == b"invalid argument"
    assert lib.moe_status_string(5) == b"device error"


def _cfg(**kw):
    from sparse_moe_bit_gb300 import moe
    base = dict(d=256, E=16, k=2, I=128, group=64, scale_dtype=1, max_tokens=16,
                has_shared=1, layouts=0)
    base.update(kw)
    return moe.MoEConfig(**base)._c()


@pytest.mark.parametrize("kw,status", [
    (dict(d=100), 1), (dict(d=0), 1), (dict(E=0), 1), (dict(E=513), 1), (dict(k=0), 1),
    (dict(k=17, E=32), 1), (dict(k=3, E=2), 1), (dict(I=100), 1), (dict(group=32), 2),
    (dict(group=96), 2), (dict(group=256), 2), (dict(scale_dtype=7), 1), (dict(max_tokens=0), 1),
    (dict(has_shared=2), 1), (dict(layouts=9), 1)])
def test_create_rejects_bad_config(lib, kw, status):
    from sparse_moe_bit_gb300 import moe
    w = moe._Weights()
    h = ctypes.c_void_p()
    assert lib.moe_create(ctypes.byref(_cfg(**kw)), ctypes.byref(w), None, ctypes.byref(h)) == status
    assert h.value is None
    assert len(lib.moe_last_error()) > 0


@pytest.mark.parametrize("kw", [dict(scale_dtype=2), dict(group=128), dict(group=128, scale_dtype=2)])
def test_bf16_scales_and_group128_pass_validation(lib, kw):
    # valid configurations: moe_create gets as far as the weight pointers
    from sparse_moe_bit_gb300 import moe
    w = moe._Weights()  # all NULL
    h = ctypes.c_void_p()
    assert lib.moe_create(ctypes.byref(_cfg(**kw)), ctypes.byref(w), None, ctypes.byref(h)) == 1
    assert b"weight" in lib.moe_last_error()


def test_create_rejects_null_or_misaligned_weights(lib):
    from sparse_moe_bit_gb300 import moe
    h = ctypes.c_void_p()
    w = moe._Weights()  # all NULL
    assert lib.moe_create(ctypes.byref(_cfg()), ctypes.byref(w), None, ctypes.byref(h)) == 1
    w = moe._Weights(*([0x1008] * 14))  # 8-byte aligned only
    assert lib.moe_create(ctypes.byref(_cfg()), ctypes.byref(w), None, ctypes.byref(h)) == 1
    assert lib.moe_create(None, ctypes.byref(w), None, ctypes.byref(h)) == 1
    assert lib.moe_create(ctypes.byref(_cfg()), ctypes.byref(w), None, None) == 1


def test_calls_on_null_handle_are_rejected(lib):
    assert lib.moe_forward(None, None, 4, None, None, None) == 1
    assert lib.moe_route(None, None, 4, None, None, None, None, None, None, None, None, None) == 1
    assert lib.moe_route_from_logits(None, None, 4, None, None, None, None, None, None, None,
                                     None) == 1
    assert lib.moe_forward_host(None, None, 4, None, None, None) == 1
    assert lib.moe_decode(None, 0, None, None, 1e-6, None, None, None) == 1
    code = ctypes.c_int()
    assert lib.moe_get_device_error(None, ctypes.byref(code)) == 1
    assert lib.moe_destroy(None) == 0


# Fake, suitably aligned device addresses: every case below is refused during
# argument checking, before anything could be enqueued.
_A = 0x10000


def _gdn_args(**kw):
    a = dict(q=_A, k=_A, v=_A, g=_A, beta=_A, scale=0.088, offsets=None, N=1, T=64, Hk=2, Hv=4,
             dk=128, dv=64, state_in=None, state_out=None, o=_A, stream=None)
    a.update(kw)
    return a


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(beta=None), 1), (dict(T=-1), 1), (dict(N=0), 1),
    (dict(Hk=0), 1), (dict(Hv=6, Hk=4), 1), (dict(N=2), 1), (dict(scale=float("nan")), 1),
    (dict(scale=float("inf")), 1), (dict(q=_A + 8), 1), (dict(state_out=_A + 4), 1),
    (dict(g=_A + 2), 1), (dict(Hv=70000, Hk=1), 1), (dict(dk=64), 2), (dict(dk=256), 2),
    (dict(dv=48), 2), (dict(dv=0), 1)])
def test_gdn_scan_rejects_bad_arguments(lib, kw, status):
    a = _gdn_args(**kw)
    r = lib.gdn_scan(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["offsets"], a["N"],
                     a["T"], a["Hk"], a["Hv"], a["dk"], a["dv"], a["state_in"], a["state_out"],
                     a["o"], a["stream"])
    assert r == status, lib.moe_last_error()
    assert lib.moe_last_error()


def test_gdn_scan_empty_without_state_is_a_no_op(lib):
    a = _gdn_args(T=0)
    assert lib.gdn_scan(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], None, 1, 0, 2, 4,
                        128, 64, None, None, a["o"], None) == 0
    assert lib.gdn_scan(None, None, None, None, None, 1.0, None, 1, 0, 2, 4, 128, 64, None, None,
                        None, None) == 0


def test_create_without_a_device_fails_cleanly(lib):
    """On a machine with no usable CUDA device moe_create returns
    MOE_ERR_CUDA with a message and no handle (it must not crash).  Skipped
    where a device exists: there the fake weight addresses would be read."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    from sparse_moe_bit_gb300 import moe
    h = ctypes.c_void_p(0x1234)
    w = moe._Weights(*([0x10000] * 14))
    r = lib.moe_create(ctypes.byref(_cfg()), ctypes.byref(w), None, ctypes.byref(h))
    assert r == 3, lib.moe_last_error()
    assert h.value is None
    assert lib.moe_last_error()


def test_gdn_binding_fails_loudly_without_a_device(lib):
    """The binding marshals the scan's arguments (N from the offsets, the
    default scale) and surfaces the library's status: with no device the call
    passes argument checking and then fails with MOE_ERR_CUDA; there is no
    CPU fallback.  Skipped where a device exists (the tensors here live on
    the host)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    import types
    import sparse_moe_bit_gb300 as M
    legacy = types.SimpleNamespace(cuda_stream=0)          # torch cannot make a stream here
    T, Hk, Hv = 8, 1, 2
    q = torch.zeros(T, Hk, 128, dtype=torch.bfloat16)
    v = torch.zeros(T, Hv, 32, dtype=torch.bfloat16)
    g = torch.zeros(T, Hv)
    off = torch.tensor([0, 3, 8], dtype=torch.int32)
    with pytest.raises(M.MoEError) as ex:
        M.gdn_scan(q, q, v, g, g, offsets=off, stream=legacy)
    assert ex.value.status == 3
    bad = torch.zeros(T, Hk, 64, dtype=torch.bfloat16)     # dk = 64: refused before any launch
    with pytest.raises(M.MoEError) as ex:
        M.gdn_scan(bad, bad, v, g, g, stream=legacy)
    assert ex.value.status == 2
