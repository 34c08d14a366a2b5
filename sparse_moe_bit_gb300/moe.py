"""Thin Python binding of libmoe.so (ctypes): argument marshalling only.

Every step of the block runs in the library's CUDA kernels; torch is used for
device memory and streams.  If libmoe.so is missing the import of this module
still works, but any use raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, fields

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_SCALE_F16 = 1
MOE_SCALE_BF16 = 2
MOE_LAYOUT_PREFILL = 1
MOE_LAYOUT_DECODE = 2
# device error word bits (include/moe.h)
MOE_DEVERR_WAIT_TIMEOUT = 1
MOE_DEVERR_NAN_LOGIT = 2
MOE_DEVERR_GRID_TIMEOUT = 4
MOE_DEVERR_RANGE = 8
MOE_DEVERR_FP16_RANGE = 16

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error",
          4: "out of device memory", 5: "device error"}

# names of the functions include/moe.h declares (checked by the ABI test)
EXPORTS = ["moe_create", "moe_destroy", "moe_route", "moe_route_from_logits", "moe_forward",
           "moe_forward_host", "moe_decode", "moe_decode_host", "moe_profile_enable",
           "moe_profile_read", "moe_route_from_logits_noalloc", "moe_get_device_error",
           "moe_status_string", "moe_last_error", "moe_version", "gdn_scan"]

STAGES = ["router", "routing", "gate_up", "down", "combine"]


class MoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class _Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("d", "E", "k", "I", "group", "scale_dtype", "max_tokens", "has_shared", "layouts")]


WEIGHT_FIELDS = ["gu_codes", "gu_scale", "gu_bias", "dn_codes", "dn_scale", "dn_bias",
                 "sh_gu_codes", "sh_gu_scale", "sh_gu_bias", "sh_dn_codes", "sh_dn_scale",
                 "sh_dn_bias", "w_router", "w_shared_gate"]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


class _Trace(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("logits", "idx", "w", "sigma", "out", "timestamps")]


_lib = None


def load_library() -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built: call sparse_moe_bit_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sig = {
        "moe_create": [ctypes.POINTER(_Config), ctypes.POINTER(_Weights), P, ctypes.POINTER(P)],
        "moe_destroy": [P],
        "moe_route": [P, P, I, P, P, P, P, P, P, P, P, P],
        "moe_route_from_logits": [P, P, I, P, P, P, P, P, P, P, P],
        "moe_forward": [P, P, I, P, P, P],
        "moe_forward_host": [P, P, I, P, P, P],
        "moe_decode": [ctypes.POINTER(P), I, P, P, F, P, ctypes.POINTER(_Trace), P],
        "moe_decode_host": [ctypes.POINTER(P), I, P, P, F, P, P],
        "moe_profile_enable": [P, I],
        "moe_profile_read": [P, ctypes.POINTER(F), I, ctypes.POINTER(I)],
        "moe_route_from_logits_noalloc": [P, I, I, I, P, P, P, P, P, P, P, P],
        "moe_get_device_error": [P, ctypes.POINTER(I)],
        "gdn_scan": [P, P, P, P, P, F, P, I, I, I, I, I, I, P, P, P, P],
        "moe_status_string": [I],
        "moe_last_error": [],
        "moe_version": [],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        msg = load_library().moe_last_error().decode(errors="replace")
        raise MoEError(status, msg)


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


@dataclass
class MoEConfig:
    d: int
    E: int
    k: int
    I: int
    group: int = 64
    scale_dtype: int = MOE_SCALE_F16
    max_tokens: int = 8192
    has_shared: int = 1
    layouts: int = 0

    def _c(self) -> _Config:
        return _Config(*[getattr(self, f.name) for f in fields(self)])


class MoE:
    """One MoE layer: a handle of the C library holding the repacked weights.

    ``weights``: dict of CUDA tensors in the canonical layout (names as in
    moe_weights: gu_codes uint8 [E,2I,d/2], gu_scale/gu_bias fp16 [E,2I,d/64],
    dn_* likewise, sh_* for the shared expert, w_router bf16 [E,d],
    w_shared_gate bf16 [d]).  They may be freed after construction."""

    def __init__(self, cfg: MoEConfig, weights: dict, stream=None):
        lib = load_library()
        self.cfg = cfg
        w = _Weights(*[_ptr(weights.get(n)) for n in WEIGHT_FIELDS])
        h = ctypes.c_void_p()
        _check(lib.moe_create(ctypes.byref(cfg._c()), ctypes.byref(w), _stream(stream),
                              ctypes.byref(h)))
        self._h = h

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            load_library().moe_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x: torch.Tensor, bias: torch.Tensor | None = None,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """y = MoE(x); x bf16 [T, d] on the GPU; bias fp32 [E] or None."""
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        _check(load_library().moe_forward(self._h, _ptr(x), T, _ptr(bias), _ptr(out),
                                          _stream(stream)))
        return out

    def forward_host(self, x_host: torch.Tensor, bias_host: torch.Tensor | None,
                     y_host: torch.Tensor, stream=None) -> torch.Tensor:
        """The same from host tensors (pinned for asynchronous copies)."""
        _check(load_library().moe_forward_host(self._h, _ptr(x_host), x_host.shape[0],
                                               _ptr(bias_host), _ptr(y_host), _stream(stream)))
        return y_host

    def _route_outputs(self, T, dev):
        c = self.cfg
        i32 = dict(dtype=torch.int32, device=dev)
        return dict(idx=torch.empty(T, c.k, **i32),
                    w=torch.empty(T, c.k, dtype=torch.float32, device=dev),
                    counts=torch.empty(c.E, **i32), offsets=torch.empty(c.E + 1, **i32),
                    perm=torch.empty(T * c.k, **i32), slot=torch.empty(T, c.k, **i32))

    def route(self, x: torch.Tensor, bias: torch.Tensor | None = None, stream=None) -> dict:
        T = x.shape[0]
        o = self._route_outputs(T, x.device)
        o["logits"] = torch.empty(T, self.cfg.E, dtype=torch.float32, device=x.device)
        _check(load_library().moe_route(
            self._h, _ptr(x), T, _ptr(bias), _ptr(o["logits"]), _ptr(o["idx"]), _ptr(o["w"]),
            _ptr(o["counts"]), _ptr(o["offsets"]), _ptr(o["perm"]), _ptr(o["slot"]),
            _stream(stream)))
        return o

    def route_from_logits(self, logits: torch.Tensor, bias: torch.Tensor | None = None,
                          stream=None) -> dict:
        T = logits.shape[0]
        o = self._route_outputs(T, logits.device)
        _check(load_library().moe_route_from_logits(
            self._h, _ptr(logits), T, _ptr(bias), _ptr(o["idx"]), _ptr(o["w"]),
            _ptr(o["counts"]), _ptr(o["offsets"]), _ptr(o["perm"]), _ptr(o["slot"]),
            _stream(stream)))
        return o

    def profile(self, enable: bool = True):
        _check(load_library().moe_profile_enable(self._h, int(enable)))

    def profile_read(self) -> tuple[dict, int]:
        """Summed milliseconds per stage since the last read, and the chunk count."""
        ms = (ctypes.c_float * len(STAGES))()
        n = ctypes.c_int(0)
        _check(load_library().moe_profile_read(self._h, ms, len(STAGES), ctypes.byref(n)))
        return dict(zip(STAGES, list(ms))), n.value

    def device_error(self) -> int:
        code = ctypes.c_int(0)
        st = load_library().moe_get_device_error(self._h, ctypes.byref(code))
        if st not in (0, 5):
            _check(st)
        return code.value


def decode(layers: list, x: torch.Tensor, bias: torch.Tensor | None = None, eps: float = 1e-6,
           trace: bool = False, stream=None):
    """Batch-1 decode through len(layers) layers in one launch.

    Returns y (bf16 [d]) and, if trace, a dict of per-layer logits, idx, w,
    sigma and out."""
    lib = load_library()
    L = len(layers)
    c = layers[0].cfg
    arr = (ctypes.c_void_p * L)(*[m.handle.value for m in layers])
    y = torch.empty(c.d, dtype=torch.bfloat16, device=x.device)
    tr = None
    t = None
    if trace:
        dev = x.device
        t = dict(logits=torch.empty(L, c.E, dtype=torch.float32, device=dev),
                 idx=torch.empty(L, c.k, dtype=torch.int32, device=dev),
                 w=torch.empty(L, c.k, dtype=torch.float32, device=dev),
                 sigma=torch.empty(L, dtype=torch.float32, device=dev),
                 out=torch.empty(L, c.d, dtype=torch.bfloat16, device=dev),
                 timestamps=torch.zeros(L, 4, dtype=torch.int64, device=dev))
        tr = _Trace(*[_ptr(t[n]) for n in ("logits", "idx", "w", "sigma", "out", "timestamps")])
    _check(lib.moe_decode(arr, L, _ptr(x), _ptr(bias), float(eps), _ptr(y),
                          ctypes.byref(tr) if tr is not None else None, _stream(stream)))
    return (y, t) if trace else y


def decode_host(layers: list, x_host: torch.Tensor, y_host: torch.Tensor,
                bias_host: torch.Tensor | None = None, eps: float = 1e-6, stream=None):
    """moe_decode on host tensors (pinned for asynchronous copies); synchronises."""
    L = len(layers)
    arr = (ctypes.c_void_p * L)(*[m.handle.value for m in layers])
    _check(load_library().moe_decode_host(arr, L, _ptr(x_host), _ptr(bias_host), float(eps),
                                          _ptr(y_host), _stream(stream)))
    return y_host


def route_from_logits_noalloc(logits: torch.Tensor, k: int, bias: torch.Tensor | None = None,
                              out: dict | None = None, stream=None) -> dict:
    """Routing from fp32 logits [T, E] through the entry point that allocates no
    device memory (T <= 2048, E <= 256).  Output tensors may be passed in
    ``out`` (keys idx, w, counts, offsets, perm, slot); otherwise they are made
    here with torch before the call."""
    T, E = logits.shape
    dev = logits.device
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        out = dict(idx=torch.empty(T, k, **i32), w=torch.empty(T, k, dtype=torch.float32, device=dev),
                   counts=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
                   perm=torch.empty(T * k, **i32), slot=torch.empty(T, k, **i32))
    _check(load_library().moe_route_from_logits_noalloc(
        _ptr(logits), T, E, k, _ptr(bias), _ptr(out["idx"]), _ptr(out["w"]), _ptr(out["counts"]),
        _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(out["slot"]), _stream(stream)))
    return out


def gdn_scan(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
             beta: torch.Tensor, scale: float | None = None, offsets: torch.Tensor | None = None,
             state: torch.Tensor | None = None, state_out: torch.Tensor | None = None,
             o: torch.Tensor | None = None, stream=None):
    """Gated DeltaNet prefill scan (include/gdn.h).

    q, k bf16 [T, Hk, dk]; v bf16 [T, Hv, dv]; g, beta fp32 [T, Hv];
    offsets int32 [N+1] (device) or None for one sequence; state fp32
    [N, Hv, dv, dk] or None (zero).  Returns (o bf16 [T, Hv, dv], final state
    fp32 [N, Hv, dv, dk]).  Outputs are made here with torch unless given."""
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = 1 if offsets is None else offsets.numel() - 1
    if scale is None:
        scale = dk ** -0.5
    dev = q.device
    if o is None:
        o = torch.empty(T, Hv, dv, dtype=torch.bfloat16, device=dev)
    if state_out is None:
        state_out = torch.empty(N, Hv, dv, dk, dtype=torch.float32, device=dev)
    _check(load_library().gdn_scan(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(offsets), N, T, Hk,
        Hv, dk, dv, _ptr(state), _ptr(state_out), _ptr(o), _stream(stream)))
    return o, state_out
