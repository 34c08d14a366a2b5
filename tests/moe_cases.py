"""Shared helpers of the GPU parity tests: seeded cases, the oracle call and
the tolerance checks (rel-L2 <= 5e-3 and max-abs <= 3e-2 * max|oracle|)."""
from __future__ import annotations

import numpy as np
import torch

import sparse_moe_bit_gb300 as M
from oracle import moe_oracle as O
from synth import device as sd
from synth import gen

REL_L2 = 5e-3
MAX_ABS_FRAC = 3e-2

TINY = gen.MoEShape(d=256, E=16, k=2, I=128)
MID = gen.MoEShape(d=512, E=32, k=4, I=256)
QWEN = gen.MoEShape(d=2048, E=256, k=8, I=512)


def bits_to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_output(out, ref, what=""):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    e = rel_l2(out, ref)
    m = float(np.max(np.abs(out - ref)))
    bound = MAX_ABS_FRAC * float(np.max(np.abs(ref)))
    assert e <= REL_L2, f"{what}: rel-L2 {e:.3e} > {REL_L2}"
    assert m <= bound, f"{what}: max-abs {m:.3e} > {bound:.3e}"
    return e, m


def near_tie_tokens(logits: np.ndarray, k: int, gap: float = 1e-4) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th largest logits differ by less than gap."""
    if logits.shape[1] <= k:
        return np.zeros(logits.shape[0], bool)
    s = -np.sort(-logits, axis=1)
    return (s[:, k - 1] - s[:, k]) < gap


def scale_dtype_code(shape) -> int:
    """The C ABI's scale_dtype for a synth.gen.MoEShape."""
    from sparse_moe_bit_gb300 import moe as _moe
    return _moe.MOE_SCALE_BF16 if shape.scale_dtype == "bf16" else _moe.MOE_SCALE_F16


class HostCase:
    """A layer generated on the host (small shapes), uploaded to the GPU."""

    def __init__(self, shape, seed=0, layer=0, has_shared=True, max_tokens=8192, layouts=0):
        self.shape = shape
        self.lw = gen.make_layer(seed, layer, shape)
        self.vals = O.layer_values(self.lw, has_shared=has_shared)
        self.w = sd.host_layer_to_device(self.lw, has_shared=has_shared)
        self.cfg = M.MoEConfig(d=shape.d, E=shape.E, k=shape.k, I=shape.I, group=shape.group,
                               scale_dtype=scale_dtype_code(shape),
                               max_tokens=max_tokens, has_shared=int(has_shared), layouts=layouts)
        self.moe = M.MoE(self.cfg, self.w)

    def oracle(self, x_bits, logits=None, bias=None):
        return O.moe_layer(O.bf16_values(x_bits), self.vals, logit_bias=bias, logits=logits)


class DeviceLayer:
    """A Qwen-shaped layer generated on the GPU; the oracle regenerates the
    experts it needs on the host (same generator, bit for bit)."""

    def __init__(self, shape, seed=0, layer=0, max_tokens=8192, layouts=0):
        self.shape, self.seed, self.layer = shape, seed, layer
        w = sd.make_layer(seed, layer, shape)
        self.cfg = M.MoEConfig(d=shape.d, E=shape.E, k=shape.k, I=shape.I,
                               max_tokens=max_tokens, layouts=layouts)
        self.moe = M.MoE(self.cfg, w)
        del w
        torch.cuda.empty_cache()
        self._cache = {}
        self.w_router = O.bf16_values(gen.bf16_matrix(seed, gen.TAG_ROUTER, layer, 0, shape.E,
                                                      shape.d, 0.02))
        self.w_sg = O.bf16_values(gen.bf16_matrix(seed, gen.TAG_SHARED_GATE, layer, 0, 1,
                                                  shape.d, 0.02)[0])

    def expert(self, e):
        if e not in self._cache:
            self._cache[e] = gen.expert_weights(self.seed, self.layer, e, self.shape)
        return self._cache[e]

    def prefetch(self, experts):
        """Generate the given experts' weights on the host, several at once
        (numpy releases the GIL inside the generator's array operations)."""
        from concurrent.futures import ThreadPoolExecutor
        need = sorted({int(e) for e in experts} - set(self._cache))
        if not need:
            return
        with ThreadPoolExecutor(max_workers=min(16, len(need))) as ex:
            for e, w in zip(need, ex.map(
                    lambda e: gen.expert_weights(self.seed, self.layer, e, self.shape), need)):
                self._cache[e] = w

    def values(self):
        s = self.shape
        return dict(E=s.E, k=s.k, group=s.group, has_shared=True, w_router=self.w_router,
                    w_shared_gate=self.w_sg, experts=None, shared=None)

    def oracle(self, x_vals, logits=None, bias=None):
        if logits is not None:
            idx, _ = O.select_top_k(np.asarray(logits, np.float64), self.shape.k)
            self.prefetch(list(np.unique(idx)) + [self.shape.E])
        return O.moe_layer(x_vals, self.values(), logit_bias=bias, logits=logits,
                           expert_source=self.expert)


def hot_cold_bias(seed, shape, T_sample=2048, target=0.5):
    """Extreme-imbalance biases: the 8 top-ranked experts share one bias b_hot,
    chosen by bisection so that they take `target` of the top-k assignments
    of a T_sample-token sample; the 64 bottom-ranked experts get -1e4 (never
    chosen); the rest 0.  Host fp64 logits of the seeded input."""
    E, k, d = shape.E, shape.k, shape.d
    rank = gen.expert_ranking(seed, E)
    hot = rank <= 8
    cold = rank > E - 64
    xs = O.bf16_values(gen.make_x(seed, T_sample, d))
    wr = O.bf16_values(gen.bf16_matrix(seed, gen.TAG_ROUTER, 0, 0, E, d, 0.02))
    lg = xs @ wr.T

    def share(bh):
        b = np.where(hot, bh, np.where(cold, -1e4, 0.0))
        idx, _ = O.select_top_k(lg + b, k)
        return hot[idx].mean()

    lo, hi = -10.0, 20.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if share(mid) < target:
            lo = mid
        else:
            hi = mid
    b_hot = 0.5 * (lo + hi)
    bias = np.where(hot, b_hot, np.where(cold, -1e4, 0.0)).astype(np.float32)
    return bias, hot, cold
