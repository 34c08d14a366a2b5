"""Plant one plausible mistake at a time in a copy of an oracle (on the CPU)
and check that its pins catch every one of them: test_oracle_pins.py for the
MoE block, test_gdn_oracle_pins.py for the Gated DeltaNet scan."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.py")
SRC_GDN = os.path.join(ROOT, "oracle", "gdn_oracle.py")

# (name, original text, planted mistake)
MUTATIONS = [
    ("dropped bias term", "return s * q + b", "return s * q"),
    ("nibble order", "out[..., 0::2] = packed & 0x0F", "out[..., 0::2] = packed >> 4"),
    ("group index", "s = np.repeat(scale_values(scale), group, axis=-1)",
     "s = np.tile(scale_values(scale), group)"),
    ("group fixed at 64", "s = np.repeat(scale_values(scale), group, axis=-1)",
     "s = np.repeat(scale_values(scale), 64, axis=-1)"),
    ("bf16 scale bits read as fp16",
     "return bf16_values(a) if a.dtype == np.uint16 else a.astype(F64)",
     "return a.view(np.float16).astype(F64) if a.dtype == np.uint16 else a.astype(F64)"),
    ("router bias sign", "lg = lg + np.asarray(logit_bias, F64)[None, :]",
     "lg = lg - np.asarray(logit_bias, F64)[None, :]"),
    ("tie-break", "order = np.lexsort((ids, -lg), axis=-1)",
     "order = np.lexsort((-ids, -lg), axis=-1)"),
    ("softmax sign", "ex = np.exp(top - m)", "ex = np.exp(m - top)"),
    ("renormalisation axis", "w = ex / ex.sum(axis=1, keepdims=True)", "w = ex / ex.sum()"),
    ("gate/up roles", "return (silu(g) * u) @ w_down.T", "return (silu(u) * g) @ w_down.T"),
    ("transposed down", "return (silu(g) * u) @ w_down.T", "return (silu(g) * u) @ w_down"),
    ("silu sign", "return z * expit(z)", "return z * expit(-z)"),
    ("gate/up halves", "return wgu[:I], wgu[I:],", "return wgu[I:], wgu[:I],"),
    ("shared gate sign", "return expit(np.asarray(x, F64) @ np.asarray(w_shared_gate, F64))",
     "return expit(-(np.asarray(x, F64) @ np.asarray(w_shared_gate, F64)))"),
    ("slot index", "out += w[:, j:j + 1] * y[:, j]", "out += w[:, j:j + 1] * y[:, 0]"),
    ("dropped shared term", "out += sigma[:, None] * swiglu_expert(x, wg, wu, wd)",
     "out += 0.0 * swiglu_expert(x, wg, wu, wd)"),
    ("perm index", "perm = (order // k).astype(np.int32)", "perm = (order % k).astype(np.int32)"),
    ("offsets shift", "offsets[1:] = np.cumsum(counts)", "offsets[:-1] = np.cumsum(counts)"),
    ("rms of v, not v^2", "np.mean(v * v, axis=-1, keepdims=True)", "np.mean(v, axis=-1, keepdims=True)"),
    ("rms eps dropped", "np.mean(v * v, axis=-1, keepdims=True) + eps)",
     "np.mean(v * v, axis=-1, keepdims=True))"),
    ("silu of the product", "return (silu(g) * u) @ w_down.T", "return silu(g * u) @ w_down.T"),
    ("scale used as bias", "return s * q + b", "return s * q + s"),
    ("full-softmax denominator", "w = ex / ex.sum(axis=1, keepdims=True)",
     "w = ex / np.exp(lg - m).sum(axis=1, keepdims=True)"),
    ("shared weighted by 1 - sigma", "out += sigma[:, None] * swiglu_expert(x, wg, wu, wd)",
     "out += (1 - sigma)[:, None] * swiglu_expert(x, wg, wu, wd)"),
    ("weight of slot 0 for every slot", "out += w[:, j:j + 1] * y[:, j]",
     "out += w[:, 0:1] * y[:, j]"),
    ("+inf logits: weight to every kept expert", "hit = (top[pos] == np.inf).astype(F64)",
     "hit = np.ones_like(top[pos])"),
    ("all -inf logits: no weight", "w[neg] = 1.0 / k", "w[neg] = 0.0"),
]


@pytest.mark.parametrize("name,orig,bad", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(name, orig, bad, tmp_path):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor not found once: {orig!r}"
    mutant = tmp_path / "moe_oracle_mutant.py"
    mutant.write_text(src.replace(orig, bad))
    env = dict(os.environ, MOE_ORACLE_FILE=str(mutant))
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle_pins.py")],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"no pin caught the planted mistake '{name}'"


WRITE = "        + beta[:, None, None] * v[:, :, None] * k[:, None, :]"
MUTATIONS_GDN = [
    ("gate applied to the write too", WRITE,
     "        + alpha * beta[:, None, None] * v[:, :, None] * k[:, None, :]"),
    ("write without beta", WRITE, "        + v[:, :, None] * k[:, None, :]"),
    ("delta sign", "(S - beta[:, None, None] * Sk", "(S + beta[:, None, None] * Sk"),
    ("readout before the write", 'o = scale * np.einsum("hij,hj->hi", S_new, q)',
     'o = scale * np.einsum("hij,hj->hi", S, q)'),
    ("readout with the key", 'o = scale * np.einsum("hij,hj->hi", S_new, q)',
     'o = scale * np.einsum("hij,hj->hi", S_new, k)'),
    ("delta read with the query", 'Sk = np.einsum("hij,hj->hi", S, k)',
     'Sk = np.einsum("hij,hj->hi", S, q)'),
    ("gate not exponentiated", "alpha = np.exp(g)[:, None, None]", "alpha = g[:, None, None]"),
    ("head grouping modulo", "head_of = np.arange(Hv) // (Hv // Hk)",
     "head_of = np.arange(Hv) % Hk"),
    ("state carried across sequences", "S = states[n].copy()",
     "S = S if n else states[n].copy()"),
    ("initial state ignored", "states[:] = np.asarray(state0, F64)", "pass"),
    ("default scale 1/dk", "scale = 1.0 / np.sqrt(dk)", "scale = 1.0 / dk"),
    ("dense rule without beta on the write",
     "S_new = S @ transition + F64(beta) * np.outer(v, k)",
     "S_new = S @ transition + np.outer(v, k)"),
    ("dense transition sign", "np.eye(dk) - F64(beta)", "np.eye(dk) + F64(beta)"),
    ("bf16 bits misplaced", "<< np.uint32(16)", "<< np.uint32(15)"),
    ("gate squared", "alpha = np.exp(g)[:, None, None]", "alpha = np.exp(2 * g)[:, None, None]"),
    ("beta twice on the erase", "(S - beta[:, None, None] * Sk",
     "(S - beta[:, None, None] ** 2 * Sk"),
    ("readout unscaled", 'o = scale * np.einsum("hij,hj->hi", S_new, q)',
     'o = np.einsum("hij,hj->hi", S_new, q)'),
    ("last sequence dropped", "for n in range(N):", "for n in range(max(N - 1, 1)):"),
    ("first initial state for every sequence", "states[:] = np.asarray(state0, F64)",
     "states[:] = np.asarray(state0, F64)[:1]"),
    ("q/k head h // Hk", "head_of = np.arange(Hv) // (Hv // Hk)", "head_of = np.arange(Hv) // Hk"),
]


@pytest.mark.parametrize("name,orig,bad", MUTATIONS_GDN, ids=[m[0] for m in MUTATIONS_GDN])
def test_gdn_pins_catch_planted_mistake(name, orig, bad, tmp_path):
    src = open(SRC_GDN).read()
    assert src.count(orig) == 1, f"mutation anchor not found once: {orig!r}"
    mutant = tmp_path / "gdn_oracle_mutant.py"
    mutant.write_text(src.replace(orig, bad))
    env = dict(os.environ, GDN_ORACLE_FILE=str(mutant))
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_gdn_oracle_pins.py")],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"no pin caught the planted mistake '{name}'"
