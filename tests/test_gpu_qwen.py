"""Qwen-shaped prefill (d=2048, E=256, k=8, I=512 + shared expert, 4-bit g64):
T=4096 with Zipf-skewed routing (outputs of every token against the oracle),
and the T=32768 extreme-imbalance stress case (outputs of 4096 sampled tokens,
every near-tie token and tokens of the hottest expert among them).  Routing is
checked bit-exact for every token."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synth import device as sd
from synth import gen
from tests.moe_cases import QWEN, DeviceLayer, check_output, hot_cold_bias, near_tie_tokens

pytestmark = pytest.mark.gpu


def _routing_exact(r, k, E):
    lg = r["logits"].cpu().numpy()
    idx, w = O.select_top_k(lg.astype(np.float64), k)
    counts, offsets, perm, slot = O.group_by_expert(idx, E)
    assert np.array_equal(r["idx"].cpu().numpy(), idx)
    assert np.array_equal(r["counts"].cpu().numpy(), counts)
    assert np.array_equal(r["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(r["perm"].cpu().numpy(), perm)
    assert np.array_equal(r["slot"].cpu().numpy(), slot)
    w32 = w.astype(np.float32)
    assert np.all(np.abs(r["w"].cpu().numpy() - w32) <= np.spacing(np.abs(w32)))
    return lg, idx, counts


def _sample_tokens(idx, counts, n_rand, n_hot, rng, lg=None):
    """n_rand random tokens, n_hot tokens of the hottest expert, the first and
    last token and (given the logits) every token whose k-th and (k+1)-th
    logits are within 1e-4."""
    T = idx.shape[0]
    hot_e = int(np.argmax(counts))
    hot_tok = np.nonzero((idx == hot_e).any(axis=1))[0]
    pick = set(rng.choice(T, min(n_rand, T), replace=False).tolist())
    pick |= set(rng.choice(hot_tok, min(n_hot, len(hot_tok)), replace=False).tolist())
    pick |= {0, T - 1}
    if lg is not None:
        pick |= set(np.nonzero(near_tie_tokens(lg, idx.shape[1]))[0].tolist())
    return np.array(sorted(pick))


def _check_sampled(layer, x_seed, lg, y, toks, bias=None):
    n = int(toks.max()) + 1
    if 4 * len(toks) >= n:  # dense: all rows at once
        bits = gen.make_x(x_seed, n, QWEN.d)[toks]
    else:
        bits = np.concatenate([gen.make_x(x_seed, 1, QWEN.d, row0=int(t)) for t in toks])
    xv = O.bf16_values(bits)
    # logits vs fp64 (tolerance of fp32 accumulation)
    ref_lg = O.router_logits(xv, layer.w_router, bias)
    absdot = np.abs(xv) @ np.abs(layer.w_router).T
    assert np.all(np.abs(lg[toks] - ref_lg) <= QWEN.d * 2.0 ** -24 * absdot + 1e-6)
    ref = layer.oracle(xv, logits=lg[toks])
    return check_output(y[toks], ref["out"], "sampled tokens")


def test_prefill_T4096_zipf():
    T = 4096
    layer = DeviceLayer(QWEN, seed=0, layer=0, max_tokens=T)
    x = sd.make_x(0, T, QWEN.d)
    bias_np = gen.zipf_bias(0, QWEN.E)
    bias = torch.from_numpy(bias_np).cuda()
    y = layer.moe.forward(x, bias)
    r = layer.moe.route(x, bias)
    torch.cuda.synchronize()
    assert layer.moe.device_error() == 0
    lg, idx, counts = _routing_exact(r, QWEN.k, QWEN.E)
    ties = near_tie_tokens(lg, QWEN.k)
    print(f"experts touched {int((counts > 0).sum())}, max load {int(counts.max())}, "
          f"near-tie tokens {int(ties.sum())}")
    toks = np.arange(T)  # every token
    e, m = _check_sampled(layer, 0, lg, y.float().cpu().numpy(), toks, bias_np)
    print(f"all {len(toks)} tokens: rel-L2 {e:.2e}, max-abs {m:.2e}")


def test_stress_T32768_imbalance_deterministic():
    T = 32768
    bias_np, hot, cold = hot_cold_bias(0, QWEN)
    bias = torch.from_numpy(bias_np).cuda()
    layer = DeviceLayer(QWEN, seed=0, layer=0, max_tokens=T)
    x = sd.make_x(0, T, QWEN.d)
    y1 = layer.moe.forward(x, bias)
    y2 = layer.moe.forward(x, bias)
    r = layer.moe.route(x, bias)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), "not bit-identical"
    lg, idx, counts = _routing_exact(r, QWEN.k, QWEN.E)
    assert np.all(counts[cold] == 0)
    share = counts[hot].sum() / (T * QWEN.k)
    assert 0.45 <= share <= 0.55, share
    toks = _sample_tokens(idx, counts, 4096, 256, np.random.default_rng(1), lg)
    assert len(toks) >= 4096
    e, m = _check_sampled(layer, 0, lg, y1.float().cpu().numpy(), toks, bias_np)
    print(f"sampled {len(toks)} tokens: rel-L2 {e:.2e}, max-abs {m:.2e}")
    # the same call in chunks of 8192 tokens gives the same bits
    chunked = DeviceLayer(QWEN, seed=0, layer=0, max_tokens=8192)
    y3 = chunked.moe.forward(x, bias)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16)), "chunking changed the output"
