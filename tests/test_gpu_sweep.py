"""The prefill length sweep at Qwen shape (d=2048, E=256, k=8, I=512 + shared
expert, 4-bit g64) under uniform and Zipf-skewed routing, processed in
chunks of 8192 tokens above that length.  The routing of every token is
checked bit-exact given the GPU's logits (chunk by chunk: a token's logits do
not depend on the chunk it shares); outputs against the fp64 oracle for every
token up to 2048 tokens and for 4096 sampled tokens from 16K on.  The sweep's
longer lengths (up to 128K tokens) are measured by bench.py; their kernels
and chunk loop are the ones exercised here."""
import numpy as np
import pytest
import torch

from synth import device as sd
from synth import gen
from tests.moe_cases import QWEN, DeviceLayer
from tests.test_gpu_qwen import _check_sampled, _routing_exact, _sample_tokens

pytestmark = pytest.mark.gpu

CHUNK = 8192


@pytest.mark.parametrize("T,zipf", [(256, False), (256, True), (2048, False), (16384, True),
                                    (32768, False)])
def test_prefill_sweep_length(T, zipf):
    chunk = min(T, CHUNK)
    layer = DeviceLayer(QWEN, seed=0, layer=0, max_tokens=chunk)
    x = sd.make_x(0, T, QWEN.d)
    bias_np = gen.zipf_bias(0, QWEN.E) if zipf else None
    bias = torch.from_numpy(bias_np).cuda() if zipf else None
    y = layer.moe.forward(x, bias)  # chunks of `chunk` tokens inside the call
    lgs, idxs = [], []
    for t0 in range(0, T, chunk):
        r = layer.moe.route(x[t0:t0 + chunk], bias)
        torch.cuda.synchronize()
        lg, idx, _ = _routing_exact(r, QWEN.k, QWEN.E)
        lgs.append(lg)
        idxs.append(idx)
    assert layer.moe.device_error() == 0
    lg = np.concatenate(lgs)
    idx = np.concatenate(idxs)
    counts = np.bincount(idx.ravel(), minlength=QWEN.E)
    # short prompts: every token; 16K and longer: 4096 sampled tokens (with
    # every near-tie token and tokens of the hottest expert)
    if T <= 2048:
        toks = np.arange(T)
    else:
        toks = _sample_tokens(idx, counts, 4096, 256, np.random.default_rng(T + zipf), lg)
        assert len(toks) >= 4096
    e, m = _check_sampled(layer, 0, lg, y.float().cpu().numpy(), toks, bias_np)
    print(f"T={T} {'zipf' if zipf else 'uniform'}: experts touched {int((counts > 0).sum())}, "
          f"sampled {len(toks)} tokens rel-L2 {e:.2e}")
