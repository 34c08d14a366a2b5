"""The device input generator reproduces the host generator bit for bit."""
import numpy as np
import pytest
import torch

from synth import device as sd
from synth import gen
from tests.moe_cases import dev_to_bits

pytestmark = pytest.mark.gpu


def test_device_matches_host_generator():
    shape = gen.MoEShape(d=512, E=4, k=2, I=256)
    wd = sd.make_layer(5, 3, shape)
    torch.cuda.synchronize()
    for e in (0, 3, 4):
        host = gen.expert_weights(5, 3, e, shape)
        if e == shape.E:
            dev = [wd[n] for n in ("sh_gu_codes", "sh_gu_scale", "sh_gu_bias",
                                   "sh_dn_codes", "sh_dn_scale", "sh_dn_bias")]
        else:
            dev = [wd[n][e] for n in ("gu_codes", "gu_scale", "gu_bias",
                                      "dn_codes", "dn_scale", "dn_bias")]
        for h, d in zip(host, dev):
            assert np.array_equal(h, d.cpu().numpy())
    assert np.array_equal(dev_to_bits(wd["w_router"]),
                          gen.bf16_matrix(5, gen.TAG_ROUTER, 3, 0, shape.E, shape.d, 0.02))
    x = sd.make_x(9, 40, shape.d, row0=17)
    assert np.array_equal(dev_to_bits(x), gen.make_x(9, 40, shape.d, row0=17))
