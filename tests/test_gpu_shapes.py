"""Parity at the edges of the supported shapes: more than 256 experts (the
routing kernel's wide variant and a router of two 256-expert units), the
largest k (16) and the largest E (512).  Prefill layout: the tensor-core
path at every T."""
import numpy as np
import pytest
import torch

import sparse_moe_bit_gb300 as M
from oracle import moe_oracle as O
from synth import gen
from tests.moe_cases import HostCase, bits_to_dev, check_output

pytestmark = pytest.mark.gpu

SHAPES = {
    "E300_k10": gen.MoEShape(d=256, E=300, k=10, I=128),
    "E64_k16": gen.MoEShape(d=256, E=64, k=16, I=128),
    "E512_k8": gen.MoEShape(d=256, E=512, k=8, I=128),
}


@pytest.fixture(scope="module", params=list(SHAPES))
def case(request):
    return HostCase(SHAPES[request.param], seed=6, layouts=M.MOE_LAYOUT_PREFILL)


def _routing_matches(r, logits, k, E):
    idx, w = O.select_top_k(logits.astype(np.float64), k)
    counts, offsets, perm, slot = O.group_by_expert(idx, E)
    assert np.array_equal(r["idx"].cpu().numpy(), idx)
    assert np.array_equal(r["counts"].cpu().numpy(), counts)
    assert np.array_equal(r["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(r["perm"].cpu().numpy(), perm)
    assert np.array_equal(r["slot"].cpu().numpy(), slot)
    w32 = w.astype(np.float32)
    assert np.all(np.abs(r["w"].cpu().numpy() - w32) <= np.spacing(np.abs(w32)))


@pytest.mark.parametrize("T", [5, 33, 500])
def test_shapes_forward_and_routing(case, T):
    bits = gen.make_x(8, T, case.shape.d)
    x = bits_to_dev(bits)
    y = case.moe.forward(x)
    r = case.moe.route(x)
    torch.cuda.synchronize()
    lg = r["logits"].cpu().numpy()
    _routing_matches(r, lg, case.shape.k, case.shape.E)
    ref = case.oracle(bits, logits=lg)
    check_output(y.float().cpu().numpy(), ref["out"], f"{case.shape} T={T}")
    assert case.moe.device_error() == 0


def test_shapes_route_from_tied_logits(case):
    rng = np.random.default_rng(3)
    T, E, k = 200, case.shape.E, case.shape.k
    lg = (np.round(rng.standard_normal((T, E)) * 2) / 2).astype(np.float32)  # many ties
    lg[:5] = 0.0
    r = case.moe.route_from_logits(torch.from_numpy(lg).cuda())
    torch.cuda.synchronize()
    _routing_matches(r, lg, k, E)
