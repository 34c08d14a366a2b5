"""The routing entry point that allocates no device memory.

It serves callers that cannot call cudaMalloc (code inside a device memory
allocator, serving loops that must avoid cudaMalloc's device synchronisation,
programs whose device memory another framework owns).  Its scratch is a
fixed device array inside the library.  This test calls it through the C ABI
twice in a row and checks each result against moe_route_from_logits (the
handle-based entry point, same tolerance as the routing parity tests:
indices, counts, offsets, perm and slot bit for bit, weights within 1 ulp).
It sits in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

import sparse_moe_bit_gb300 as M
from oracle import moe_oracle as O
from sparse_moe_bit_gb300 import moe as MM
from tests.moe_cases import MID, HostCase

pytestmark = pytest.mark.gpu


def _same(a, b):
    for key in ("idx", "counts", "offsets", "perm", "slot"):
        assert torch.equal(a[key], b[key]), key
    wa, wb = a["w"].cpu().numpy(), b["w"].cpu().numpy()
    assert np.all(np.abs(wa - wb) <= np.spacing(np.abs(wb)))


def test_noalloc_routing_matches_handle_routing_twice():
    case = HostCase(MID, seed=5, max_tokens=2048)
    rng = np.random.default_rng(17)
    for call, T in enumerate((2048, 700)):
        lg = (rng.standard_normal((T, MID.E)) * 2).astype(np.float32)
        lg[:5] = np.round(lg[:5])  # exact ties
        logits = torch.from_numpy(lg).cuda()
        bias = torch.linspace(-0.5, 0.5, MID.E, device="cuda") if call else None
        ref = case.moe.route_from_logits(logits, bias)
        got = MM.route_from_logits_noalloc(logits, MID.k, bias)
        torch.cuda.synchronize()
        _same(got, ref)


def _matches_oracle(got, lg, k, E):
    """Routing of fp32 logits against the oracle's selection and grouping:
    indices, counts, offsets, perm and slot bit for bit, weights within 1 ulp
    of fp32 of the fp64 weights."""
    idx, w = O.select_top_k(lg.astype(np.float64), k)
    counts, offsets, perm, slot = O.group_by_expert(idx, E)
    assert np.array_equal(got["idx"].cpu().numpy(), idx)
    assert np.array_equal(got["counts"].cpu().numpy(), counts)
    assert np.array_equal(got["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(got["perm"].cpu().numpy(), perm)
    assert np.array_equal(got["slot"].cpu().numpy(), slot)
    w32 = w.astype(np.float32)
    assert np.all(np.abs(got["w"].cpu().numpy() - w32) <= np.spacing(np.abs(w32)))


@pytest.mark.parametrize("E,k", [(256, 16), (256, 8)])
def test_noalloc_routing_at_its_limits(E, k):
    """The largest sizes the entry point takes (T = 2048 with E = 256 and
    k = 16: every lane slot of the selection, the largest tile map and scratch
    offsets) and the Qwen-shaped router (E = 256, k = 8), twice in a row."""
    rng = np.random.default_rng(E + k)
    for T in (2048, 1999):
        lg = (rng.standard_normal((T, E)) * 1.5).astype(np.float32)
        lg[:64] = np.round(lg[:64] * 2) / 2  # exact ties
        hot = rng.choice(E, 4, replace=False)
        lg[:, hot] += 3.0  # a few experts take most rows: several full tiles
        got = MM.route_from_logits_noalloc(torch.from_numpy(lg).cuda(), k)
        torch.cuda.synchronize()
        _matches_oracle(got, lg, k, E)


def test_noalloc_rejects_misaligned_pointers():
    lib = M.load_library()
    x = torch.zeros(64, 16, device="cuda")
    o = torch.zeros(1 << 16, dtype=torch.int32, device="cuda")
    p = o.data_ptr()
    assert lib.moe_route_from_logits_noalloc(x.data_ptr() + 2, 4, 16, 2, None, p, p, p, p, p, p,
                                             None) == 1
    assert lib.moe_route_from_logits_noalloc(x.data_ptr(), 4, 16, 2, None, p + 1, p, p, p, p, p,
                                             None) == 1
    assert lib.moe_route_from_logits_noalloc(x.data_ptr(), 4, 16, 2, x.data_ptr() + 2, p, p, p,
                                             p, p, p, None) == 1


def test_noalloc_rejects_sizes_beyond_its_limit():
    lib = M.load_library()
    x = torch.zeros(4, 16, device="cuda")
    o = torch.zeros(1 << 16, dtype=torch.int32, device="cuda")
    p = o.data_ptr()
    assert lib.moe_route_from_logits_noalloc(x.data_ptr(), 2049, 16, 2, None, p, p, p, p, p, p,
                                             None) == 1
    assert lib.moe_route_from_logits_noalloc(x.data_ptr(), 4, 257, 2, None, p, p, p, p, p, p,
                                             None) == 1
    assert lib.moe_route_from_logits_noalloc(x.data_ptr(), 4, 16, 17, None, p, p, p, p, p, p,
                                             None) == 1
