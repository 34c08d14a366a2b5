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
