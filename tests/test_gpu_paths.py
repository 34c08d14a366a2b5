"""The one-CTA GEMM variants (no CTA pairs: MOE_GEMM_2SM=0) against the
oracle.  The variant is chosen once per process from the environment, so it
runs in a child process."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
sys.path.insert(0, %r)
import numpy as np, torch
from oracle import moe_oracle as O
from synth import gen
from tests.moe_cases import MID, HostCase, bits_to_dev, rel_l2
import sparse_moe_bit_gb300 as M
case = HostCase(MID, seed=1, layouts=M.MOE_LAYOUT_PREFILL)
res = {}
for T in (7, 300):
    bits = gen.make_x(9, T, MID.d)
    x = bits_to_dev(bits)
    y = case.moe.forward(x)
    r = case.moe.route(x)
    torch.cuda.synchronize()
    ref = case.oracle(bits, logits=r["logits"].cpu().numpy())["out"]
    out = y.float().cpu().numpy()
    res[T] = [rel_l2(out, ref), float(np.max(np.abs(out - ref)) / np.max(np.abs(ref))),
              bool(np.all(np.isfinite(out)))]
print(json.dumps({"res": res, "err": case.moe.device_error()}))
""" % ROOT


def test_one_cta_gemm_variants():
    env = dict(os.environ, MOE_GEMM_2SM="0")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["err"] == 0
    for T, (e, m, finite) in out["res"].items():
        assert finite, f"T={T}: non-finite output"
        assert e <= 5e-3, f"T={T}: rel-L2 {e:.3e}"
        assert m <= 3e-2, f"T={T}: max-abs {m:.3e} of max|oracle|"
