"""Failure detection on the GPU without a fault: every wait of the decode
kernel on another CTA is bounded.  A child process sets a short limit and the
test-only flag that makes the kernel wait for one router-sum arrival that no
CTA makes; the wait must run out, the kernel must end and report
MOE_DEVERR_GRID_TIMEOUT in the device error word, and the CUDA context must
stay usable (a later handle without the flag computes normally)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys, time
sys.path.insert(0, %r)
import torch
import sparse_moe_bit_gb300 as M
from synth import gen
from tests.moe_cases import TINY, HostCase, bits_to_dev
x = bits_to_dev(gen.make_x(0, 1, TINY.d))
stalled = HostCase(TINY, seed=0, max_tokens=4, layouts=M.MOE_LAYOUT_DECODE)
t0 = time.time()
M.decode([stalled.moe], x[0])
torch.cuda.synchronize()
dt = time.time() - t0
err = stalled.moe.device_error()
os.environ.pop("MOE_TEST_UNSET_FLAG")
fine = HostCase(TINY, seed=0, max_tokens=4, layouts=M.MOE_LAYOUT_DECODE)
y = M.decode([fine.moe], x[0])
torch.cuda.synchronize()
err2 = fine.moe.device_error()
z = float((torch.ones(1000, device="cuda") * 2).sum().item())
print(json.dumps({"err": err, "dt": dt, "err2": err2, "finite": bool(torch.isfinite(y.float()).all()), "z": z}))
""" % ROOT


def test_decode_wait_runs_out_and_is_reported():
    import sparse_moe_bit_gb300 as M
    env = dict(os.environ, MOE_WAIT_LIMIT_NS="20000000", MOE_TEST_UNSET_FLAG="1")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["err"] & M.MOE_DEVERR_GRID_TIMEOUT, out
    assert out["dt"] < 10.0, out  # ended soon after the 20 ms limit (plus start-up)
    assert out["err2"] == 0 and out["finite"], out
    assert out["z"] == 2000.0
