"""The roofline denominators bench.py reports, against their derivation
from the layer's shapes (4-bit codes plus one fp16 scale and bias per 64
weights; bf16 router and shared gate; SwiGLU expert FLOPs)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

d, E, k, I = 2048, 256, 8, 512


def _matrix_bytes(rows, cols, group=64):
    return rows * cols // 2 + rows * (cols // group) * 2 * 2  # codes + fp16 s, beta


def test_expert_and_layer_bytes():
    expert = _matrix_bytes(2 * I, d) + _matrix_bytes(d, I)
    assert expert == bench.EXPERT_BYTES == 1769472  # 4.5 bits per weight
    assert expert * 16 == 9 * (2 * I * d + d * I)  # 4.5 bits, i.e. 9/16 byte, per weight
    decode_layer = 9 * expert + E * d * 2 + d * 2 + 2 * d * 2  # experts, router, w_sg, x + y
    assert decode_layer == bench.LAYER_BYTES_DECODE == 16986112


def test_flops_per_token_and_row():
    per_expert = 2 * d * 2 * I + 2 * I * d
    assert bench.GATEUP_FLOP_PER_ROW == 2 * d * 2 * I == 4194304
    assert bench.FLOP_PER_TOKEN == 2 * d * E + 9 * per_expert + 2 * d == 57675776


def test_point_roofline_bound_and_value():
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}
    # T = 1, every expert cold: bytes dominate
    t, bound = bench.point_roofline(1, 9, 1, peaks)
    nbytes = 9 * bench.EXPERT_BYTES + bench.ROUTER_BYTES + 4 * d
    assert bound == "hbm" and abs(t - nbytes / 8000e9) < 1e-15
    # large T, few experts: FLOPs dominate
    t, bound = bench.point_roofline(65536, 64, 8, peaks)
    assert bound == "tensor" and abs(t - bench.FLOP_PER_TOKEN * 65536 / 2000e12) < 1e-12


def test_gdn_scan_alu_roofline():
    # per state element and token: S.k, S.q (one multiply-add each) and the
    # update alpha S + c k (two operations)
    assert bench.gdn_alu_ops(2048, 32, 128, 128) == 4 * 2048 * 32 * 128 * 128
    # 152 SMs x 128 fp32 lanes x 2.07 GHz
    assert abs(bench.gdn_alu_peak(152) - 40.27392) < 1e-9


def test_gdn_scan_bytes():
    # q, k 16 heads x 128, v and o 32 heads x 128 (bf16), g and beta (fp32), state (fp32)
    assert bench.gdn_bytes(2048, 16, 32, 128, 128) == (
        2 * 2048 * 16 * 128 * 2 + 2 * 2048 * 32 * 128 * 2 + 2 * 2048 * 32 * 4 + 32 * 128 * 128 * 4)
    assert bench.gdn_bytes(2048, 16, 32, 128, 128) == 52953088
