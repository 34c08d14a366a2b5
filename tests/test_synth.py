"""The seeded input generator: determinism, shape of the distribution and the
quantiser's error bound.  (Inputs only; no MoE arithmetic is tested here.)"""
import numpy as np

from synth import gen


def test_splitmix64_reference_values():
    # SplitMix64 seeded with 0 (state advances by GAMMA before each output):
    # the first outputs of the published generator.
    assert gen.mix64_int(gen.GAMMA) == 0xE220A8397B1DCDAF
    assert gen.mix64_int((2 * gen.GAMMA) & gen.MASK64) == 0x6E789E6AA1B965F4
    v = gen.draws(0, np.array([0, 1], dtype=np.uint64))
    assert int(v[0]) == 0xE220A8397B1DCDAF and int(v[1]) == 0x6E789E6AA1B965F4


def test_streams_deterministic_and_distinct():
    a = gen.normal_fp32(gen.stream_key(0, gen.TAG_X), 0, 1000, 1.0)
    b = gen.normal_fp32(gen.stream_key(0, gen.TAG_X), 0, 1000, 1.0)
    c = gen.normal_fp32(gen.stream_key(0, gen.TAG_X, 1), 0, 1000, 1.0)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c)
    # counter based: a window equals the slice of a longer draw
    w = gen.normal_fp32(gen.stream_key(0, gen.TAG_X), 100, 50, 1.0)
    assert np.array_equal(w, a[100:150])


def test_normal_shape_moments():
    v = gen.normal_fp32(gen.stream_key(3, gen.TAG_GATE_UP), 0, 400000, 0.02).astype(np.float64)
    assert abs(v.mean()) < 2e-4
    assert abs(v.std() - 0.02) < 2e-4
    k = ((v - v.mean()) ** 4).mean() / v.var() ** 2
    assert 2.7 < k < 3.0  # Irwin-Hall(8): excess kurtosis -0.15


def test_bf16_rounding_is_rne():
    v = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e-3], dtype=np.float32)
    b = gen.round_to_bf16_bits(v)
    back = gen.bf16_bits_to_fp32(b)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: rounds to even (1.0)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0078125 and back[3] == -2.5
    assert abs(back[4] - 3.0e-3) <= 2.0 ** -8 * 3.0e-3  # half an ulp (8 significant bits)


def test_quantiser_hand_group():
    # values -1 + k/15 * 3 for k = 0..15 (repeated): s = 3/15, beta = -1
    k = np.arange(64) % 16
    w = (-1.0 + k * (3.0 / 15.0)).astype(np.float32)[None, :]
    packed, s, b = gen.quantize_rows(w, 64)
    assert float(b[0, 0]) == -1.0
    assert float(s[0, 0]) == float(np.float16(np.float32(3.0) / np.float32(15.0)))
    q = np.empty(64, np.uint8); q[0::2] = packed[0] & 15; q[1::2] = packed[0] >> 4
    assert np.array_equal(q, k.astype(np.uint8))


def test_quantiser_error_bound_and_constant_group():
    w = gen.normal_fp32(gen.stream_key(1, gen.TAG_DOWN), 0, 64 * 256, 0.02).reshape(64, 256)
    packed, s, b = gen.quantize_rows(w, 64)
    q = np.empty(w.shape, np.float64); q[:, 0::2] = packed & 15; q[:, 1::2] = packed >> 4
    sf = np.repeat(s.astype(np.float64), 64, axis=1)
    bf = np.repeat(b.astype(np.float64), 64, axis=1)
    err = np.abs(sf * q + bf - w)
    # half a step, plus the fp16 rounding of beta and of 15*s
    bound = sf / 2 + np.abs(bf) * 2.0 ** -11 + 15 * sf * 2.0 ** -11 + 1e-9
    assert np.all(err <= bound)
    c = np.full((1, 64), 0.25, np.float32)
    pc, sc, bc = gen.quantize_rows(c, 64)
    assert float(sc[0, 0]) == 0.0 and float(bc[0, 0]) == 0.25 and not pc.any()


def test_zipf_bias():
    b = gen.zipf_bias(0, 256)
    rank = gen.expert_ranking(0, 256)
    assert sorted(rank.tolist()) == list(range(1, 257))
    assert b[rank == 1][0] == 0.0
    np.testing.assert_allclose(b, (1.5 * np.log(1.0 / rank)).astype(np.float32))


def test_quantiser_bf16_scales_group128():
    # bf16 scale/bias (bit patterns), 128-wide groups: s and beta are the RNE
    # bf16 roundings of (max - min)/15 and min; the error bound grows by the
    # coarser rounding (2^-8 relative) of beta and of 15 s
    w = gen.normal_fp32(gen.stream_key(2, gen.TAG_GATE_UP), 0, 32 * 512, 0.02).reshape(32, 512)
    packed, s, b = gen.quantize_rows(w, 128, "bf16")
    assert s.dtype == np.uint16 and b.dtype == np.uint16 and s.shape == (32, 4)
    g = w.reshape(32, 4, 128)
    assert np.array_equal(s, gen.round_to_bf16_bits((g.max(2) - g.min(2)) / np.float32(15.0)))
    assert np.array_equal(b, gen.round_to_bf16_bits(g.min(2)))
    q = np.empty(w.shape, np.float64); q[:, 0::2] = packed & 15; q[:, 1::2] = packed >> 4
    sf = np.repeat(gen.bf16_bits_to_fp32(s).astype(np.float64), 128, axis=1)
    bf = np.repeat(gen.bf16_bits_to_fp32(b).astype(np.float64), 128, axis=1)
    err = np.abs(sf * q + bf - w)
    bound = sf / 2 + np.abs(bf) * 2.0 ** -8 + 15 * sf * 2.0 ** -8 + 1e-9
    assert np.all(err <= bound)


def test_gdn_inputs_recipe():
    from synth import gdn
    shape = gdn.GdnShape(Hk=2, Hv=4, dk=128, dv=64)
    a = gdn.make_inputs(0, [5, 0, 11], shape, state_std=0.1)
    b = gdn.make_inputs(0, [5, 0, 11], shape, state_std=0.1)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v), (a.g, b.g), (a.beta, b.beta)):
        assert np.array_equal(x, y)                       # seeded, reproducible
    assert a.q.shape == (16, 2, 128) and a.v.shape == (16, 4, 64)
    assert a.state0.shape == (3, 4, 64, 128)
    assert list(a.offsets) == [0, 5, 5, 16]
    qn = np.linalg.norm(gen.bf16_bits_to_fp32(a.q).astype(np.float64), axis=-1)
    assert np.all(np.abs(qn - 1) < 4e-3)                  # unit norm up to bf16 rounding
    alpha = np.exp(a.g.astype(np.float64))
    assert np.all((alpha >= 0.9 - 1e-6) & (alpha < 1.0))
    assert np.all((a.beta > 0) & (a.beta < 1))
    assert not np.array_equal(a.q, a.k)
